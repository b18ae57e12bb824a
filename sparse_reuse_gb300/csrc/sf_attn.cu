// Folded self-attention of one layer, exact against each branch's own keys.
//
// "SpecFold" (arXiv 2610.04875v2 summary) §A.1: a folded row's attention is
// the child's attention state exactly; App. B: attention kernels process the
// recomputed queries and keep per-head softmax max/denominator state; the
// onedev.kr review ("How to use it"): FlashAttention-style streaming, the
// shared prefix KV seen by every branch through a zero-copy strided view, GQA.
//
// Kernels (BF16 contexts on the 5th-generation tensor cores, tcgen05 MMAs
// into tensor memory; FP32 contexts on CUDA cores with fp32 operands):
//   short prefixes, direct mode: one fused kernel per (branch, KV head, query
//     tile): every row's query against the shared prefix (TMA-streamed) and
//     against its branch's own block keys (gathered through the source slots),
//     one streaming softmax, the normalised output written directly;
//   otherwise:
//     1. prefix partial per recomputed query: streaming softmax state
//        (max, denominator, unnormalised output) of q against the request's
//        prefix keys, the prefix split over S chunks (a cluster of S CTAs per
//        query tile);
//     2. per (row, head): the query is the one of the row's resolved source;
//        its block part runs over the branch's own L block keys/values, read
//        through the source slots of the branch's positions, and is merged
//        with the query's prefix partial by log-sum-exp;
//   SF_ATTN_CORRECT: step 2 for the recompute rows only, then the §A.1
//     subtract/add correction for the folded rows.
// The GQA group's query heads are packed into the M dimension so every
// key/value tile is read once per KV head.
#include "sf_internal.h"
#include "sf_tc.cuh"

namespace sf {
namespace {

constexpr int kMaxHd = 128;
constexpr int kMaxSplits = 8;
constexpr int kQT = 64;  // query tile of the CUDA-core path's split count
constexpr int kKB = 64;  // keys per block

// Number of prefix splits and keys per split for this pass.
struct Splits {
  int S, len;
};

__device__ __forceinline__ Splits prefix_splits(const AttnArgs& a) {
  if (a.P <= 0) return {0, 0};
  const int G = a.nq / a.nkv;
  int tiles = 0;
  for (int r = 0; r < a.R; ++r) tiles += (((a.meta[2 + r] - a.meta[1 + r]) * G) + kQT - 1) / kQT;
  tiles *= a.nkv;
  int S = tiles > 0 ? (a.target_ctas + tiles - 1) / tiles : 1;
  S = max(1, min(S, min(kMaxSplits, (a.P + kKB - 1) / kKB)));
  const int len = (((a.P + S - 1) / S) + kKB - 1) / kKB * kKB;
  return {(a.P + len - 1) / len, len};
}

// ------------------------------------------------------------ tensor-core path

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared through L2 only (zero-filled
// when !valid; src must still point into a live allocation).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------ tcgen05 prefix path
//
// Prefix partials on the 5th-generation tensor cores: CTA = (128 query vectors
// of one request and KV head = the 128 TMEM lanes, one split of the prefix).
// The queries are written once into TMEM as bf16 pairs; per block of 64 keys:
//   S = Q K^T       tcgen05.mma with Q from TMEM and K K-major in shared
//                   memory, S in TMEM (three buffers: the scores two blocks
//                   ahead are computed while this block's softmax runs);
//   P = exp2(S - m) by the softmax warps, one query row per thread, written
//                   back to TMEM as bf16 pairs (two buffers);
//   O += P V        tcgen05.mma with P from TMEM and V MN-major as the TMA
//                   box leaves it, O in TMEM.
// Shared memory then carries only the K and V rings, so each block costs
// the TMA writes and one tensor-core read of its keys and values.
// The running max m of a row only moves when a block's max exceeds it by more
// than 2^8, and O is then rescaled in TMEM; the partial state (m, l, O) stays
// exact because m is whatever reference the exponentials used.
// Warp 0 streams the keys through a kTcStages-deep ring of TMA loads (a stage
// is freed once its scores are computed), warp 10 the values (freed once P V
// is done), warp 1 owns TMEM and issues the score MMAs, warp 11 the P V MMAs,
// warps 2-9 load Q and run the softmax and the epilogue: the two warps on the
// same 32 TMEM lanes take half of each row's 64 scores and half of its output
// columns, and exchange only the row's block maximum.  Every role that waits
// on barriers has a warp of its own: a lane spinning on one barrier holds back
// a diverged lane of its warp, and one thread issuing both MMA groups leaves
// the tensor core idle during its barrier waits (its queue is short).
// With several splits, the splits of a query tile form a cluster: every split
// stores its partial state in a slot of its own (part_o / part_ml slots
// 1..S), the cluster meets at a barrier, and split s merges rows
// [s per, (s + 1) per) of the tile from the S slots.
constexpr int kTcQ = 128;
constexpr int kTcStages = 4;
// warp 0 K loads, warp 1 S = Q K^T, warps 2-9 softmax (two per row group), warp 10 V loads, warp 11 O += P V
constexpr int kTcThreads = 384;
constexpr int kTcVWarp = 10;
constexpr int kTcPVWarp = 11;
constexpr int kTcMinKeysPerSplit = 512;
constexpr int kTcMaxSplits = 4;
static_assert(1 + kTcMaxSplits <= kMaxSplits, "split slots of the partial buffers");
constexpr float kTcRescaleLog2 = 8.f;

// Few long splits: the fixed cost of a CTA (TMEM, barriers, the first scores,
// the epilogue) is paid once per split, so S is the smallest count that still
// fills about one wave of SMs.  A folded pass leaves about two live query
// tiles per (request, KV head) -- the main branch and a ragged remainder --
// so the host aims at target / (2 R nkv) splits, never below 512 keys each.
// The kernel reads S back from the grid, so both sides agree by construction.
__host__ __device__ __forceinline__ Splits tc_split_len(int P, int S) {
  if (P <= 0 || S <= 0) return {0, 0};
  const int len = (((P + S - 1) / S) + kKB - 1) / kKB * kKB;
  return {(P + len - 1) / len, len};
}

inline Splits tc_splits(int P, int groups, int target_ctas) {
  int S = target_ctas / (2 * (groups > 0 ? groups : 1));
  // long prefixes: at least 512 keys a split; short ones (a latency-bound
  // job with few query tiles) split down to two 64-key blocks
  const int by_len = P / (P >= 2048 ? kTcMinKeysPerSplit : 2 * kKB);
  S = S > by_len ? by_len : S;
  S = S < 1 ? 1 : (S > kTcMaxSplits ? kTcMaxSplits : S);
  return tc_split_len(P, S);
}

// Fused kernel (short prefixes): every query tile is live, so S is the split
// count that brings the grid to about one wave, with at least two 64-key
// blocks a split.
constexpr double kFusedMaxFlops = 6.0e9;
inline Splits fused_splits(int P, int ctas, int target_ctas) {
  int S = target_ctas / (ctas > 0 ? ctas : 1);
  const int by_len = P / (2 * kKB);
  S = S > by_len ? by_len : S;
  S = S < 1 ? 1 : (S > kTcMaxSplits ? kTcMaxSplits : S);
  return tc_split_len(P, S);
}

template <int HD>
struct TcLayout {
  static constexpr int ST = kTcStages;                  // K (and V) ring stages
  static constexpr int QH = HD / 64;                    // 64-dim halves
  static constexpr int KV_TILE = kKB * 128;             // one 64-dim half of a K or V block
  static constexpr int STAGE = QH * KV_TILE;            // K (or V) of one block
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = ST * STAGE;
  static constexpr int OFF_BAR = 2 * ST * STAGE;
  static constexpr int BYTES = OFF_BAR + 256 + 1024;   // + alignment of the dynamic window
  // fused variant: the branch's own block keys and values (one 64-key block,
  // gathered), after the barriers; 128-byte-swizzled tiles start on a
  // 1024-byte boundary, where the MMA descriptors place the swizzle atoms
  static constexpr int OFF_BK = (OFF_BAR + 256 + 1023) / 1024 * 1024;
  static constexpr int OFF_BV = OFF_BK + STAGE;
  static constexpr int BYTES_FUSED = OFF_BV + STAGE + 1024;
  static constexpr int SBUF = 3;                        // score buffers: columns [64 s, 64 s + 64)
  static constexpr int Q_COL = SBUF * kKB;              // Q: HD / 2 columns of bf16 pairs
  static constexpr int O_COL = 256;                     // O: columns [256, 256 + HD)
  static constexpr int P_COL = O_COL + HD;              // P: two buffers of kKB / 2 columns of bf16 pairs
  static constexpr int TMEM_COLS = 512;
  static_assert(Q_COL + HD / 2 <= O_COL && P_COL + kKB <= TMEM_COLS, "TMEM columns");
  static_assert((4 * ST + 2 * SBUF + 6) * 8 + 8 <= 256, "barrier area");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_BK % 1024 == 0 && OFF_BV % 1024 == 0,
                "swizzled tiles on 1024-byte boundaries");
  static_assert(BYTES_FUSED <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void tmem_ld32_raw(uint32_t taddr, float (&v)[32]) { tc::tmem_ld32(taddr, v); }

// 2^x on the special-function unit (flushes subnormal results to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// kFused: the whole attention of every row of a branch in one kernel, for
// short prefixes.  The CTA's 128 query vectors are rows of one branch (row
// (b, v / G), query head kvh * G + v % G, the query of the row's source), the
// last split appends the branch's own block keys and values as one more
// 64-key block (gathered like Q, zero past L), and the merged state is
// normalised and written as the attention output: no partial state and no
// block kernel.  Folded rows repeat their source's prefix scores, which costs
// little while the prefix is short.
template <int HD, bool kFused>
__global__ void __launch_bounds__(kTcThreads, 1) attn_prefix_tc(const __grid_constant__ CUtensorMap tmK,
                                                                const __grid_constant__ CUtensorMap tmV,
                                                                const AttnArgs a) {
  using Lay = TcLayout<HD>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* sK = base + Lay::OFF_K;
  unsigned char* sV = base + Lay::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + Lay::OFF_BAR);
  uint64_t* kfull = bar;                   // [Lay::ST] K landed
  uint64_t* vfull = bar + Lay::ST;         // [Lay::ST] V landed
  uint64_t* kempty = bar + 2 * Lay::ST;    // [Lay::ST] K consumed by S = Q K^T
  uint64_t* vempty = bar + 3 * Lay::ST;    // [Lay::ST] V consumed by O += P V
  uint64_t* sfull = bar + 4 * Lay::ST;     // [SBUF] scores in TMEM
  uint64_t* sempty = sfull + Lay::SBUF;    // [SBUF] scores read
  uint64_t* pfull = sempty + Lay::SBUF;    // [2] P written
  uint64_t* pvdone = pfull + 2;            // [2] P V of that buffer done
  uint64_t* qready = pvdone + 2;
  uint64_t* ofull = qready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ofull + 1);
  __shared__ float xmax[2][2][kTcQ];             // [block parity][half][row]: partial block maxima

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid: x = split, y = (request, KV head) -- fused: (branch, KV head) --,
  // z = query tile; the splits of a tile and the first query tiles of every y
  // are dispatched first, the tiles that only a larger recompute set would
  // fill come last
  const int xr = blockIdx.y / a.nkv, kvh = blockIdx.y % a.nkv;
  const int r = kFused ? xr / a.Bp : xr;
  const Splits sp = tc_split_len(a.P, (int)gridDim.x);
  const int G = a.nq / a.nkv;
  // recompute offsets from the gate kernel (complete once this grid runs), past L1
  const int off_r = kFused ? 0 : __ldcg(a.meta + 1 + r);
  const int nqv = kFused ? a.L * G : (__ldcg(a.meta + 2 + r) - off_r) * G;
  const int q0 = blockIdx.z * kTcQ;
  // An empty tile leaves without the dependency wait: it reads nothing of the
  // previous kernel, and the live tiles (the main branch always recomputes,
  // so there is one per request and KV head) still hold the next kernel back
  // until they have waited.  Every split of a tile agrees.
  if (q0 >= nqv) return;
  const int s = (int)blockIdx.x;
  const int k_lo = s * sp.len, k_hi = min(a.P, k_lo + sp.len);
  const int nblk_p = (k_hi - k_lo + kKB - 1) / kKB;  // prefix blocks of this split
  // fused: the last split takes the branch's block keys as one more block
  const bool with_block = kFused && s == sp.S - 1;
  const int nblk = nblk_p + (with_block ? 1 : 0);

  if (tid == 0) {
    for (int i = 0; i < Lay::ST; ++i) {
      tc::mbar_init(&kfull[i], 1);
      tc::mbar_init(&vfull[i], 1);
      tc::mbar_init(&kempty[i], 1);
      tc::mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < Lay::SBUF; ++i) {
      tc::mbar_init(&sfull[i], 1);
      tc::mbar_init(&sempty[i], 256);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&pfull[i], 256);
      tc::mbar_init(&pvdone[i], 1);
    }
    tc::mbar_init(qready, 256);
    tc::mbar_init(ofull, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, Lay::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // lane 0 of warp 0 loads key block b into K stage b % Lay::ST, lane 0 of
  // warp 10 the value block into the V ring
  auto issue = [&](int b, bool keys) {
    const int st = b % Lay::ST;
    unsigned char* dst = (keys ? sK : sV) + st * Lay::STAGE;
    uint64_t* full = keys ? &kfull[st] : &vfull[st];
    const int z = r * a.P + k_lo + b * kKB;
    tc::mbar_expect_tx(full, Lay::QH * Lay::KV_TILE);
#pragma unroll
    for (int h = 0; h < Lay::QH; ++h) tc::tma_load_3d(dst + h * Lay::KV_TILE, keys ? &tmK : &tmV, h * 64, kvh, z, full);
  };
  // the prefix keys and values are inputs of the pass
  const bool producer = (warp == 0 || warp == kTcVWarp);
  if (producer && lane == 0)
    for (int b = 0; b < min(Lay::ST, nblk_p); ++b) issue(b, warp == 0);
  pdl_wait();
  pdl_trigger();

  const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);
  if (producer) {
    if (lane == 0) {
      const bool keys = warp == 0;
      for (int b = Lay::ST; b < nblk_p; ++b) {
        // the stage is free once the MMA that read block b - Lay::ST has completed
        tc::mbar_wait(keys ? &kempty[b % Lay::ST] : &vempty[b % Lay::ST], ((b / Lay::ST) - 1) & 1, a.err);
        issue(b, keys);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kTcPVWarp) {
    if (lane == 0) {
      // A descriptor's address field is the shared-memory address in 16-byte
      // units, so the descriptor of any tile of a ring is its first tile's
      // plus the offset / 16: built once here
      tc::mbar_wait(qready, 0, a.err);
      tc::fence_after_sync();
      if (warp == 1) {
        const uint32_t idesc_s = tc::idesc_bf16_f32(kTcQ, kKB);
        const uint64_t dk0 = tc::sw128_kmajor_desc(smem_addr(sK));
        const uint64_t dbk = tc::sw128_kmajor_desc(smem_addr(base + Lay::OFF_BK));
        // S(b) = Q K(b)^T into score buffer b % SBUF, up to SBUF blocks ahead of the softmax
        for (int b = 0; b < nblk; ++b) {
          const int st = b % Lay::ST, sb = b % Lay::SBUF;
          const bool blk = b >= nblk_p;  // fused: the branch's block keys, ready with Q
          if (!blk) tc::mbar_wait(&kfull[st], (b / Lay::ST) & 1, a.err);
          if (b >= Lay::SBUF) tc::mbar_wait(&sempty[sb], ((b / Lay::SBUF) - 1) & 1, a.err);
          tc::fence_after_sync();
          const uint64_t dk = blk ? dbk : dk0 + (uint64_t)((st * Lay::STAGE) >> 4);
          const uint32_t ds = tmem + sb * kKB;
          // 16 query dimensions a step = 8 TMEM columns of bf16 pairs
          tc::mma_bf16_ts(ds, tmem + Lay::Q_COL, dk, idesc_s, 0u);
#pragma unroll
          for (int kk = 1; kk < HD / 16; ++kk)
            tc::mma_bf16_ts(ds, tmem + Lay::Q_COL + kk * 8,
                            dk + (uint64_t)(((kk >> 2) * Lay::KV_TILE + (kk & 3) * 32) >> 4), idesc_s, 1u);
          tc::mma_commit(&sfull[sb]);
          if (!blk) tc::mma_commit(&kempty[st]);
        }
      } else {
        const uint32_t idesc_pv = tc::idesc_bf16_f32(kTcQ, HD) | (1u << 16);  // V is MN-major
        const uint64_t dv0 = tc::sw128_mnmajor_desc(smem_addr(sV), Lay::KV_TILE);
        const uint64_t dbv = tc::sw128_mnmajor_desc(smem_addr(base + Lay::OFF_BV), Lay::KV_TILE);
        for (int j = 0; j < nblk; ++j) {
          // O += P(j) V(j)
          const int st = j % Lay::ST, pb = j & 1;
          const bool blk = j >= nblk_p;
          tc::mbar_wait(&pfull[pb], (j >> 1) & 1, a.err);
          if (!blk) tc::mbar_wait(&vfull[st], (j / Lay::ST) & 1, a.err);
          tc::fence_after_sync();
          const uint64_t dv = blk ? dbv : dv0 + (uint64_t)((st * Lay::STAGE) >> 4);
          const uint32_t dp = tmem + Lay::P_COL + pb * (kKB / 2);
          tc::mma_bf16_ts(tmem + Lay::O_COL, dp, dv, idesc_pv, j > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < kKB / 16; ++kk)  // 16 keys a step: 2048 bytes of V, 8 columns of P
            tc::mma_bf16_ts(tmem + Lay::O_COL, dp + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), idesc_pv, 1u);
          tc::mma_commit(&pvdone[pb]);
          if (!blk) tc::mma_commit(&vempty[st]);
        }
        tc::mma_commit(ofull);
      }
    }
    __syncwarp();
  } else {
    // softmax warps: TMEM lanes 32 * (warp % 4) .. + 31, one query row per
    // thread pair; `half` selects 32 of the row's 64 scores and HD / 2 of its
    // query and output columns
    const int grp = warp & 3, half = (warp - 2) >> 2;
    const int row = 32 * grp + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * grp) << 16);
    const int v = q0 + row;
    {
      const bool ok = v < nqv;
      // fused: row (b, v / G) of the branch, whose query is its source's
      const int g = kFused ? __ldcg(a.rcslot + xr * a.L + (ok ? v / G : 0)) : off_r + (ok ? v / G : 0);
      const int h = kvh * G + (ok ? v % G : 0);
      const uint4* src = reinterpret_cast<const uint4*>(qkv + (size_t)g * a.ld_qkv + h * HD + half * (HD / 2));
      if constexpr (kFused) {
        if (with_block) {
          // the branch's block keys and values: key m of the branch's table is
          // the K/V row of its source slot (zero past L); 256 threads, 64 keys
          const int koff = (a.nq + kvh) * HD, voff = (a.nq + a.nkv + kvh) * HD;
          const int t = tid - 64;
          for (int idx = t; idx < kKB * (HD / 8); idx += 256) {
            const int m = idx / (HD / 8), c = idx % (HD / 8);
            const int gm = m < a.L ? __ldcg(a.rcslot + xr * a.L + m) : 0;
            const bf16* kr = qkv + (size_t)gm * a.ld_qkv;
            const int off = (c >> 3) * Lay::KV_TILE + m * 128 + (((c & 7) ^ (m & 7)) << 4);
            cp_async16(base + Lay::OFF_BK + off, kr + koff + c * 8, m < a.L);
            cp_async16(base + Lay::OFF_BV + off, kr + voff + c * 8, m < a.L);
          }
        }
        cp_async_commit();
      }
      // this thread's HD / 2 query dimensions as HD / 4 columns of bf16 pairs
      uint32_t qr[HD / 4];
#pragma unroll
      for (int c = 0; c < HD / 16; ++c) {
        const uint4 u = ok ? __ldcg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        qr[4 * c] = u.x;
        qr[4 * c + 1] = u.y;
        qr[4 * c + 2] = u.z;
        qr[4 * c + 3] = u.w;
      }
      tc::tmem_st_u32<HD / 4>(tl + Lay::Q_COL + half * (HD / 4), qr);
      tc::tmem_wait_st();
      if constexpr (kFused) {
        cp_async_wait<0>();
        tc::fence_proxy_async_smem();
      }
      tc::fence_before_sync();
      tc::mbar_arrive(qready);
    }
    const float scale = a.scale_log2;
    // running max in raw score units, partial denominator of this thread's keys
    float m_ref = -INFINITY, l = 0.f;
    for (int b = 0; b < nblk; ++b) {
      const int sb = b % Lay::SBUF, pbuf = b & 1;
      tc::mbar_wait(&sfull[sb], (b / Lay::SBUF) & 1, a.err);
      tc::fence_after_sync();
      float sc[32];
      tmem_ld32_raw(tl + sb * kKB + 32 * half, sc);
      tc::fence_before_sync();
      tc::mbar_arrive(&sempty[sb]);
      if (kFused && b >= nblk_p) {  // the branch's block keys: 64 slots, L of them real
        const int m0 = 32 * half;
        if (m0 + 32 > a.L) {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (m0 + k >= a.L) sc[k] = -INFINITY;
        }
      } else {
        const int kb0 = k_lo + b * kKB + 32 * half;
        if (kb0 + 32 > k_hi) {  // the split's last block may be ragged
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (kb0 + k >= k_hi) sc[k] = -INFINITY;
        }
      }
      // tree reduction: five dependent steps instead of 31
      float mt[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) mt[k] = fmaxf(sc[k], sc[k + 16]);
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) mt[k] = fmaxf(mt[k], mt[k + w]);
      const float mx = mt[0];
      // the row's block maximum: exchange with the partner warp (double-buffered by block parity)
      xmax[pbuf][half][row] = mx;
      tc::named_bar_sync(1 + grp, 64);
      const float mb = fmaxf(mx, xmax[pbuf][half ^ 1][row]);
      if (b == 0) {
        m_ref = mb;
      } else {
        const bool need = (mb - m_ref) * scale > kTcRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {  // warp-wide: the TMEM accesses are collective
          const float m_new = need ? mb : m_ref;
          const float f = ex2_approx((m_ref - m_new) * scale);
          // O holds every block before b once P V of block b - 1 is done
          tc::mbar_wait(&pvdone[(b - 1) & 1], ((b - 1) >> 1) & 1, a.err);
          tc::fence_after_sync();
#pragma unroll
          for (int c0 = half * (HD / 2); c0 < (half + 1) * (HD / 2); c0 += 32) {
            float o[32];
            tmem_ld32_raw(tl + Lay::O_COL + c0, o);
#pragma unroll
            for (int i2 = 0; i2 < 32; ++i2) o[i2] *= f;
            tc::tmem_st32(tl + Lay::O_COL + c0, o);
          }
          tc::tmem_wait_st();
          l *= f;
          m_ref = m_new;
        }
      }
      const float mneg = -m_ref * scale;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float p0 = ex2_approx(fmaf(sc[k], scale, mneg)), p1 = ex2_approx(fmaf(sc[k + 1], scale, mneg));
        ls[(k >> 1) & 3] += p0 + p1;
        pk[k / 2] = pack_bf16(p0, p1);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // P buffer b % 2 is free once P V of block b - 2 is done
      if (b >= 2) {
        tc::mbar_wait(&pvdone[pbuf], ((b - 2) >> 1) & 1, a.err);
        tc::fence_after_sync();
      }
      // keys 32 half .. + 31 of the block: columns 16 half .. + 15 of the buffer
      tc::tmem_st_u32<16>(tl + Lay::P_COL + pbuf * (kKB / 2) + 16 * half, pk);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&pfull[pbuf]);
    }
    // the row's denominator: both halves (through the buffer of the next
    // block parity, which the partner no longer reads)
    xmax[nblk & 1][half][row] = l;
    tc::named_bar_sync(1 + grp, 64);
    const float lrow = l + xmax[nblk & 1][half ^ 1][row];
    const float mrow = m_ref * scale;
    tc::mbar_wait(ofull, 0, a.err);
    tc::fence_after_sync();
    // Epilogue.  The rows go through shared memory (the K and V rings, idle
    // once every MMA has completed) so that a warp stores and loads whole
    // rows: one 16-byte piece a lane, 32 lanes on consecutive addresses.
    constexpr int HO = HD / 2, XLD = HD + 4;  // padded rows: the staging stores hit distinct banks
    float* xs = reinterpret_cast<float*>(base + Lay::OFF_K);
    float* xml = xs + kTcQ * XLD;  // per row: m (log2 units), l
    static_assert(kTcQ * (XLD + 2) * 4 <= 2 * Lay::ST * Lay::STAGE, "staging area within the rings");
#pragma unroll
    for (int c0 = 0; c0 < HO; c0 += 32) {
      float o[32];
      tmem_ld32_raw(tl + Lay::O_COL + half * HO + c0, o);
      float* dst = xs + row * XLD + half * HO + c0;
#pragma unroll
      for (int c = 0; c < 32; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
    }
    if (half == 0) *reinterpret_cast<float2*>(xml + 2 * row) = make_float2(m_ref * scale, lrow);
    tc::named_bar_sync(5, 256);
    // rows of the tile by warp: row rr = sw, sw + 8, ...; lane c4 < HD / 4 holds columns 4 c4 .. + 3
    const int sw = warp - 2;
    const int c4 = lane;
    const bool col_ok = c4 < HD / 4;
    const int rows = min(kTcQ, nqv - q0);
    auto vec_index = [&](int rr) {  // query vector (row of the layer) * nq + query head
      const int vv = q0 + rr;
      return (size_t)((kFused ? xr * a.L : off_r) + vv / G) * a.nq + kvh * G + vv % G;
    };
    auto write_final = [&](int rr, float4 acc, float M, float lsum) {
      const size_t qv = vec_index(rr);
      if constexpr (kFused) {
        const float inv = 1.f / lsum;
        const int vv = q0 + rr;
        bf16* dst = reinterpret_cast<bf16*>(a.attn) + (size_t)(xr * a.L + vv / G) * a.ld_attn + (kvh * G + vv % G) * HD;
        if (col_ok)
          *reinterpret_cast<uint2*>(dst + 4 * c4) =
              make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
      } else {
        if (col_ok) *reinterpret_cast<float4*>(a.part_o + qv * HD + 4 * c4) = acc;
        if (lane == 0) *reinterpret_cast<float2*>(a.part_ml + qv * 2) = make_float2(M, lsum);
      }
    };
    // a warp takes its rows four at a time (rr, rr + 8, rr + 16, rr + 24), all
    // four rows' loads in flight before their stores
    constexpr int RB = 4;
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (sp.S == 1) {
      for (int r0 = sw; r0 < rows; r0 += 8 * RB) {
        float4 acc[RB];
        float2 ml[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int rr = r0 + 8 * u;
          acc[u] = rr < rows && col_ok ? *reinterpret_cast<const float4*>(xs + rr * XLD + 4 * c4) : zero4;
          ml[u] = rr < rows ? *reinterpret_cast<const float2*>(xml + 2 * rr) : make_float2(0.f, 1.f);
        }
#pragma unroll
        for (int u = 0; u < RB; ++u)
          if (r0 + 8 * u < rows) write_final(r0 + 8 * u, acc[u], ml[u].x, ml[u].y);
      }
    } else {
      // publish this split's partial state in slot 1 + s
      const size_t TQ = (size_t)a.T * a.nq;
      for (int r0 = sw; r0 < rows; r0 += 8 * RB) {
        float4 val[RB];
        float2 ml[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int rr = r0 + 8 * u;
          val[u] = rr < rows && col_ok ? *reinterpret_cast<const float4*>(xs + rr * XLD + 4 * c4) : zero4;
          ml[u] = rr < rows ? *reinterpret_cast<const float2*>(xml + 2 * rr) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int rr = r0 + 8 * u;
          if (rr < rows) {
            const size_t qv = (1 + s) * TQ + vec_index(rr);
            if (col_ok) *reinterpret_cast<float4*>(a.part_o + qv * HD + 4 * c4) = val[u];
            if (lane == 0) *reinterpret_cast<float2*>(a.part_ml + qv * 2) = ml[u];
          }
        }
      }
      __threadfence();
      // every split of the tile has published once the cluster has met
      tc::cluster_sync_all();
      // merge rows [s per, (s + 1) per): this split's own state from shared memory, the others' through L2
      const int per = (kTcQ + sp.S - 1) / sp.S;
      const int m_hi = min(rows, (s + 1) * per);
      for (int r0 = s * per + sw; r0 < m_hi; r0 += 8 * RB) {
        size_t qv[RB];
        float2 ml[RB][kTcMaxSplits];
        float4 part[RB][kTcMaxSplits];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int rr = r0 + 8 * u;
          qv[u] = rr < m_hi ? vec_index(rr) : 0;
#pragma unroll
          for (int t = 0; t < kTcMaxSplits; ++t) {
            if (rr >= m_hi || t >= sp.S) {
              ml[u][t] = make_float2(-INFINITY, 0.f);
              part[u][t] = zero4;
            } else if (t == s) {
              ml[u][t] = *reinterpret_cast<const float2*>(xml + 2 * rr);
              part[u][t] = col_ok ? *reinterpret_cast<const float4*>(xs + rr * XLD + 4 * c4) : zero4;
            } else {
              const size_t q = (1 + t) * TQ + qv[u];
              ml[u][t] = __ldcg(reinterpret_cast<const float2*>(a.part_ml + q * 2));
              part[u][t] = col_ok ? __ldcg(reinterpret_cast<const float4*>(a.part_o + q * HD + 4 * c4)) : zero4;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int rr = r0 + 8 * u;
          if (rr >= m_hi) continue;
          float M = -INFINITY;
#pragma unroll
          for (int t = 0; t < kTcMaxSplits; ++t) M = fmaxf(M, ml[u][t].x);
          float lsum = 0.f;
          float4 acc = zero4;
#pragma unroll
          for (int t = 0; t < kTcMaxSplits; ++t) {
            if (t < sp.S) {
              const float w = exp2f(ml[u][t].x - M);
              lsum += w * ml[u][t].y;
              acc.x += w * part[u][t].x;
              acc.y += w * part[u][t].y;
              acc.z += w * part[u][t].z;
              acc.w += w * part[u][t].w;
            }
          }
          write_final(rr, acc, M, lsum);
        }
      }
    }
  }
  // the other warps meet the cluster too (the softmax warps did above)
  if (sp.S > 1 && (warp < 2 || warp == kTcVWarp || warp == kTcPVWarp)) tc::cluster_sync_all();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Lay::TMEM_COLS);
  }
}

// ------------------------------------------------------------ tcgen05 block path
//
// Block attention + merge on the 5th-generation tensor cores: CTA = 128 query
// vectors of one branch and KV head (one per TMEM lane and thread), query
// vector v = block position v / G with query head kvh * G + v % G, its query
// the one of the row's resolved source.  Keys and values are the branch's own
// block table K_i[m] = QKV[rcslot(i, m)], gathered with asynchronous copies
// into 128-byte-swizzled tiles of NK = 32 or 64 keys (zero past L):
//   S = Q K^T   one tcgen05.mma chain (K-major Q and K), S in TMEM;
//   P = exp2(S - m_b) per row by its thread, bf16 into swizzled shared memory;
//   O = P V     tcgen05.mma (V MN-major), O in the same TMEM columns as S,
//               which every thread has read by then;
// then each thread merges its row with the query's prefix partial state by
// log-sum-exp and writes the normalised bf16 output.
constexpr int kBlkQ = 128;
constexpr int kBlkMaxKeys = 64;

// Shared memory: Q (128 rows x HD, as 64-dim halves), then the K and V tiles
// of NK keys (per 64-dim half NK rows of 128 bytes), then two mbarriers and
// the TMEM address.  P (128 rows x NK keys, bf16) reuses Q's space once
// S = Q K^T has completed.
template <int HD>
struct BlkLayout {
  static constexpr int QH = HD / 64;
  static constexpr int Q_HALF = kBlkQ * 128;  // 128 rows x 64 dims
  static constexpr int TMEM_COLS = HD;        // S in columns [0, NK), then O in [0, HD)
  static __host__ __device__ constexpr int kv_half(int nk) { return nk * 128; }
  static __host__ __device__ constexpr int off_k() { return QH * Q_HALF; }
  static __host__ __device__ constexpr int off_v(int nk) { return off_k() + QH * kv_half(nk); }
  static __host__ __device__ constexpr int off_bar(int nk) { return off_v(nk) + QH * kv_half(nk); }
  static __host__ __device__ constexpr int bytes(int nk) { return off_bar(nk) + 64 + 1024; }
  static_assert(QH * Q_HALF % 1024 == 0 && kv_half(32) % 1024 == 0, "swizzled tiles on 1024-byte boundaries");
};

template <int HD>
__global__ void __launch_bounds__(kBlkQ) attn_block_tc(const AttnArgs a) {
  using Lay = BlkLayout<HD>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int NK = a.L <= 32 ? 32 : 64;
  const int KVH = Lay::kv_half(NK);
  unsigned char* sQ = base;
  unsigned char* sK = base + Lay::off_k();
  unsigned char* sV = base + Lay::off_v(NK);
  unsigned char* sP = base;  // over Q once S = Q K^T has completed
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + Lay::off_bar(NK));  // [0] S done, [1] O done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  __shared__ int slot[kBlkMaxKeys];
  __shared__ int pos[kBlkMaxKeys];  // block positions of this CTA's query rows
  __shared__ int s_npos;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int rb = blockIdx.y / a.nkv, kvh = blockIdx.y % a.nkv;  // rb = r * Bp + i
  const int G = a.nq / a.nkv, L = a.L;
  const int q0 = blockIdx.x * kBlkQ;
  const bool correct = a.mode == SF_ATTN_CORRECT;
  // Every kernel of the pass lets its dependants start only after its own
  // dependency wait, so the kernels before the previous one have completed
  // when this grid starts: with a prefix kernel in between, the source slots
  // and the recompute list (gate kernel) and the projected rows are read
  // before the wait, past L1.
  if (a.P == 0) {
    pdl_wait();
    pdl_trigger();
  }
  const int cnt = __ldcg(a.meta);
  for (int m = tid; m < kBlkMaxKeys; m += kBlkQ) {
    int g = m < L ? __ldcg(a.rcslot + rb * L + m) : 0;
    if (g < 0 || g >= cnt) {
      raise_error(a.err, kErrAttn);
      g = 0;
    }
    slot[m] = g;
  }
  __syncthreads();
  // the rows of the branch this kernel answers for: all of them, or with the
  // correction mode only the rows that recompute (their own source)
  if (tid == 0) {
    int np = 0;
    for (int m = 0; m < L; ++m)
      if (!correct || __ldcg(a.rc + slot[m]) == rb * L + m) pos[np++] = m;
    s_npos = np;
  }
  __syncthreads();
  const int nqv = s_npos * G;
  if (q0 >= nqv) return;  // uniform over the CTA
  const int v = q0 + tid;
  const bool live = v < nqv;
  const int vn = live ? pos[v / G] : 0;  // block position of this thread's query row
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, Lay::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // gather: this thread's query row, and keys/values m = tid / 2 (two threads
  // per key, one per 64-dim half when HD = 128)
  const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);
  {
    const bf16* src = qkv + (size_t)slot[vn] * a.ld_qkv + (kvh * G + (live ? v % G : 0)) * HD;
#pragma unroll
    for (int c = 0; c < HD / 8; ++c)
      cp_async16(sQ + (c >> 3) * Lay::Q_HALF + tid * 128 + (((c & 7) ^ (tid & 7)) << 4), src + c * 8, live);
    const int koff = (a.nq + kvh) * HD, voff = (a.nq + a.nkv + kvh) * HD;
    for (int idx = tid; idx < NK * (HD / 8); idx += kBlkQ) {
      const int m = idx / (HD / 8), c = idx % (HD / 8);
      const bf16* row = qkv + (size_t)slot[m] * a.ld_qkv;
      const int off = (c >> 3) * KVH + m * 128 + (((c & 7) ^ (m & 7)) << 4);
      cp_async16(sK + off, row + koff + c * 8, m < L);
      cp_async16(sV + off, row + voff + c * 8, m < L);
    }
    cp_async_commit();
  }
  size_t qi = 0;
  if (live) qi = (size_t)slot[vn] * a.nq + kvh * G + v % G;
  cp_async_wait<0>();
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(kBlkQ, NK);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const uint64_t dq = tc::sw128_kmajor_desc(smem_addr(sQ + (kk >> 2) * Lay::Q_HALF + (kk & 3) * 32));
      const uint64_t dk = tc::sw128_kmajor_desc(smem_addr(sK + (kk >> 2) * KVH + (kk & 3) * 32));
      tc::mma_bf16(tmem, dq, dk, idesc, kk > 0 ? 1u : 0u);
    }
    tc::mma_commit(&bar[0]);
  }
  const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
  tc::mbar_wait(&bar[0], 0, a.err);
  tc::fence_after_sync();
  // softmax of the row over its L block keys (log2 units)
  float sc[kBlkMaxKeys];
  tc::tmem_ld32(tl, *reinterpret_cast<float(*)[32]>(sc));
  if (NK > 32) tc::tmem_ld32(tl + 32, *reinterpret_cast<float(*)[32]>(sc + 32));
  float mb = -INFINITY;
#pragma unroll
  for (int k = 0; k < kBlkMaxKeys; ++k) {
    if (k < NK) {
      sc[k] = k < L ? sc[k] * a.scale_log2 : -INFINITY;
      mb = fmaxf(mb, sc[k]);
    }
  }
  float lb = 0.f;
  unsigned char* prow = sP + tid * 128;
#pragma unroll
  for (int c = 0; c < kBlkMaxKeys / 8; ++c) {
    if (c * 8 < NK) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = exp2f(sc[c * 8 + 2 * e] - mb), p1 = exp2f(sc[c * 8 + 2 * e + 1] - mb);
        lb += p0 + p1;
        pk[e] = pack_bf16(p0, p1);
      }
      *reinterpret_cast<uint4*>(prow + ((c ^ (tid & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();  // every row's P is written and every S read
  tc::fence_after_sync();
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(kBlkQ, HD) | (1u << 16);  // V is MN-major
    for (int kk = 0; kk < NK / 16; ++kk) {
      const uint64_t dp = tc::sw128_kmajor_desc(smem_addr(sP + kk * 32));
      const uint64_t dv = tc::sw128_mnmajor_desc(smem_addr(sV + kk * 2048), KVH);
      tc::mma_bf16(tmem, dp, dv, idesc, kk > 0 ? 1u : 0u);
    }
    tc::mma_commit(&bar[1]);
  }
  // Everything above reads only the projected rows and the gate's slots
  // (complete when this grid starts); the prefix kernel's partial state is
  // read from here on.  A CTA that starts while the prefix kernel still runs
  // has its block part done by the time the partial is ready.
  float mp = 0.f, lp = 0.f;
  if (a.P > 0) {
    pdl_wait();
    pdl_trigger();
    if (live) {
      mp = a.part_ml[qi * 2];
      lp = a.part_ml[qi * 2 + 1];
    }
  }
  // merge weights of the block part and the prefix partial
  float wb = 1.f, wp = 0.f, l = lb;
  if (a.P > 0) {
    const float M = fmaxf(mb, mp);
    wb = exp2f(mb - M);
    wp = exp2f(mp - M);
    l = lb * wb + lp * wp;
  }
  const float inv = 1.f / l;
  bf16* dst = reinterpret_cast<bf16*>(a.attn) + (size_t)(rb * L + vn) * a.ld_attn + (kvh * G + (live ? v % G : 0)) * HD;
  float* po = a.part_o + qi * HD;
  // correction mode: the row's merged state (max in log2 units, denominator,
  // unnormalised output) replaces its prefix partial for the correction kernel
  if (correct && live) {
    a.part_ml[qi * 2] = a.P > 0 ? fmaxf(mb, mp) : mb;
    a.part_ml[qi * 2 + 1] = l;
  }
  // the prefix partial is read 32 columns at a time, each chunk's loads issued
  // before the previous chunk is applied (the first while P V runs)
  const bool pre = a.P > 0 && live;
  float4 cur[8], nxt[8];
  if (pre) {
#pragma unroll
    for (int e = 0; e < 8; ++e) cur[e] = *reinterpret_cast<const float4*>(po + 4 * e);
  }
  tc::mbar_wait(&bar[1], 0, a.err);
  tc::fence_after_sync();
#pragma unroll
  for (int c0 = 0; c0 < HD; c0 += 32) {
    if (pre && c0 + 32 < HD) {
#pragma unroll
      for (int e = 0; e < 8; ++e) nxt[e] = *reinterpret_cast<const float4*>(po + c0 + 32 + 4 * e);
    }
    float o[32];
    tc::tmem_ld32(tl + c0, o);
    if (live) {
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = o[c + e] * wb;
        if (a.P > 0) {
          const float4 p0 = cur[c / 4], p1 = cur[c / 4 + 1];
          x[0] += wp * p0.x; x[1] += wp * p0.y; x[2] += wp * p0.z; x[3] += wp * p0.w;
          x[4] += wp * p1.x; x[5] += wp * p1.y; x[6] += wp * p1.z; x[7] += wp * p1.w;
        }
        *reinterpret_cast<uint4*>(dst + c0 + c) =
            make_uint4(pack_bf16(x[0] * inv, x[1] * inv), pack_bf16(x[2] * inv, x[3] * inv),
                       pack_bf16(x[4] * inv, x[5] * inv), pack_bf16(x[6] * inv, x[7] * inv));
        if (correct) {
          *reinterpret_cast<float4*>(po + c0 + c) = make_float4(x[0], x[1], x[2], x[3]);
          *reinterpret_cast<float4*>(po + c0 + c + 4) = make_float4(x[4], x[5], x[6], x[7]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) cur[e] = nxt[e];
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Lay::TMEM_COLS);
  }
}

// ------------------------------------------------------------ CUDA-core path (fp32 contexts)

template <typename TAct>
__global__ void __launch_bounds__(128) attn_prefix_simt(const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float qs[4][kMaxHd];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qv = blockIdx.x * 4 + warp;
  const int g = qv / a.nq, h = qv % a.nq;
  const Splits sp = prefix_splits(a);
  const int s = blockIdx.y;
  if (s >= sp.S) return;
  const int count = a.meta[0];
  if (g >= count) return;
  int r = 0;
  while (r + 1 < a.R && a.meta[2 + r] <= g) ++r;
  const int G = a.nq / a.nkv, kvh = h / G, hd = a.hd, per = hd / 32;
  const TAct* qkv = reinterpret_cast<const TAct*>(a.qkv);
  for (int j = lane; j < hd; j += 32) qs[warp][j] = to_f32<TAct>(qkv[(size_t)g * a.ld_qkv + h * hd + j]);
  __syncwarp();
  const int k_lo = s * sp.len, k_hi = min(a.P, k_lo + sp.len);
  const TAct* K = reinterpret_cast<const TAct*>(a.pk) + (size_t)r * a.P * a.nkv * hd + kvh * hd;
  const TAct* V = reinterpret_cast<const TAct*>(a.pv) + (size_t)r * a.P * a.nkv * hd + kvh * hd;
  const size_t kstride = (size_t)a.nkv * hd;
  float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int kb = k_lo; kb < k_hi; kb += 32) {
    const int key = kb + lane;
    float sc = -INFINITY;
    if (key < k_hi) {
      const TAct* kr = K + key * kstride;
      float dot = 0.f;
      for (int j = 0; j < hd; j += 4) {
        const float4 kv = load4<TAct>(kr + j);
        dot += qs[warp][j] * kv.x + qs[warp][j + 1] * kv.y + qs[warp][j + 2] * kv.z + qs[warp][j + 3] * kv.w;
      }
      sc = dot * a.scale_log2;
    }
    const float m_new = fmaxf(m, warp_max(sc));
    const float p = key < k_hi ? exp2f(sc - m_new) : 0.f;
    const float corr = exp2f(m - m_new);
    l = l * corr + warp_sum(p);
    for (int c = 0; c < per; ++c) acc[c] *= corr;
    const int nk = min(32, k_hi - kb);
    for (int t = 0; t < nk; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p, t);
      const TAct* vr = V + (kb + t) * kstride;
      for (int c = 0; c < per; ++c) acc[c] += pt * to_f32<TAct>(vr[lane + 32 * c]);
    }
    m = m_new;
  }
  const size_t qi = ((size_t)s * a.T + g) * a.nq + h;
  for (int c = 0; c < per; ++c) a.part_o[qi * hd + lane + 32 * c] = acc[c];
  if (lane == 0) {
    a.part_ml[qi * 2 + 0] = m;
    a.part_ml[qi * 2 + 1] = l;
  }
}

template <typename TAct>
__global__ void __launch_bounds__(128) attn_block_simt(const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float qs[4][kMaxHd];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * 4 + warp;
  const int row = w / a.nq, h = w % a.nq;
  if (row >= a.T) return;
  const int count = a.meta[0];
  const int G = a.nq / a.nkv, kvh = h / G, hd = a.hd, per = hd / 32, L = a.L;
  const int g = a.rcslot[row];
  if (g < 0 || g >= count) {
    raise_error(a.err, kErrAttn);
    return;
  }
  // correction mode: only the rows that recompute (their own source)
  if (a.mode == SF_ATTN_CORRECT && a.rc[g] != row) return;
  const TAct* qkv = reinterpret_cast<const TAct*>(a.qkv);
  for (int j = lane; j < hd; j += 32) qs[warp][j] = to_f32<TAct>(qkv[(size_t)g * a.ld_qkv + h * hd + j]);
  __syncwarp();
  const int base = (row / L) * L;
  const int koff = (a.nq + kvh) * hd, voff = (a.nq + a.nkv + kvh) * hd;
  float sc[2] = {-INFINITY, -INFINITY};
  int ks[2] = {0, 0};
  for (int rr = 0; rr < 2; ++rr) {
    const int mk = lane + 32 * rr;
    if (mk < L) {
      const int kslot = a.rcslot[base + mk];
      ks[rr] = kslot;
      const TAct* kr = qkv + (size_t)kslot * a.ld_qkv + koff;
      float dot = 0.f;
      for (int j = 0; j < hd; j += 4) {
        const float4 kv = load4<TAct>(kr + j);
        dot += qs[warp][j] * kv.x + qs[warp][j + 1] * kv.y + qs[warp][j + 2] * kv.z + qs[warp][j + 3] * kv.w;
      }
      sc[rr] = dot * a.scale_log2;
    }
  }
  const Splits sp = prefix_splits(a);
  float M = warp_max(fmaxf(sc[0], sc[1]));
  for (int s = 0; s < sp.S; ++s) M = fmaxf(M, a.part_ml[(((size_t)s * a.T + g) * a.nq + h) * 2]);
  float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < sp.S; ++s) {
    const size_t qi = ((size_t)s * a.T + g) * a.nq + h;
    const float wgt = exp2f(a.part_ml[qi * 2] - M);
    l += wgt * a.part_ml[qi * 2 + 1];
    for (int c = 0; c < per; ++c) acc[c] += wgt * a.part_o[qi * hd + lane + 32 * c];
  }
  float p[2];
  for (int rr = 0; rr < 2; ++rr) p[rr] = (lane + 32 * rr < L) ? exp2f(sc[rr] - M) : 0.f;
  l += warp_sum(p[0] + p[1]);
  for (int rr = 0; rr < 2; ++rr) {
    const int nk = min(32, L - 32 * rr);
    for (int t = 0; t < nk; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p[rr], t);
      const int vslot = __shfl_sync(0xffffffffu, ks[rr], t);
      const TAct* vr = qkv + (size_t)vslot * a.ld_qkv + voff;
      for (int c = 0; c < per; ++c) acc[c] += pt * to_f32<TAct>(vr[lane + 32 * c]);
    }
  }
  const float inv = 1.f / l;
  TAct* out = reinterpret_cast<TAct*>(a.attn) + (size_t)row * a.ld_attn + h * hd;
  for (int c = 0; c < per; ++c) out[lane + 32 * c] = from_f32<TAct>(acc[c] * inv);
  if (a.mode == SF_ATTN_CORRECT) {
    // the merged state replaces the first split's prefix partial (index
    // slot * nq + head), which only this row read
    __syncwarp();
    const size_t qi = (size_t)g * a.nq + h;
    for (int c = 0; c < per; ++c) a.part_o[qi * hd + lane + 32 * c] = acc[c];
    if (lane == 0) {
      a.part_ml[qi * 2] = M;
      a.part_ml[qi * 2 + 1] = l;
    }
  }
}

// The subtract/add correction of a folded row ("SpecFold" §A.1, applied
// against the nearest recomputed ancestor as in §A.3): one warp per (row,
// query head).  The row's source row recomputed its query and left its merged
// softmax state (max M in log2 units, denominator l, unnormalised output acc)
// over the shared prefix and the source branch's block keys.  At the block
// positions where the row's own branch reads a different key/value slot than
// the source branch, the source's contribution is removed and the branch's
// own added:
//   M' = max(M, new scores);  l' = l 2^(M-M') - sum 2^(s_old-M') + sum 2^(s_new-M')
//   acc' = acc 2^(M-M') - sum 2^(s_old-M') v_old + sum 2^(s_new-M') v_new
// and the output is acc' / l'.  Recompute rows were written by the block
// kernel and are skipped.
template <typename TAct>
__global__ void __launch_bounds__(128) attn_correct_kernel(const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * 4 + warp;
  const int row = w / a.nq, h = w % a.nq;
  if (row >= a.T) return;
  const int count = a.meta[0];
  const int g = a.rcslot[row];
  if (g < 0 || g >= count) {
    raise_error(a.err, kErrAttn);
    return;
  }
  const int srow = a.rc[g];
  if (srow == row) return;  // a recompute row
  if (srow < 0 || srow >= a.T) {
    raise_error(a.err, kErrAttn);
    return;
  }
  const int G = a.nq / a.nkv, kvh = h / G, hd = a.hd, per = hd / 32, L = a.L;
  const int base_i = (row / L) * L, base_s = (srow / L) * L;
  const TAct* qkv = reinterpret_cast<const TAct*>(a.qkv);
  float q[kMaxHd / 32];
  for (int c = 0; c < per; ++c) q[c] = to_f32<TAct>(qkv[(size_t)g * a.ld_qkv + h * hd + lane + 32 * c]);
  const size_t qi = (size_t)g * a.nq + h;
  const float M = a.part_ml[qi * 2], l0 = a.part_ml[qi * 2 + 1];
  // block positions whose key/value slot differs between the branch and the source branch
  int ki[2] = {0, 0}, ks[2] = {0, 0};
  unsigned dmask[2] = {0u, 0u};
  for (int rr = 0; rr < 2; ++rr) {
    const int m = lane + 32 * rr;
    bool diff = false;
    if (m < L) {
      ki[rr] = a.rcslot[base_i + m];
      ks[rr] = a.rcslot[base_s + m];
      diff = ki[rr] != ks[rr];
    }
    dmask[rr] = __ballot_sync(0xffffffffu, diff);
  }
  const int koff = (a.nq + kvh) * hd, voff = (a.nq + a.nkv + kvh) * hd;
  auto score = [&](int slot) {
    const TAct* kr = qkv + (size_t)slot * a.ld_qkv + koff;
    float dot = 0.f;
    for (int c = 0; c < per; ++c) dot += q[c] * to_f32<TAct>(kr[lane + 32 * c]);
    return warp_sum(dot) * a.scale_log2;
  };
  // pass 1: the scores at the changed positions (lane m % 32 keeps those of position m)
  float s_old[2] = {0.f, 0.f}, s_new[2] = {0.f, 0.f};
  float Mn = M;
  for (int rr = 0; rr < 2; ++rr) {
    for (unsigned mk = dmask[rr]; mk; mk &= mk - 1) {
      const int t = __ffs(mk) - 1;
      const float so = score(__shfl_sync(0xffffffffu, ks[rr], t));
      const float sn = score(__shfl_sync(0xffffffffu, ki[rr], t));
      if (lane == t) {
        s_old[rr] = so;
        s_new[rr] = sn;
      }
      Mn = fmaxf(Mn, sn);
    }
  }
  // pass 2: rescale to the new max, remove the old contributions, add the new
  const float f = exp2f(M - Mn);
  float l = l0 * f;
  float acc[kMaxHd / 32];
  for (int c = 0; c < per; ++c) acc[c] = a.part_o[qi * hd + lane + 32 * c] * f;
  for (int rr = 0; rr < 2; ++rr) {
    for (unsigned mk = dmask[rr]; mk; mk &= mk - 1) {
      const int t = __ffs(mk) - 1;
      const float wo = exp2f(__shfl_sync(0xffffffffu, s_old[rr], t) - Mn);
      const float wn = exp2f(__shfl_sync(0xffffffffu, s_new[rr], t) - Mn);
      const TAct* vo = qkv + (size_t)__shfl_sync(0xffffffffu, ks[rr], t) * a.ld_qkv + voff;
      const TAct* vn = qkv + (size_t)__shfl_sync(0xffffffffu, ki[rr], t) * a.ld_qkv + voff;
      l += wn - wo;
      for (int c = 0; c < per; ++c)
        acc[c] += wn * to_f32<TAct>(vn[lane + 32 * c]) - wo * to_f32<TAct>(vo[lane + 32 * c]);
    }
  }
  const float inv = 1.f / l;
  TAct* out = reinterpret_cast<TAct*>(a.attn) + (size_t)row * a.ld_attn + h * hd;
  for (int c = 0; c < per; ++c) out[lane + 32 * c] = from_f32<TAct>(acc[c] * inv);
}

template <int HD>
cudaError_t attention_tc(Launch& lc, const AttnArgs& a) {
  const int G = a.nq / a.nkv;
  static cudaError_t attr = [&] {
    cudaError_t e = cudaFuncSetAttribute(attn_prefix_tc<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcLayout<HD>::BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_prefix_tc<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               TcLayout<HD>::BYTES_FUSED);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_block_tc<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, BlkLayout<HD>::bytes(64));
    return e;
  }();
  if (attr != cudaSuccess) return lc.err = attr;
  // short prefixes, direct mode: one fused kernel does every row's whole
  // attention, repeating the prefix scores of folded rows (at most about
  // kFusedMaxFlops of score and value products for all rows of the layer)
  const bool fused = a.P > 0 && a.mode == SF_ATTN_DIRECT &&
                     4.0 * a.T * a.nq * a.hd * (double)a.P <= kFusedMaxFlops;
  if (a.P > 0) {
    alignas(64) CUtensorMap tmK, tmV;
    if (!make_tmap_kv(&tmK, a.pk, HD, a.nkv, (uint64_t)a.R * a.P) ||
        !make_tmap_kv(&tmV, a.pv, HD, a.nkv, (uint64_t)a.R * a.P))
      return lc.err = cudaErrorInvalidValue;
    // fused: the whole attention of every row in the prefix kernel (short
    // prefixes, direct mode); the grid covers every row of every branch
    if (fused) {
      const int tiles = (a.L * G + kTcQ - 1) / kTcQ;
      const Splits sp = fused_splits(a.P, a.R * a.Bp * a.nkv * tiles, a.target_ctas);
      dim3 grid(sp.S, a.R * a.Bp * a.nkv, tiles);
      lc.before(SF_K_ATTN_PREFIX);
      lc.check(launch_pdl_cluster(lc.st, grid, dim3(kTcThreads), (size_t)TcLayout<HD>::BYTES_FUSED, dim3(sp.S, 1, 1),
                                  attn_prefix_tc<HD, true>, tmK, tmV, a));
      lc.after(SF_K_ATTN_PREFIX);
      return lc.err;
    }
    // worst case: every row of a request recomputes
    lc.before(SF_K_ATTN_PREFIX);
    {
      const Splits sp = tc_splits(a.P, a.R * a.nkv, a.target_ctas);
      dim3 grid(sp.S, a.R * a.nkv, (a.Bp * a.L * G + kTcQ - 1) / kTcQ);
      lc.check(launch_pdl_cluster(lc.st, grid, dim3(kTcThreads), (size_t)TcLayout<HD>::BYTES, dim3(sp.S, 1, 1),
                                  attn_prefix_tc<HD, false>, tmK, tmV, a));
    }
    lc.after(SF_K_ATTN_PREFIX);
  }
  dim3 grid((a.L * G + kBlkQ - 1) / kBlkQ, a.R * a.Bp * a.nkv);
  lc.before(SF_K_ATTN_BLOCK);
  lc.check(launch_pdl(lc.st, grid, dim3(kBlkQ), (size_t)BlkLayout<HD>::bytes(a.L <= 32 ? 32 : 64), 1,
                      attn_block_tc<HD>, a));
  lc.after(SF_K_ATTN_BLOCK);
  if (a.mode == SF_ATTN_CORRECT) {
    lc.before(SF_K_ATTN_CORRECT);
    lc.check(launch_pdl(lc.st, dim3((a.T * a.nq + 3) / 4), dim3(128), 0, 1, attn_correct_kernel<bf16>, a));
    lc.after(SF_K_ATTN_CORRECT);
  }
  return lc.err;
}

template <typename TAct>
cudaError_t attention_simt(Launch& lc, const AttnArgs& a) {
  if (a.P > 0) {
    dim3 grid((a.T * a.nq + 3) / 4, kMaxSplits);
    lc.before(SF_K_ATTN_PREFIX);
    lc.check(launch_pdl(lc.st, grid, dim3(128), 0, 1, attn_prefix_simt<TAct>, a));
    lc.after(SF_K_ATTN_PREFIX);
  }
  lc.before(SF_K_ATTN_BLOCK);
  lc.check(launch_pdl(lc.st, dim3((a.T * a.nq + 3) / 4), dim3(128), 0, 1, attn_block_simt<TAct>, a));
  lc.after(SF_K_ATTN_BLOCK);
  if (a.mode == SF_ATTN_CORRECT) {
    lc.before(SF_K_ATTN_CORRECT);
    lc.check(launch_pdl(lc.st, dim3((a.T * a.nq + 3) / 4), dim3(128), 0, 1, attn_correct_kernel<TAct>, a));
    lc.after(SF_K_ATTN_CORRECT);
  }
  return lc.err;
}

}  // namespace

cudaError_t launch_attention(Launch& lc, int act_bf16, const AttnArgs& a) {
  if (a.hd > kMaxHd || a.hd % 32 != 0 || a.L > kKB) return cudaErrorInvalidValue;
  if (!act_bf16) return attention_simt<float>(lc, a);
  if (a.hd == 128) return attention_tc<128>(lc, a);
  if (a.hd == 64) return attention_tc<64>(lc, a);
  return cudaErrorInvalidValue;
}

}  // namespace sf
