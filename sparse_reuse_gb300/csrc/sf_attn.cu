// Folded self-attention of one layer, exact against each branch's own keys.
//
// "SpecFold" (arXiv 2610.04875v2 summary) §A.1: a folded row's attention is
// the child's attention state exactly; App. B: attention kernels process the
// recomputed queries and keep per-head softmax max/denominator state; the
// onedev.kr review ("How to use it"): FlashAttention-style streaming, the
// shared prefix KV seen by every branch through a zero-copy strided view, GQA.
//
// Decomposition used here (same result, different order of work):
//   1. prefix partial per recomputed query: streaming softmax state
//      (max, denominator, unnormalised output) of q against the request's
//      prefix keys, the prefix split over S chunks;
//   2. per (row, head): the query is the one of the row's resolved source;
//      its block part runs over the branch's own L block keys/values, read
//      through the source slots of the branch's positions, and is merged with
//      the query's prefix partials by log-sum-exp.
// The tensor-core path fixes the split count S from the prefix length (a
// cluster of S CTAs per query tile); the CUDA-core path derives S on the
// device from the live recompute count, identically in both of its kernels.
//
// BF16 contexts run both kernels on the tensor cores (mma.sync m16n8k16, bf16
// in, fp32 accumulate); the GQA group's query heads are packed into the M
// dimension so every key/value tile is read once per KV head.  FP32 contexts
// use CUDA-core kernels that keep fp32 operands.
#include "sf_internal.h"
#include "sf_tc.cuh"

namespace sf {
namespace {

constexpr int kMaxHd = 128;
constexpr int kMaxSplits = 8;
constexpr int kQT = 64;  // query vectors per CTA (16 per warp)
constexpr int kKB = 64;  // keys per block

// Number of prefix splits and keys per split for this pass.
struct Splits {
  int S, len;
};

// Tensor-core path: the split count is fixed on the host from the prefix
// length alone, so the split CTAs of a query tile form a cluster of exactly
// that size.  Up to 512 keys a split is two 64-key blocks (more CTAs for a
// short, latency-bound job); longer prefixes take four blocks per split,
// which halves the partial states the cluster exchanges and merges.
__host__ __device__ __forceinline__ int keys_per_split(int P) { return P <= 512 ? 128 : 256; }
// K/V stages of the mma.sync prefix kernel: every block of a split is in
// flight before the dependency wait.
__host__ __device__ __forceinline__ int mma_prefix_stages(int P) { return keys_per_split(P) / 64; }
__host__ __device__ __forceinline__ Splits fixed_splits(int P) {
  if (P <= 0) return {0, 0};
  const int kps = keys_per_split(P);
  int S = (P + kps - 1) / kps;
  S = S < 1 ? 1 : (S > kMaxSplits ? kMaxSplits : S);
  const int len = (((P + S - 1) / S) + kKB - 1) / kKB * kKB;
  return {(P + len - 1) / len, len};
}

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

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

using bf16 = __nv_bfloat16;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v2(uint32_t addr, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float x) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(x) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Scores of this warp's 16 query rows against KB keys in smem (rows = keys).
template <int HD, int KB>
__device__ __forceinline__ void qk_scores(float (&sc)[KB / 8][4], const uint32_t (&qf)[HD / 16][4], const bf16* K,
                                          int lane) {
  constexpr int LD = HD + 8;
#pragma unroll
  for (int nt = 0; nt < KB / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  const int j = lane >> 3;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
    for (int n2 = 0; n2 < KB / 16; ++n2) {
      uint32_t kf[4];
      ldsm_x4(kf, K + (n2 * 16 + (j >> 1) * 8 + (lane & 7)) * LD + kk * 16 + (j & 1) * 8);
      mma16816(sc[2 * n2], qf[kk], kf[0], kf[1]);
      mma16816(sc[2 * n2 + 1], qf[kk], kf[2], kf[3]);
    }
  }
}

// o += P V for this warp's 16 rows; P in the score accumulators (bf16-rounded).
template <int HD, int KB>
__device__ __forceinline__ void pv_accum(float (&o)[HD / 8][4], const float (&p)[KB / 8][4], const bf16* V,
                                         int lane) {
  constexpr int LD = HD + 8;
  const int j = lane >> 3;
#pragma unroll
  for (int kt = 0; kt < KB / 16; ++kt) {
    uint32_t pa[4] = {pack_bf16(p[2 * kt][0], p[2 * kt][1]), pack_bf16(p[2 * kt][2], p[2 * kt][3]),
                      pack_bf16(p[2 * kt + 1][0], p[2 * kt + 1][1]), pack_bf16(p[2 * kt + 1][2], p[2 * kt + 1][3])};
#pragma unroll
    for (int d2 = 0; d2 < HD / 16; ++d2) {
      uint32_t vf[4];
      ldsm_x4_t(vf, V + (kt * 16 + (j & 1) * 8 + (lane & 7)) * LD + d2 * 16 + (j >> 1) * 8);
      mma16816(o[2 * d2], pa, vf[0], vf[1]);
      mma16816(o[2 * d2 + 1], pa, vf[2], vf[3]);
    }
  }
}

// The same two products with K and V tiles written by TMA: per 64-dim half a
// [64 keys][128 bytes] tile with 128-byte swizzling (16-byte chunk c of key
// row k stored at chunk c ^ (k & 7)).
__device__ __forceinline__ const unsigned char* sw_addr(const unsigned char* tile, int row, int chunk) {
  return tile + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <int HD>
__device__ __forceinline__ void qk_scores_sw(float (&sc)[kKB / 8][4], const uint32_t (&qf)[HD / 16][4],
                                             const unsigned char* K, int lane) {
#pragma unroll
  for (int nt = 0; nt < kKB / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  const int j = lane >> 3;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const unsigned char* tile = K + (kk >> 2) * (kKB * 128);
#pragma unroll
    for (int n2 = 0; n2 < kKB / 16; ++n2) {
      uint32_t kf[4];
      ldsm_x4(kf, sw_addr(tile, n2 * 16 + (j >> 1) * 8 + (lane & 7), (kk & 3) * 2 + (j & 1)));
      mma16816(sc[2 * n2], qf[kk], kf[0], kf[1]);
      mma16816(sc[2 * n2 + 1], qf[kk], kf[2], kf[3]);
    }
  }
}

template <int HD>
__device__ __forceinline__ void pv_accum_sw(float (&o)[HD / 8][4], const float (&p)[kKB / 8][4],
                                            const unsigned char* V, int lane) {
  const int j = lane >> 3;
#pragma unroll
  for (int kt = 0; kt < kKB / 16; ++kt) {
    uint32_t pa[4] = {pack_bf16(p[2 * kt][0], p[2 * kt][1]), pack_bf16(p[2 * kt][2], p[2 * kt][3]),
                      pack_bf16(p[2 * kt + 1][0], p[2 * kt + 1][1]), pack_bf16(p[2 * kt + 1][2], p[2 * kt + 1][3])};
#pragma unroll
    for (int d2 = 0; d2 < HD / 16; ++d2) {
      uint32_t vf[4];
      ldsm_x4_t(vf, sw_addr(V + (d2 >> 2) * (kKB * 128), kt * 16 + (j & 1) * 8 + (lane & 7), (d2 & 3) * 2 + (j >> 1)));
      mma16816(o[2 * d2], pa, vf[0], vf[1]);
      mma16816(o[2 * d2 + 1], pa, vf[2], vf[3]);
    }
  }
}

template <int HD>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[HD / 16][4], const bf16* Q, int warp, int lane) {
  constexpr int LD = HD + 8;
  const int j = lane >> 3;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk)
    ldsm_x4(qf[kk], Q + (warp * 16 + (j & 1) * 8 + (lane & 7)) * LD + kk * 16 + (j >> 1) * 8);
}

// Prefix partials: CTA = (64 query vectors of one request and KV head, one
// split of the prefix).  Query vector v of the request is recompute slot
// off_r + v / G, query head kvh * G + v % G.  K/V blocks of 64 keys stream
// through a STAGES-deep ring of TMA loads (one (64-dim, 1-head, 64-key) box
// per 64-dim half); the split CTAs of a query tile form one cluster (along z):
// after their streaming loops every CTA sends its partial state (max,
// denominator, unnormalised output) of each query row to the CTA that owns
// the row, and each owner merges the S states in rank order and writes one
// merged state per query.
template <int HD, int STAGES>
constexpr int prefix_smem_bytes() {
  return STAGES * 2 * (HD / 64) * (kKB * 128) + kQT * (HD + 8) * 2 + 64 + 1024;
}

template <int HD, int STAGES>
__global__ void __launch_bounds__(128) attn_prefix_mma(const __grid_constant__ CUtensorMap tmK,
                                                       const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  constexpr int LD = HD + 8;
  constexpr int XLD = HD + 2;  // exchange row: o[HD], m, l
  constexpr int KTILE = kKB * 128;
  constexpr int STAGE = 2 * (HD / 64) * KTILE;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  bf16* sQ = reinterpret_cast<bf16*>(base + STAGES * STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + STAGES * STAGE + kQT * LD * 2);
  float* xbuf = reinterpret_cast<float*>(base);  // exchange area, reused after the loop
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid: x = (request, KV head), y = query tile, z = split; the first query
  // tiles of every (request, KV head) are dispatched first, and the tiles that
  // only a larger recompute set would fill come last
  const int r = blockIdx.x / a.nkv, kvh = blockIdx.x % a.nkv;
  const Splits sp = fixed_splits(a.P);
  const int G = a.nq / a.nkv;
  // Every kernel of the pass lets its dependants start only after its own
  // dependency wait, so the kernels before the previous one have completed
  // when this grid starts: the recompute offsets (gate kernel) can be read
  // before the wait, past L1.  Only the queries (previous kernel) wait.
  const int off_r = __ldcg(a.meta + 1 + r), nqv = (__ldcg(a.meta + 2 + r) - off_r) * G;
  const int q0 = blockIdx.y * kQT;
  // An empty tile leaves without the dependency wait: it reads nothing of the
  // previous kernel, and the live tiles (the main branch always recomputes,
  // so there is one per request and KV head) still hold the next kernel back
  // until they have waited.  Uniform over the cluster.
  if (q0 >= nqv) return;
  const int s = sp.S > 1 ? (int)cluster_rank() : 0;
  const int k_lo = s * sp.len, k_hi = min(a.P, k_lo + sp.len);
  const int nblk = k_hi > k_lo ? (k_hi - k_lo + kKB - 1) / kKB : 0;
  const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);

  if (tid == 0) {
    for (int st = 0; st < STAGES; ++st) tc::mbar_init(&full[st], 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int b) {  // thread 0: K and V of key block b into its stage
    const int st = b % STAGES;
    unsigned char* sk = base + st * STAGE;
    const int z = r * a.P + k_lo + b * kKB;
    tc::mbar_expect_tx(&full[st], STAGE);
#pragma unroll
    for (int h = 0; h < HD / 64; ++h) {
      tc::tma_load_3d(sk + h * KTILE, &tmK, h * 64, kvh, z, &full[st]);
      tc::tma_load_3d(sk + (HD / 64 + h) * KTILE, &tmV, h * 64, kvh, z, &full[st]);
    }
  };
  // the prefix keys and values are inputs of the pass: every stage is filled
  // before the wait (with P <= 1024 that is the whole split)
  if (tid == 0)
    for (int b = 0; b < min(STAGES, nblk); ++b) issue(b);
  pdl_wait();
  pdl_trigger();

  for (int idx = tid; idx < kQT * (HD / 8); idx += 128) {
    const int row = idx / (HD / 8), c8 = idx % (HD / 8), v = q0 + row;
    const bool ok = v < nqv;
    const int g = off_r + (ok ? v / G : 0), h = kvh * G + (ok ? v % G : 0);
    cp_async16(sQ + row * LD + c8 * 8, qkv + (size_t)g * a.ld_qkv + h * HD + c8 * 8, ok);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  uint32_t qf[HD / 16][4];
  load_q_frags<HD>(qf, sQ, warp, lane);

  float o[HD / 8][4];
#pragma unroll
  for (int nt = 0; nt < HD / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  for (int b = 0; b < nblk; ++b) {
    // block b + STAGES - 1 goes to the stage the last barrier freed (the
    // first STAGES blocks were issued before the wait)
    if (tid == 0 && b >= 1 && b + STAGES - 1 < nblk) issue(b + STAGES - 1);
    // a wait that gives up raises the error word but does not leave the loop,
    // so every warp keeps reaching the same barriers
    tc::mbar_wait(&full[b % STAGES], (b / STAGES) & 1, a.err);
    const unsigned char* sk = base + (b % STAGES) * STAGE;
    float sc[kKB / 8][4];
    qk_scores_sw<HD>(sc, qf, sk, lane);
    const int kb0 = k_lo + b * kKB;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kKB / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kb0 + nt * 8 + (lane & 3) * 2 + (e & 1);
        sc[nt][e] = key < k_hi ? sc[nt][e] * a.scale_log2 : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
    const float n0 = fmaxf(m0, quad_max(mx0)), n1 = fmaxf(m1, quad_max(mx1));
    const float c0 = exp2f(m0 - n0), c1 = exp2f(m1 - n1);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < kKB / 8; ++nt) {
      sc[nt][0] = exp2f(sc[nt][0] - n0);
      sc[nt][1] = exp2f(sc[nt][1] - n0);
      sc[nt][2] = exp2f(sc[nt][2] - n1);
      sc[nt][3] = exp2f(sc[nt][3] - n1);
      s0 += sc[nt][0] + sc[nt][1];
      s1 += sc[nt][2] + sc[nt][3];
    }
    l0 = l0 * c0 + s0;
    l1 = l1 * c1 + s1;
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int nt = 0; nt < HD / 8; ++nt) {
      o[nt][0] *= c0;
      o[nt][1] *= c0;
      o[nt][2] *= c1;
      o[nt][3] *= c1;
    }
    pv_accum_sw<HD>(o, sc, sk + (HD / 64) * KTILE, lane);
    __syncthreads();
  }
  l0 = quad_sum(l0);
  l1 = quad_sum(l1);

  if (sp.S == 1) {  // a single split: the partial is already the merged state
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int v = q0 + warp * 16 + (lane >> 2) + half * 8;
      if (v >= nqv) continue;
      const size_t qi = (size_t)(off_r + v / G) * a.nq + kvh * G + v % G;
      float* po = a.part_o + qi * HD + (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < HD / 8; ++nt)
        *reinterpret_cast<float2*>(po + nt * 8) = make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
      if ((lane & 3) == 0) {
        a.part_ml[qi * 2 + 0] = half ? m1 : m0;
        a.part_ml[qi * 2 + 1] = half ? l1 : l0;
      }
    }
    return;
  }
  // rows [rank * per, (rank + 1) * per) of the tile are merged by `rank`
  const int per = (kQT + sp.S - 1) / sp.S;
  cluster_sync_all();  // every CTA is past its loop: exchange areas are free
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int vr = warp * 16 + (lane >> 2) + half * 8;  // row within the tile
    const int owner = vr / per;
    const uint32_t dst = map_rank(smem_addr(xbuf + ((size_t)s * per + (vr - owner * per)) * XLD), (uint32_t)owner);
#pragma unroll
    for (int nt = 0; nt < HD / 8; ++nt)
      st_cluster_v2(dst + (nt * 8 + (lane & 3) * 2) * 4, o[nt][2 * half], o[nt][2 * half + 1]);
    if ((lane & 3) == 0) {
      st_cluster_f32(dst + HD * 4, half ? m1 : m0);
      st_cluster_f32(dst + (HD + 1) * 4, half ? l1 : l0);
    }
  }
  cluster_sync_all();  // every partial has arrived
  // one warp per merged row: the split weights are formed once per row, each
  // lane combines features lane + 32c
  const int rows = min(per, kQT - s * per);
  for (int rl = warp; rl < rows; rl += 4) {
    const int v = q0 + s * per + rl;
    if (v >= nqv) break;
    float mt[kMaxSplits], w[kMaxSplits];
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < kMaxSplits; ++t) {
      mt[t] = t < sp.S ? xbuf[((size_t)t * per + rl) * XLD + HD] : -INFINITY;
      M = fmaxf(M, mt[t]);
    }
    float l = 0.f;
#pragma unroll
    for (int t = 0; t < kMaxSplits; ++t) {
      w[t] = t < sp.S ? exp2f(mt[t] - M) : 0.f;
      if (t < sp.S) l += w[t] * xbuf[((size_t)t * per + rl) * XLD + HD + 1];
    }
    const size_t qi = (size_t)(off_r + v / G) * a.nq + kvh * G + v % G;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      const int dd = lane + 32 * c;
      float acc = 0.f;
#pragma unroll
      for (int t = 0; t < kMaxSplits; ++t)
        if (t < sp.S) acc += w[t] * xbuf[((size_t)t * per + rl) * XLD + dd];
      a.part_o[qi * HD + dd] = acc;
    }
    if (lane == 0) {
      a.part_ml[qi * 2 + 0] = M;
      a.part_ml[qi * 2 + 1] = l;
    }
  }
}

// ------------------------------------------------------------ tcgen05 prefix path
//
// Prefix partials on the 5th-generation tensor cores: CTA = (128 query vectors
// of one request and KV head = the 128 TMEM lanes, one split of the prefix).
// Per block of 64 keys:
//   S = Q K^T       tcgen05.mma, Q and K K-major in shared memory, S in TMEM
//                   (three buffers: the scores two blocks ahead are computed
//                   while this block's softmax runs);
//   P = exp2(S - m) by the softmax warps, one query row per thread, written as
//                   bf16 to shared memory (K-major, 128-byte swizzle);
//   O += P V        tcgen05.mma, V MN-major as the TMA box leaves it, O in TMEM.
// The running max m of a row only moves when a block's max exceeds it by more
// than 2^8, and O is then rescaled in TMEM; the partial state (m, l, O) stays
// exact because m is whatever reference the exponentials used.
// Warp 0 streams K and V through two kTcStages-deep rings of TMA loads (lane 0
// the keys, freed once their scores are computed; lane 1 the values, freed
// once P V is done), warp 1 owns TMEM and issues the MMAs, warps 2-9 load Q and
// run the softmax and the epilogue: the two warps on the same 32 TMEM lanes
// take half of each row's 64 scores and half of its output columns, and
// exchange only the row's block maximum.
// The split CTAs of a tile form a cluster and merge as the CUDA-core path does.
constexpr int kTcQ = 128;
constexpr int kTcStages = 4;
constexpr int kTcThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 softmax (two per row group)
constexpr int kTcMinKeysPerSplit = 512;
constexpr int kTcMaxSplits = 4;
// Prefixes of at least this many keys take the tcgen05 kernel.
constexpr int kTcMinPrefix = 1;
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

template <int HD>
struct TcLayout {
  static constexpr int QH = HD / 64;                    // 64-dim halves
  static constexpr int HALF = kTcQ * 128;               // one 64-dim half of Q: 128 rows x 128 B
  static constexpr int KV_TILE = kKB * 128;             // one 64-dim half of a K or V block
  static constexpr int STAGE = QH * KV_TILE;            // K (or V) of one block
  static constexpr int P_TILE = kTcQ * 128;             // P: 128 rows x 64 keys (bf16)
  static constexpr int OFF_K = QH * HALF;
  static constexpr int OFF_V = OFF_K + kTcStages * STAGE;
  static constexpr int OFF_P = OFF_V + kTcStages * STAGE;
  static constexpr int OFF_BAR = OFF_P + 2 * P_TILE;
  static constexpr int BYTES = OFF_BAR + 256 + 1024;   // + alignment of the dynamic window
  static constexpr int XLD = HD + 4;                    // merge exchange row: o[HD], m, l (16-byte rows)
  static constexpr int SBUF = 3;                        // score buffers: columns [64 s, 64 s + 64)
  static constexpr int O_COL = 256;                     // O: columns [256, 256 + HD)
  static constexpr int TMEM_COLS = 512;
  static_assert((kTcQ + kMaxSplits - 1) * XLD * 4 <= OFF_P, "merge exchange area");
};

__device__ __forceinline__ void tmem_ld32_raw(uint32_t taddr, float (&v)[32]) { tc::tmem_ld32(taddr, v); }

// 2^x on the special-function unit (flushes subnormal results to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int HD>
__global__ void __launch_bounds__(kTcThreads, 1) attn_prefix_tc(const __grid_constant__ CUtensorMap tmK,
                                                                const __grid_constant__ CUtensorMap tmV,
                                                                const AttnArgs a) {
  using Lay = TcLayout<HD>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* sQ = base;
  unsigned char* sK = base + Lay::OFF_K;
  unsigned char* sV = base + Lay::OFF_V;
  unsigned char* sP = base + Lay::OFF_P;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + Lay::OFF_BAR);
  uint64_t* kfull = bar;                   // [kTcStages] K landed
  uint64_t* vfull = bar + kTcStages;       // [kTcStages] V landed
  uint64_t* kempty = bar + 2 * kTcStages;  // [kTcStages] K consumed by S = Q K^T
  uint64_t* vempty = bar + 3 * kTcStages;  // [kTcStages] V consumed by O += P V
  uint64_t* sfull = bar + 4 * kTcStages;   // [SBUF] scores in TMEM
  uint64_t* sempty = sfull + Lay::SBUF;    // [SBUF] scores read
  uint64_t* pfull = sempty + Lay::SBUF;    // [2] P written
  uint64_t* pvdone = pfull + 2;            // [2] P V of that buffer done
  uint64_t* qready = pvdone + 2;
  uint64_t* ofull = qready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ofull + 1);
  float* xbuf = reinterpret_cast<float*>(base);  // merge exchange, over Q and the ring once they are dead
  __shared__ float xmax[2][2][kTcQ];             // [block parity][half][row]: partial block maxima

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid: x = (request, KV head), y = query tile, z = split; the first query
  // tiles of every (request, KV head) are dispatched first, and the tiles that
  // only a larger recompute set would fill come last
  const int r = blockIdx.x / a.nkv, kvh = blockIdx.x % a.nkv;
  const Splits sp = tc_split_len(a.P, (int)gridDim.z);
  const int G = a.nq / a.nkv;
  // recompute offsets from the gate kernel (complete once this grid runs), past L1
  const int off_r = __ldcg(a.meta + 1 + r), nqv = (__ldcg(a.meta + 2 + r) - off_r) * G;
  const int q0 = blockIdx.y * kTcQ;
  // An empty tile leaves without the dependency wait: it reads nothing of the
  // previous kernel, and the live tiles (the main branch always recomputes,
  // so there is one per request and KV head) still hold the next kernel back
  // until they have waited.  Uniform over the cluster.
  if (q0 >= nqv) return;
  const int s = sp.S > 1 ? (int)tc::cluster_ctarank() : 0;
  const int k_lo = s * sp.len, k_hi = min(a.P, k_lo + sp.len);
  const int nblk = (k_hi - k_lo + kKB - 1) / kKB;

  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
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

  // warp 0: lane 0 loads key block b into K stage b % kTcStages, lane 1 the
  // value block into the V ring
  auto issue = [&](int b, bool keys) {
    const int st = b % kTcStages;
    unsigned char* dst = (keys ? sK : sV) + st * Lay::STAGE;
    uint64_t* full = keys ? &kfull[st] : &vfull[st];
    const int z = r * a.P + k_lo + b * kKB;
    tc::mbar_expect_tx(full, Lay::QH * Lay::KV_TILE);
#pragma unroll
    for (int h = 0; h < Lay::QH; ++h) tc::tma_load_3d(dst + h * Lay::KV_TILE, keys ? &tmK : &tmV, h * 64, kvh, z, full);
  };
  // the prefix keys and values are inputs of the pass
  if (warp == 0 && lane < 2)
    for (int b = 0; b < min(kTcStages, nblk); ++b) issue(b, lane == 0);
  pdl_wait();
  pdl_trigger();

  const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);
  if (warp == 0) {
    if (lane < 2) {
      const bool keys = lane == 0;
      for (int b = kTcStages; b < nblk; ++b) {
        // the stage is free once the MMA that read block b - kTcStages has completed
        tc::mbar_wait(keys ? &kempty[b % kTcStages] : &vempty[b % kTcStages], ((b / kTcStages) - 1) & 1, a.err);
        issue(b, keys);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(kTcQ, kKB);
      const uint32_t idesc_pv = tc::idesc_bf16_f32(kTcQ, HD) | (1u << 16);  // V is MN-major
      tc::mbar_wait(qready, 0, a.err);
      auto issue_s = [&](int b) {  // S(b) = Q K(b)^T into score buffer b % SBUF
        const int st = b % kTcStages, sb = b % Lay::SBUF;
        tc::mbar_wait(&kfull[st], (b / kTcStages) & 1, a.err);
        if (b >= Lay::SBUF) tc::mbar_wait(&sempty[sb], ((b / Lay::SBUF) - 1) & 1, a.err);
        tc::fence_after_sync();
        const unsigned char* sk = sK + st * Lay::STAGE;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t dq = tc::sw128_kmajor_desc(smem_addr(sQ + (kk >> 2) * Lay::HALF + (kk & 3) * 32));
          const uint64_t dk = tc::sw128_kmajor_desc(smem_addr(sk + (kk >> 2) * Lay::KV_TILE + (kk & 3) * 32));
          tc::mma_bf16(tmem + sb * kKB, dq, dk, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sfull[sb]);
        tc::mma_commit(&kempty[st]);
      };
      for (int b = 0; b < min(Lay::SBUF - 1, nblk); ++b) issue_s(b);
      for (int j = 0; j < nblk; ++j) {
        // the scores SBUF - 1 blocks ahead, as soon as their buffer is read
        if (j + Lay::SBUF - 1 < nblk) issue_s(j + Lay::SBUF - 1);
        // O += P(j) V(j)
        const int st = j % kTcStages, pb = j & 1;
        tc::mbar_wait(&pfull[pb], (j >> 1) & 1, a.err);
        tc::mbar_wait(&vfull[st], (j / kTcStages) & 1, a.err);
        tc::fence_after_sync();
        const unsigned char* sv = sV + st * Lay::STAGE;
#pragma unroll
        for (int kk = 0; kk < kKB / 16; ++kk) {
          const uint64_t dp = tc::sw128_kmajor_desc(smem_addr(sP + pb * Lay::P_TILE + kk * 32));
          const uint64_t dv = tc::sw128_mnmajor_desc(smem_addr(sv + kk * 2048), Lay::KV_TILE);
          tc::mma_bf16(tmem + Lay::O_COL, dp, dv, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&pvdone[pb]);
        tc::mma_commit(&vempty[st]);
      }
      tc::mma_commit(ofull);
    }
    __syncwarp();
  } else {
    // softmax warps: TMEM lanes 32 * (warp % 4) .. + 31, one query row per
    // thread pair; `half` selects 32 of the row's 64 scores and HD / 2 of its
    // output columns
    const int grp = warp & 3, half = (warp - 2) >> 2;
    const int row = 32 * grp + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * grp) << 16);
    const int v = q0 + row;
    {
      const bool ok = v < nqv;
      const int g = off_r + (ok ? v / G : 0), h = kvh * G + (ok ? v % G : 0);
      const bf16* src = qkv + (size_t)g * a.ld_qkv + h * HD;
#pragma unroll
      for (int c = half * (HD / 16); c < (half + 1) * (HD / 16); ++c)
        cp_async16(sQ + (c >> 3) * Lay::HALF + row * 128 + (((c & 7) ^ (row & 7)) << 4), src + c * 8, ok);
      cp_async_commit();
      cp_async_wait<0>();
      tc::fence_proxy_async_smem();
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
      const int kb0 = k_lo + b * kKB + 32 * half;
      if (kb0 + 32 > k_hi) {  // the split's last block may be ragged
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (kb0 + k >= k_hi) sc[k] = -INFINITY;
      }
      float mx = sc[0];
#pragma unroll
      for (int k = 1; k < 32; ++k) mx = fmaxf(mx, sc[k]);
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
      float ls = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float p0 = ex2_approx(fmaf(sc[k], scale, mneg)), p1 = ex2_approx(fmaf(sc[k + 1], scale, mneg));
        ls += p0 + p1;
        pk[k / 2] = pack_bf16(p0, p1);
      }
      l += ls;
      // P buffer b % 2 is free once P V of block b - 2 is done
      if (b >= 2) tc::mbar_wait(&pvdone[pbuf], ((b - 2) >> 1) & 1, a.err);
      unsigned char* prow = sP + pbuf * Lay::P_TILE + row * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(prow + (((4 * half + c) ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      tc::fence_proxy_async_smem();
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
    constexpr int HO = HD / 2;
    float o[HO];
#pragma unroll
    for (int c0 = 0; c0 < HO; c0 += 32)
      tmem_ld32_raw(tl + Lay::O_COL + half * HO + c0, *reinterpret_cast<float(*)[32]>(o + c0));
    if (sp.S == 1) {  // a single split: the partial is already the merged state
      if (v < nqv) {
        const size_t qi = (size_t)(off_r + v / G) * a.nq + kvh * G + v % G;
        float* po = a.part_o + qi * HD + half * HO;
#pragma unroll
        for (int c = 0; c < HO; c += 4) *reinterpret_cast<float4*>(po + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
        if (half == 0) {
          a.part_ml[qi * 2 + 0] = mrow;
          a.part_ml[qi * 2 + 1] = lrow;
        }
      }
    } else {
      // rows [rank * per, (rank + 1) * per) of the tile are merged by `rank`
      const int per = (kTcQ + sp.S - 1) / sp.S;
      // (the exchange area covers Q and the ring: wait until every split is past its loop)
      asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
      const int owner = row / per;
      const uint32_t dst =
          tc::map_to_rank(smem_addr(xbuf + ((size_t)s * per + (row - owner * per)) * Lay::XLD), (uint32_t)owner);
#pragma unroll
      for (int c = 0; c < HO; c += 4)
        asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + (half * HO + c) * 4), "f"(o[c]),
                     "f"(o[c + 1]), "f"(o[c + 2]), "f"(o[c + 3])
                     : "memory");
      if (half == 0)
        asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(dst + HD * 4), "f"(mrow), "f"(lrow) : "memory");
    }
  }
  if (sp.S > 1) {
    if (warp < 2)  // the producer and MMA warps take part in the cluster barriers too
      asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    // merge: one warp per row (all warps), split weights formed once per row
    const int rows = min((kTcQ + sp.S - 1) / sp.S, kTcQ - s * ((kTcQ + sp.S - 1) / sp.S));
    const int per = (kTcQ + sp.S - 1) / sp.S;
    for (int rl = warp; rl < rows; rl += kTcThreads / 32) {
      const int v = q0 + s * per + rl;
      if (v >= nqv) break;
      float mt[kMaxSplits], w[kMaxSplits];
      float M = -INFINITY;
#pragma unroll
      for (int t = 0; t < kMaxSplits; ++t) {
        mt[t] = t < sp.S ? xbuf[((size_t)t * per + rl) * Lay::XLD + HD] : -INFINITY;
        M = fmaxf(M, mt[t]);
      }
      float lsum = 0.f;
#pragma unroll
      for (int t = 0; t < kMaxSplits; ++t) {
        w[t] = t < sp.S ? exp2f(mt[t] - M) : 0.f;
        if (t < sp.S) lsum += w[t] * xbuf[((size_t)t * per + rl) * Lay::XLD + HD + 1];
      }
      const size_t qi = (size_t)(off_r + v / G) * a.nq + kvh * G + v % G;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        const int dd = lane + 32 * c;
        float acc = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxSplits; ++t)
          if (t < sp.S) acc += w[t] * xbuf[((size_t)t * per + rl) * Lay::XLD + dd];
        a.part_o[qi * HD + dd] = acc;
      }
      if (lane == 0) {
        a.part_ml[qi * 2 + 0] = M;
        a.part_ml[qi * 2 + 1] = lsum;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Lay::TMEM_COLS);
  }
}

// Block attention + merge: CTA = (32 query vectors of one branch and KV head,
// two warps).  Query vector v is block position n = v / G with query head
// kvh * G + v % G; its query is the one of the row's resolved source; its
// block keys/values are the branch's own table K_i[m] = QKV[rcslot(i, m)].
constexpr int kBQT = 32;

template <int HD, int KB>
__global__ void __launch_bounds__(64) attn_block_mma(const AttnArgs a) {
  constexpr int LD = HD + 8;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int slot[KB];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + kBQT * LD;
  bf16* sV = sK + KB * LD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.y / a.nkv, kvh = blockIdx.y % a.nkv;  // rb = r * Bp + i
  const int G = a.nq / a.nkv, L = a.L;
  const int q0 = blockIdx.x * kBQT, nqv = L * G;
  if (q0 >= nqv) {
    pdl_wait();
    return;
  }
  // Every kernel of the pass lets its dependants start only after its own
  // dependency wait, so the kernels before the previous one have completed
  // when this grid starts: the source slots (gate kernel) are read before the
  // wait, past L1, and so are the projected rows when the prefix kernel sits
  // between the projection and this one.
  const int count = __ldcg(a.meta);
  const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);
  const int koff = (a.nq + kvh) * HD, voff = (a.nq + a.nkv + kvh) * HD;
  for (int m = tid; m < KB; m += 64) {
    int g = m < L ? __ldcg(a.rcslot + rb * L + m) : 0;
    if (g < 0 || g >= count) {
      raise_error(a.err, kErrAttn);
      g = 0;
    }
    slot[m] = g;
  }
  __syncthreads();
  auto load_rows = [&] {
    for (int idx = tid; idx < kBQT * (HD / 8); idx += 64) {
      const int row = idx / (HD / 8), c8 = idx % (HD / 8), v = q0 + row;
      const bool ok = v < nqv;
      cp_async16(sQ + row * LD + c8 * 8,
                 qkv + (size_t)slot[ok ? v / G : 0] * a.ld_qkv + (kvh * G + (ok ? v % G : 0)) * HD + c8 * 8, ok);
    }
    for (int idx = tid; idx < KB * (HD / 8); idx += 64) {
      const int m = idx / (HD / 8), c8 = idx % (HD / 8);
      const bf16* src = qkv + (size_t)slot[m] * a.ld_qkv;
      cp_async16(sK + m * LD + c8 * 8, src + koff + c8 * 8, m < L);
      cp_async16(sV + m * LD + c8 * 8, src + voff + c8 * 8, m < L);
    }
    cp_async_commit();
  };
  if (a.P > 0) load_rows();
  pdl_wait();
  pdl_trigger();
  if (a.P == 0) load_rows();
  // the merged prefix state of this thread's two query vectors (previous
  // kernel), needed only after the block part: loaded into registers while it
  // runs
  float mp[2] = {0.f, 0.f}, lp[2] = {0.f, 0.f};
  float2 pp[2][HD / 8];
  if (a.P > 0) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int v = q0 + warp * 16 + (lane >> 2) + half * 8;
      const size_t qi = v < nqv ? (size_t)slot[v / G] * a.nq + kvh * G + v % G : (size_t)slot[0] * a.nq + kvh * G;
      const float* po = a.part_o + qi * HD + (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < HD / 8; ++nt) pp[half][nt] = *reinterpret_cast<const float2*>(po + nt * 8);
      mp[half] = a.part_ml[qi * 2];
      lp[half] = a.part_ml[qi * 2 + 1];
    }
  }
  cp_async_wait<0>();  // the projected rows have landed
  __syncthreads();
  uint32_t qf[HD / 16][4];
  load_q_frags<HD>(qf, sQ, warp, lane);
  float sc[KB / 8][4];
  qk_scores<HD, KB>(sc, qf, sK, lane);
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < KB / 8; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = nt * 8 + (lane & 3) * 2 + (e & 1);
      sc[nt][e] = m < L ? sc[nt][e] * a.scale_log2 : -INFINITY;
    }
    mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
    mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
  }
  const float mb0 = quad_max(mx0), mb1 = quad_max(mx1);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < KB / 8; ++nt) {
    sc[nt][0] = exp2f(sc[nt][0] - mb0);
    sc[nt][1] = exp2f(sc[nt][1] - mb0);
    sc[nt][2] = exp2f(sc[nt][2] - mb1);
    sc[nt][3] = exp2f(sc[nt][3] - mb1);
    s0 += sc[nt][0] + sc[nt][1];
    s1 += sc[nt][2] + sc[nt][3];
  }
  const float lb0 = quad_sum(s0), lb1 = quad_sum(s1);
  float o[HD / 8][4];
#pragma unroll
  for (int nt = 0; nt < HD / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  pv_accum<HD, KB>(o, sc, sV, lane);

  bf16* out = reinterpret_cast<bf16*>(a.attn);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int v = q0 + warp * 16 + (lane >> 2) + half * 8;
    if (v >= nqv) continue;
    const int row = rb * L + v / G, h = kvh * G + v % G;
    const float mb = half ? mb1 : mb0, lb = half ? lb1 : lb0;
    float acc[HD / 8][2];
    float l, wb;
    if (a.P > 0) {
      // merge with the prefix state of this query (one per recompute slot and head)
      const float M = fmaxf(mb, mp[half]);
      wb = exp2f(mb - M);
      const float wp = exp2f(mp[half] - M);
      l = lb * wb + lp[half] * wp;
#pragma unroll
      for (int nt = 0; nt < HD / 8; ++nt) {
        acc[nt][0] = o[nt][2 * half] * wb + wp * pp[half][nt].x;
        acc[nt][1] = o[nt][2 * half + 1] * wb + wp * pp[half][nt].y;
      }
    } else {
      l = lb;
#pragma unroll
      for (int nt = 0; nt < HD / 8; ++nt) {
        acc[nt][0] = o[nt][2 * half];
        acc[nt][1] = o[nt][2 * half + 1];
      }
    }
    const float inv = 1.f / l;
    bf16* dst = out + (size_t)row * a.ld_attn + h * HD + (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < HD / 8; ++nt)
      *reinterpret_cast<__nv_bfloat162*>(dst + nt * 8) = __floats2bfloat162_rn(acc[nt][0] * inv, acc[nt][1] * inv);
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
  if (a.P > 0) {
    pdl_wait();
    pdl_trigger();
  }
  // the prefix state of this thread's query (previous kernel)
  size_t qi = 0;
  float mp = 0.f, lp = 0.f;
  if (live) qi = (size_t)slot[vn] * a.nq + kvh * G + v % G;
  if (a.P > 0 && live) {
    mp = a.part_ml[qi * 2];
    lp = a.part_ml[qi * 2 + 1];
  }
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
  // merge weights of the block part and the prefix partial
  float wb = 1.f, wp = 0.f, l = lb;
  if (a.P > 0) {
    const float M = fmaxf(mb, mp);
    wb = exp2f(mb - M);
    wp = exp2f(mp - M);
    l = lb * wb + lp * wp;
  }
  const float inv = 1.f / l;
  tc::mbar_wait(&bar[1], 0, a.err);
  tc::fence_after_sync();
  bf16* dst = reinterpret_cast<bf16*>(a.attn) + (size_t)(rb * L + vn) * a.ld_attn + (kvh * G + (live ? v % G : 0)) * HD;
  float* po = a.part_o + qi * HD;
  // correction mode: the row's merged state (max in log2 units, denominator,
  // unnormalised output) replaces its prefix partial for the correction kernel
  if (correct && live) {
    a.part_ml[qi * 2] = a.P > 0 ? fmaxf(mb, mp) : mb;
    a.part_ml[qi * 2 + 1] = l;
  }
#pragma unroll
  for (int c0 = 0; c0 < HD; c0 += 32) {
    float o[32];
    tc::tmem_ld32(tl + c0, o);
    if (live) {
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = o[c + e] * wb;
        if (a.P > 0) {
          const float4 p0 = *reinterpret_cast<const float4*>(po + c0 + c);
          const float4 p1 = *reinterpret_cast<const float4*>(po + c0 + c + 4);
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
cudaError_t attention_mma(Launch& lc, const AttnArgs& a) {
  constexpr int LD = HD + 8;
  const int G = a.nq / a.nkv;
  // block keys per CTA tile: 32 when the block length allows, else 64
  const int kb = a.L <= 32 ? 32 : kKB;
  const size_t smem_b = (size_t)(kBQT + 2 * kb) * LD * sizeof(bf16);
  static cudaError_t attr = [&] {
    cudaError_t e = cudaFuncSetAttribute(attn_prefix_tc<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcLayout<HD>::BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_prefix_mma<HD, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               prefix_smem_bytes<HD, 2>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_prefix_mma<HD, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               prefix_smem_bytes<HD, 4>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_block_tc<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, BlkLayout<HD>::bytes(64));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_block_mma<HD, kKB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)((kBQT + 2 * kKB) * LD * sizeof(bf16)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_block_mma<HD, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)((kBQT + 2 * 32) * LD * sizeof(bf16)));
    return e;
  }();
  if (attr != cudaSuccess) return lc.err = attr;
  if (a.P > 0) {
    alignas(64) CUtensorMap tmK, tmV;
    if (!make_tmap_kv(&tmK, a.pk, HD, a.nkv, (uint64_t)a.R * a.P) ||
        !make_tmap_kv(&tmV, a.pv, HD, a.nkv, (uint64_t)a.R * a.P))
      return lc.err = cudaErrorInvalidValue;
    // worst case: every row of a request recomputes
    lc.before(SF_K_ATTN_PREFIX);
    if (a.P >= kTcMinPrefix) {
      const Splits sp = tc_splits(a.P, a.R * a.nkv, a.target_ctas);
      dim3 grid(a.R * a.nkv, (a.Bp * a.L * G + kTcQ - 1) / kTcQ, sp.S);
      lc.check(launch_pdl(lc.st, grid, dim3(kTcThreads), (size_t)TcLayout<HD>::BYTES, sp.S, attn_prefix_tc<HD>,
                          tmK, tmV, a));
    } else {
      const Splits sp = fixed_splits(a.P);
      dim3 grid(a.R * a.nkv, (a.Bp * a.L * G + kQT - 1) / kQT, sp.S);
      if (mma_prefix_stages(a.P) == 2)
        lc.check(launch_pdl(lc.st, grid, dim3(128), (size_t)prefix_smem_bytes<HD, 2>(), sp.S, attn_prefix_mma<HD, 2>,
                            tmK, tmV, a));
      else
        lc.check(launch_pdl(lc.st, grid, dim3(128), (size_t)prefix_smem_bytes<HD, 4>(), sp.S, attn_prefix_mma<HD, 4>,
                            tmK, tmV, a));
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
  if (a.hd == 128) return attention_mma<128>(lc, a);
  if (a.hd == 64) return attention_mma<64>(lc, a);
  return cudaErrorInvalidValue;
}

}  // namespace sf
