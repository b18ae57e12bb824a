// tcgen05 / TMEM GEMM over the rows of the compacted recompute set (BF16).
//
// Y[g][o] = sum_k X[g][k] W[o][k] for g < count (count read on the device).
// The weight is the M operand: each CTA owns 128 output features (TMEM lanes)
// and up to 256 rows (TMEM columns), so a weight tile is streamed once for all
// rows of a layer; the rows are the N operand, loaded in 64-row TMA boxes only
// up to the live row count, and as many pipeline stages as the shared memory
// holds for that count.  Narrow GEMMs split K over the CTAs of a thread block
// cluster (along grid z); after the main loops every CTA pushes the partial
// accumulator of row j into the shared memory of cluster rank j % S, which
// finishes that row (distributed shared memory): each owner adds the partials
// in cluster-rank order before the epilogue, so the result does not depend on
// scheduling, no global workspace is used and the epilogue work is spread over
// every rank of the cluster.  The epilogue's own global reads (rotary table,
// residual rows) are issued while the main loop runs.
//
// Warp roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues the
// MMAs, warps 2-5 drain TMEM into the layer epilogue.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "sf_epilogue.cuh"
#include "sf_internal.h"
#include "sf_tc.cuh"
#include "specfold_kernels.h"

namespace sf {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = 256;
constexpr int RC = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_CHUNK = RC * BK * 2;
constexpr int THREADS = 192;
// The pipeline's shared memory holds a ring of weight (A) tiles growing up from
// its start and a ring of row (B) tiles growing down from its end; the number
// of stages follows from the live row count, so a small recompute set keeps
// up to MAX_STAGES weight tiles in flight.  Its size is a launch parameter:
// PIPE_BYTES gives one CTA per SM, PIPE_BYTES_PAIR two (for GEMMs with more
// tiles than SMs, which then run in one wave).  Weight tiles fetched before
// the row count is known go to the first slots of the A ring that even a full
// 256-row tile keeps.
constexpr int MAX_STAGES = 12;
constexpr int PIPE_BYTES = 216 * 1024;
constexpr int PIPE_BYTES_PAIR = 110 * 1024;
constexpr int SMEM_BYTES = PIPE_BYTES + 1024 + 256;
static_assert(2 * MAX_STAGES * 8 + 8 + 4 <= 256, "barrier area");

// Stages of a pipeline of `pipe` bytes for row tiles of n_chunks 64-row boxes
// (n_chunks <= 0: a full tile, the fewest stages).
__host__ __device__ constexpr int stages_for(int pipe, int n_chunks) {
  return pipe / (A_BYTES + (n_chunks > 0 ? n_chunks : BN / RC) * B_CHUNK) < MAX_STAGES
             ? pipe / (A_BYTES + (n_chunks > 0 ? n_chunks : BN / RC) * B_CHUNK)
             : MAX_STAGES;
}
static_assert(stages_for(PIPE_BYTES, 0) >= 4 && stages_for(PIPE_BYTES_PAIR, 0) >= 2, "a full row tile's stages");
constexpr int STAGE_LD = 129;            // epilogue staging row stride (floats)

// Split counts whose exchange buffers fit the pipeline's shared memory for a
// full 256-row tile: S * ceil(256 / S) rows of 128 fp32 partials.
__host__ __device__ constexpr bool split_fits(int S) {
  return S >= 1 && S <= 8 && S * ((BN + S - 1) / S) * BM * 4 <= PIPE_BYTES;
}

struct Params {
  int M, K;
  const int32_t* count;
  int dense_count;
  int splits;  // cluster size along z (1 = no split)
  unsigned* err;
  int pipe;    // pipeline bytes (PIPE_BYTES or PIPE_BYTES_PAIR)
  int count_early;  // *count is final when the grid starts (written two or more launches back)
  int tile;    // rows per row tile (BN; a dense count is split evenly, in multiples of 16)
};

template <class Epi>
__global__ void __launch_bounds__(THREADS, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const Params p, const typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int pipe = p.pipe;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pipe);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* tfull = empty + MAX_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x, n_tile = blockIdx.y;
  const int S = p.splits;
  const int z = S > 1 ? (int)cluster_ctarank() : 0;
  const int row0 = n_tile * p.tile;
  const int nk = p.K / BK;
  const int kb0 = (int)((long long)z * nk / S);
  const int kb1 = (int)((long long)(z + 1) * nk / S);
  const int m0 = m_tile * BM;
  // The first row tile always has rows unless the count is zero; later row
  // tiles learn from the live count whether they have work before they
  // allocate anything (the decision is uniform over a cluster).  A count that
  // is final when the grid starts is read before the dependency wait, so an
  // empty tile leaves at once instead of holding an SM until the previous
  // kernel completes: the live tiles still hold the next kernel back.
  if (n_tile > 0) {
    if (p.count_early) {
      if (row0 >= __ldcg(p.count)) return;
    } else {
      pdl_wait();
      pdl_trigger();
      const int c0 = p.count ? *p.count : p.dense_count;
      if (row0 >= c0) return;
    }
  }
  const bool lead = n_tile == 0 || p.count_early;  // not waited for yet

  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, BN);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // weight tiles of the first stages do not depend on earlier kernels: start
  // streaming them before waiting for the kernel that produced the rows
  const int npre = lead ? min(stages_for(pipe, 0), kb1 - kb0) : 0;
  if (warp == 0 && lane == 0) {
    for (int it = 0; it < npre; ++it) {
      mbar_expect_tx_only(&full[it], A_BYTES);
      tma_load_2d(smem + it * A_BYTES, &tmA, (kb0 + it) * BK, m0, &full[it]);
    }
  }
  if (lead) {
    pdl_wait();
    pdl_trigger();
  }
  const int count = p.count ? *p.count : p.dense_count;
  const bool active = row0 < count;  // uniform over the cluster
  const int n_rows = active ? min(p.tile, count - row0) : 0;
  const int n_mma = (n_rows + 15) & ~15;
  const int n_chunks = (n_rows + RC - 1) / RC;
  const int nst = stages_for(pipe, n_chunks);  // uniform over the cluster
  auto sA = [&](int st) { return smem + st * A_BYTES; };
  auto sB = [&](int st) { return smem + pipe - (st + 1) * n_chunks * B_CHUNK; };
  const int q = warp & 3;
  const int f = q * 32 + lane;
  const int ew = warp - 2;
  const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
  bool go = true;
  // rows own0 + S * t (t < n_own) of the tile are finished by this CTA: all of
  // them without a split, every S-th one (cluster rank z first) with one
  const int own0 = S > 1 ? z : 0;
  const int n_own = n_rows > own0 ? (n_rows - own0 + S - 1) / S : 0;
  // An epilogue whose rows read global memory issues the reads of the next 32
  // rows before it applies the current ones (two register sets); a staged
  // one reads shared memory and needs no look-ahead.
  constexpr bool kAhead = !epilogue_rolled<Epi>();
  typename Epi::Pre pre[8], pre2[8];
  typename Epi::Params epl = ep;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      if (!active) {
        // no rows: let the prefetched weight tiles land before leaving
        for (; it < npre; ++it) {
          mbar_arrive(&full[it]);
          mbar_wait(&full[it], 0, p.err);
        }
      } else {
        int s = 0;
        uint32_t ph = 0;  // stage it % nst and parity of it / nst, advanced without division
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if (it < npre) {
            mbar_expect_tx(&full[s], n_chunks * B_CHUNK);
          } else {
            if (!mbar_wait(&empty[s], ph ^ 1, p.err)) break;
            mbar_expect_tx(&full[s], A_BYTES + n_chunks * B_CHUNK);
            tma_load_2d(sA(s), &tmA, kb * BK, m0, &full[s]);
          }
          for (int c = 0; c < n_chunks; ++c)
            tma_load_2d(sB(s) + c * B_CHUNK, &tmB, kb * BK, row0 + c * RC, &full[s]);
          if (++s == nst) {
            s = 0;
            ph ^= 1;
          }
        }
        // every copy this CTA issued lands before its shared memory is reused
        for (int j = max(0, it - nst); j < it; ++j) mbar_wait(&full[j % nst], (j / nst) & 1, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && active) {
      const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
      int it = 0, s = 0;
      uint32_t ph = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        if (!mbar_wait(&full[s], ph, p.err)) break;
        fence_after_sync();
        const uint64_t da = sw128_kmajor_desc(smem_u32(sA(s)));
        const uint64_t db = sw128_kmajor_desc(smem_u32(sB(s)));
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_bf16(tmem, da + 2 * k, db + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
        if (++s == nst) {
          s = 0;
          ph ^= 1;
        }
      }
      mma_commit(tfull);
      // TMEM and shared memory are reused only after every MMA has completed
      mbar_wait(tfull, 0, p.err);
    }
    __syncwarp();
  } else if (active) {
    // the epilogue's tables (staged) or its global reads for this warp's
    // first rows are fetched while the main loop streams the weights
    if constexpr (Epi::kStaged) {
      Epi::stage(epl, smem + pipe + 256, row0, n_rows, threadIdx.x - 64);
      named_bar_sync(1, 128);
    }
    epilogue_prefetch<Epi>(epl, row0 + own0, S, min(32, n_own), m0, ew, lane, pre);
    go = mbar_wait(tfull, 0, p.err);
    fence_after_sync();
    if (S == 1 && go) {
      float* stage = reinterpret_cast<float*>(smem);
      auto chunk = [&](int j0, typename Epi::Pre(&cur)[8], typename Epi::Pre(&next)[8]) {
        const int nxt = min(32, n_rows - j0 - 32);
        if (kAhead && nxt > 0) epilogue_prefetch<Epi>(epl, row0 + j0 + 32, 1, nxt, m0, ew, lane, next);
        float v[32];
        tmem_ld32(tbase + j0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) stage[j * STAGE_LD + f] = v[j];
        named_bar_sync(1, 128);
        if (!kAhead && j0 > 0) epilogue_prefetch<Epi>(epl, row0 + j0, 1, min(32, n_rows - j0), m0, ew, lane, cur);
        epilogue_apply<Epi>(epl, row0 + j0, 1, min(32, n_rows - j0), m0, ew, lane, cur,
                            [&](int jj, float (&vv)[4]) {
#pragma unroll
                              for (int c = 0; c < 4; ++c) vv[c] = stage[jj * STAGE_LD + lane + 32 * c];
                            });
        named_bar_sync(1, 128);
      };
      for (int j0 = 0; j0 < n_rows; j0 += 64) {
        chunk(j0, pre, pre2);
        if (j0 + 32 < n_rows) {
          if constexpr (kAhead)
            chunk(j0 + 32, pre2, pre);
          else
            chunk(j0 + 32, pre, pre2);
        }
      }
    }
  }

  if (S > 1 && active) {
    // row j of the tile is finished by cluster rank j % S, which keeps the
    // partials of every rank for it at buf[rank][j / S][feature]
    const int n_slot = (n_rows + S - 1) / S;
    float* buf = reinterpret_cast<float*>(smem);
    const bool fits = (size_t)S * n_slot * BM * 4 <= (size_t)pipe;  // S * ceil(256 / S) rows fit PIPE_BYTES
    if (threadIdx.x == 0 && !fits) raise_error(p.err, kErrGemm);
    fence_before_sync();
    cluster_sync_all();  // every CTA of the tile is past its main loop
    if (warp >= 2 && go && fits) {
      const uint32_t mine = smem_u32(buf + (size_t)z * n_slot * BM + f);
      int owner = 0, slot = 0;  // of row c * 32 + j, advanced row by row
      for (int c = 0; c * 32 < n_rows; ++c) {
        float v[32];
        tmem_ld32(tbase + c * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (c * 32 + j < n_rows)
            st_cluster_f32(map_to_rank(mine + slot * BM * 4, (uint32_t)owner), v[j]);
          if (++owner == S) {
            owner = 0;
            ++slot;
          }
        }
      }
    }
    cluster_sync_all();  // every partial has been delivered
    if (warp >= 2 && go && fits) {
      auto part = [&](int t0, typename Epi::Pre(&cur)[8], typename Epi::Pre(&next)[8]) {
        const int nxt = min(32, n_own - t0 - 32);
        if (kAhead && nxt > 0)
          epilogue_prefetch<Epi>(epl, row0 + own0 + S * (t0 + 32), S, nxt, m0, ew, lane, next);
        if (!kAhead && t0 > 0)
          epilogue_prefetch<Epi>(epl, row0 + own0 + S * t0, S, min(32, n_own - t0), m0, ew, lane, cur);
        epilogue_apply<Epi>(epl, row0 + own0 + S * t0, S, min(32, n_own - t0), m0, ew, lane, cur,
                            [&](int jj, float (&vv)[4]) {
                              vv[0] = vv[1] = vv[2] = vv[3] = 0.f;
                              const float* src = buf + (size_t)(t0 + jj) * BM + lane;
                              // partials in cluster-rank order (a rolled loop: cold code)
#pragma unroll 1
                              for (int r = 0; r < S; ++r, src += (size_t)n_slot * BM) {
#pragma unroll
                                for (int cc = 0; cc < 4; ++cc) vv[cc] += src[32 * cc];
                              }
                            });
      };
      for (int t0 = 0; t0 < n_own; t0 += 64) {
        part(t0, pre, pre2);
        if (t0 + 32 < n_own) {
          if constexpr (kAhead)
            part(t0 + 32, pre2, pre);
          else
            part(t0 + 32, pre, pre2);
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, BN);
  }
}

}  // namespace tc

// ---------------------------------------------------------------- host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

template <class Epi>
cudaError_t set_smem_attr() {
  static cudaError_t e = cudaFuncSetAttribute(tc::gemm_tc_kernel<Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              tc::SMEM_BYTES);
  return e;
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

// Row-major bf16 matrix [rows][inner] as a TMA source with 64-element x
// box_rows boxes and 128-byte swizzling.
bool make_tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || inner % 64 != 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest number of clusters of size s (2..8) that can be resident at once.
int max_active_clusters(int s) {
  static int cache[9] = {0};
  static std::once_flag once;
  std::call_once(once, [] {
    set_smem_attr<EpiStore>();
    for (int c = 2; c <= 8; ++c) {
      if (!tc::split_fits(c)) continue;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, 1, c);
      cfg.blockDim = dim3(tc::THREADS);
      cfg.dynamicSmemBytes = tc::SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = (unsigned)c;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, tc::gemm_tc_kernel<EpiStore>, &cfg) != cudaSuccess) n = 0;
      cache[c] = n;
    }
    cudaGetLastError();
  });
  return (s >= 2 && s <= 8) ? cache[s] : 0;
}

// Prefix keys or values of one layer, [rows = R * P][nkv][hd] bf16, as a 3-D
// TMA source with (64 dims, 1 head, 64 keys) boxes and 128-byte swizzling.
bool make_tmap_kv(CUtensorMap* tm, const void* base, int hd, int nkv, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn || hd % 64 != 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)nkv, rows};
  cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)nkv * hd * 2};
  cuuint32_t box[3] = {64u, 1u, 64u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K splits for an M x K weight over n_tiles row tiles: the largest cluster
// size that keeps every (m, n) tile resident in one wave and gives each CTA
// at least one K block.
int gemm_tc_splits(int M, int K, int n_tiles) {
  const int m_tiles = M / tc::BM, nk = K / tc::BK, tiles = std::max(1, m_tiles * n_tiles);
  const int want = std::min(sm_count() / tiles, nk);
  for (int s = 8; s > 1; --s)
    if (s <= want && tc::split_fits(s) && max_active_clusters(s) >= tiles) return s;
  return 1;
}

namespace {

template <class Epi>
cudaError_t launch_tc(const TcGemm& g, const typename Epi::Params& ep, cudaStream_t st) {
  cudaError_t e = set_smem_attr<Epi>();
  if (e != cudaSuccess) return e;
  // a single-split GEMM with more tiles than SMs runs two CTAs per SM, all in
  // one wave; an epilogue's staged tables sit past the barriers and come out
  // of the pipeline
  int staged = 0;
  if constexpr (Epi::kStaged) staged = Epi::stage_bytes(ep);
  const int m_tiles_live = (g.M / tc::BM) * (g.count ? 1 : (g.dense_count + tc::BN - 1) / tc::BN);
  const int base = g.splits == 1 && m_tiles_live > sm_count() && !staged ? tc::PIPE_BYTES_PAIR : tc::PIPE_BYTES;
  const int pipe = base - ((staged + 1023) & ~1023);
  if (tc::stages_for(pipe, 0) < 2) return cudaErrorInvalidValue;
  // a dense row count is split into equal row tiles (multiples of 16, the
  // MMA's N step), so no tile carries a short remainder; with more tiles than
  // SMs the tile count is the one with the shortest busiest SM: tiles per SM
  // (rounded up) times rows per tile
  int tile = tc::BN, n_tiles = (g.max_rows + tc::BN - 1) / tc::BN;
  if (!g.count && g.dense_count > 0) {
    n_tiles = (g.dense_count + tc::BN - 1) / tc::BN;
    tile = ((g.dense_count + n_tiles - 1) / n_tiles + 15) & ~15;
    if (base == tc::PIPE_BYTES_PAIR) {
      const int m_tiles = g.M / tc::BM, sms = sm_count();
      long best = -1;
      for (int n = n_tiles; n <= 2 * n_tiles + 4; ++n) {
        const int t = ((g.dense_count + n - 1) / n + 15) & ~15;
        const int used = (g.dense_count + t - 1) / t;
        if (t < 64 || m_tiles * used > 2 * sms) continue;  // all tiles resident, two per SM at most
        const long cost = (long)((m_tiles * used + sms - 1) / sms) * t;
        if (best < 0 || cost < best) {
          best = cost;
          n_tiles = used;
          tile = t;
        }
      }
    }
  }
  tc::Params p{g.M, g.K, g.count, g.dense_count, g.splits, g.err, pipe, g.count_early ? 1 : 0, tile};
  return launch_pdl(st, dim3(g.M / tc::BM, n_tiles, g.splits), dim3(tc::THREADS),
                    (size_t)pipe + 1024 + 256 + staged, g.splits, tc::gemm_tc_kernel<Epi>, *g.tmA, *g.tmB, p,
                    ep);
}

}  // namespace

cudaError_t launch_gemm_tc(Launch& lc, int fam, const TcGemm& g, EpiKind kind, const EpiArgs& e) {
  if (g.M % tc::BM != 0 || g.K % tc::BK != 0 || !tc::split_fits(g.splits) || g.splits > g.K / tc::BK)
    return lc.err = cudaErrorInvalidValue;
  cudaError_t err = cudaSuccess;
  lc.before(fam);
  switch (kind) {
    case kEpiQKV: {
      using E = EpiQKV<__nv_bfloat16>;
      err = launch_tc<E>(g, E::Params{(__nv_bfloat16*)e.qkv, e.qkv_ld, e.qk_dim, e.qkv_M, e.hd, e.rc, e.L, e.P, e.rope},
                         lc.st);
      break;
    }
    case kEpiResidual:
      err = launch_tc<EpiResidual>(g, EpiResidual::Params{e.h, e.H, e.h_ld}, lc.st);
      break;
    case kEpiSwiGLU: {
      using E = EpiSwiGLU<__nv_bfloat16>;
      err = launch_tc<E>(g, E::Params{(__nv_bfloat16*)e.u, e.u_ld}, lc.st);
      break;
    }
    case kEpiStore:
      err = launch_tc<EpiStore>(g, EpiStore::Params{e.y, e.y_ld}, lc.st);
      break;
    case kEpiArgmax:
      err = launch_tc<EpiArgmax>(g, EpiArgmax::Params{e.part, e.part_ld, e.vocab}, lc.st);
      break;
  }
  if (err != cudaSuccess && lc.err == cudaSuccess) lc.err = err;
  lc.after(fam);
  return lc.err;
}

}  // namespace sf

extern "C" sf_status sfk_gemm_bf16(void* stream, const void* X, int rows_cap, const void* W, int M, int K,
                                   const int32_t* count, int dense_count, float* Y, int ldy, int splits,
                                   uint32_t* err) {
  using namespace sf;
  if (!X || !W || !Y || rows_cap <= 0 || M <= 0 || K <= 0 || M % tc::BM != 0 || K % tc::BK != 0 || ldy < M ||
      !tc::split_fits(splits) || splits > K / tc::BK || (!count && dense_count > rows_cap) || dense_count < 0)
    return SF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(W) & 15u)) return SF_ERR_INVALID_ARG;
  alignas(64) CUtensorMap tmA, tmB;
  if (!make_tmap_bf16(&tmA, W, K, M, tc::BM) || !make_tmap_bf16(&tmB, X, K, rows_cap, tc::RC)) return SF_ERR_CUDA;
  TcGemm g{&tmA, &tmB, M, K, count, dense_count, rows_cap, splits, err};
  EpiArgs e{};
  e.y = Y;
  e.y_ld = ldy;
  Launch lc{nullptr, (cudaStream_t)stream};
  launch_gemm_tc(lc, SF_K_AUX, g, kEpiStore, e);
  return lc.err == cudaSuccess ? SF_OK : SF_ERR_CUDA;
}
