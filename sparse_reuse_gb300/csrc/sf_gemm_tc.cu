// tcgen05 / TMEM GEMM over the rows of the compacted recompute set (BF16).
//
// Y[g][o] = sum_k X[g][k] W[o][k] for g < count (count read on the device).
// The weight is the M operand: each CTA owns 128 output features (TMEM lanes)
// and up to 256 rows (TMEM columns), so a weight tile is streamed once for all
// rows of a layer; the rows are the N operand, loaded in 64-row TMA boxes only
// up to the live row count.  Narrow GEMMs split K over CTAs; the partial sums
// go to a workspace and the last CTA of a tile (atomic ticket, no waiting)
// adds them in split order, so results do not depend on scheduling.
//
// Warp roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues the
// MMAs, warps 2-5 drain TMEM through shared memory into the layer epilogue.
#include <cudaTypedefs.h>

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
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_CHUNK = RC * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = STAGES * (A_BYTES + B_BYTES) + 1024 + 256;
constexpr int STAGE_LD = 129;  // epilogue staging row stride (floats)

struct Params {
  int M, K;
  const int32_t* count;
  int dense_count;
  int max_rows;
  int splits;
  float* ws;           // [splits][max_rows][M] partial sums (splits > 1)
  unsigned* tile_ctr;  // [n_tiles][m_tiles] arrival tickets, zero between launches
  unsigned* err;
};

template <class Epi>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const Params p, const typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int count = p.count ? *p.count : p.dense_count;
  const int m_tile = blockIdx.x, n_tile = blockIdx.y, z = blockIdx.z;
  const int row0 = n_tile * BN;
  if (row0 >= count) return;
  const int n_rows = min(BN, count - row0);
  const int n_mma = (n_rows + 15) & ~15;
  const int n_chunks = (n_rows + RC - 1) / RC;
  const int nk = p.K / BK;
  const int kb0 = (int)((long long)z * nk / p.splits);
  const int kb1 = (int)((long long)(z + 1) * nk / p.splits);
  const int m0 = m_tile * BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, p.err)) break;
        mbar_expect_tx(&full[s], A_BYTES + n_chunks * B_CHUNK);
        tma_load_2d(sA + s * A_BYTES, &tmA, kb * BK, m0, &full[s]);
        for (int c = 0; c < n_chunks; ++c)
          tma_load_2d(sB + s * B_BYTES + c * B_CHUNK, &tmB, kb * BK, row0 + c * RC, &full[s]);
      }
      // every copy this CTA issued lands before it can exit
      for (int j = max(0, it - STAGES); j < it; ++j) mbar_wait(&full[j % STAGES], (j / STAGES) & 1, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
      int it = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait(&full[s], ph, p.err)) break;
        fence_after_sync();
        const uint64_t da = sw128_kmajor_desc(smem_u32(sA + s * A_BYTES));
        const uint64_t db = sw128_kmajor_desc(smem_u32(sB + s * B_BYTES));
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_bf16(tmem, da + 2 * k, db + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
      }
      mma_commit(tfull);
      // TMEM is released only after every MMA of this CTA has completed
      mbar_wait(tfull, 0, p.err);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int f = q * 32 + lane;
    const int ew = warp - 2;
    float* stage = reinterpret_cast<float*>(smem);
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
    bool go = mbar_wait(tfull, 0, p.err);
    fence_after_sync();
    if (go && p.splits > 1) {
      for (int j0 = 0; j0 < n_rows; j0 += 32) {
        float v[32];
        tmem_ld32(tbase + j0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j0 + j < n_rows) p.ws[((size_t)z * p.max_rows + row0 + j0 + j) * p.M + m0 + f] = v[j];
      }
      __threadfence();
      named_bar_sync(1, 128);
      if (threadIdx.x == 64) {
        unsigned* ctr = p.tile_ctr + (size_t)n_tile * gridDim.x + m_tile;
        const unsigned t = atomicAdd(ctr, 1u);
        *last_flag = (t == (unsigned)p.splits - 1) ? 1 : 0;
        if (*last_flag) *ctr = 0u;
      }
      named_bar_sync(1, 128);
      go = *last_flag != 0;
      if (go) __threadfence();
    }
    if (go) {
      for (int j0 = 0; j0 < n_rows; j0 += 32) {
        float v[32];
        if (p.splits == 1) {
          tmem_ld32(tbase + j0, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
          for (int s = 0; s < p.splits; ++s) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j0 + j < n_rows) v[j] += __ldcg(p.ws + ((size_t)s * p.max_rows + row0 + j0 + j) * p.M + m0 + f);
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) stage[j * STAGE_LD + f] = v[j];
        named_bar_sync(1, 128);
        for (int jj = ew; jj < 32 && j0 + jj < n_rows; jj += 4) {
          float vv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) vv[c] = stage[jj * STAGE_LD + lane + 32 * c];
          Epi::apply(ep, row0 + j0 + jj, m0, lane, vv);
        }
        named_bar_sync(1, 128);
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

int gemm_tc_splits(int M, int K, int n_tiles, size_t ws_floats, int max_rows) {
  const int m_tiles = M / tc::BM, nk = K / tc::BK;
  int s = sm_count() / std::max(1, m_tiles * n_tiles);
  s = std::min(s, std::max(1, nk / 2));
  s = std::min(s, 16);
  const size_t per = (size_t)max_rows * M;
  if (per > 0) s = (int)std::min<size_t>((size_t)s, ws_floats / per);
  return std::max(1, s);
}

cudaError_t launch_gemm_tc(Launch& lc, int fam, const TcGemm& g, EpiKind kind, const EpiArgs& e) {
  if (g.M % tc::BM != 0 || g.K % tc::BK != 0 || g.splits < 1 || g.splits > g.K / tc::BK) return cudaErrorInvalidValue;
  tc::Params p{g.M, g.K, g.count, g.dense_count, g.max_rows, g.splits, g.ws, g.tile_ctr, g.err};
  dim3 grid(g.M / tc::BM, (g.max_rows + tc::BN - 1) / tc::BN, g.splits);
  cudaError_t err = cudaSuccess;
  lc.before(fam);
  switch (kind) {
    case kEpiQKV: {
      using E = EpiQKV<__nv_bfloat16>;
      E::Params ep{(__nv_bfloat16*)e.qkv, e.qkv_ld, e.qk_dim, e.qkv_M, e.hd, e.rc, e.L, e.P, e.rope};
      err = set_smem_attr<E>();
      if (err == cudaSuccess) tc::gemm_tc_kernel<E><<<grid, tc::THREADS, tc::SMEM_BYTES, lc.st>>>(*g.tmA, *g.tmB, p, ep);
      break;
    }
    case kEpiResidual: {
      using E = EpiResidual;
      E::Params ep{e.h, e.H, e.h_ld};
      err = set_smem_attr<E>();
      if (err == cudaSuccess) tc::gemm_tc_kernel<E><<<grid, tc::THREADS, tc::SMEM_BYTES, lc.st>>>(*g.tmA, *g.tmB, p, ep);
      break;
    }
    case kEpiSwiGLU: {
      using E = EpiSwiGLU<__nv_bfloat16>;
      E::Params ep{(__nv_bfloat16*)e.u, e.u_ld};
      err = set_smem_attr<E>();
      if (err == cudaSuccess) tc::gemm_tc_kernel<E><<<grid, tc::THREADS, tc::SMEM_BYTES, lc.st>>>(*g.tmA, *g.tmB, p, ep);
      break;
    }
    case kEpiStore: {
      using E = EpiStore;
      E::Params ep{e.y, e.y_ld};
      err = set_smem_attr<E>();
      if (err == cudaSuccess) tc::gemm_tc_kernel<E><<<grid, tc::THREADS, tc::SMEM_BYTES, lc.st>>>(*g.tmA, *g.tmB, p, ep);
      break;
    }
  }
  if (err != cudaSuccess && lc.err == cudaSuccess) lc.err = err;
  lc.after(fam);
  return lc.err;
}

}  // namespace sf

extern "C" sf_status sfk_gemm_bf16(void* stream, const void* X, int rows_cap, const void* W, int M, int K,
                                   const int32_t* count, int dense_count, float* Y, int ldy, int splits, float* ws,
                                   uint32_t* tile_ctr, uint32_t* err) {
  using namespace sf;
  if (!X || !W || !Y || rows_cap <= 0 || M <= 0 || K <= 0 || M % tc::BM != 0 || K % tc::BK != 0 || ldy < M ||
      splits < 1 || splits > K / tc::BK || (splits > 1 && (!ws || !tile_ctr)) || (!count && dense_count > rows_cap) ||
      dense_count < 0)
    return SF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(W) & 15u)) return SF_ERR_INVALID_ARG;
  alignas(64) CUtensorMap tmA, tmB;
  if (!make_tmap_bf16(&tmA, W, K, M, tc::BM) || !make_tmap_bf16(&tmB, X, K, rows_cap, tc::RC)) return SF_ERR_CUDA;
  TcGemm g{&tmA, &tmB, M, K, count, dense_count, rows_cap, splits, ws, tile_ctr, err};
  EpiArgs e{};
  e.y = Y;
  e.y_ld = ldy;
  Launch lc{nullptr, (cudaStream_t)stream};
  launch_gemm_tc(lc, SF_K_AUX, g, kEpiStore, e);
  return lc.err == cudaSuccess ? SF_OK : SF_ERR_CUDA;
}
