// Row-gathered GEMMs of the folded layer: Y[g][o] = sum_k X[g][k] W[o][k] for
// the g < count rows of the compacted recompute set (QKV, gate/up, down) or
// all rows (output projection), followed by the layer's epilogue.
//
// FP32 contexts use this CUDA-core kernel (fp32 operands keep the pass within
// fp32 rounding); BF16 contexts use the tcgen05 kernel in sf_gemm_tc.cu.
#include "sf_epilogue.cuh"
#include "sf_internal.h"

namespace sf {


namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16;

// 64 rows x 64 outputs per block, 256 threads, 4 x 4 outputs per thread.
template <typename TAct>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const TAct* __restrict__ X, int ldx,
                                                        const TAct* __restrict__ W, int ldw,
                                                        float* __restrict__ Y, int ldy,
                                                        const int32_t* count_ptr, int dense_count, int K) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs[kBK][kBN + 4];
  pdl_wait();
  pdl_trigger();
  const int count = count_ptr ? *count_ptr : dense_count;
  const int g0 = blockIdx.y * kBM, o0 = blockIdx.x * kBN;
  if (g0 >= count) return;
  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;  // 16 x 16 thread grid
  const int lr = tid / 4, lk = (tid % 4) * 4;  // loader: row lr, k lk..lk+3
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kBK) {
    {
      const int g = g0 + lr;
      float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g < count) xv = load4<TAct>(X + (size_t)g * ldx + k0 + lk);
      As[lk + 0][lr] = xv.x; As[lk + 1][lr] = xv.y; As[lk + 2][lr] = xv.z; As[lk + 3][lr] = xv.w;
      const float4 wv = load4<TAct>(W + (size_t)(o0 + lr) * ldw + k0 + lk);
      Bs[lk + 0][lr] = wv.x; Bs[lk + 1][lr] = wv.y; Bs[lk + 2][lr] = wv.z; Bs[lk + 3][lr] = wv.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int g = g0 + tr * 4 + i;
    if (g < count)
      *reinterpret_cast<float4*>(Y + (size_t)g * ldy + o0 + tc * 4) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

// One warp per (row, 128-feature tile) applies the epilogue to fp32 results.
template <class Epi>
__global__ void __launch_bounds__(128) epilogue_kernel(const float* __restrict__ Y, int ldy, int n_tiles,
                                                      const int32_t* count_ptr, int dense_count,
                                                      const typename Epi::Params p) {
  pdl_wait();
  pdl_trigger();
  const int count = count_ptr ? *count_ptr : dense_count;
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int g = w / n_tiles, t = w % n_tiles;
  if (g >= count) return;
  float v[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) v[c] = Y[(size_t)g * ldy + t * 128 + lane + 32 * c];
  typename Epi::Pre pre;
  Epi::prefetch(p, g, t * 128, lane, pre);
  Epi::apply(p, g, t * 128, lane, v, pre);
}

template <typename TAct>
cudaError_t gemm_simt(Launch& lc, int fam, const GemmArgs& g, EpiKind kind, const EpiArgs& e, float* y32) {
  const int ldy = g.M;
  dim3 grid(g.M / kBN, (g.max_rows + kBM - 1) / kBM);
  lc.before(fam);
  lc.check(launch_pdl(lc.st, grid, dim3(256), 0, 1, gemm_simt_kernel<TAct>, (const TAct*)g.X, g.ldx,
                      (const TAct*)g.W, g.ldw, y32, ldy, g.count, g.dense_count, g.K));
  lc.after(fam);
  const int n_tiles = g.M / 128;
  const int blocks = (g.max_rows * n_tiles + 3) / 4;
  lc.before(SF_K_AUX);
  switch (kind) {
    case kEpiQKV: {
      typename EpiQKV<TAct>::Params p{(TAct*)e.qkv, e.qkv_ld, e.qk_dim, e.qkv_M, e.hd, e.rc, e.L, e.P, e.rope};
      lc.check(launch_pdl(lc.st, dim3(blocks), dim3(128), 0, 1, epilogue_kernel<EpiQKV<TAct>>, (const float*)y32, ldy, n_tiles, g.count, g.dense_count, p));
      break;
    }
    case kEpiResidual: {
      EpiResidual::Params p{e.h, e.H, e.h_ld};
      lc.check(launch_pdl(lc.st, dim3(blocks), dim3(128), 0, 1, epilogue_kernel<EpiResidual>, (const float*)y32, ldy, n_tiles, g.count, g.dense_count, p));
      break;
    }
    case kEpiSwiGLU: {
      typename EpiSwiGLU<TAct>::Params p{(TAct*)e.u, e.u_ld};
      lc.check(launch_pdl(lc.st, dim3(blocks), dim3(128), 0, 1, epilogue_kernel<EpiSwiGLU<TAct>>, (const float*)y32, ldy, n_tiles, g.count, g.dense_count, p));
      break;
    }
    case kEpiStore: {
      EpiStore::Params p{e.y, e.y_ld};
      lc.check(launch_pdl(lc.st, dim3(blocks), dim3(128), 0, 1, epilogue_kernel<EpiStore>, (const float*)y32, ldy, n_tiles, g.count, g.dense_count, p));
      break;
    }
    case kEpiArgmax: {
      EpiArgmax::Params p{e.part, e.part_ld, e.vocab};
      lc.check(launch_pdl(lc.st, dim3(blocks), dim3(128), 0, 1, epilogue_kernel<EpiArgmax>, (const float*)y32, ldy, n_tiles, g.count, g.dense_count, p));
      break;
    }
  }
  lc.after(SF_K_AUX);
  return lc.err;
}

}  // namespace

cudaError_t launch_gemm(Launch& lc, int fam, int act_bf16, const GemmArgs& g, EpiKind kind, const EpiArgs& e,
                        float* y32) {
  if (g.M % 128 != 0 || g.K % kBK != 0) return cudaErrorInvalidValue;
  if (act_bf16) return gemm_simt<__nv_bfloat16>(lc, fam, g, kind, e, y32);
  return gemm_simt<float>(lc, fam, g, kind, e, y32);
}

}  // namespace sf
