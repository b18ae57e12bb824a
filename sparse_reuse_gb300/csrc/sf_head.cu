// Verification head: final RMSNorm, LM head with a greedy-token epilogue, and
// draft acceptance ("SpecFold", arXiv 2610.04875v2 summary, §1 and §2.2: a
// matching draft supplies logits that skip later denoising passes; App. B:
// the LM head runs outside the layer kernels).
//
//   head_norm_kernel      RMSNorm of every output row -> xn (context dtype)
//   GEMM + EpiArgmax      logits tile by tile; per (row, 128-entry vocabulary
//                         tile) the largest logit and its index
//   head_reduce_kernel    one warp per row: greedy token over the tiles
//   head_accept_kernel    one warp per request: branches in index order
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <new>
#include <string>

#include "sf_internal.h"
#include "specfold_head.h"

struct sf_head {
  int d = 0, vocab = 0, V_pad = 0, n_vt = 0, dtype = SF_BF16, rows_cap = 0, rows_pad = 0, sm_count = 148;
  float eps = 0.f;
  float* gain = nullptr;
  void* w = nullptr;        // [V_pad][d] W_lm^T, zero rows past vocab
  void* xn = nullptr;       // [rows_pad][d] normalised rows (context dtype)
  float2* part = nullptr;   // [rows_cap][n_vt] (largest logit, index) per vocabulary tile
  float* y32 = nullptr;     // [rows_cap][V_pad] logits (FP32 heads)
  unsigned* err_dev = nullptr;
  unsigned* err_host = nullptr;
  alignas(64) CUtensorMap tm_w, tm_x;
  std::string last_error;
};

namespace sf {
namespace {

constexpr int kHeadThreads = 256;

template <typename TIn, typename TAct>
__global__ void __launch_bounds__(kHeadThreads) head_norm_kernel(const TIn* X, int rows, int d, const float* gain,
                                                                 float eps, TAct* out) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const int d4 = d >> 2;
  for (int g = blockIdx.x; g < rows; g += gridDim.x) {
    const TIn* x = X + (size_t)g * d;
    float ss = 0.f;
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      const float4 v = load4<TIn>(x + c * 4);
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum(ss, red);
    const float rstd = rsqrtf(ss / (float)d + eps);
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      const float4 v = load4<TIn>(x + c * 4);
      const float4 w = *reinterpret_cast<const float4*>(gain + c * 4);
      store4<TAct>(out + (size_t)g * d + c * 4,
                   make_float4(v.x * rstd * w.x, v.y * rstd * w.y, v.z * rstd * w.z, v.w * rstd * w.w));
    }
  }
}

// One warp per row: the greedy token over the row's vocabulary-tile partials
// (largest value, the lowest index on a tie).
__global__ void __launch_bounds__(kHeadThreads) head_reduce_kernel(const float2* part, int n_vt, int rows, int vocab,
                                                                   int32_t* pred, unsigned* err) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x * (kHeadThreads / 32) + (threadIdx.x >> 5);
  if (g >= rows) return;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  const float2* p = part + (size_t)g * n_vt;
  for (int t = lane; t < n_vt; t += 32) {  // tiles rise with t, so the first maximum wins in a lane
    const float2 v = p[t];
    const int vi = __float_as_int(v.y);
    if (vi != 0x7fffffff && (bi == 0x7fffffff || v.x > best)) {
      best = v.x;
      bi = vi;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (oi != 0x7fffffff && (bi == 0x7fffffff || ob > best || (ob == best && oi < bi))) {
      best = ob;
      bi = oi;
    }
  }
  if (lane == 0) {
    if (bi < 0 || bi >= vocab) {
      raise_error(err, kErrGemm);
      bi = 0;
    }
    pred[g] = bi;
  }
}

// One warp per request: acceptance of every branch in index order, then the
// deepest accepted branch.
constexpr int kAcceptWarps = 4;

__global__ void __launch_bounds__(32 * kAcceptWarps) head_accept_kernel(const __grid_constant__ Tree tree, int L,
                                                                        const int32_t* tokens, const int32_t* pred,
                                                                        uint8_t* accepted, int32_t* chosen) {
  __shared__ uint8_t acc[kAcceptWarps][128];
  __shared__ uint8_t dep[kAcceptWarps][128];
  pdl_wait();
  pdl_trigger();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kAcceptWarps + w;
  if (r >= tree.R) return;
  const int Bp = tree.Bp;
  for (int i = 0; i < Bp; ++i) {
    bool ok = true;
    const int p = i > 0 ? tree.parent[r * Bp + i] : -1;
    if (p >= 0) {
      const int32_t* ti = tokens + (size_t)(r * Bp + i) * L;
      const int32_t* tp = tokens + (size_t)(r * Bp + p) * L;
      const int32_t* pp = pred + (size_t)(r * Bp + p) * L;
      for (int n = lane; n < L; n += 32)
        if (ti[n] != tp[n] && ti[n] != pp[n]) ok = false;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) {
      acc[w][i] = p < 0 ? 1 : (acc[w][p] && ok ? 1 : 0);
      dep[w][i] = p < 0 ? 0 : dep[w][p] + 1;
      if (accepted) accepted[r * Bp + i] = acc[w][i];
    }
    __syncwarp();
  }
  if (lane == 0 && chosen) {
    int best = 0;
    for (int i = 1; i < Bp; ++i)
      if (acc[w][i] && dep[w][i] > dep[w][best]) best = i;
    chosen[r] = best;
  }
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

bool misaligned(const void* p, uintptr_t align) { return p && (reinterpret_cast<uintptr_t>(p) & (align - 1)); }

sf_status fail(sf_head* h, sf_status st, const char* fmt, ...) __attribute__((format(printf, 3, 4)));
sf_status fail(sf_head* h, sf_status st, const char* fmt, ...) {
  if (h) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    h->last_error = buf;
  }
  return st;
}

void free_head(sf_head* h) {
  if (!h) return;
  void* bufs[] = {h->gain, h->w, h->xn, h->part, h->y32, h->err_dev};
  for (void* b : bufs) cudaFree(b);
  if (h->err_host) cudaFreeHost(h->err_host);
  delete h;
}

template <typename T>
cudaError_t halloc(T** p, size_t bytes) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes > 0 ? bytes : 16);
  if (e == cudaSuccess) e = cudaMemset(q, 0, bytes > 0 ? bytes : 16);
  *p = static_cast<T*>(q);
  return e;
}

}  // namespace
}  // namespace sf

using namespace sf;

extern "C" {

sf_status sf_head_create(const sf_head_shapes* shapes, const float* final_norm, const void* w_lm, sf_head** out) {
  if (!out) return SF_ERR_INVALID_ARG;
  *out = nullptr;
  if (!shapes || !final_norm || !w_lm) return SF_ERR_INVALID_ARG;
  const sf_head_shapes s = *shapes;
  if (s.vocab < 1 || s.max_rows < 1 || !(s.rms_eps >= 0.f) || (s.dtype != SF_F32 && s.dtype != SF_BF16) ||
      s.d_model <= 0)
    return SF_ERR_INVALID_ARG;
  if (s.d_model % 128 != 0 || s.d_model > 16384 || s.max_rows > kMaxRows) return SF_ERR_UNSUPPORTED;
  sf_head* h = new (std::nothrow) sf_head();
  if (!h) return SF_ERR_OOM;
  h->d = s.d_model;
  h->vocab = s.vocab;
  h->V_pad = round_up(s.vocab, 128);
  h->n_vt = h->V_pad / 128;
  h->dtype = s.dtype;
  h->eps = s.rms_eps;
  h->rows_cap = s.max_rows;
  h->rows_pad = round_up(s.max_rows, 256);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (h->sm_count <= 0) h->sm_count = 148;
  const int ab = s.dtype == SF_BF16 ? 2 : 4, d = h->d;
  cudaError_t e = cudaSuccess;
#define SF_HTRY(x)                                                                        \
  do {                                                                                    \
    e = (x);                                                                              \
    if (e != cudaSuccess) {                                                               \
      sf_status st_ = e == cudaErrorMemoryAllocation ? SF_ERR_OOM : SF_ERR_CUDA;          \
      free_head(h);                                                                       \
      cudaGetLastError();                                                                 \
      return st_;                                                                         \
    }                                                                                     \
  } while (0)
  SF_HTRY(halloc(&h->gain, (size_t)d * 4));
  SF_HTRY(cudaMemcpy(h->gain, final_norm, (size_t)d * 4, cudaMemcpyDeviceToDevice));
  SF_HTRY(halloc(&h->w, (size_t)h->V_pad * d * ab));
  SF_HTRY(launch_pack_transpose(0, w_lm, d, s.vocab, h->w, d, 0, 0, s.dtype == SF_BF16));
  SF_HTRY(halloc(&h->xn, (size_t)h->rows_pad * d * ab));
  SF_HTRY(halloc(&h->part, (size_t)h->rows_cap * h->n_vt * sizeof(float2)));
  if (s.dtype == SF_F32) SF_HTRY(halloc(&h->y32, (size_t)h->rows_cap * h->V_pad * 4));
  SF_HTRY(halloc(&h->err_dev, 64));
  SF_HTRY(cudaHostAlloc((void**)&h->err_host, 64, cudaHostAllocDefault));
  *h->err_host = 0;
  if (s.dtype == SF_BF16 &&
      (!make_tmap_bf16(&h->tm_w, h->w, d, h->V_pad, 128) || !make_tmap_bf16(&h->tm_x, h->xn, d, h->rows_pad, 64))) {
    free_head(h);
    return SF_ERR_CUDA;
  }
  SF_HTRY(cudaDeviceSynchronize());
#undef SF_HTRY
  *out = h;
  return SF_OK;
}

sf_status sf_head_verify(sf_head* h, void* stream, const void* hidden, const int32_t* tokens, const int32_t* parent,
                         int R, int B, int L, int32_t* pred, uint8_t* accepted, int32_t* chosen) {
  if (!h) return SF_ERR_INVALID_ARG;
  if (!hidden || !tokens || !parent || !pred) return fail(h, SF_ERR_INVALID_ARG, "null hidden/tokens/parent/pred");
  if (R < 0 || B < 0 || L < 1) return fail(h, SF_ERR_INVALID_ARG, "negative R or B, or L < 1");
  if (misaligned(hidden, 16) || misaligned(tokens, 4) || misaligned(pred, 4) || misaligned(chosen, 4))
    return fail(h, SF_ERR_INVALID_ARG, "hidden needs 16-byte alignment, tokens/pred/chosen 4-byte");
  const int Bp = B + 1;
  if (Bp > 127 || (long)R * Bp > kMaxTreeSlots || (long)R * Bp * L > h->rows_cap)
    return fail(h, SF_ERR_SHAPE, "R=%d B=%d L=%d beyond the head's capacity (%d rows)", R, B, L, h->rows_cap);
  Tree tree{};
  tree.R = R;
  tree.Bp = Bp;
  for (int r = 0; r < R; ++r) {
    if (parent[r * Bp] != -1) return fail(h, SF_ERR_TREE, "request %d: parent[0] must be -1", r);
    for (int i = 1; i < Bp; ++i) {
      const int pi = parent[r * Bp + i];
      if (pi < 0 || pi >= i) return fail(h, SF_ERR_TREE, "request %d: parent[%d] = %d not in [0, %d)", r, i, pi, i);
      tree.parent[r * Bp + i] = (int8_t)pi;
    }
    tree.parent[r * Bp] = -1;
  }
  if (*h->err_host) return fail(h, SF_ERR_DEVICE_ASSERT, "device check word 0x%x", *h->err_host);
  if (R == 0) return SF_OK;
  const int T = R * Bp * L, d = h->d, bf16 = h->dtype == SF_BF16;
  cudaStream_t st = (cudaStream_t)stream;
  Launch lc{nullptr, st};
  lc.before(SF_K_AUX);
  const int grid = T < 8 * h->sm_count ? T : 8 * h->sm_count;
  if (bf16)
    lc.check(launch_pdl(st, dim3(grid), dim3(kHeadThreads), 0, 1, head_norm_kernel<__nv_bfloat16, __nv_bfloat16>,
                        (const __nv_bfloat16*)hidden, T, d, (const float*)h->gain, h->eps, (__nv_bfloat16*)h->xn));
  else
    lc.check(launch_pdl(st, dim3(grid), dim3(kHeadThreads), 0, 1, head_norm_kernel<float, float>, (const float*)hidden,
                        T, d, (const float*)h->gain, h->eps, (float*)h->xn));
  lc.after(SF_K_AUX);
  EpiArgs e{};
  e.part = h->part;
  e.part_ld = h->n_vt;
  e.vocab = h->vocab;
  if (bf16) {
    TcGemm t{};
    t.tmA = &h->tm_w;
    t.tmB = &h->tm_x;
    t.M = h->V_pad;
    t.K = d;
    t.count = nullptr;
    t.dense_count = T;
    t.max_rows = T;
    t.splits = gemm_tc_splits(h->V_pad, d, (T + 255) / 256);
    t.err = h->err_dev;
    t.count_early = false;
    launch_gemm_tc(lc, SF_K_AUX, t, kEpiArgmax, e);
  } else {
    GemmArgs g{};
    g.X = h->xn;
    g.ldx = d;
    g.W = h->w;
    g.ldw = d;
    g.M = h->V_pad;
    g.K = d;
    g.count = nullptr;
    g.dense_count = T;
    g.max_rows = T;
    launch_gemm(lc, SF_K_AUX, 0, g, kEpiArgmax, e, h->y32);
  }
  lc.before(SF_K_AUX);
  lc.check(launch_pdl(st, dim3((T + kHeadThreads / 32 - 1) / (kHeadThreads / 32)), dim3(kHeadThreads), 0, 1,
                      head_reduce_kernel, (const float2*)h->part, h->n_vt, T, h->vocab, pred, h->err_dev));
  lc.after(SF_K_AUX);
  if (accepted || chosen) {
    lc.before(SF_K_AUX);
    lc.check(launch_pdl(st, dim3((R + kAcceptWarps - 1) / kAcceptWarps), dim3(32 * kAcceptWarps), 0, 1,
                        head_accept_kernel, tree, L, tokens, (const int32_t*)pred, accepted, chosen));
    lc.after(SF_K_AUX);
  }
  if (lc.err == cudaSuccess)
    lc.err = cudaMemcpyAsync(h->err_host, h->err_dev, sizeof(unsigned), cudaMemcpyDeviceToHost, st);
  if (lc.err != cudaSuccess) return fail(h, SF_ERR_CUDA, "launch failed: %s", cudaGetErrorString(lc.err));
  return SF_OK;
}

const char* sf_head_last_error(const sf_head* h) { return h ? h->last_error.c_str() : ""; }

sf_status sf_head_destroy(sf_head* h) {
  if (!h) return SF_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  unsigned w = 0;
  if (e == cudaSuccess) cudaMemcpy(&w, h->err_dev, sizeof(unsigned), cudaMemcpyDeviceToHost);
  free_head(h);
  if (e != cudaSuccess) return SF_ERR_CUDA;
  return w ? SF_ERR_DEVICE_ASSERT : SF_OK;
}

}  // extern "C"
