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
//      prefix keys, split over the prefix;
//   2. per (row, head): the query is the one of the row's resolved source;
//      its block part runs over the branch's own L block keys/values, read
//      through the source slots of the branch's positions, and is merged with
//      the query's prefix partials by log-sum-exp.
#include "sf_internal.h"

namespace sf {
namespace {

constexpr int kMaxHd = 128;

template <typename TAct>
__global__ void __launch_bounds__(128) attn_prefix_kernel(const AttnArgs a) {
  __shared__ float qs[4][kMaxHd];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qv = blockIdx.x * 4 + warp;
  const int g = qv / a.nq, h = qv % a.nq;
  const int count = a.meta[0];
  if (g >= count) return;
  int r = 0;
  while (r + 1 < a.R && a.meta[2 + r] <= g) ++r;
  const int G = a.nq / a.nkv, kvh = h / G, hd = a.hd, per = hd / 32;
  const TAct* qkv = reinterpret_cast<const TAct*>(a.qkv);
  for (int j = lane; j < hd; j += 32) qs[warp][j] = to_f32<TAct>(qkv[(size_t)g * a.ld_qkv + h * hd + j]);
  __syncwarp();
  const int s = blockIdx.y;
  const int k_lo = s * a.split_len, k_hi = min(a.P, k_lo + a.split_len);
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
__global__ void __launch_bounds__(128) attn_block_kernel(const AttnArgs a) {
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
  const TAct* qkv = reinterpret_cast<const TAct*>(a.qkv);
  for (int j = lane; j < hd; j += 32) qs[warp][j] = to_f32<TAct>(qkv[(size_t)g * a.ld_qkv + h * hd + j]);
  __syncwarp();
  const int base = (row / L) * L;  // first row of this branch
  const int koff = (a.nq + kvh) * hd, voff = (a.nq + a.nkv + kvh) * hd;
  // block scores, one key per lane per round (L <= 64)
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
  float M = warp_max(fmaxf(sc[0], sc[1]));
  for (int s = 0; s < a.n_splits; ++s) M = fmaxf(M, a.part_ml[(((size_t)s * a.T + g) * a.nq + h) * 2]);
  float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < a.n_splits; ++s) {
    const size_t qi = ((size_t)s * a.T + g) * a.nq + h;
    const float ms = a.part_ml[qi * 2], ls = a.part_ml[qi * 2 + 1];
    const float wgt = exp2f(ms - M);  // 0 for an empty split (ms = -inf)
    l += wgt * ls;
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
}

template <typename TAct>
cudaError_t attention_impl(Launch& lc, const AttnArgs& a) {
  if (a.P > 0 && a.n_splits > 0) {
    dim3 grid((a.T * a.nq + 3) / 4, a.n_splits);
    lc.before(SF_K_ATTN_PREFIX);
    attn_prefix_kernel<TAct><<<grid, 128, 0, lc.st>>>(a);
    lc.after(SF_K_ATTN_PREFIX);
  }
  lc.before(SF_K_ATTN_BLOCK);
  attn_block_kernel<TAct><<<(a.T * a.nq + 3) / 4, 128, 0, lc.st>>>(a);
  lc.after(SF_K_ATTN_BLOCK);
  return lc.err;
}

}  // namespace

cudaError_t launch_attention(Launch& lc, int act_bf16, const AttnArgs& a) {
  if (a.hd > kMaxHd || a.hd % 32 != 0 || a.L > 64) return cudaErrorInvalidValue;
  if (act_bf16) return attention_impl<__nv_bfloat16>(lc, a);
  return attention_impl<float>(lc, a);
}

}  // namespace sf
