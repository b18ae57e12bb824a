// GEMM epilogues of the folded layer.  Each works on one output row g and one
// 128-wide tile of output features [m0, m0 + 128): lane l of a warp holds the
// fp32 accumulators of features m0 + l + 32c, c = 0..3, so the rotary pair
// (j, j + hd/2) of a head and the gate/up pair of a SwiGLU tile sit in the
// same thread for hd in {64, 128}.
//
// prefetch() issues the row's global reads (residual input, rotary table)
// and apply() consumes them, so a warp can start the reads of several rows
// before it waits on any of them.
#pragma once

#include "sf_common.cuh"

namespace sf {

// Packed Q|K|V projection of recompute row g: rotary encoding of q and k at
// absolute position P + n (n = rc[g] mod L), then a store of the row into the
// physical QKV table [T_rc][Mqkv].  Features past Mqkv are zero padding of
// the packed weight and are dropped.
template <typename TAct>
struct EpiQKV {
  struct Params {
    TAct* qkv;
    int ld;          // row stride of the table (elements)
    int qk_dim;      // (nq + nkv) * hd: features that are rotary-encoded
    int M;           // (nq + 2 nkv) * hd: real features
    int hd;
    const int32_t* rc;
    int L;
    int P;
    const float2* rope;  // [pos][hd/2] (cos, sin)
  };
  struct Pre {
    float2 cs[4];
  };
  static __device__ __forceinline__ void prefetch(const Params& p, int g, int m0, int lane, Pre& pre) {
    const int pos = p.P + (p.rc[g] % p.L);
    const int half = p.hd >> 1;
    // m0 is a multiple of 128 and hd divides 128, so j % half = (lane + 32c) % half
    const float2* row = p.rope + (size_t)pos * half;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int f = m0 + lane + 32 * c;
      pre.cs[c] = f < p.qk_dim ? row[(lane + 32 * c) & (half - 1)] : make_float2(1.f, 0.f);
    }
  }
  // hd = 128: a tile is one head, feature l + 32c pairs with l + 32(c ^ 2);
  // hd = 64: a tile is two heads, the pair is l + 32(c ^ 1).  The partner is a
  // compile-time index in both cases, so v stays in registers.
  template <int PAIR>
  static __device__ __forceinline__ void rotate_store(const Params& p, int g, int m0, int lane, const float v[4],
                                                      const Pre& pre) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int f = m0 + lane + 32 * c;
      if (f >= p.M) continue;
      float o = v[c];
      if (f < p.qk_dim) {
        const float2 cs = pre.cs[c];
        const float w = v[c ^ PAIR];
        // the first half of each head subtracts the partner, the second adds it
        o = ((c & PAIR) == 0) ? (v[c] * cs.x - w * cs.y) : (v[c] * cs.x + w * cs.y);
      }
      p.qkv[(size_t)g * p.ld + f] = from_f32<TAct>(o);
    }
  }
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4],
                                               const Pre& pre) {
    if (p.hd == 128)
      rotate_store<2>(p, g, m0, lane, v, pre);
    else
      rotate_store<1>(p, g, m0, lane, v, pre);
  }
};

// Output projection of every row plus the branch's own residual:
// h[g] = H[g] + attn[g] W_o.
struct EpiResidual {
  struct Params {
    float* h;
    const float* H;
    int ld;
  };
  struct Pre {
    float H[4];
  };
  static __device__ __forceinline__ void prefetch(const Params& p, int g, int m0, int lane, Pre& pre) {
#pragma unroll
    for (int c = 0; c < 4; ++c) pre.H[c] = p.H[(size_t)g * p.ld + m0 + lane + 32 * c];
  }
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4],
                                               const Pre& pre) {
#pragma unroll
    for (int c = 0; c < 4; ++c) p.h[(size_t)g * p.ld + m0 + lane + 32 * c] = pre.H[c] + v[c];
  }
};

// Gate/up tile t = m0 / 128 holds gate features 64t..64t+63 in its first half
// and the matching up features in its second half; u = silu(gate) * up.
template <typename TAct>
struct EpiSwiGLU {
  struct Params {
    TAct* u;
    int ld;
  };
  struct Pre {};
  static __device__ __forceinline__ void prefetch(const Params&, int, int, int, Pre&) {}
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4],
                                               const Pre&) {
    const int t = m0 >> 7;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = lane + 32 * c;
      p.u[(size_t)g * p.ld + t * 64 + j] = from_f32<TAct>(silu(v[c]) * v[c + 2]);
    }
  }
};

// Plain fp32 store (down projection of the recompute rows, and the kernel
// test entry point).
struct EpiStore {
  struct Params {
    float* y;
    int ld;
  };
  struct Pre {};
  static __device__ __forceinline__ void prefetch(const Params&, int, int, int, Pre&) {}
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4],
                                               const Pre&) {
#pragma unroll
    for (int c = 0; c < 4; ++c) p.y[(size_t)g * p.ld + m0 + lane + 32 * c] = v[c];
  }
};

// Epilogue of up to 32 rows row0 + stride * jj, jj < nvalid; epilogue warp ew
// handles jj = ew + 4b (b = 0..7).  epilogue_prefetch() issues the global reads
// of all of them (it can run before the accumulators are ready, e.g. while the
// main loop streams the weights); epilogue_apply() consumes them, with getv(jj,
// v) supplying the fp32 accumulators of row jj for this lane's four features.
template <class Epi>
__device__ __forceinline__ void epilogue_prefetch(const typename Epi::Params& ep, int row0, int stride, int nvalid,
                                                  int m0, int ew, int lane, typename Epi::Pre (&pre)[8]) {
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const int jj = ew + 4 * b;
    if (jj < nvalid) Epi::prefetch(ep, row0 + jj * stride, m0, lane, pre[b]);
  }
}

template <class Epi, class GetV>
__device__ __forceinline__ void epilogue_apply(const typename Epi::Params& ep, int row0, int stride, int nvalid,
                                               int m0, int ew, int lane, const typename Epi::Pre (&pre)[8],
                                               GetV getv) {
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const int jj = ew + 4 * b;
    if (jj < nvalid) {
      float vv[4];
      getv(jj, vv);
      Epi::apply(ep, row0 + jj * stride, m0, lane, vv, pre[b]);
    }
  }
}

}  // namespace sf
