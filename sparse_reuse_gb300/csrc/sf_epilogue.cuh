// GEMM epilogues of the folded layer.  Each works on one output row g and one
// 128-wide tile of output features [m0, m0 + 128): lane l of a warp holds the
// fp32 accumulators of features m0 + l + 32c, c = 0..3, so the rotary pair
// (j, j + hd/2) of a head and the gate/up pair of a SwiGLU tile sit in the
// same thread for hd in {64, 128}.
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
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4]) {
    const int pos = p.P + (p.rc[g] % p.L);
    const int half = p.hd >> 1;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int f = m0 + lane + 32 * c;
      if (f >= p.M) continue;
      float o = v[c];
      if (f < p.qk_dim) {
        const int j = f % p.hd;
        const int pc = (p.hd == 128) ? (c ^ 2) : (c ^ 1);
        const float2 cs = p.rope[(size_t)pos * half + (j % half)];
        o = (j < half) ? (v[c] * cs.x - v[pc] * cs.y) : (v[c] * cs.x + v[pc] * cs.y);
      }
      p.qkv[(size_t)g * p.ld + f] = from_f32<TAct>(o);
    }
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
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const size_t o = (size_t)g * p.ld + m0 + lane + 32 * c;
      p.h[o] = p.H[o] + v[c];
    }
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
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4]) {
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
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) p.y[(size_t)g * p.ld + m0 + lane + 32 * c] = v[c];
  }
};

}  // namespace sf
