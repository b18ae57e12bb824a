// GEMM epilogues of the folded layer.  Each works on one output row g and one
// 128-wide tile of output features [m0, m0 + 128): lane l of a warp holds the
// fp32 accumulators of features m0 + l + 32c, c = 0..3, so the rotary pair
// (j, j + hd/2) of a head and the gate/up pair of a SwiGLU tile sit in the
// same thread for hd in {64, 128}.
//
// prefetch() issues the row's global reads (residual input, rotary table)
// and apply() consumes them, so a warp can start the reads of several rows
// before it waits on any of them.  An epilogue with kStaged set copies the
// small tables it reads into shared memory once per tile instead (stage(),
// while the main loop runs), so its rows read only shared memory.
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
    // bound by stage(): the rotary rows of positions P..P+L-1 and the block
    // position n of rows row_base.. in shared memory (null: global reads)
    const float2* s_cs = nullptr;
    const int* s_n = nullptr;
    int row_base = 0;
  };
  struct Pre {
    float2 cs[4];
  };
  static constexpr bool kStaged = true;
  // shared memory of the staged tables for a tile of up to 256 rows
  static __host__ __device__ int stage_bytes(const Params& p) { return p.L * (p.hd >> 1) * 8 + 256 * 4; }
  // Run by the 128 epilogue threads (t = 0..127) of a tile of n_rows rows
  // from row0; the rows sit at P + n with n < L, so L rotary rows cover all.
  static __device__ __forceinline__ void stage(Params& p, unsigned char* sm, int row0, int n_rows, int t) {
    const int nf4 = p.L * (p.hd >> 1) / 2;  // float2 pairs as float4
    float4* cs = reinterpret_cast<float4*>(sm);
    int* sn = reinterpret_cast<int*>(sm + (size_t)nf4 * 16);
    const float4* src = reinterpret_cast<const float4*>(p.rope + (size_t)p.P * (p.hd >> 1));
    for (int i = t; i < nf4; i += 128) cs[i] = src[i];
    for (int j = t; j < n_rows; j += 128) sn[j] = p.rc[row0 + j] % p.L;
    p.s_cs = reinterpret_cast<const float2*>(cs);
    p.s_n = sn;
    p.row_base = row0;
  }
  static __device__ __forceinline__ void prefetch(const Params& p, int g, int m0, int lane, Pre& pre) {
    const int half = p.hd >> 1;
    // m0 is a multiple of 128 and hd divides 128, so j % half = (lane + 32c) % half
    const float2* row = p.s_cs ? p.s_cs + (size_t)p.s_n[g - p.row_base] * half
                               : p.rope + (size_t)(p.P + (p.rc[g] % p.L)) * half;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int f = m0 + lane + 32 * c;
      pre.cs[c] = f < p.qk_dim ? row[(lane + 32 * c) & (half - 1)] : make_float2(1.f, 0.f);
    }
  }
  // hd = 128: a tile is one head, feature l + 32c pairs with l + 32(c ^ 2);
  // hd = 64: a tile is two heads, the pair is l + 32(c ^ 1).  Both partners
  // are register operands and the choice is a select, so one copy of the code
  // serves both widths.
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4],
                                               const Pre& pre) {
    const bool h128 = p.hd == 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int f = m0 + lane + 32 * c;
      if (f >= p.M) continue;
      float o = v[c];
      if (f < p.qk_dim) {
        const float2 cs = pre.cs[c];
        const float w = h128 ? v[c ^ 2] : v[c ^ 1];
        // the first half of each head subtracts the partner, the second adds it
        const bool first = h128 ? (c & 2) == 0 : (c & 1) == 0;
        o = first ? (v[c] * cs.x - w * cs.y) : (v[c] * cs.x + w * cs.y);
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
  struct Pre {
    float H[4];
  };
  static constexpr bool kStaged = false;
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
  static constexpr bool kStaged = false;
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
  static constexpr bool kStaged = false;
  static __device__ __forceinline__ void prefetch(const Params&, int, int, int, Pre&) {}
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4],
                                               const Pre&) {
#pragma unroll
    for (int c = 0; c < 4; ++c) p.y[(size_t)g * p.ld + m0 + lane + 32 * c] = v[c];
  }
};

// Greedy-token partial of the LM head: for output row g and the 128 vocabulary
// entries [m0, m0 + 128) of this tile, the largest logit and its index (the
// lowest index on a tie; entries at or past `vocab` are zero padding of the
// packed weight and are skipped), stored at part[g * ld + m0 / 128] as
// (value, index bits).  All 32 lanes of the warp take part.
struct EpiArgmax {
  struct Params {
    float2* part;
    int ld;     // vocabulary tiles per row
    int vocab;
  };
  struct Pre {};
  static constexpr bool kStaged = false;
  static __device__ __forceinline__ void prefetch(const Params&, int, int, int, Pre&) {}
  static __device__ __forceinline__ void apply(const Params& p, int g, int m0, int lane, const float v[4],
                                               const Pre&) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // features rise with c, so the first maximum wins
      const int f = m0 + lane + 32 * c;
      if (f < p.vocab && (v[c] > best || bi == 0x7fffffff)) {
        best = v[c];
        bi = f;
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
    if (lane == 0) p.part[(size_t)g * p.ld + (m0 >> 7)] = make_float2(best, __int_as_float(bi));
  }
};

// Epilogue of up to 32 rows row0 + stride * jj, jj < nvalid; epilogue warp ew
// handles jj = ew + 4b (b = 0..7).  epilogue_prefetch() issues the global reads
// of all of them (it can run before the accumulators are ready, e.g. while the
// main loop streams the weights); epilogue_apply() consumes them, with getv(jj,
// v) supplying the fp32 accumulators of row jj for this lane's four features.
//
// The epilogue runs once per CTA, so its code is fetched cold: an epilogue
// whose per-row reads are cheap (none, or staged in shared memory) runs its
// rows in a rolled loop and reads them just before use; only one with global
// reads per row keeps eight unrolled rows and their reads in registers.
template <class Epi>
constexpr bool epilogue_rolled() {
  return Epi::kStaged || sizeof(typename Epi::Pre) <= 1;
}

template <class Epi>
__device__ __forceinline__ void epilogue_prefetch(const typename Epi::Params& ep, int row0, int stride, int nvalid,
                                                  int m0, int ew, int lane, typename Epi::Pre (&pre)[8]) {
  if constexpr (!epilogue_rolled<Epi>()) {  // a rolled epilogue reads each row just before use
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int jj = ew + 4 * b;
      if (jj < nvalid) Epi::prefetch(ep, row0 + jj * stride, m0, lane, pre[b]);
    }
  }
}

template <class Epi, class GetV>
__device__ __forceinline__ void epilogue_apply(const typename Epi::Params& ep, int row0, int stride, int nvalid,
                                               int m0, int ew, int lane, const typename Epi::Pre (&pre)[8],
                                               GetV getv) {
  if constexpr (epilogue_rolled<Epi>()) {
#pragma unroll 1
    for (int jj = ew; jj < nvalid; jj += 4) {
      typename Epi::Pre one;
      Epi::prefetch(ep, row0 + jj * stride, m0, lane, one);
      float vv[4];
      getv(jj, vv);
      Epi::apply(ep, row0 + jj * stride, m0, lane, vv, one);
    }
  } else {
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
}

}  // namespace sf
