// Gate, compaction and source resolution of one folded layer, plus the row
// kernels around the GEMMs (RMSNorm gather, final residual) and the weight
// repacking done at context creation.
//
// Gate: "SpecFold" (arXiv 2610.04875v2 summary) §3.1-§3.2 and App. B — every
// draft position is gated by the parent-child relative residual
// rho = ||H_i[n] - H_par(i)[n]|| / ||H_par(i)[n]|| (formula as printed in the
// onedev.kr review, "What is different"); rho <= delta folds; the main branch
// bypasses the gate.  Compaction: App. B, recomputed indices go to a global
// and per-branch list.  Resolution: §A.3 / App. B, a folded position follows
// its chain to the nearest ancestor that recomputed it.
#include <cmath>
#include <mutex>

#include "sf_internal.h"
#include "specfold_kernels.h"

namespace sf {
namespace {

constexpr int kGateThreads = 256;  // every kernel of this file

// One row of the layer input in fp32, 4 features at column c4 * 4.
template <bool kLayer0, typename TIn>
__device__ __forceinline__ float4 layer_input4(const GateArgs& a, int row, int c4) {
  if constexpr (kLayer0) {
    return load4<TIn>(reinterpret_cast<const TIn*>(a.x_in) + (size_t)row * a.d + c4 * 4);
  } else {
    // the previous layer's last residual add: H = h + f[source slot]
    const int s = a.rcslot_prev[row];
    const float4 x = *reinterpret_cast<const float4*>(a.h_prev + (size_t)row * a.d + c4 * 4);
    const float4 f = *reinterpret_cast<const float4*>(a.f_prev + (size_t)s * a.d + c4 * 4);
    return make_float4(x.x + f.x, x.y + f.y, x.z + f.z, x.w + f.w);
  }
}

// Exclusive scan over the block of one int per thread; returns the prefix and
// writes the total to *total.  `tmp` holds 32 ints.
__device__ int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) tmp[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int base = warp > 0 ? tmp[warp - 1] : 0;
  *total = tmp[nw - 1];
  return base + x - v;
}

// Compaction (stable, ascending row id): the recompute list, the slot of every
// recompute row (its own source slot) and the per-request offsets.  Run by the
// last thread block of the gate kernel once every fold flag is in memory;
// slot[] (shared) receives each row's slot, -1 for a folded row.
__device__ void compact(const GateArgs& a, uint8_t* flags, int* slot, int* tmp) {
  const int T = a.T, L = a.L, Bp = a.tree.Bp, R = a.tree.R;
  for (int row = threadIdx.x; row < T; row += blockDim.x) flags[row] = __ldcg(a.fold + row);
  __syncthreads();
  const int chunk = (T + blockDim.x - 1) / blockDim.x;
  const int lo = min(T, (int)threadIdx.x * chunk), hi = min(T, lo + chunk);
  int cnt = 0;
  for (int row = lo; row < hi; ++row) cnt += flags[row] ? 0 : 1;
  int total = 0;
  int s = block_exclusive_scan(cnt, tmp, &total);
  for (int row = lo; row < hi; ++row) {
    if (!flags[row]) {
      slot[row] = s;
      a.rc[s] = row;
      a.rcslot[row] = s;
      if (a.rc_user) a.rc_user[s] = row;
      ++s;
    } else {
      slot[row] = -1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.meta[0] = total;
    for (int r = 0; r < R; ++r) a.meta[1 + r] = slot[r * Bp * L];  // main row n = 0 always recomputes
    a.meta[1 + R] = total;
    if (a.rc_count_user) *a.rc_count_user = total;
  }
}

// Source resolution of the folded rows (a folded (i, n) follows its chain to
// the nearest ancestor that recomputed n) and every row's source branch.
__device__ void resolve(const GateArgs& a, const uint8_t* flags, const int* slot) {
  const int T = a.T, L = a.L, Bp = a.tree.Bp;
  for (int row = threadIdx.x; row < T; row += blockDim.x) {
    const int n = row % L, rb = row / L, i = rb % Bp, r = rb / Bp;
    int b = i, steps = 0;
    while (flags[(r * Bp + b) * L + n]) {
      b = a.tree.parent[r * Bp + b];
      if (b < 0 || ++steps > Bp) {  // cannot happen for a validated tree
        raise_error(a.err, kErrGate);
        b = 0;
        break;
      }
    }
    if (b != i) {
      const int sl = slot[(r * Bp + b) * L + n];
      if (sl < 0) raise_error(a.err, kErrGate);
      a.rcslot[row] = sl < 0 ? 0 : sl;
    }
    if (a.src_user) a.src_user[row] = b;
  }
}

__device__ void compact_and_resolve(const GateArgs& a, uint8_t* flags, int* slot, int* tmp) {
  compact(a, flags, slot, tmp);
  resolve(a, flags, slot);
}

// One block per row (r, i, n): the row's layer input H (previous layer's
// residual applied) and its gate decision against the parent row.  For short
// rows (VEC > 0) every thread first loads its VEC float4 of the row and of the
// parent row, then reduces and stores them, so all its loads are in flight at
// once; long rows (VEC == 0) are streamed in a loop at full occupancy.
template <bool kLayer0, typename TIn, int VEC>
__global__ void __launch_bounds__(kGateThreads) gate_kernel(const __grid_constant__ GateArgs a) {
  __shared__ float red[32];
  __shared__ int tmp[32];
  __shared__ bool is_last;
  extern __shared__ __align__(16) unsigned char dyn[];
  pdl_wait();
  pdl_trigger();

  const int row = blockIdx.x;
  const int L = a.L, Bp = a.tree.Bp;
  const int n = row % L, rb = row / L, i = rb % Bp, r = rb / Bp;
  const int prow = i > 0 ? (r * Bp + a.tree.parent[r * Bp + i]) * L + n : -1;
  const int d4 = a.d >> 2;

  float diff2 = 0.f, par2 = 0.f;
  if constexpr (VEC > 0) {
    float4 xs[VEC], ys[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int c = threadIdx.x + k * blockDim.x;
      if (c < d4) {
        xs[k] = layer_input4<kLayer0, TIn>(a, row, c);
        // the parent's input is recomputed from the same operands, so it is
        // bit-identical to what the parent's block writes
        if (prow >= 0) ys[k] = layer_input4<kLayer0, TIn>(a, prow, c);
      }
    }
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int c = threadIdx.x + k * blockDim.x;
      if (c < d4) {
        const float4 x = xs[k];
        *reinterpret_cast<float4*>(a.H_out + (size_t)row * a.d + c * 4) = x;
        if (a.dbg) *reinterpret_cast<float4*>(a.dbg + (size_t)row * a.d + c * 4) = x;
        if (prow >= 0) {
          const float4 y = ys[k];
          const float dx = x.x - y.x, dy = x.y - y.y, dz = x.z - y.z, dw = x.w - y.w;
          diff2 += dx * dx + dy * dy + dz * dz + dw * dw;
          par2 += y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
        }
      }
    }
  } else {
    // long rows: stream the row at full occupancy
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      const float4 x = layer_input4<kLayer0, TIn>(a, row, c);
      *reinterpret_cast<float4*>(a.H_out + (size_t)row * a.d + c * 4) = x;
      if (a.dbg) *reinterpret_cast<float4*>(a.dbg + (size_t)row * a.d + c * 4) = x;
      if (prow >= 0) {
        const float4 y = layer_input4<kLayer0, TIn>(a, prow, c);
        const float dx = x.x - y.x, dy = x.y - y.y, dz = x.z - y.z, dw = x.w - y.w;
        diff2 += dx * dx + dy * dy + dz * dz + dw * dw;
        par2 += y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
      }
    }
  }
  if (prow >= 0) {
    diff2 = block_sum(diff2, red);
    par2 = block_sum(par2, red);
  }
  if (threadIdx.x == 0) {
    // rho <= delta  <=>  ||diff||^2 <= delta^2 ||parent||^2 (covers a zero parent)
    const uint8_t f = (prow >= 0 && a.delta > 0.f && diff2 <= a.delta * a.delta * par2) ? 1 : 0;
    a.fold[row] = f;
    if (a.fold_user) a.fold_user[row] = f;
    // only the flag has to be visible before this block's ticket is counted
    __threadfence();
    is_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  uint8_t* flags = dyn;
  int* slot = reinterpret_cast<int*>(dyn + ((a.T + 15) & ~15));
  compact_and_resolve(a, flags, slot, tmp);
  __syncthreads();
  if (threadIdx.x == 0) {
    *a.ticket = 0u;
    // a resolution check that fired is reported through the count as well
    if (a.rc_count_user && a.err && (atomicOr(a.err, 0u) & kErrGate)) *a.rc_count_user = -1;
  }
}

// ---------------------------------------------------------------- fused gate

// Tag of this layer of this pass: (pass epoch * 1024 + layer) * 2 + 1 is
// unique to it (at most 1024 layers) and never zero, so the rows' scan words
// need no clearing between layers or passes.
__device__ __forceinline__ unsigned scan_tag(const GateArgs& a) {
  return ((*a.epoch) * 1024u + (unsigned)a.layer) * 2u + 1u;
}

// A row's gate word: the layer's tag in the high half, and in bit 0 whether
// the row recomputes.
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long gate_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr unsigned long long kScanWaitNs = 2000000000ull;  // a wait that gives up raises kErrTimeout

// Whether row j recomputes (bit 0 of its word, once the word carries this
// layer's tag; spinning, bounded).  `v` is a first read of the word.  A wait
// that gives up raises kErrTimeout and answers "recomputes", so the caller
// still finishes with in-range values.
__device__ __noinline__ unsigned gate_word_wait(const GateArgs& a, int j, unsigned tag, unsigned long long v) {
  const unsigned long long t0 = gate_timer_ns();
  while ((unsigned)(v >> 32) != tag) {
    __nanosleep(64);
    v = ld_acquire_u64(a.scan + j);
    if ((unsigned)(v >> 32) != tag && gate_timer_ns() - t0 > kScanWaitNs) {
      raise_error(a.err, kErrTimeout);
      return 1u;
    }
  }
  return (unsigned)v & 1u;
}

__device__ __forceinline__ unsigned gate_word(const GateArgs& a, int j, unsigned tag) {
  const unsigned long long v = ld_acquire_u64(a.scan + j);
  return (unsigned)(v >> 32) == tag ? ((unsigned)v & 1u) : gate_word_wait(a, j, tag, v);
}

// Gate, compaction, source resolution and attention RMSNorm of one layer in
// one launch, one CTA per row.  Each CTA takes an arrival ticket and handles
// row = ticket, so rows are handed out in ascending order and every lower row
// belongs to a CTA that is already running:
//   1. the row's layer input H (previous layer's residual applied, written
//      out) and its gate decision against the parent row: VEC float4 columns
//      a thread (256 threads cover rows of up to VEC * 1024 features), every
//      load of the row and of its parent row issued before the first is used;
//   2. it publishes the decision in its gate word (release);
//   3. warp 0 finds the row's source, the nearest row up its chain (itself,
//      its parent's row, ...) that recomputes, from those rows' words, and the
//      CTA counts the recompute rows below the row and below the source from
//      the words of all lower rows (256 threads read them at once): the counts
//      are the slots of the row and of its source in the stable ascending
//      recompute list;
//   4. a recompute row writes its list entry and its normalised row at its
//      slot, from the registers that still hold H.
// A CTA waits only for lower rows, whose CTAs never wait for higher ones, so
// every wait ends whatever the number of resident CTAs; the waits are
// bounded all the same.
template <bool kLayer0, typename TIn, int VEC, typename TAct>
__global__ void __launch_bounds__(kGateThreads, VEC <= 2 ? 5 : 3) gate_scan_kernel(const __grid_constant__ GateArgs a) {
  __shared__ float red[3][32];
  __shared__ int cnt[2][32];
  __shared__ int s_row, s_srow, s_src, s_slot;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    const unsigned t = atomicAdd(a.ticket, 1u);
    if (t == (unsigned)a.T - 1u) *a.ticket = 0u;  // every ticket of this launch is taken
    s_row = (int)t;
  }
  __syncthreads();
  const int row = s_row;
  const int L = a.L, Bp = a.tree.Bp;
  const int n = row % L, rb = row / L, i = rb % Bp, r = rb / Bp;
  const int prow = i > 0 ? (r * Bp + a.tree.parent[r * Bp + i]) * L + n : -1;
  const int d4 = a.d >> 2;
  const unsigned tag = scan_tag(a);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kGateThreads / 32;

  // 1. the layer input of the row and of its parent row
  float4 xs[VEC], ys[VEC];
  if constexpr (kLayer0) {
    const TIn* xr = reinterpret_cast<const TIn*>(a.x_in) + (size_t)row * a.d;
    const TIn* yr = reinterpret_cast<const TIn*>(a.x_in) + (size_t)(prow >= 0 ? prow : row) * a.d;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int c = threadIdx.x + k * kGateThreads;
      if (c < d4) {
        xs[k] = load4<TIn>(xr + c * 4);
        if (prow >= 0) ys[k] = load4<TIn>(yr + c * 4);
      }
    }
  } else {
    // the previous layer's last residual add: H = h + f[source slot]; the
    // parent's input is recomputed from the same operands, so it is
    // bit-identical to what the parent's CTA writes
    const float4* hx = reinterpret_cast<const float4*>(a.h_prev + (size_t)row * a.d);
    const float4* fx = reinterpret_cast<const float4*>(a.f_prev + (size_t)a.rcslot_prev[row] * a.d);
    const float4* hy = reinterpret_cast<const float4*>(a.h_prev + (size_t)(prow >= 0 ? prow : row) * a.d);
    const float4* fy =
        reinterpret_cast<const float4*>(a.f_prev + (size_t)a.rcslot_prev[prow >= 0 ? prow : row] * a.d);
    float4 fxs[VEC], fys[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int c = threadIdx.x + k * kGateThreads;
      if (c < d4) {
        xs[k] = hx[c];
        fxs[k] = fx[c];
        if (prow >= 0) {
          ys[k] = hy[c];
          fys[k] = fy[c];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      xs[k] = make_float4(xs[k].x + fxs[k].x, xs[k].y + fxs[k].y, xs[k].z + fxs[k].z, xs[k].w + fxs[k].w);
      if (prow >= 0)
        ys[k] = make_float4(ys[k].x + fys[k].x, ys[k].y + fys[k].y, ys[k].z + fys[k].z, ys[k].w + fys[k].w);
    }
  }
  float diff2 = 0.f, par2 = 0.f, ss = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int c = threadIdx.x + k * kGateThreads;
    if (c < d4) {
      const float4 x = xs[k];
      *reinterpret_cast<float4*>(a.H_out + (size_t)row * a.d + c * 4) = x;
      if (a.dbg) *reinterpret_cast<float4*>(a.dbg + (size_t)row * a.d + c * 4) = x;
      ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
      if (prow >= 0) {
        const float4 y = ys[k];
        const float dx = x.x - y.x, dy = x.y - y.y, dz = x.z - y.z, dw = x.w - y.w;
        diff2 += dx * dx + dy * dy + dz * dz + dw * dw;
        par2 += y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
      }
    }
  }
  // the three sums in one exchange, added in the same order as block_sum
  diff2 = warp_sum(diff2);
  par2 = warp_sum(par2);
  ss = warp_sum(ss);
  if (lane == 0) {
    red[0][warp] = diff2;
    red[1][warp] = par2;
    red[2][warp] = ss;
  }
  __syncthreads();
  diff2 = warp_sum(lane < kWarps ? red[0][lane] : 0.f);
  par2 = warp_sum(lane < kWarps ? red[1][lane] : 0.f);
  ss = warp_sum(lane < kWarps ? red[2][lane] : 0.f);
  // rho <= delta  <=>  ||diff||^2 <= delta^2 ||parent||^2 (covers a zero parent)
  const int f = (prow >= 0 && a.delta > 0.f && diff2 <= a.delta * a.delta * par2) ? 1 : 0;

  // 2. the decision
  if (threadIdx.x == 0) {
    a.fold[row] = (uint8_t)f;
    if (a.fold_user) a.fold_user[row] = (uint8_t)f;
    if (a.rho_user)
      a.rho_user[row] = prow < 0 ? __int_as_float(0x7fc00000)
                                 : (par2 > 0.f ? sqrtf(diff2 / par2) : (diff2 > 0.f ? __int_as_float(0x7f800000) : 0.f));
    if (!(a.stall && row == 0))  // failure injection: row 0 never reports
      st_release_u64(a.scan + row, ((unsigned long long)tag << 32) | (f ? 0u : 1u));
  }

  // 3. the source, then the recompute rows below the row and below the source
  if (warp == 0) {
    if (!f) {
      if (lane == 0) {
        s_srow = row;
        s_src = i;
      }
    } else {
      // lane k reads the word of the k-th row up the chain from the parent
      // (32 at a time); the main branch always recomputes
      int start = a.tree.parent[r * Bp + i];
      for (;;) {
        int b = start;
        for (int k = 0; k < lane && b >= 0; ++k) b = a.tree.parent[r * Bp + b];
        const bool on = b >= 0;
        const unsigned rc = on ? gate_word(a, (r * Bp + b) * L + n, tag) : 0u;
        const unsigned hits = __ballot_sync(0xffffffffu, on && rc);
        if (hits) {
          const int src = __shfl_sync(0xffffffffu, b, __ffs(hits) - 1);
          if (lane == 0) {
            s_srow = (r * Bp + src) * L + n;
            s_src = src;
          }
          break;
        }
        const int last = __shfl_sync(0xffffffffu, b, 31);
        start = last >= 0 ? a.tree.parent[r * Bp + last] : -1;
        if (start < 0) {  // cannot happen for a validated tree
          if (lane == 0) {
            raise_error(a.err, kErrGate);
            s_srow = r * Bp * L + n;
            s_src = 0;
          }
          break;
        }
      }
    }
  }
  __syncthreads();
  const int srow = s_srow;
  int below = 0, below_src = 0;
  for (int j0 = 0; j0 < row; j0 += 4 * kGateThreads) {
    unsigned long long w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = j0 + threadIdx.x + k * kGateThreads;
      w[k] = j < row ? ld_acquire_u64(a.scan + j) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = j0 + threadIdx.x + k * kGateThreads;
      if (j < row) {
        const unsigned rc = (unsigned)(w[k] >> 32) == tag ? ((unsigned)w[k] & 1u) : gate_word_wait(a, j, tag, w[k]);
        below += rc;
        below_src += j < srow ? rc : 0;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    below += __shfl_xor_sync(0xffffffffu, below, o);
    below_src += __shfl_xor_sync(0xffffffffu, below_src, o);
  }
  if (lane == 0) {
    cnt[0][warp] = below;
    cnt[1][warp] = below_src;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tot = 0, tot_src = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      tot += cnt[0][w];
      tot_src += cnt[1][w];
    }
    const int slot = f ? tot_src : tot;
    if (!f) {
      a.rc[slot] = row;
      if (a.rc_user) a.rc_user[slot] = row;
      if (i == 0 && n == 0) a.meta[1 + r] = slot;  // first recompute row of request r
    }
    a.rcslot[row] = slot;
    if (a.src_user) a.src_user[row] = s_src;
    if (row == a.T - 1) {
      const int total = tot + (f ? 0 : 1);
      a.meta[0] = total;
      a.meta[1 + a.tree.R] = total;
      if (a.rc_count_user) *a.rc_count_user = total;
    }
    s_slot = slot;
  }
  if (f) return;
  __syncthreads();

  // 4. the normalised row of a recompute row
  const float rstd = rsqrtf(ss / (float)a.d + a.eps);
  TAct* out = reinterpret_cast<TAct*>(a.xn) + (size_t)s_slot * a.d;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int c = threadIdx.x + k * kGateThreads;
    if (c < d4) {
      const float4 v = xs[k];
      const float4 w = *reinterpret_cast<const float4*>(a.gain + c * 4);
      store4<TAct>(out + c * 4, make_float4(v.x * rstd * w.x, v.y * rstd * w.y, v.z * rstd * w.z, v.w * rstd * w.w));
    }
  }
}

// Wide rows (more than 4 float4 a thread): the gate in two launches, which
// overlap better than one kernel whose register-heavy CTAs run in several
// waves.
//
// Gate, part 1: the layer input and the gate decision of every row.  CTA =
// one row, VEC float4 columns per thread (256 threads cover rows of up to
// VEC * 1024 features), every load of the row and of its parent row issued
// before the first is used: the row's layer input H (previous layer's
// residual applied, written out), ||H - H_parent||^2, ||H_parent||^2 and
// ||H||^2, the fold decision, and the row's gate word (release).  Nothing
// here waits, so every CTA finishes whatever else is resident.
template <bool kLayer0, typename TIn, int VEC>
__global__ void __launch_bounds__(kGateThreads) gate_rows_kernel(const __grid_constant__ GateArgs a) {
  __shared__ float red[3][32];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const int L = a.L, Bp = a.tree.Bp;
  const int n = row % L, rb = row / L, i = rb % Bp, r = rb / Bp;
  const int prow = i > 0 ? (r * Bp + a.tree.parent[r * Bp + i]) * L + n : -1;
  const int d4 = a.d >> 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  float4 xs[VEC], ys[VEC];
  if constexpr (kLayer0) {
    const TIn* xr = reinterpret_cast<const TIn*>(a.x_in) + (size_t)row * a.d;
    const TIn* yr = reinterpret_cast<const TIn*>(a.x_in) + (size_t)(prow >= 0 ? prow : row) * a.d;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int c = threadIdx.x + k * kGateThreads;
      if (c < d4) {
        xs[k] = load4<TIn>(xr + c * 4);
        if (prow >= 0) ys[k] = load4<TIn>(yr + c * 4);
      }
    }
  } else {
    // the previous layer's last residual add: H = h + f[source slot]; the
    // parent's input is recomputed from the same operands, so it is
    // bit-identical to what the parent's CTA writes
    const float4* hx = reinterpret_cast<const float4*>(a.h_prev + (size_t)row * a.d);
    const float4* fx = reinterpret_cast<const float4*>(a.f_prev + (size_t)a.rcslot_prev[row] * a.d);
    const float4* hy = reinterpret_cast<const float4*>(a.h_prev + (size_t)(prow >= 0 ? prow : row) * a.d);
    const float4* fy =
        reinterpret_cast<const float4*>(a.f_prev + (size_t)a.rcslot_prev[prow >= 0 ? prow : row] * a.d);
    float4 fxs[VEC], fys[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int c = threadIdx.x + k * kGateThreads;
      if (c < d4) {
        xs[k] = hx[c];
        fxs[k] = fx[c];
        if (prow >= 0) {
          ys[k] = hy[c];
          fys[k] = fy[c];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      xs[k] = make_float4(xs[k].x + fxs[k].x, xs[k].y + fxs[k].y, xs[k].z + fxs[k].z, xs[k].w + fxs[k].w);
      if (prow >= 0)
        ys[k] = make_float4(ys[k].x + fys[k].x, ys[k].y + fys[k].y, ys[k].z + fys[k].z, ys[k].w + fys[k].w);
    }
  }
  float diff2 = 0.f, par2 = 0.f, ss = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int c = threadIdx.x + k * kGateThreads;
    if (c < d4) {
      const float4 x = xs[k];
      *reinterpret_cast<float4*>(a.H_out + (size_t)row * a.d + c * 4) = x;
      if (a.dbg) *reinterpret_cast<float4*>(a.dbg + (size_t)row * a.d + c * 4) = x;
      ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
      if (prow >= 0) {
        const float4 y = ys[k];
        const float dx = x.x - y.x, dy = x.y - y.y, dz = x.z - y.z, dw = x.w - y.w;
        diff2 += dx * dx + dy * dy + dz * dz + dw * dw;
        par2 += y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
      }
    }
  }
  // the three sums in one exchange, added in the same order as block_sum
  diff2 = warp_sum(diff2);
  par2 = warp_sum(par2);
  ss = warp_sum(ss);
  if (lane == 0) {
    red[0][warp] = diff2;
    red[1][warp] = par2;
    red[2][warp] = ss;
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  constexpr int kWarps = kGateThreads / 32;
  diff2 = par2 = ss = 0.f;
  // thread 0 adds the warps' sums as a warp_sum over lanes 0..7 would:
  // pairwise at distance 16, 8, 4, 2, 1 (zeros above lane 7)
  float d8[kWarps], p8[kWarps], s8[kWarps];
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    d8[w] = red[0][w];
    p8[w] = red[1][w];
    s8[w] = red[2][w];
  }
#pragma unroll
  for (int o = kWarps / 2; o > 0; o >>= 1)
#pragma unroll
    for (int w = 0; w < o; ++w) {
      d8[w] += d8[w + o];
      p8[w] += p8[w + o];
      s8[w] += s8[w + o];
    }
  diff2 = d8[0];
  par2 = p8[0];
  ss = s8[0];
  // rho <= delta  <=>  ||diff||^2 <= delta^2 ||parent||^2 (covers a zero parent)
  const int f = (prow >= 0 && a.delta > 0.f && diff2 <= a.delta * a.delta * par2) ? 1 : 0;
  a.fold[row] = (uint8_t)f;
  if (a.fold_user) a.fold_user[row] = (uint8_t)f;
  if (a.rho_user)
    a.rho_user[row] = prow < 0 ? __int_as_float(0x7fc00000)
                               : (par2 > 0.f ? sqrtf(diff2 / par2) : (diff2 > 0.f ? __int_as_float(0x7f800000) : 0.f));
  a.row_ss[row] = ss;
  // the release covers this row's H, which the CTA's barrier ordered before
  // it, and its sums
  __threadfence();
  if (!(a.stall && row == 0))  // failure injection: row 0 never reports
    st_release_u64(a.scan + row, ((unsigned long long)scan_tag(a) << 32) | (f ? 0u : 1u));
}

// Gate, part 2: compaction, source resolution and attention RMSNorm.  CTA =
// one row.  It starts while part 1 still runs (it lets its own dependants go
// at once and waits for part 1's completion only before it exits), and
// reads part 1's results through the rows' gate words (acquire, bounded
// spin): part 1 has all its CTAs running before this grid can start, and
// they never wait, so every word arrives.
//   - a folded row follows its chain up the tree (the ancestors are lower
//     rows at the same position) to the nearest ancestor that recomputes;
//   - the CTA counts the recompute rows below the row, and below its source,
//     from the words of all lower rows (256 threads read them at once): the
//     counts are the slots of the row and of its source in the stable
//     ascending recompute list;
//   - a recompute row writes its list entry and its normalised row at its
//     slot (H from part 1, through L2).
template <typename TAct>
__global__ void __launch_bounds__(kGateThreads) gate_compact_kernel(const __grid_constant__ GateArgs a) {
  __shared__ int cnt[2][32];
  __shared__ int s_srow, s_src, s_slot;
  pdl_trigger();
  const int row = blockIdx.x;
  const int L = a.L, Bp = a.tree.Bp;
  const int n = row % L, rb = row / L, i = rb % Bp, r = rb / Bp;
  const unsigned tag = scan_tag(a);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kGateThreads / 32;

  if (warp == 0) {
    // lane k reads the word of the k-th row up the chain (the row itself,
    // its parent's row, ...; 32 at a time); the source is the nearest one
    // that recomputes, and the main branch always does
    int start = i;
    for (;;) {
      int b = start;
      for (int k = 0; k < lane && b >= 0; ++k) b = a.tree.parent[r * Bp + b];
      const bool on = b >= 0;
      const unsigned rc = on ? gate_word(a, (r * Bp + b) * L + n, tag) : 0u;
      const unsigned hits = __ballot_sync(0xffffffffu, on && rc);
      if (hits) {
        const int src = __shfl_sync(0xffffffffu, b, __ffs(hits) - 1);
        if (lane == 0) {
          s_srow = (r * Bp + src) * L + n;
          s_src = src;
        }
        break;
      }
      const int next = __shfl_sync(0xffffffffu, b, 31);
      if (next < 0 || __shfl_sync(0xffffffffu, on, 31) == 0) {  // cannot happen for a validated tree
        if (lane == 0) {
          raise_error(a.err, kErrGate);
          s_srow = r * Bp * L + n;
          s_src = 0;
        }
        break;
      }
      start = a.tree.parent[r * Bp + next];
      if (start < 0) {
        if (lane == 0) {
          raise_error(a.err, kErrGate);
          s_srow = r * Bp * L + n;
          s_src = 0;
        }
        break;
      }
    }
  }
  __syncthreads();
  const int srow = s_srow;
  const bool own = srow == row;
  // recompute rows below this row and below the source row, 4 words a thread at a time
  int below = 0, below_src = 0;
  for (int j0 = 0; j0 < row; j0 += 4 * kGateThreads) {
    unsigned long long w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = j0 + threadIdx.x + k * kGateThreads;
      w[k] = j < row ? ld_acquire_u64(a.scan + j) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = j0 + threadIdx.x + k * kGateThreads;
      if (j < row) {
        const unsigned rc = (unsigned)(w[k] >> 32) == tag ? ((unsigned)w[k] & 1u) : gate_word_wait(a, j, tag, w[k]);
        below += rc;
        below_src += j < srow ? rc : 0;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    below += __shfl_xor_sync(0xffffffffu, below, o);
    below_src += __shfl_xor_sync(0xffffffffu, below_src, o);
  }
  if (lane == 0) {
    cnt[0][warp] = below;
    cnt[1][warp] = below_src;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tot = 0, tot_src = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      tot += cnt[0][w];
      tot_src += cnt[1][w];
    }
    const int slot = own ? tot : tot_src;
    if (own) {
      a.rc[slot] = row;
      if (a.rc_user) a.rc_user[slot] = row;
      if (i == 0 && n == 0) a.meta[1 + r] = slot;  // first recompute row of request r
    }
    a.rcslot[row] = slot;
    if (a.src_user) a.src_user[row] = s_src;
    if (row == a.T - 1) {
      const int total = tot + (own ? 1 : 0);
      a.meta[0] = total;
      a.meta[1 + a.tree.R] = total;
      if (a.rc_count_user) *a.rc_count_user = total;
    }
    s_slot = slot;
  }
  __syncthreads();
  if (own) {
    const int sl = s_slot;
    const float rstd = rsqrtf(__ldcg(a.row_ss + row) / (float)a.d + a.eps);
    const float4* Hrow = reinterpret_cast<const float4*>(a.H_out + (size_t)row * a.d);
    TAct* out = reinterpret_cast<TAct*>(a.xn) + (size_t)sl * a.d;
    for (int c = threadIdx.x; c < (a.d >> 2); c += kGateThreads) {
      const float4 v = __ldcg(Hrow + c);
      const float4 w = *reinterpret_cast<const float4*>(a.gain + c * 4);
      store4<TAct>(out + c * 4, make_float4(v.x * rstd * w.x, v.y * rstd * w.y, v.z * rstd * w.z, v.w * rstd * w.w));
    }
  }
  // part 1 has completed before this grid does, so every kernel after this
  // one sees both grids finished when its own dependency wait returns
  pdl_wait();
}

// RMSNorm of rows rc[g] (or g when rc is null), g < count, gathered into a
// dense [count][d] activation matrix.
template <typename TAct>
__global__ void __launch_bounds__(kGateThreads) rmsnorm_gather_kernel(const float* X, const int32_t* rc, const int32_t* count_ptr,
                                                             int max_rows, const float* gain, float eps, TAct* out,
                                                             int d, unsigned* err) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const int count = count_ptr ? *count_ptr : max_rows;
  const int d4 = d >> 2;
  for (int g = blockIdx.x; g < count; g += gridDim.x) {
    int row = rc ? rc[g] : g;
    if (row < 0 || row >= max_rows) {
      raise_error(err, kErrNorm);
      row = 0;
    }
    const float* x = X + (size_t)row * d;
    float ss = 0.f;
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      const float4 v = *reinterpret_cast<const float4*>(x + c * 4);
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum(ss, red);
    const float rstd = rsqrtf(ss / (float)d + eps);
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      const float4 v = *reinterpret_cast<const float4*>(x + c * 4);
      const float4 w = *reinterpret_cast<const float4*>(gain + c * 4);
      store4<TAct>(out + (size_t)g * d + c * 4,
                   make_float4(v.x * rstd * w.x, v.y * rstd * w.y, v.z * rstd * w.z, v.w * rstd * w.w));
    }
  }
}

// Last layer's residual add for every row, cast to the output type.
template <typename TOut>
__global__ void __launch_bounds__(kGateThreads) final_residual_kernel(const float* h, const float* f, const int32_t* rcslot,
                                                             TOut* out, float* dbg, int T, int d, unsigned* epoch,
                                                             unsigned* err) {
  pdl_wait();
  pdl_trigger();
  // every gate of this pass has completed: the next pass tags its decisions anew
  if (epoch && blockIdx.x == 0 && threadIdx.x == 0) *epoch += 1u;
  const int d4 = d >> 2;
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    int s = rcslot[row];
    if (s < 0 || s >= T) {
      raise_error(err, kErrResid);
      s = 0;
    }
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      const float4 x = *reinterpret_cast<const float4*>(h + (size_t)row * d + c * 4);
      const float4 y = *reinterpret_cast<const float4*>(f + (size_t)s * d + c * 4);
      const float4 o = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
      store4<TOut>(out + (size_t)row * d + c * 4, o);
      if (dbg) *reinterpret_cast<float4*>(dbg + (size_t)row * d + c * 4) = o;
    }
  }
}

// dst[map(n)][k] = src[k][n] for src [K][N]; map(n) = row_base + n, or with
// interleave = 1 (gate) / 2 (up): (n / 64) * 128 + (interleave - 1) * 64 + n % 64.
template <typename T>
__global__ void pack_transpose_kernel(const T* src, int K, int N, T* dst, int ld_dst, int row_base, int interleave) {
  __shared__ T tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {
    const int k = k0 + y, n = n0 + threadIdx.x;
    if (k < K && n < N) tile[y][threadIdx.x] = src[(size_t)k * N + n];
  }
  __syncthreads();
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {
    const int n = n0 + y, k = k0 + threadIdx.x;
    if (k < K && n < N) {
      const int drow = interleave ? (n / 64) * 128 + (interleave - 1) * 64 + (n % 64) : row_base + n;
      dst[(size_t)drow * ld_dst + k] = tile[threadIdx.x][y];
    }
  }
}

int grid_rows(int rows) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return rows < 8 * sms ? (rows > 0 ? rows : 1) : 8 * sms;
}

}  // namespace

namespace {

template <int VEC>
cudaError_t launch_gate_vec(Launch& lc, const GateArgs& a, int in_bf16, int threads, size_t dyn) {
  const dim3 grid(a.T), block(threads);
  if (a.x_in == nullptr) return launch_pdl(lc.st, grid, block, dyn, 1, gate_kernel<false, float, VEC>, a);
  if (in_bf16) return launch_pdl(lc.st, grid, block, dyn, 1, gate_kernel<true, __nv_bfloat16, VEC>, a);
  return launch_pdl(lc.st, grid, block, dyn, 1, gate_kernel<true, float, VEC>, a);
}

}  // namespace

cudaError_t launch_gate(Launch& lc, const GateArgs& a, int in_bf16) {
  const int d4 = a.d / 4;
  if (a.d % 4 != 0) return lc.err = cudaErrorInvalidValue;
  const size_t dyn = ((a.T + 15) & ~15) + (size_t)a.T * sizeof(int);
  // rows of up to 512 float4: 256 threads holding 2 float4 each (and 2 of the
  // parent); longer rows: the streaming loop
  lc.before(SF_K_GATE);
  if (d4 <= 512)
    lc.check(launch_gate_vec<2>(lc, a, in_bf16, kGateThreads, dyn));
  else
    lc.check(launch_gate_vec<0>(lc, a, in_bf16, kGateThreads, dyn));
  lc.after(SF_K_GATE);
  return lc.err;
}

namespace {

template <int VEC>
cudaError_t launch_gate_scan(Launch& lc, const GateArgs& a, int bf16) {
  // layer 0 reads the block input, which has the context dtype like the
  // normalised rows
  auto k = a.x_in == nullptr
               ? (bf16 ? gate_scan_kernel<false, float, VEC, __nv_bfloat16> : gate_scan_kernel<false, float, VEC, float>)
               : (bf16 ? gate_scan_kernel<true, __nv_bfloat16, VEC, __nv_bfloat16>
                       : gate_scan_kernel<true, float, VEC, float>);
  return launch_pdl(lc.st, dim3(a.T), dim3(kGateThreads), 0, 1, k, a);
}

}  // namespace

namespace {

template <int VEC>
cudaError_t launch_gate_rows(Launch& lc, const GateArgs& a, int bf16) {
  auto k = a.x_in == nullptr ? gate_rows_kernel<false, float, VEC>
                             : (bf16 ? gate_rows_kernel<true, __nv_bfloat16, VEC> : gate_rows_kernel<true, float, VEC>);
  return launch_pdl(lc.st, dim3(a.T), dim3(kGateThreads), 0, 1, k, a);
}

}  // namespace

cudaError_t launch_gate_norm(Launch& lc, const GateArgs& a, int bf16) {
  const int per = (a.d / 4 + kGateThreads - 1) / kGateThreads;  // float4 columns a thread
  if (a.d % 4 != 0 || per > 16 || !a.xn || !a.gain || !a.scan || !a.epoch || !a.ticket || !a.row_ss || a.T < 1)
    return lc.err = cudaErrorInvalidValue;
  if (per <= 4) {
    lc.before(SF_K_GATE);
    if (per <= 2)
      lc.check(launch_gate_scan<2>(lc, a, bf16));
    else
      lc.check(launch_gate_scan<4>(lc, a, bf16));
    lc.after(SF_K_GATE);
    return lc.err;
  }
  // wide rows: two launches, each bracketed (counted and, when selected,
  // timed) on its own
  lc.before(SF_K_GATE);
  if (per <= 6)
    lc.check(launch_gate_rows<6>(lc, a, bf16));
  else if (per <= 8)
    lc.check(launch_gate_rows<8>(lc, a, bf16));
  else
    lc.check(launch_gate_rows<16>(lc, a, bf16));
  lc.after(SF_K_GATE);
  lc.before(SF_K_GATE);
  lc.check(launch_pdl(lc.st, dim3(a.T), dim3(kGateThreads), 0, 1,
                      bf16 ? gate_compact_kernel<__nv_bfloat16> : gate_compact_kernel<float>, a));
  lc.after(SF_K_GATE);
  return lc.err;
}

cudaError_t launch_rmsnorm_gather(Launch& lc, int fam, const float* X, const int32_t* rc, const int32_t* count,
                                  int max_rows, const float* gain, float eps, void* out, int d, int act_bf16,
                                  unsigned* err) {
  lc.before(fam);
  const int grid = grid_rows(max_rows);
  if (act_bf16)
    lc.check(launch_pdl(lc.st, dim3(grid), dim3(kGateThreads), 0, 1, rmsnorm_gather_kernel<__nv_bfloat16>, X, rc, count,
                        max_rows, gain, eps, (__nv_bfloat16*)out, d, err));
  else
    lc.check(launch_pdl(lc.st, dim3(grid), dim3(kGateThreads), 0, 1, rmsnorm_gather_kernel<float>, X, rc, count, max_rows,
                        gain, eps, (float*)out, d, err));
  lc.after(fam);
  return lc.err;
}

cudaError_t launch_final_residual(Launch& lc, const float* h, const float* f, const int32_t* rcslot, void* out,
                                  int out_bf16, float* dbg, int T, int d, unsigned* epoch, unsigned* err) {
  lc.before(SF_K_RESIDUAL);
  const int grid = grid_rows(T);
  if (out_bf16)
    lc.check(launch_pdl(lc.st, dim3(grid), dim3(kGateThreads), 0, 1, final_residual_kernel<__nv_bfloat16>, h, f, rcslot,
                        (__nv_bfloat16*)out, dbg, T, d, epoch, err));
  else
    lc.check(launch_pdl(lc.st, dim3(grid), dim3(kGateThreads), 0, 1, final_residual_kernel<float>, h, f, rcslot, (float*)out,
                        dbg, T, d, epoch, err));
  lc.after(SF_K_RESIDUAL);
  return lc.err;
}

cudaError_t launch_pack_transpose(cudaStream_t st, const void* src, int K, int N, void* dst, int ld_dst, int row_base,
                                  int interleave, int bf16) {
  dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
  if (bf16)
    pack_transpose_kernel<__nv_bfloat16><<<grid, block, 0, st>>>((const __nv_bfloat16*)src, K, N,
                                                                 (__nv_bfloat16*)dst, ld_dst, row_base, interleave);
  else
    pack_transpose_kernel<float><<<grid, block, 0, st>>>((const float*)src, K, N, (float*)dst, ld_dst, row_base,
                                                         interleave);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free entry point of the gate / compaction / resolution step.
//
// The kernel above needs a little scratch besides its inputs and outputs: the
// arrival ticket that elects the last block, the fold flags the last block
// re-reads, the per-request offset table and a device error word.  Here that
// scratch is one file-scope device array, so the call allocates nothing.

namespace {

constexpr size_t kScratchTicket = 0;                        // unsigned
constexpr size_t kScratchErr = 4;                           // unsigned
constexpr size_t kScratchMeta = 256;                        // int32 [2 + kMaxTreeSlots]
constexpr size_t kScratchFlags = kScratchMeta + 4352;       // uint8 [kMaxRows]
constexpr size_t kScratchBytes = kScratchFlags + sf::kMaxRows;  // 12800 bytes

// Shared by every call on a device and kept until the process exits.
static __device__ __align__(256) unsigned char g_gate_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_gate_scratch on the current device (looked up once per
// device; the host-side symbol itself is not a device address).  The cached
// address belongs to the device's primary context: it does not survive a
// device reset, after which the library must be reloaded.
cudaError_t gate_scratch(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gate_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace sf

extern "C" sf_status sfk_gate_noalloc(void* stream, const void* hidden, int dtype, const int32_t* parent, int R,
                                      int B, int L, int d, float delta, float* H_out, uint8_t* fold, int32_t* rc,
                                      int32_t* rcslot, int32_t* src, int32_t* rc_count) {
  using namespace sf;
  if (!hidden || !parent || !H_out || !fold || !rc || !rcslot || !src || !rc_count) return SF_ERR_INVALID_ARG;
  if ((dtype != SF_F32 && dtype != SF_BF16) || R < 1 || B < 0 || L < 1 || d <= 0 || d % 4 != 0 ||
      !std::isfinite(delta) || delta < 0.f)
    return SF_ERR_INVALID_ARG;
  // rows are read as 4-element vectors and H_out is written as float4
  auto misaligned = [](const void* p, uintptr_t align) { return (reinterpret_cast<uintptr_t>(p) & (align - 1)) != 0; };
  if (misaligned(hidden, dtype == SF_F32 ? 16 : 8) || misaligned(H_out, 16) || misaligned(rc, 4) ||
      misaligned(rcslot, 4) || misaligned(src, 4) || misaligned(rc_count, 4))
    return SF_ERR_INVALID_ARG;
  const int Bp = B + 1;
  if (Bp > 127 || (long)R * Bp > kMaxTreeSlots || (long)R * Bp * L > kMaxRows) return SF_ERR_SHAPE;
  for (int r = 0; r < R; ++r) {
    if (parent[r * Bp] != -1) return SF_ERR_TREE;
    for (int i = 1; i < Bp; ++i)
      if (parent[r * Bp + i] < 0 || parent[r * Bp + i] >= i) return SF_ERR_TREE;
  }
  unsigned char* scratch = nullptr;
  if (gate_scratch(&scratch) != cudaSuccess) return SF_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  // the ticket and the error word must start at zero; the rest is overwritten
  if (cudaMemsetAsync(scratch, 0, 8, st) != cudaSuccess) return SF_ERR_CUDA;
  GateArgs a{};
  a.tree.R = R;
  a.tree.Bp = Bp;
  for (int k = 0; k < R * Bp; ++k) a.tree.parent[k] = (int8_t)parent[k];
  a.x_in = hidden;
  a.H_out = H_out;
  a.fold = scratch + kScratchFlags;
  a.fold_user = fold;
  a.rc = rc;
  a.rcslot = rcslot;
  a.src_user = src;
  a.meta = reinterpret_cast<int32_t*>(scratch + kScratchMeta);
  a.rc_count_user = rc_count;
  a.ticket = reinterpret_cast<unsigned*>(scratch + kScratchTicket);
  a.err = reinterpret_cast<unsigned*>(scratch + kScratchErr);
  a.delta = delta;
  a.T = R * Bp * L;
  a.d = d;
  a.L = L;
  Launch lc{nullptr, st};
  launch_gate(lc, a, dtype == SF_BF16);
  return lc.err == cudaSuccess ? SF_OK : SF_ERR_CUDA;
}
