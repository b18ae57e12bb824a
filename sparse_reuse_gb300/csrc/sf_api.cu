// C ABI of libspecfold: context lifetime, argument validation and the
// per-layer launch sequence of one folded verification pass.
//
// Per layer ("SpecFold", arXiv 2610.04875v2 summary, App. B: gate/compaction,
// source resolution, RMSNorm + packed QKV + rotary, attention with folded
// rows, FFN on recomputed rows, per-branch residual):
//   gate (+ previous layer's residual)  -> fold flags, recompute list, source slots
//   RMSNorm gather of recompute rows    -> xn
//   QKV GEMM + rotary epilogue          -> physical Q|K|V table of recompute rows
//   prefix attention partials           -> per recomputed query
//   block attention + merge             -> attention output of every row
//   O GEMM + residual epilogue          -> h
//   RMSNorm gather of recompute rows    -> xn
//   gate/up GEMM + SwiGLU epilogue      -> u
//   down GEMM                           -> FFN table of recompute rows
// then the last layer's residual writes hidden_out.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "sf_internal.h"

using namespace sf;

namespace {

const char* kStatusText[] = {"ok", "invalid argument", "shape outside the context's capacity",
                             "invalid draft tree", "unsupported shape", "out of device memory",
                             "CUDA error", "device-side check fired"};

sf_status fail(sf_ctx* c, sf_status st, const char* fmt, ...) __attribute__((format(printf, 3, 4)));
sf_status fail(sf_ctx* c, sf_status st, const char* fmt, ...) {
  if (c) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    c->last_error = buf;
  }
  return st;
}

// A non-null pointer that does not start on an `align`-byte boundary.
bool misaligned(const void* p, uintptr_t align) { return p && (reinterpret_cast<uintptr_t>(p) & (align - 1)); }

template <typename T>
cudaError_t dalloc(T** p, size_t bytes) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes > 0 ? bytes : 16);
  if (e == cudaSuccess) e = cudaMemset(q, 0, bytes > 0 ? bytes : 16);
  *p = static_cast<T*>(q);
  return e;
}

void free_ctx(sf_ctx* c) {
  if (!c) return;
  for (auto& L : c->layers) {
    cudaFree(L.wqkv); cudaFree(L.wo); cudaFree(L.wgu); cudaFree(L.wd); cudaFree(L.g1); cudaFree(L.g2);
  }
  void* bufs[] = {c->H, c->h, c->fphys, c->xn, c->qkv, c->attn, c->u, c->y32, c->part_o, c->part_ml,
                  c->fold, c->rc, c->rcslot[0], c->rcslot[1], c->meta, c->ticket, c->epoch, c->scan, c->gate_ss,

                  c->err_dev, c->rope};
  for (void* b : bufs) cudaFree(b);
  if (c->err_host) cudaFreeHost(c->err_host);
  for (auto e : c->ev_start) cudaEventDestroy(e);
  for (auto e : c->ev_stop) cudaEventDestroy(e);
  if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
  if (c->timing_exec) cudaGraphExecDestroy(c->timing_exec);
  delete c;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

namespace sf {

void Launch::before(int fam) {
  if (ctx && ctx->timing_mask & (1u << fam)) {
    if (ctx->ev_used == ctx->ev_start.size()) {
      cudaEvent_t a, b;
      cudaEventCreate(&a);
      cudaEventCreate(&b);
      ctx->ev_start.push_back(a);
      ctx->ev_stop.push_back(b);
      ctx->ev_family.push_back(fam);
    }
    ctx->ev_family[ctx->ev_used] = fam;
    if (external_events)
      cudaEventRecordWithFlags(ctx->ev_start[ctx->ev_used], st, cudaEventRecordExternal);
    else
      cudaEventRecord(ctx->ev_start[ctx->ev_used], st);
  }
}

void Launch::after(int fam) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess && err == cudaSuccess) err = e;
  ++launches;
  ++family[fam];
  if (ctx && ctx->timing_mask & (1u << fam)) {
    if (external_events)
      cudaEventRecordWithFlags(ctx->ev_stop[ctx->ev_used], st, cudaEventRecordExternal);
    else
      cudaEventRecord(ctx->ev_stop[ctx->ev_used], st);
    ++ctx->ev_used;
  }
}

}  // namespace sf

namespace {

struct PassArgs {
  const void* hidden_in;
  const void* prefix_k;
  const void* prefix_v;
  int R, B, P;
  float delta;
  void* hidden_out;
  uint8_t* fold;
  int32_t* src;
  int32_t* rc_count;
  const int32_t* parent;
};

// One GEMM of the layer: tcgen05 kernel for BF16 contexts, CUDA-core fp32
// kernel for FP32 contexts.
cudaError_t run_gemm(sf_ctx* c, Launch& lc, int fam, const GemmArgs& g, const CUtensorMap* tmA,
                     const CUtensorMap* tmB, EpiKind kind, const EpiArgs& e) {
  if (c->s.dtype != SF_BF16) return launch_gemm(lc, fam, 0, g, kind, e, c->y32);
  TcGemm t{};
  t.tmA = tmA;
  t.tmB = tmB;
  t.M = g.M;
  t.K = g.K;
  t.count = g.count;
  t.dense_count = g.dense_count;
  t.max_rows = g.max_rows;
  const int n_tiles = g.count ? 1 : (g.dense_count + 255) / 256;
  t.splits = gemm_tc_splits(g.M, g.K, n_tiles);
  t.err = c->err_dev;
  t.count_early = g.count && g.count_early;
  return launch_gemm_tc(lc, fam, t, kind, e);
}

cudaError_t enqueue_pass(sf_ctx* c, Launch& lc, const PassArgs& p) {
  const sf_shapes& s = c->s;
  const int Bp = p.B + 1, L = s.block_len, T = p.R * Bp * L, d = s.d_model;
  const int nl = s.n_layers, bf16 = s.dtype == SF_BF16;
  const size_t kv_layer = (size_t)p.R * p.P * s.n_kv_heads * s.head_dim * c->act_bytes;
  GateArgs ga{};
  ga.tree.R = p.R;
  ga.tree.Bp = Bp;
  for (int r = 0; r < p.R; ++r)
    for (int i = 0; i < Bp; ++i) ga.tree.parent[r * Bp + i] = (int8_t)p.parent[r * Bp + i];
  for (int l = 0; l < nl; ++l) {
    const sf_layer_dev& W = c->layers[l];
    int32_t* rcslot = c->rcslot[l & 1];
    ga.x_in = l == 0 ? p.hidden_in : nullptr;
    ga.h_prev = c->h;
    ga.f_prev = c->fphys;
    ga.rcslot_prev = c->rcslot[(l + 1) & 1];
    ga.H_out = c->H;
    ga.dbg = c->dbg_hidden ? c->dbg_hidden + (size_t)l * T * d : nullptr;
    ga.fold = c->fold;
    ga.fold_user = p.fold ? p.fold + (size_t)l * T : nullptr;
    ga.rc = c->rc;
    ga.rcslot = rcslot;
    ga.src_user = p.src ? p.src + (size_t)l * T : nullptr;
    ga.meta = c->meta;
    ga.rc_count_user = p.rc_count ? p.rc_count + l : nullptr;
    ga.rc_user = c->dbg_rc ? c->dbg_rc + (size_t)l * T : nullptr;
    ga.ticket = c->ticket;
    ga.err = c->err_dev;
    ga.delta = p.delta;
    ga.T = T;
    ga.d = d;
    ga.L = L;
    ga.xn = c->xn;
    ga.gain = W.g1;
    ga.eps = s.rms_eps;
    ga.scan = c->scan;
    ga.row_ss = c->gate_ss;
    ga.rho_user = c->dbg_rho ? c->dbg_rho + (size_t)l * T : nullptr;
    ga.stall = c->inject_stall && l == 0;
    ga.epoch = c->epoch;
    ga.layer = l;
    if (launch_gate_norm(lc, ga, bf16) != cudaSuccess) return lc.err;

    GemmArgs g{};
    EpiArgs e{};
    g.X = c->xn; g.ldx = d; g.W = W.wqkv; g.ldw = d; g.M = c->Mqkv_pad; g.K = d;
    g.count = c->meta; g.dense_count = T; g.max_rows = T;
    e.qkv = c->qkv; e.qkv_ld = c->Mqkv_pad; e.qk_dim = c->q_dim + c->kv_dim; e.qkv_M = c->Mqkv;
    e.hd = s.head_dim; e.rc = c->rc; e.L = L; e.P = p.P; e.rope = c->rope;
    if (run_gemm(c, lc, SF_K_GEMM_QKV, g, &W.tm_wqkv, &c->tm_xn, kEpiQKV, e) != cudaSuccess) return lc.err;

    AttnArgs a{};
    a.qkv = c->qkv; a.ld_qkv = c->Mqkv_pad;
    a.pk = p.P > 0 ? (const char*)p.prefix_k + l * kv_layer : nullptr;
    a.pv = p.P > 0 ? (const char*)p.prefix_v + l * kv_layer : nullptr;
    a.meta = c->meta; a.rcslot = rcslot; a.part_o = c->part_o; a.part_ml = c->part_ml;
    a.attn = c->attn; a.ld_attn = c->q_dim;
    a.R = p.R; a.Bp = Bp; a.L = L; a.P = p.P; a.T = T;
    a.nq = s.n_q_heads; a.nkv = s.n_kv_heads; a.hd = s.head_dim;
    a.target_ctas = c->sm_count;
    a.mode = c->attn_mode;
    a.rc = c->rc;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.head_dim));
    a.err = c->err_dev;
    if (launch_attention(lc, bf16, a) != cudaSuccess) return lc.err;

    g = GemmArgs{};
    e = EpiArgs{};
    g.X = c->attn; g.ldx = c->q_dim; g.W = W.wo; g.ldw = c->q_dim; g.M = d; g.K = c->q_dim;
    g.count = nullptr; g.dense_count = T; g.max_rows = T;
    e.h = c->h; e.H = c->H; e.h_ld = d;
    if (run_gemm(c, lc, SF_K_GEMM_O, g, &W.tm_wo, &c->tm_attn, kEpiResidual, e) != cudaSuccess) return lc.err;

    launch_rmsnorm_gather(lc, SF_K_NORM, c->h, c->rc, c->meta, T, W.g2, s.rms_eps, c->xn, d, bf16, c->err_dev);

    g = GemmArgs{};
    e = EpiArgs{};
    g.X = c->xn; g.ldx = d; g.W = W.wgu; g.ldw = d; g.M = c->Mgu; g.K = d;
    g.count = c->meta; g.dense_count = T; g.max_rows = T;
    g.count_early = true;  // from the gate kernel, before the projection
    e.u = c->u; e.u_ld = c->Fp;
    if (run_gemm(c, lc, SF_K_GEMM_GATEUP, g, &W.tm_wgu, &c->tm_xn, kEpiSwiGLU, e) != cudaSuccess) return lc.err;

    g = GemmArgs{};
    e = EpiArgs{};
    g.X = c->u; g.ldx = c->Fp; g.W = W.wd; g.ldw = c->Fp; g.M = d; g.K = c->Fp;
    g.count = c->meta; g.dense_count = T; g.max_rows = T;
    g.count_early = true;
    e.y = c->fphys; e.y_ld = d;
    if (run_gemm(c, lc, SF_K_GEMM_DOWN, g, &W.tm_wd, &c->tm_u, kEpiStore, e) != cudaSuccess) return lc.err;
  }
  launch_final_residual(lc, c->h, c->fphys, c->rcslot[(nl - 1) & 1], p.hidden_out, bf16,
                        c->dbg_hidden ? c->dbg_hidden + (size_t)nl * T * d : nullptr, T, d, c->epoch, c->err_dev);
  if (lc.err == cudaSuccess) lc.err = cudaMemcpyAsync(c->err_host, c->err_dev, sizeof(unsigned),
                                                      cudaMemcpyDeviceToHost, lc.st);
  return lc.err;
}

void add_stats(sf_ctx* c, const Launch& lc) {
  c->stats.kernel_launches += lc.launches;
  for (int f = 0; f < SF_K_COUNT; ++f) c->stats.family_launches[f] += lc.family[f];
}

}  // namespace

extern "C" {

const char* sf_status_str(sf_status s) {
  const int i = (int)s;
  return (i >= 0 && i < (int)(sizeof(kStatusText) / sizeof(kStatusText[0]))) ? kStatusText[i] : "unknown status";
}

const char* sf_last_error(const sf_ctx* c) { return c ? c->last_error.c_str() : ""; }

sf_status sf_create(const sf_shapes* shapes, const sf_layer_weights* layers, sf_ctx** out) {
  if (!out) return SF_ERR_INVALID_ARG;
  *out = nullptr;
  if (!shapes || !layers) return SF_ERR_INVALID_ARG;
  const sf_shapes s = *shapes;
  if (s.n_layers <= 0 || s.d_model <= 0 || s.n_q_heads <= 0 || s.n_kv_heads <= 0 || s.head_dim <= 0 ||
      s.d_ffn <= 0 || s.block_len <= 0 || s.max_requests <= 0 || s.max_branches <= 0 || s.max_prefix < 0 ||
      !(s.rms_eps >= 0.f) || !(s.rope_theta > 0.f) || (s.dtype != SF_F32 && s.dtype != SF_BF16))
    return SF_ERR_INVALID_ARG;
  if ((s.head_dim != 64 && s.head_dim != 128) || s.d_model % 128 != 0 || s.d_model > 16384 || s.n_layers > 1024 ||
      s.n_q_heads % s.n_kv_heads != 0 ||
      s.block_len > 64 || s.max_branches > 127 || (long)s.max_requests * s.max_branches > kMaxTreeSlots ||
      (long)s.max_requests * s.max_branches * s.block_len > kMaxRows)
    return SF_ERR_UNSUPPORTED;
  for (int l = 0; l < s.n_layers; ++l) {
    const sf_layer_weights& w = layers[l];
    if (!w.attn_norm || !w.wq || !w.wk || !w.wv || !w.wo || !w.ffn_norm || !w.w_gate || !w.w_up || !w.w_down)
      return SF_ERR_INVALID_ARG;
  }
  sf_ctx* c = new (std::nothrow) sf_ctx();
  if (!c) return SF_ERR_OOM;
  c->s = s;
  cudaGetDevice(&c->device);
  const int bf16 = s.dtype == SF_BF16;
  c->act_bytes = bf16 ? 2 : 4;
  c->q_dim = s.n_q_heads * s.head_dim;
  c->kv_dim = s.n_kv_heads * s.head_dim;
  c->Mqkv = c->q_dim + 2 * c->kv_dim;
  c->Mqkv_pad = round_up(c->Mqkv, 128);
  c->Fp = round_up(s.d_ffn, 64);
  c->Mgu = 2 * c->Fp;
  c->T_max = s.max_requests * s.max_branches * s.block_len;
  c->max_pos = s.max_prefix + s.block_len;
  c->max_splits = 8;
  cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
  if (c->sm_count <= 0) c->sm_count = 148;
  const int d = s.d_model, T = c->T_max, ab = c->act_bytes;
  const size_t maxM = (size_t)std::max(std::max(c->Mqkv_pad, c->Mgu), d);
  cudaError_t e = cudaSuccess;
#define SF_TRY(x)                                                                             \
  do {                                                                                        \
    e = (x);                                                                                  \
    if (e != cudaSuccess) {                                                                   \
      sf_status st_ = e == cudaErrorMemoryAllocation ? SF_ERR_OOM : SF_ERR_CUDA;              \
      free_ctx(c);                                                                            \
      cudaGetLastError();                                                                     \
      return st_;                                                                             \
    }                                                                                         \
  } while (0)
  SF_TRY(dalloc(&c->H, (size_t)T * d * 4));
  SF_TRY(dalloc(&c->h, (size_t)T * d * 4));
  SF_TRY(dalloc(&c->fphys, (size_t)T * d * 4));
  c->rows_cap = round_up(T, 256);
  const int RC = c->rows_cap;
  SF_TRY(dalloc(&c->xn, (size_t)RC * d * ab));
  SF_TRY(dalloc(&c->qkv, (size_t)T * c->Mqkv_pad * ab));
  SF_TRY(dalloc(&c->attn, (size_t)RC * c->q_dim * ab));
  SF_TRY(dalloc(&c->u, (size_t)RC * c->Fp * ab));
  if (bf16) {
    if (!make_tmap_bf16(&c->tm_xn, c->xn, d, RC, 64) || !make_tmap_bf16(&c->tm_attn, c->attn, c->q_dim, RC, 64) ||
        !make_tmap_bf16(&c->tm_u, c->u, c->Fp, RC, 64)) {
      free_ctx(c);
      return SF_ERR_CUDA;
    }
  } else {
    SF_TRY(dalloc(&c->y32, (size_t)T * maxM * 4));
  }
  SF_TRY(dalloc(&c->part_o, (size_t)c->max_splits * T * c->q_dim * 4));
  SF_TRY(dalloc(&c->part_ml, (size_t)c->max_splits * T * s.n_q_heads * 2 * 4));
  SF_TRY(dalloc(&c->fold, (size_t)T));
  SF_TRY(dalloc(&c->rc, (size_t)T * 4));
  SF_TRY(dalloc(&c->rcslot[0], (size_t)T * 4));
  SF_TRY(dalloc(&c->rcslot[1], (size_t)T * 4));
  SF_TRY(dalloc(&c->meta, (size_t)(s.max_requests + 2) * 4));
  SF_TRY(dalloc(&c->ticket, 64));
  SF_TRY(dalloc(&c->epoch, 64));
  SF_TRY(dalloc(&c->scan, (size_t)T * 8));
  SF_TRY(dalloc(&c->gate_ss, (size_t)T * 4));
  SF_TRY(dalloc(&c->err_dev, 64));
  SF_TRY(cudaHostAlloc((void**)&c->err_host, 64, cudaHostAllocDefault));
  *c->err_host = 0;
  {
    const int half = s.head_dim / 2;
    std::vector<float2> cs((size_t)c->max_pos * half);
    for (int pos = 0; pos < c->max_pos; ++pos)
      for (int j = 0; j < half; ++j) {
        const double a = pos * std::pow((double)s.rope_theta, -2.0 * j / s.head_dim);
        cs[(size_t)pos * half + j] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    SF_TRY(dalloc(&c->rope, cs.size() * sizeof(float2)));
    SF_TRY(cudaMemcpy(c->rope, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice));
  }
  c->layers.resize(s.n_layers);
  for (int l = 0; l < s.n_layers; ++l) {
    const sf_layer_weights& w = layers[l];
    sf_layer_dev& D = c->layers[l];
    SF_TRY(dalloc(&D.wqkv, (size_t)c->Mqkv_pad * d * ab));
    SF_TRY(dalloc(&D.wo, (size_t)d * c->q_dim * ab));
    SF_TRY(dalloc(&D.wgu, (size_t)c->Mgu * d * ab));
    SF_TRY(dalloc(&D.wd, (size_t)d * c->Fp * ab));
    SF_TRY(dalloc(&D.g1, (size_t)d * 4));
    SF_TRY(dalloc(&D.g2, (size_t)d * 4));
    SF_TRY(launch_pack_transpose(0, w.wq, d, c->q_dim, D.wqkv, d, 0, 0, bf16));
    SF_TRY(launch_pack_transpose(0, w.wk, d, c->kv_dim, D.wqkv, d, c->q_dim, 0, bf16));
    SF_TRY(launch_pack_transpose(0, w.wv, d, c->kv_dim, D.wqkv, d, c->q_dim + c->kv_dim, 0, bf16));
    SF_TRY(launch_pack_transpose(0, w.wo, c->q_dim, d, D.wo, c->q_dim, 0, 0, bf16));
    SF_TRY(launch_pack_transpose(0, w.w_gate, d, s.d_ffn, D.wgu, d, 0, 1, bf16));
    SF_TRY(launch_pack_transpose(0, w.w_up, d, s.d_ffn, D.wgu, d, 0, 2, bf16));
    SF_TRY(launch_pack_transpose(0, w.w_down, s.d_ffn, d, D.wd, c->Fp, 0, 0, bf16));
    if (bf16 && (!make_tmap_bf16(&D.tm_wqkv, D.wqkv, d, c->Mqkv_pad, 128) ||
                 !make_tmap_bf16(&D.tm_wo, D.wo, c->q_dim, d, 128) ||
                 !make_tmap_bf16(&D.tm_wgu, D.wgu, d, c->Mgu, 128) || !make_tmap_bf16(&D.tm_wd, D.wd, c->Fp, d, 128))) {
      free_ctx(c);
      return SF_ERR_CUDA;
    }
    SF_TRY(cudaMemcpy(D.g1, w.attn_norm, (size_t)d * 4, cudaMemcpyDeviceToDevice));
    SF_TRY(cudaMemcpy(D.g2, w.ffn_norm, (size_t)d * 4, cudaMemcpyDeviceToDevice));
  }
  SF_TRY(cudaDeviceSynchronize());
#undef SF_TRY
  *out = c;
  return SF_OK;
}

sf_status sf_verify(sf_ctx* c, void* stream, const void* hidden_in, const int32_t* parent, const void* prefix_k,
                    const void* prefix_v, int R, int B, int P, float delta, void* hidden_out, uint8_t* fold_mask,
                    int32_t* src, int32_t* rc_count) {
  if (!c) return SF_ERR_INVALID_ARG;
  if (!hidden_in || !hidden_out || !parent) return fail(c, SF_ERR_INVALID_ARG, "null hidden_in/hidden_out/parent");
  if (!std::isfinite(delta) || delta < 0.f) return fail(c, SF_ERR_INVALID_ARG, "delta must be finite and >= 0");
  if (R < 0 || B < 0 || P < 0) return fail(c, SF_ERR_INVALID_ARG, "negative R, B or P");
  if (R > c->s.max_requests || B + 1 > c->s.max_branches || P > c->s.max_prefix)
    return fail(c, SF_ERR_SHAPE, "R=%d B=%d P=%d beyond capacity (%d, %d, %d)", R, B, P, c->s.max_requests,
                c->s.max_branches - 1, c->s.max_prefix);
  if (P > 0 && (!prefix_k || !prefix_v)) return fail(c, SF_ERR_INVALID_ARG, "null prefix K/V with P > 0");
  // rows move as 16-byte vectors (and the prefix through TMA): a misaligned
  // buffer is refused here rather than met by a kernel
  if (misaligned(hidden_in, 16) || misaligned(hidden_out, 16) || misaligned(prefix_k, 16) ||
      misaligned(prefix_v, 16) || misaligned(src, 4) || misaligned(rc_count, 4))
    return fail(c, SF_ERR_INVALID_ARG, "hidden and prefix buffers need 16-byte alignment, src/rc_count 4-byte");
  const int Bp = B + 1;
  for (int r = 0; r < R; ++r) {
    if (parent[r * Bp] != -1) return fail(c, SF_ERR_TREE, "request %d: parent[0] must be -1", r);
    for (int i = 1; i < Bp; ++i) {
      const int pi = parent[r * Bp + i];
      if (pi < 0 || pi >= i) return fail(c, SF_ERR_TREE, "request %d: parent[%d] = %d not in [0, %d)", r, i, pi, i);
    }
  }
  if (*c->err_host) return fail(c, SF_ERR_DEVICE_ASSERT, "device check word 0x%x", *c->err_host);
  if (R == 0) return SF_OK;
  cudaStream_t st = (cudaStream_t)stream;
  PassArgs pa{hidden_in, prefix_k, prefix_v, R, B, P, delta, hidden_out, fold_mask, src, rc_count, parent};

  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (st) cudaStreamIsCapturing(st, &cap);
  const bool graphs = c->use_graphs && c->timing_mask == 0 && st != nullptr && cap == cudaStreamCaptureStatusNone;
  if (graphs) {
    sf_graph_key key;
    key.hidden_in = hidden_in; key.prefix_k = prefix_k; key.prefix_v = prefix_v; key.hidden_out = hidden_out;
    key.fold = fold_mask; key.src = src; key.rc_count = rc_count; key.dbg_hidden = c->dbg_hidden;
    key.stall = c->inject_stall;
    key.attn_mode = c->attn_mode;
    key.dbg_rc = c->dbg_rc; key.dbg_rho = c->dbg_rho; key.stream = stream; key.R = R; key.B = B; key.P = P; key.delta = delta;
    key.parent.assign(parent, parent + R * Bp);
    if (!(c->graph_valid && key == c->graph_key)) {
      c->graph_valid = false;
      if (c->graph_exec) {
        cudaGraphExecDestroy(c->graph_exec);
        c->graph_exec = nullptr;
      }
      cudaGraph_t graph = nullptr;
      cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
      Launch lc{c, st};
      if (e == cudaSuccess) enqueue_pass(c, lc, pa);
      cudaError_t e2 = e == cudaSuccess ? cudaStreamEndCapture(st, &graph) : e;
      if (e == cudaSuccess && lc.err == cudaSuccess && e2 == cudaSuccess)
        e2 = cudaGraphInstantiate(&c->graph_exec, graph, 0);
      if (graph) cudaGraphDestroy(graph);
      if (e != cudaSuccess || lc.err != cudaSuccess || e2 != cudaSuccess) {
        cudaGetLastError();
        c->graph_exec = nullptr;
        return fail(c, SF_ERR_CUDA, "graph capture failed: %s",
                    cudaGetErrorString(e != cudaSuccess ? e : (lc.err != cudaSuccess ? lc.err : e2)));
      }
      c->graph_valid = true;
      c->graph_key = key;
      c->graph_nodes = lc.launches;
      for (int f = 0; f < SF_K_COUNT; ++f) c->graph_family[f] = lc.family[f];
    }
    cudaError_t e = cudaGraphLaunch(c->graph_exec, st);
    if (e != cudaSuccess) return fail(c, SF_ERR_CUDA, "graph launch: %s", cudaGetErrorString(e));
    c->stats.passes++;
    c->stats.graph_replays++;
    c->stats.kernel_launches += c->graph_nodes;
    for (int f = 0; f < SF_K_COUNT; ++f) c->stats.family_launches[f] += c->graph_family[f];
    return SF_OK;
  }
  if (c->timing_mask != 0 && st != nullptr && cap == cudaStreamCaptureStatusNone) {
    // timed pass: the same kernels as a graph replay, with an event-record
    // node around every launch of the selected families, so the events see
    // back-to-back device execution rather than host launch gaps
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    Launch lc{c, st};
    lc.external_events = true;
    cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) enqueue_pass(c, lc, pa);
    cudaError_t e2 = e == cudaSuccess ? cudaStreamEndCapture(st, &graph) : e;
    if (e == cudaSuccess && lc.err == cudaSuccess && e2 == cudaSuccess) e2 = cudaGraphInstantiate(&exec, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess || lc.err != cudaSuccess || e2 != cudaSuccess) {
      cudaGetLastError();
      return fail(c, SF_ERR_CUDA, "timing capture failed: %s",
                  cudaGetErrorString(e != cudaSuccess ? e : (lc.err != cudaSuccess ? lc.err : e2)));
    }
    e = cudaGraphLaunch(exec, st);
    if (c->timing_exec) {
      cudaStreamSynchronize(st);
      cudaGraphExecDestroy(c->timing_exec);
    }
    c->timing_exec = exec;
    if (e != cudaSuccess) return fail(c, SF_ERR_CUDA, "timing graph launch: %s", cudaGetErrorString(e));
    add_stats(c, lc);
    c->stats.passes++;
    return SF_OK;
  }
  Launch lc{c, st};
  enqueue_pass(c, lc, pa);
  add_stats(c, lc);
  c->stats.passes++;
  if (lc.err != cudaSuccess) return fail(c, SF_ERR_CUDA, "launch failed: %s", cudaGetErrorString(lc.err));
  return SF_OK;
}

sf_status sf_set_debug(sf_ctx* c, float* layer_hidden, int32_t* rc_rows) {
  if (!c) return SF_ERR_INVALID_ARG;
  if (misaligned(layer_hidden, 16) || misaligned(rc_rows, 4))
    return fail(c, SF_ERR_INVALID_ARG, "layer_hidden needs 16-byte alignment, rc_rows 4-byte");
  c->dbg_hidden = layer_hidden;
  c->dbg_rc = rc_rows;
  return SF_OK;
}

sf_status sf_set_attention_mode(sf_ctx* c, int mode) {
  if (!c || (mode != SF_ATTN_DIRECT && mode != SF_ATTN_CORRECT && mode != SF_ATTN_DIRECT_SPLIT))
    return SF_ERR_INVALID_ARG;
  c->attn_mode = mode;
  return SF_OK;
}

sf_status sf_set_rho_dump(sf_ctx* c, float* rho) {
  if (!c) return SF_ERR_INVALID_ARG;
  if (misaligned(rho, 4)) return fail(c, SF_ERR_INVALID_ARG, "rho needs 4-byte alignment");
  c->dbg_rho = rho;
  return SF_OK;
}

sf_status sf_sync_status(sf_ctx* c, void* stream) {
  if (!c) return SF_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(c, SF_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
  unsigned w = 0;
  e = cudaMemcpy(&w, c->err_dev, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(c, SF_ERR_CUDA, "reading the device check word: %s", cudaGetErrorString(e));
  if (w) {
    // reported once: the word is cleared so that the caller can continue
    e = cudaMemset(c->err_dev, 0, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    *c->err_host = 0;
    if (e != cudaSuccess) return fail(c, SF_ERR_CUDA, "clearing the device check word: %s", cudaGetErrorString(e));
    return fail(c, SF_ERR_DEVICE_ASSERT, "device check word 0x%x", w);
  }
  *c->err_host = 0;
  return SF_OK;
}

sf_status sf_inject_stall(sf_ctx* c, int on) {
  if (!c) return SF_ERR_INVALID_ARG;
  c->inject_stall = on ? 1 : 0;
  return SF_OK;
}

sf_status sf_destroy(sf_ctx* c) {
  if (!c) return SF_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  unsigned w = 0;
  if (e == cudaSuccess) cudaMemcpy(&w, c->err_dev, sizeof(unsigned), cudaMemcpyDeviceToHost);
  free_ctx(c);
  if (e != cudaSuccess) return SF_ERR_CUDA;
  return w ? SF_ERR_DEVICE_ASSERT : SF_OK;
}

sf_status sf_get_stats(const sf_ctx* c, sf_stats* out) {
  if (!c || !out) return SF_ERR_INVALID_ARG;
  *out = c->stats;
  return SF_OK;
}

sf_status sf_set_graphs(sf_ctx* c, int use_graphs) {
  if (!c) return SF_ERR_INVALID_ARG;
  c->use_graphs = use_graphs != 0;
  if (!c->use_graphs) c->graph_valid = false;
  return SF_OK;
}

sf_status sf_timing_begin(sf_ctx* c, unsigned family_mask) {
  if (!c) return SF_ERR_INVALID_ARG;
  c->timing_mask = family_mask;
  c->ev_used = 0;
  return SF_OK;
}

sf_status sf_timing_read(sf_ctx* c, double* total_ms, int64_t* launches) {
  if (!c || !total_ms || !launches) return SF_ERR_INVALID_ARG;
  for (int f = 0; f < SF_K_COUNT; ++f) {
    total_ms[f] = 0.0;
    launches[f] = 0;
  }
  for (size_t i = 0; i < c->ev_used; ++i) {
    cudaError_t e = cudaEventSynchronize(c->ev_stop[i]);
    if (e != cudaSuccess) return fail(c, SF_ERR_CUDA, "event sync: %s", cudaGetErrorString(e));
    float ms = 0.f;
    cudaEventElapsedTime(&ms, c->ev_start[i], c->ev_stop[i]);
    total_ms[c->ev_family[i]] += ms;
    launches[c->ev_family[i]] += 1;
  }
  return SF_OK;
}

sf_status sf_timing_list(sf_ctx* c, int family, double* ms, int max_n, int* n) {
  if (!c || !n || max_n < 0 || (max_n > 0 && !ms) || family < 0 || family >= SF_K_COUNT) return SF_ERR_INVALID_ARG;
  int k = 0;
  for (size_t i = 0; i < c->ev_used; ++i) {
    if (c->ev_family[i] != family) continue;
    cudaError_t e = cudaEventSynchronize(c->ev_stop[i]);
    if (e != cudaSuccess) return fail(c, SF_ERR_CUDA, "event sync: %s", cudaGetErrorString(e));
    float t = 0.f;
    cudaEventElapsedTime(&t, c->ev_start[i], c->ev_stop[i]);
    if (k < max_n) ms[k] = t;
    ++k;
  }
  *n = k;
  return SF_OK;
}

}  // extern "C"
