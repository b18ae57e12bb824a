// Host-side internals of libspecfold: the context and the launch functions of
// every kernel family.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <string>
#include <vector>

#include "sf_common.cuh"
#include "specfold.h"

struct sf_layer_dev {
  void* wqkv = nullptr;  // [Mqkv_pad][d]      packed Wq^T | Wk^T | Wv^T | 0
  void* wo = nullptr;    // [d][q_dim]         Wo^T
  void* wgu = nullptr;   // [2*Fp][d]          tiles of 64 gate rows + 64 up rows
  void* wd = nullptr;    // [d][Fp]            Wd^T, zero columns past F
  float* g1 = nullptr;   // [d] attention RMSNorm gain
  float* g2 = nullptr;   // [d] FFN RMSNorm gain
  // TMA descriptors of the packed weights (BF16 contexts)
  alignas(64) CUtensorMap tm_wqkv, tm_wo, tm_wgu, tm_wd;
};

struct sf_graph_key {
  const void* hidden_in = nullptr;
  const void* prefix_k = nullptr;
  const void* prefix_v = nullptr;
  void* hidden_out = nullptr;
  void* fold = nullptr;
  void* src = nullptr;
  void* rc_count = nullptr;
  void* dbg_hidden = nullptr;
  void* dbg_rc = nullptr;
  void* dbg_rho = nullptr;
  void* stream = nullptr;
  int R = 0, B = 0, P = 0;
  float delta = 0.f;
  int stall = 0;
  int attn_mode = 0;
  std::vector<int> parent;
  bool operator==(const sf_graph_key& o) const {
    return hidden_in == o.hidden_in && prefix_k == o.prefix_k && prefix_v == o.prefix_v &&
           hidden_out == o.hidden_out && fold == o.fold && src == o.src && rc_count == o.rc_count &&
           dbg_hidden == o.dbg_hidden && dbg_rc == o.dbg_rc && dbg_rho == o.dbg_rho && stream == o.stream && R == o.R &&
           B == o.B && P == o.P && delta == o.delta && stall == o.stall && attn_mode == o.attn_mode &&
           parent == o.parent;
  }
};

struct sf_ctx {
  sf_shapes s{};
  int device = 0;
  int act_bytes = 4;
  int q_dim = 0, kv_dim = 0, Mqkv = 0, Mqkv_pad = 0, Fp = 0, Mgu = 0;
  int T_max = 0, max_pos = 0;
  int sm_count = 148;
  std::vector<sf_layer_dev> layers;

  // workspaces (device)
  float* H = nullptr;       // [T_max][d] layer input (fp32 residual stream)
  float* h = nullptr;       // [T_max][d] after attention + residual
  float* fphys = nullptr;   // [T_max][d] FFN output of the recompute rows
  void* xn = nullptr;       // [T_max][max(d, Fp)] normalised gathered rows (act dtype)
  void* qkv = nullptr;      // [T_max][Mqkv_pad] physical Q|K|V table of the recompute rows
  void* attn = nullptr;     // [T_max][q_dim] attention output of every row
  void* u = nullptr;        // [T_max][Fp] SwiGLU activations of the recompute rows
  float* y32 = nullptr;     // [T_max][max M] fp32 GEMM accumulators (FP32 contexts)
  int rows_cap = 0;         // activation buffers' row capacity (T_max rounded to 256)
  alignas(64) CUtensorMap tm_xn, tm_attn, tm_u;  // activation operands (BF16 contexts)
  float* part_o = nullptr;  // [max_splits][T_max][nq][hd] prefix-attention partials
  float* part_ml = nullptr; // [max_splits][T_max][nq][2]  (running max, denominator)
  int max_splits = 0;
  uint8_t* fold = nullptr;  // [T_max]
  int32_t* rc = nullptr;    // [T_max]
  int32_t* rcslot[2] = {nullptr, nullptr};  // [T_max], ping-pong between layers
  int32_t* meta = nullptr;  // [0] = rc count, [1 + r] = first recompute slot of request r
  unsigned* ticket = nullptr;
  unsigned* epoch = nullptr;  // [0] pass counter
  unsigned long long* scan = nullptr;  // [T_max] the gate's per-row words
  float* gate_ss = nullptr;            // [T_max] ||H||^2 per row (wide-row gate)
  unsigned* err_dev = nullptr;
  unsigned* err_host = nullptr;  // pinned mirror, refreshed at the end of every pass
  float2* rope = nullptr;   // [max_pos][hd/2] (cos, sin), computed in double on the host

  float* dbg_hidden = nullptr;
  int32_t* dbg_rc = nullptr;
  float* dbg_rho = nullptr;  // [n_layers][T] gate rho dump, or nullptr
  int inject_stall = 0;  // failure injection: layer 0's first row never reports its gate decision
  int attn_mode = SF_ATTN_DIRECT;

  sf_stats stats{};
  bool use_graphs = true;
  unsigned timing_mask = 0;
  std::vector<cudaEvent_t> ev_start, ev_stop;
  std::vector<int> ev_family;
  size_t ev_used = 0;
  std::string last_error;

  // cached graph of the last argument set
  bool graph_valid = false;
  sf_graph_key graph_key;
  cudaGraphExec_t graph_exec = nullptr;
  uint64_t graph_nodes = 0;
  uint64_t graph_family[SF_K_COUNT] = {};
  cudaGraphExec_t timing_exec = nullptr;  // last timed pass (kept until its events are read)
};

namespace sf {

// Bracket for every kernel launch: counts it, records timing events when the
// family is selected, and turns a launch error into SF_ERR_CUDA.
struct Launch {
  sf_ctx* ctx;
  cudaStream_t st;
  cudaError_t err = cudaSuccess;
  bool external_events = false;  // recording into a graph under capture
  uint64_t launches = 0;
  uint64_t family[SF_K_COUNT] = {};
  void before(int fam);
  void after(int fam);
  void check(cudaError_t e) {
    if (e != cudaSuccess && err == cudaSuccess) err = e;
  }
};

struct GemmArgs {
  const void* X;           // [rows][K] activations (act dtype), K contiguous
  int ldx;
  const void* W;           // [M][K] packed weight (act dtype), K contiguous
  int ldw;
  int M, K;
  const int32_t* count;    // device row count, or nullptr to use dense_count
  int dense_count;
  int max_rows;            // capacity of X / outputs
  bool count_early;        // count written two or more launches back (final when the grid starts)
};

enum EpiKind { kEpiQKV = 0, kEpiResidual = 1, kEpiSwiGLU = 2, kEpiStore = 3, kEpiArgmax = 4 };

struct EpiArgs {
  // kEpiQKV
  void* qkv = nullptr; int qkv_ld = 0; int qk_dim = 0; int qkv_M = 0; int hd = 0;
  const int32_t* rc = nullptr; int L = 0; int P = 0; const float2* rope = nullptr;
  // kEpiResidual
  float* h = nullptr; const float* H = nullptr; int h_ld = 0;
  // kEpiSwiGLU
  void* u = nullptr; int u_ld = 0;
  // kEpiStore
  float* y = nullptr; int y_ld = 0;
  // kEpiArgmax
  float2* part = nullptr; int part_ld = 0; int vocab = 0;
};

struct GateArgs {
  const void* x_in;            // layer 0: hidden_in [T][d] (dtype); else nullptr
  const float* h_prev;         // layer > 0: previous layer's h [T][d]
  const float* f_prev;         // layer > 0: previous layer's FFN table [T_rc][d]
  const int32_t* rcslot_prev;  // layer > 0: previous layer's source slots [T]
  float* H_out;                // [T][d]
  float* dbg;                  // [T][d] or nullptr
  uint8_t* fold;               // [T]
  uint8_t* fold_user;          // [T] or nullptr
  int32_t* rc;                 // [T]
  int32_t* rcslot;             // [T]
  int32_t* src_user;           // [T] or nullptr
  int32_t* meta;               // [1 + R + 1]
  int32_t* rc_count_user;      // one int or nullptr
  int32_t* rc_user;            // [T] or nullptr
  unsigned* ticket;
  unsigned* err;
  float delta;
  int T, d, L;
  Tree tree;
  // fused gate + attention RMSNorm (gate_norm_kernel) only
  void* xn;               // [T_rc][d] context dtype: normalised recompute rows
  const float* gain;      // [d] attention RMSNorm gain
  float eps;
  unsigned long long* scan;  // [T] per-row gate words (tag | recompute bit)
  float* row_ss;             // [T] ||H||^2 of every row (wide-row gate: part 1 to part 2)
  float* rho_user;           // [T] or nullptr: rho of every row (NaN for the main branch)
  int stall;                 // failure injection: row 0 never reports, so the waits on it run out
  const unsigned* epoch;     // pass counter, advanced by the final residual kernel
  int layer;
};

// sf_gate.cu
cudaError_t launch_gate(Launch& lc, const GateArgs& a, int in_bf16);
cudaError_t launch_rmsnorm_gather(Launch& lc, int fam, const float* X, const int32_t* rc,
                                  const int32_t* count, int max_rows, const float* gain, float eps,
                                  void* out, int d, int act_bf16, unsigned* err);
cudaError_t launch_gate_norm(Launch& lc, const GateArgs& a, int bf16);
cudaError_t launch_final_residual(Launch& lc, const float* h, const float* f, const int32_t* rcslot,
                                  void* out, int out_bf16, float* dbg, int T, int d, unsigned* epoch,
                                  unsigned* err);
cudaError_t launch_pack_transpose(cudaStream_t st, const void* src, int K, int N, void* dst, int ld_dst,
                                  int row_base, int interleave, int bf16);

// sf_gemm_tc.cu (BF16 contexts)
struct TcGemm {
  const CUtensorMap* tmA;  // weight [M][K]
  const CUtensorMap* tmB;  // activations [rows][K]
  int M, K;
  const int32_t* count;
  int dense_count;
  int max_rows;
  int splits;  // K split over a cluster of this many CTAs (1..6 or 8)
  unsigned* err;
  bool count_early;  // *count is final before the dependency wait
};
bool make_tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
int gemm_tc_splits(int M, int K, int n_tiles);
bool make_tmap_kv(CUtensorMap* tm, const void* base, int hd, int nkv, uint64_t rows);
cudaError_t launch_gemm_tc(Launch& lc, int fam, const TcGemm& g, EpiKind kind, const EpiArgs& e);

// sf_gemm.cu (FP32 contexts)
cudaError_t launch_gemm(Launch& lc, int fam, int act_bf16, const GemmArgs& g, EpiKind kind,
                        const EpiArgs& e, float* y32);

// sf_attn.cu
struct AttnArgs {
  const void* qkv; int ld_qkv;
  const void* pk; const void* pv;  // this layer's [R][P][nkv][hd]
  const int32_t* meta;
  const int32_t* rcslot;
  float* part_o; float* part_ml;
  void* attn; int ld_attn;
  int R, Bp, L, P, T, nq, nkv, hd;
  int target_ctas;  // prefix splits are chosen on the device to reach about this many CTAs
  float scale_log2;
  unsigned* err;
  // SF_ATTN_CORRECT: the block kernels run only the recompute rows and leave
  // their merged softmax state in part_o / part_ml (index slot * nq + head);
  // the correction kernel derives every folded row from its source's state
  int mode;
  const int32_t* rc;  // recompute list (row of every slot)
};
cudaError_t launch_attention(Launch& lc, int act_bf16, const AttnArgs& a);

}  // namespace sf
