"""Python binding of libspecfold (the C ABI in include/specfold.h).

Argument marshalling only: every step of the verification pass runs in the
library's CUDA kernels.  The in-tree libspecfold.so is loaded on the first
call into the binding; if it is missing that call raises ImportError (build it with
``python -c "import __graft_entry__ as g; g.build()"`` or
``python sparse_reuse_gb300/build.py``).  PyTorch provides device memory and
streams only.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecfold.so")

SF_OK, SF_ERR_INVALID_ARG, SF_ERR_SHAPE, SF_ERR_TREE, SF_ERR_UNSUPPORTED, SF_ERR_OOM, SF_ERR_CUDA, \
    SF_ERR_DEVICE_ASSERT = range(8)
SF_F32, SF_BF16 = 0, 1
FAMILIES = ["gate", "norm", "gemm_qkv", "attn_prefix", "attn_block", "gemm_o", "gemm_gateup", "gemm_down",
            "residual", "aux", "attn_correct"]
SF_ATTN_DIRECT, SF_ATTN_CORRECT, SF_ATTN_DIRECT_SPLIT = 0, 1, 2
SF_K_COUNT = len(FAMILIES)

# every symbol include/specfold.h declares
EXPORTS = ["sf_create", "sf_verify", "sf_set_debug", "sf_set_rho_dump", "sf_set_attention_mode", "sf_sync_status", "sf_destroy", "sf_status_str",
           "sf_last_error", "sf_get_stats", "sf_set_graphs", "sf_timing_begin", "sf_timing_read", "sf_timing_list",
           "sfk_gemm_bf16", "sfk_gate_noalloc", "sf_inject_stall",
           "sf_head_create", "sf_head_verify", "sf_head_last_error", "sf_head_destroy"]


class SfShapes(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("d_ffn", ctypes.c_int),
                ("dtype", ctypes.c_int), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("block_len", ctypes.c_int), ("max_requests", ctypes.c_int), ("max_branches", ctypes.c_int),
                ("max_prefix", ctypes.c_int)]


class SfLayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")]


class SfHeadShapes(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("vocab", ctypes.c_int), ("dtype", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("max_rows", ctypes.c_int)]


class SfStats(ctypes.Structure):
    _fields_ = [("passes", ctypes.c_uint64), ("kernel_launches", ctypes.c_uint64),
                ("graph_replays", ctypes.c_uint64), ("family_launches", ctypes.c_uint64 * SF_K_COUNT)]


class SpecFoldError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libspecfold.so is not built ({LIB_PATH}); run sparse_reuse_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32p, c_int, c_float = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_float
    lib.sf_create.argtypes = [ctypes.POINTER(SfShapes), ctypes.POINTER(SfLayerWeights), ctypes.POINTER(vp)]
    lib.sf_verify.argtypes = [vp, vp, vp, i32p, vp, vp, c_int, c_int, c_int, c_float, vp, vp, vp, vp]
    lib.sf_set_debug.argtypes = [vp, vp, vp]
    lib.sf_set_rho_dump.argtypes = [vp, vp]
    lib.sf_set_attention_mode.argtypes = [vp, c_int]
    lib.sf_sync_status.argtypes = [vp, vp]
    lib.sf_inject_stall.argtypes = [vp, c_int]
    lib.sf_destroy.argtypes = [vp]
    lib.sf_status_str.argtypes = [c_int]
    lib.sf_status_str.restype = ctypes.c_char_p
    lib.sf_last_error.argtypes = [vp]
    lib.sf_last_error.restype = ctypes.c_char_p
    lib.sf_get_stats.argtypes = [vp, ctypes.POINTER(SfStats)]
    lib.sf_set_graphs.argtypes = [vp, c_int]
    lib.sf_timing_begin.argtypes = [vp, ctypes.c_uint]
    lib.sf_timing_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
    lib.sf_timing_list.argtypes = [vp, c_int, ctypes.POINTER(ctypes.c_double), c_int, ctypes.POINTER(c_int)]
    lib.sfk_gemm_bf16.argtypes = [vp, vp, c_int, vp, c_int, c_int, vp, c_int, vp, c_int, c_int, vp]
    lib.sfk_gate_noalloc.argtypes = [vp, vp, c_int, i32p, c_int, c_int, c_int, c_int, c_float, vp, vp, vp, vp, vp,
                                     vp]
    lib.sf_head_create.argtypes = [ctypes.POINTER(SfHeadShapes), vp, vp, ctypes.POINTER(vp)]
    lib.sf_head_verify.argtypes = [vp, vp, vp, vp, i32p, c_int, c_int, c_int, vp, vp, vp]
    lib.sf_head_last_error.argtypes = [vp]
    lib.sf_head_last_error.restype = ctypes.c_char_p
    lib.sf_head_destroy.argtypes = [vp]
    for name in EXPORTS:
        fn = getattr(lib, name)
        if name not in ("sf_status_str", "sf_last_error", "sf_head_last_error"):
            fn.restype = c_int
    return lib


class _LazyLib:
    """Loads libspecfold.so on first use so that the build module inside this
    package can be imported on a machine where it is not built yet; any call
    into the binding without the library raises ImportError."""

    _cdll = None

    def __getattr__(self, name):
        if _LazyLib._cdll is None:
            _LazyLib._cdll = _load()
        return getattr(_LazyLib._cdll, name)


lib = _LazyLib()


def _check(st: int, ctx=None, what: str = "", head=None):
    if st != SF_OK:
        msg = lib.sf_status_str(st).decode()
        if ctx or head:
            extra = (lib.sf_last_error(ctx) if ctx else lib.sf_head_last_error(head)).decode()
            if extra:
                msg += f": {extra}"
        raise SpecFoldError(st, f"{what}: {msg}" if what else msg)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    h = int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)
    return h or None


# ---------------------------------------------------------------- C-ABI mirrors

def sf_create(shapes: SfShapes, layers: Sequence[SfLayerWeights]) -> int:
    arr = (SfLayerWeights * len(layers))(*layers)
    ctx = ctypes.c_void_p()
    _check(lib.sf_create(ctypes.byref(shapes), arr, ctypes.byref(ctx)), None, "sf_create")
    return ctx.value


def sf_verify(ctx, stream, hidden_in, parent, prefix_k, prefix_v, R, B, P, delta, hidden_out,
              fold_mask=None, src=None, rc_count=None) -> None:
    par = np.ascontiguousarray(parent, dtype=np.int32)
    _check(lib.sf_verify(ctx, stream, hidden_in, par.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), prefix_k,
                         prefix_v, int(R), int(B), int(P), float(delta), hidden_out, fold_mask, src, rc_count),
           ctx, "sf_verify")


def sf_set_debug(ctx, layer_hidden, rc_rows) -> None:
    _check(lib.sf_set_debug(ctx, layer_hidden, rc_rows), ctx, "sf_set_debug")


def sf_set_attention_mode(ctx, mode: int) -> None:
    _check(lib.sf_set_attention_mode(ctx, int(mode)), ctx, "sf_set_attention_mode")


def sf_set_rho_dump(ctx, rho) -> None:
    _check(lib.sf_set_rho_dump(ctx, rho), ctx, "sf_set_rho_dump")


def sf_sync_status(ctx, stream) -> None:
    _check(lib.sf_sync_status(ctx, stream), ctx, "sf_sync_status")


def sf_inject_stall(ctx, on: bool) -> None:
    _check(lib.sf_inject_stall(ctx, int(bool(on))), ctx, "sf_inject_stall")


def sf_destroy(ctx) -> None:
    _check(lib.sf_destroy(ctx), None, "sf_destroy")


def sf_get_stats(ctx) -> dict:
    s = SfStats()
    _check(lib.sf_get_stats(ctx, ctypes.byref(s)), ctx, "sf_get_stats")
    return {"passes": s.passes, "kernel_launches": s.kernel_launches, "graph_replays": s.graph_replays,
            "family_launches": {FAMILIES[i]: s.family_launches[i] for i in range(SF_K_COUNT)}}


def sf_set_graphs(ctx, on: bool) -> None:
    _check(lib.sf_set_graphs(ctx, int(bool(on))), ctx, "sf_set_graphs")


def sf_timing_begin(ctx, families: Sequence[str]) -> None:
    mask = 0
    for f in families:
        mask |= 1 << FAMILIES.index(f)
    _check(lib.sf_timing_begin(ctx, mask), ctx, "sf_timing_begin")


def sf_timing_read(ctx) -> dict:
    ms = (ctypes.c_double * SF_K_COUNT)()
    n = (ctypes.c_int64 * SF_K_COUNT)()
    _check(lib.sf_timing_read(ctx, ms, n), ctx, "sf_timing_read")
    return {FAMILIES[i]: (ms[i], n[i]) for i in range(SF_K_COUNT) if n[i] > 0}


def sf_timing_list(ctx, family: str) -> List[float]:
    """Durations (ms) of the timed launches of one family, in launch order."""
    n = ctypes.c_int(0)
    _check(lib.sf_timing_list(ctx, FAMILIES.index(family), None, 0, ctypes.byref(n)), ctx, "sf_timing_list")
    buf = (ctypes.c_double * max(1, n.value))()
    _check(lib.sf_timing_list(ctx, FAMILIES.index(family), buf, n.value, ctypes.byref(n)), ctx, "sf_timing_list")
    return [buf[i] for i in range(n.value)]


def sfk_gemm_bf16(stream, X, rows_cap, W, M, K, count, dense_count, Y, ldy, splits, err=None) -> None:
    _check(lib.sfk_gemm_bf16(stream, X, int(rows_cap), W, int(M), int(K), count, int(dense_count), Y, int(ldy),
                             int(splits), err), None, "sfk_gemm_bf16")


def sfk_gate_noalloc(stream, hidden, dtype, parent, R, B, L, d, delta, H_out, fold, rc, rcslot, src,
                     rc_count) -> None:
    par = np.ascontiguousarray(parent, dtype=np.int32)
    _check(lib.sfk_gate_noalloc(stream, hidden, int(dtype), par.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                int(R), int(B), int(L), int(d), float(delta), H_out, fold, rc, rcslot, src,
                                rc_count), None, "sfk_gate_noalloc")


def sf_head_create(shapes: SfHeadShapes, final_norm, w_lm) -> int:
    h = ctypes.c_void_p()
    _check(lib.sf_head_create(ctypes.byref(shapes), final_norm, w_lm, ctypes.byref(h)), None, "sf_head_create")
    return h.value


def sf_head_verify(head, stream, hidden, tokens, parent, R, B, L, pred, accepted=None, chosen=None) -> None:
    par = np.ascontiguousarray(parent, dtype=np.int32)
    _check(lib.sf_head_verify(head, stream, hidden, tokens, par.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                              int(R), int(B), int(L), pred, accepted, chosen), None, "sf_head_verify", head=head)


def sf_head_destroy(head) -> None:
    _check(lib.sf_head_destroy(head), None, "sf_head_destroy")


# ---------------------------------------------------------------- torch convenience

class SpecFold:
    """A context over torch tensors.

    weights: per layer a dict with attn_norm, wq, wk, wv, wo, ffn_norm,
    w_gate, w_up, w_down (CUDA tensors, [in, out] row-major; gains fp32)."""

    def __init__(self, *, n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn, dtype, block_len,
                 max_requests, max_branches, max_prefix, weights: List[dict], rms_eps=1e-6,
                 rope_theta=10000.0):
        self.shapes = SfShapes(n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn,
                               SF_BF16 if dtype in ("bf16", SF_BF16) else SF_F32, rms_eps, rope_theta,
                               block_len, max_requests, max_branches, max_prefix)
        layers = []
        for w in weights:
            for k, t in w.items():
                if not t.is_cuda or not t.is_contiguous():
                    raise ValueError(f"weight {k} must be a contiguous CUDA tensor")
            layers.append(SfLayerWeights(*[_ptr(w[n]) for n in
                                           ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate",
                                            "w_up", "w_down")]))
        self.ctx = sf_create(self.shapes, layers)

    def close(self):
        if getattr(self, "ctx", None):
            sf_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def verify(self, hidden, parent, prefix_k, prefix_v, delta, *, out=None, fold=None, src=None,
               rc_count=None, stream=None, want_masks=True):
        """Enqueue one pass; returns (out, fold_mask, src, rc_count) tensors."""
        import torch
        parent = np.asarray(parent, dtype=np.int32)
        R, Bp = parent.shape
        L, nl = self.shapes.block_len, self.shapes.n_layers
        P = 0 if prefix_k is None else int(prefix_k.shape[2])
        dev = hidden.device
        if out is None:
            out = torch.empty_like(hidden)
        if want_masks:
            if fold is None:
                fold = torch.empty((nl, R, Bp, L), dtype=torch.uint8, device=dev)
            if src is None:
                src = torch.empty((nl, R, Bp, L), dtype=torch.int32, device=dev)
            if rc_count is None:
                rc_count = torch.empty((nl,), dtype=torch.int32, device=dev)
        sf_verify(self.ctx, _stream_handle(stream), _ptr(hidden), parent, _ptr(prefix_k), _ptr(prefix_v), R,
                  Bp - 1, P, delta, _ptr(out), _ptr(fold), _ptr(src), _ptr(rc_count))
        return out, fold, src, rc_count

    def set_debug(self, layer_hidden=None, rc_rows=None):
        sf_set_debug(self.ctx, _ptr(layer_hidden), _ptr(rc_rows))

    def set_attention_mode(self, mode: int):
        sf_set_attention_mode(self.ctx, mode)

    def set_rho_dump(self, rho=None):
        sf_set_rho_dump(self.ctx, _ptr(rho))

    def sync(self, stream=None):
        sf_sync_status(self.ctx, _stream_handle(stream))

    def stats(self):
        return sf_get_stats(self.ctx)

    def set_graphs(self, on: bool):
        sf_set_graphs(self.ctx, on)


class Head:
    """The verification head over torch tensors: final RMSNorm, LM head,
    greedy tokens and draft acceptance of a pass output.

    final_norm: fp32 CUDA tensor [d]; w_lm: CUDA tensor [d, vocab] in the
    context dtype."""

    def __init__(self, *, d_model, vocab, dtype, max_rows, final_norm, w_lm, rms_eps=1e-6):
        for name, t in (("final_norm", final_norm), ("w_lm", w_lm)):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CUDA tensor")
        self.shapes = SfHeadShapes(d_model, vocab, SF_BF16 if dtype in ("bf16", SF_BF16) else SF_F32, rms_eps,
                                   max_rows)
        self.head = sf_head_create(self.shapes, _ptr(final_norm), _ptr(w_lm))

    def close(self):
        if getattr(self, "head", None):
            sf_head_destroy(self.head)
            self.head = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def verify(self, hidden, tokens, parent, *, pred=None, accepted=None, chosen=None, stream=None):
        """Enqueue the head for one pass output; returns (pred, accepted, chosen)."""
        import torch
        parent = np.asarray(parent, dtype=np.int32)
        R, Bp = parent.shape
        L = int(hidden.shape[2])
        dev = hidden.device
        if pred is None:
            pred = torch.empty((R, Bp, L), dtype=torch.int32, device=dev)
        if accepted is None:
            accepted = torch.empty((R, Bp), dtype=torch.uint8, device=dev)
        if chosen is None:
            chosen = torch.empty((R,), dtype=torch.int32, device=dev)
        sf_head_verify(self.head, _stream_handle(stream), _ptr(hidden), _ptr(tokens), parent, R, Bp - 1, L,
                       _ptr(pred), _ptr(accepted), _ptr(chosen))
        return pred, accepted, chosen


def from_config(cfg, weights, max_requests=None, max_branches=None, max_prefix=None) -> SpecFold:
    """Context for a workload description with the fields of synth.Config."""
    return SpecFold(n_layers=cfg.n_layers, d_model=cfg.d_model, n_q_heads=cfg.n_q_heads,
                    n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, d_ffn=cfg.d_ffn, dtype=cfg.dtype,
                    block_len=cfg.block_len, max_requests=max_requests or cfg.n_requests,
                    max_branches=max_branches or cfg.n_branches, max_prefix=max_prefix or cfg.prefix_len,
                    weights=weights, rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta)
