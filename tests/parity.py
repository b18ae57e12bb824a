"""Helpers shared by the GPU parity tests: run the CUDA path through the
C-ABI binding and compare it with the float64 oracle on the same seeded
inputs.

Tolerances (the comparison the workload description fixes):
* fold masks, compaction lists and resolved sources: bit-exact, except for
  positions whose oracle rho lies within 1e-4 * delta of delta, where either
  decision is accepted and the oracle takes the GPU's;
* hidden states: per row ||gpu - ref||_inf / max(||ref||_inf, 1e-6), maximum
  over rows, at most 1e-4 for fp32 contexts and 2e-2 for bf16 contexts.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

TOL = {"f32": 1e-4, "bf16": 2e-2}
BAND = 1e-4


def rel_err_rows(got: np.ndarray, want: np.ndarray) -> float:
    got = got.reshape(-1, got.shape[-1])
    want = want.reshape(-1, want.shape[-1])
    num = np.abs(got - want).max(axis=1)
    den = np.maximum(np.abs(want).max(axis=1), 1e-6)
    return float((num / den).max()) if got.size else 0.0


def run_gpu(cfg, wl, delta, debug=True, graphs=True, ctx=None):
    import torch
    import sparse_reuse_gb300 as sf
    own = ctx is None
    if own:
        ctx = sf.from_config(cfg, wl.weights)
    ctx.set_graphs(graphs)
    T, d, nl = cfg.rows, cfg.d_model, cfg.n_layers
    dbg = rcs = None
    if debug:
        dbg = torch.zeros((nl + 1, T, d), dtype=torch.float32, device="cuda")
        rcs = torch.full((nl, T), -1, dtype=torch.int32, device="cuda")
        ctx.set_debug(dbg, rcs)
    out, fold, src, rc_count = ctx.verify(wl.hidden, wl.parents, wl.prefix_k if cfg.prefix_len else None,
                                          wl.prefix_v if cfg.prefix_len else None, delta)
    ctx.sync()
    res = {"out": out.float().cpu().numpy(), "fold": fold.cpu().numpy().astype(bool),
           "src": src.cpu().numpy().astype(np.int64), "rc_count": rc_count.cpu().numpy().astype(np.int64),
           "stats": ctx.stats()}
    if debug:
        res["layer_hidden"] = dbg.cpu().numpy()
        res["rc_rows"] = rcs.cpu().numpy().astype(np.int64)
        ctx.set_debug(None, None)
    if own:
        ctx.close()
    return res


def oracle_inputs(wl):
    return (wl.hidden.double().cpu().numpy(), wl.prefix_k.double().cpu().numpy(),
            wl.prefix_v.double().cpu().numpy())


def check_free_running(cfg, wl, gpu, delta, tol=None, exact_masks=True):
    """Whole pass of the oracle from the same inputs; returns the oracle result."""
    H0, pk, pv = oracle_inputs(wl)
    Ws = {}

    def get_layer(l):
        if l not in Ws:
            Ws[l] = oracle.layer_weights_f64(wl.weights[l])
        return Ws[l]

    ref = oracle.verify_pass(H0, wl.parents, delta, get_layer, pk, pv, cfg, form="tables")
    if exact_masks:
        assert np.array_equal(gpu["fold"], ref["fold"]), _mask_diff(gpu["fold"], ref["fold"])
        assert np.array_equal(gpu["src"], ref["src"])
        assert gpu["rc_count"].tolist() == ref["rc_count"].tolist()
        if "rc_rows" in gpu:
            for l, rc in enumerate(ref["rc"]):
                assert np.array_equal(gpu["rc_rows"][l, :rc.size], rc)
    tol = TOL[cfg.dtype] if tol is None else tol
    err = rel_err_rows(gpu["out"], ref["out"])
    assert err <= tol, f"free-running hidden rel err {err:.3e} > {tol}"
    return ref, err


def _mask_diff(a, b):
    idx = np.argwhere(a != b)
    return f"{len(idx)} fold decisions differ, first at (layer, r, i, n) = {idx[:5].tolist()}"


def check_teacher_forced(cfg, wl, gpu, delta, layers, tol=None):
    """For each sampled layer l, run the oracle's layer l from the GPU's own
    fp32 layer input and compare decisions, lists and the layer output.
    Returns the max relative error over the sampled layers."""
    _, pk_all, pv_all = None, wl.prefix_k, wl.prefix_v
    tol = TOL[cfg.dtype] if tol is None else tol
    R, Bp, L, d = cfg.n_requests, cfg.n_branches, cfg.block_len, cfg.d_model
    worst = 0.0
    for l in layers:
        W = oracle.layer_weights_f64(wl.weights[l])
        H_in = gpu["layer_hidden"][l].astype(np.float64).reshape(R, Bp, L, d)
        want_out = gpu["layer_hidden"][l + 1].reshape(R, Bp, L, d)
        folds = np.zeros((R, Bp, L), bool)
        for r in range(R):
            pk = pk_all[l, r].double().cpu().numpy() if cfg.prefix_len else np.zeros((0, cfg.n_kv_heads, cfg.head_dim))
            pv = pv_all[l, r].double().cpu().numpy() if cfg.prefix_len else np.zeros((0, cfg.n_kv_heads, cfg.head_dim))
            _, rho = oracle.gate_request(H_in[r], wl.parents[r], delta)
            forced = -np.ones((Bp, L), dtype=np.int64)
            if delta > 0:
                band = np.abs(rho - delta) <= BAND * delta
                forced[band] = gpu["fold"][l, r][band]
            out, fold, rho, src = oracle.folded_layer_resolved(H_in[r], wl.parents[r], delta, W, pk, pv, cfg,
                                                               forced)
            assert np.array_equal(gpu["fold"][l, r], fold), f"layer {l} request {r}: fold masks differ"
            assert np.array_equal(gpu["src"][l, r], src), f"layer {l} request {r}: sources differ"
            folds[r] = fold
            err = rel_err_rows(want_out[r], out)
            worst = max(worst, err)
            assert err <= tol, f"layer {l} request {r}: rel err {err:.3e} > {tol}"
        rc, _, _ = oracle.compaction(folds)
        assert gpu["rc_count"][l] == rc.size
        if "rc_rows" in gpu:
            assert np.array_equal(gpu["rc_rows"][l, :rc.size], rc), f"layer {l}: recompute lists differ"
    return worst
