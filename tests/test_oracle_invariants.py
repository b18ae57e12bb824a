"""Whole-layer pins of the oracle (CPU only).

* delta = 0 recovers dense per-branch recomputation (SpecFold summary §4.3:
  delta -> 0 approaches Spiffy, i.e. dense verification; App. C: serialized
  per-branch verification), and that dense layer equals an independent
  textbook layer written here with torch primitives (sdpa, rms_norm, complex
  rotary, silu).
* A child whose tokens equal its parent's folds everything and reproduces the
  parent bit for bit (§3.2 / §A.2: folded positions reuse the parent's outputs).
* The main branch never depends on delta (App. B: the main branch bypasses the gate).
* The topological table form (§A.3) equals the order-free resolved-source
  form (App. B) and a scalar brute force.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _setup(cfg, seed=0):
    wl = synth.make_workload(cfg, seed)
    Ws = [oracle.layer_weights_f64(w) for w in wl.weights]
    H = wl.hidden.double().numpy()
    pk = wl.prefix_k.double().numpy()
    pv = wl.prefix_v.double().numpy()
    return wl, Ws, H, pk, pv


def textbook_layer(x, W, pk, pv, cfg):
    """Independent dense layer in torch: [L, d] -> [L, d]."""
    x = torch.tensor(x)
    L, d = x.shape
    nq, nkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    Wt = {k: torch.tensor(v) for k, v in W.items()}
    P = pk.shape[0]
    xn = torch.nn.functional.rms_norm(x, (d,), Wt["attn_norm"], eps=cfg.rms_eps)
    q = (xn @ Wt["wq"]).view(L, nq, hd)
    k = (xn @ Wt["wk"]).view(L, nkv, hd)
    v = (xn @ Wt["wv"]).view(L, nkv, hd)
    freqs = torch.tensor(cfg.rope_theta, dtype=torch.float64) ** (
        -torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    ang = torch.arange(P, P + L, dtype=torch.float64)[:, None, None] * freqs
    rot = torch.polar(torch.ones_like(ang), ang)

    def rope(t):
        z = torch.complex(t[..., : hd // 2], t[..., hd // 2:]) * rot
        return torch.cat([z.real, z.imag], -1)

    q, k = rope(q), rope(k)
    K = torch.cat([torch.tensor(pk), k], 0).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
    V = torch.cat([torch.tensor(pv), v], 0).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
    a = torch.nn.functional.scaled_dot_product_attention(q.permute(1, 0, 2), K, V)
    h = x + a.permute(1, 0, 2).reshape(L, nq * hd) @ Wt["wo"]
    hn = torch.nn.functional.rms_norm(h, (d,), Wt["ffn_norm"], eps=cfg.rms_eps)
    f = (torch.nn.functional.silu(hn @ Wt["w_gate"]) * (hn @ Wt["w_up"])) @ Wt["w_down"]
    return (h + f).numpy()


CFG = synth.small_config(n_layers=2, n_drafts=4, prefix_len=5)


def test_dense_layer_matches_textbook():
    wl, Ws, H, pk, pv = _setup(CFG)
    for i in range(CFG.n_branches):
        got = oracle.dense_layer(H[0, i], Ws[0], pk[0, 0], pv[0, 0], CFG)
        ref = textbook_layer(H[0, i], Ws[0], pk[0, 0], pv[0, 0], CFG)
        np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-13)


def test_textbook_catches_plausible_mistakes():
    """The textbook comparison is sensitive to a transposed W_o, a dropped
    residual or a swapped rotary pairing (applied to the oracle's inputs)."""
    wl, Ws, H, pk, pv = _setup(CFG)
    ref = textbook_layer(H[0, 1], Ws[0], pk[0, 0], pv[0, 0], CFG)
    bad = dict(Ws[0])
    bad["w_gate"], bad["w_up"] = Ws[0]["w_up"], Ws[0]["w_gate"]
    got = oracle.dense_layer(H[0, 1], bad, pk[0, 0], pv[0, 0], CFG)
    assert np.max(np.abs(got - ref)) > 1e-6


@pytest.mark.parametrize("form", ["tables", "resolved"])
def test_delta_zero_is_dense_per_branch(form):
    wl, Ws, H, pk, pv = _setup(CFG)
    res = oracle.verify_pass(H, wl.parents, 0.0, lambda l: Ws[l], pk, pv, CFG, form=form)
    assert not res["fold"].any()
    for i in range(CFG.n_branches):
        x = H[0, i]
        for l in range(CFG.n_layers):
            x = textbook_layer(x, Ws[l], pk[l, 0], pv[l, 0], CFG)
        np.testing.assert_allclose(res["out"][0, i], x, rtol=1e-10, atol=1e-12)


def test_identical_child_folds_everything_and_reproduces_parent():
    cfg = CFG.with_(n_drafts=3, tree="chain")
    wl, Ws, H, pk, pv = _setup(cfg)
    H = H.copy()
    H[0, 3] = H[0, 2]                      # branch 3's block equals its parent's
    res = oracle.verify_pass(H, wl.parents, 0.1, lambda l: Ws[l], pk, pv, cfg)
    assert res["fold"][:, 0, 3].all()
    assert np.array_equal(res["out"][0, 3], res["out"][0, 2])
    # and its sources are the parent's sources at every layer
    assert np.array_equal(res["src"][:, 0, 3], res["src"][:, 0, 2])


def test_main_branch_independent_of_delta():
    wl, Ws, H, pk, pv = _setup(CFG)
    outs = [oracle.verify_pass(H, wl.parents, d, lambda l: Ws[l], pk, pv, CFG)["out"][0, 0]
            for d in (0.0, 0.05, 0.5, 10.0)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def _mixed_delta(wl, Ws, H, pk, pv, cfg):
    """A delta near the median draft rho of layer 0 so both decisions occur."""
    _, rho = oracle.gate_request(H[0], wl.parents[0], 1.0)
    r = rho[1:].ravel()
    r = r[np.isfinite(r) & (r > 0)]
    return float(np.median(r)) if r.size else 0.1


def test_table_form_equals_resolved_form():
    for seed in range(3):
        cfg = CFG.with_(n_drafts=6, max_depth=3)
        wl, Ws, H, pk, pv = _setup(cfg, seed)
        delta = max(_mixed_delta(wl, Ws, H, pk, pv, cfg), 0.3)
        a = oracle.verify_pass(H, wl.parents, delta, lambda l: Ws[l], pk, pv, cfg, form="tables")
        b = oracle.verify_pass(H, wl.parents, delta, lambda l: Ws[l], pk, pv, cfg, form="resolved")
        assert np.array_equal(a["fold"], b["fold"])
        assert np.array_equal(a["src"], b["src"])
        assert a["fold"].any() and (~a["fold"][:, :, 1:]).any()
        np.testing.assert_allclose(a["out"], b["out"], rtol=1e-12, atol=1e-13)


def test_folding_changes_results_where_it_should():
    """Folded rows inherit outputs, so at a positive delta the draft outputs
    differ from dense recomputation while the main branch does not."""
    cfg = CFG.with_(n_drafts=4)
    wl, Ws, H, pk, pv = _setup(cfg, 1)
    a = oracle.verify_pass(H, wl.parents, 0.0, lambda l: Ws[l], pk, pv, cfg)
    b = oracle.verify_pass(H, wl.parents, 0.5, lambda l: Ws[l], pk, pv, cfg)
    assert b["fold"].any()
    assert np.array_equal(a["out"][0, 0], b["out"][0, 0])
    assert np.max(np.abs(a["out"][0, 1:] - b["out"][0, 1:])) > 0


def test_multi_request_is_per_request():
    cfg = CFG.with_(n_requests=2, n_drafts=3, n_layers=1)
    wl, Ws, H, pk, pv = _setup(cfg)
    both = oracle.verify_pass(H, wl.parents, 0.2, lambda l: Ws[l], pk, pv, cfg)
    for r in range(2):
        one = oracle.verify_pass(H[r:r + 1], wl.parents[r:r + 1], 0.2, lambda l: Ws[l],
                                 pk[:, r:r + 1], pv[:, r:r + 1], cfg.with_(n_requests=1))
        assert np.array_equal(one["out"][0], both["out"][r])
        assert np.array_equal(one["fold"][:, 0], both["fold"][:, r])


def test_bruteforce_matches_tables():
    cfg = synth.small_config(n_layers=1, d_model=16, n_q_heads=4, n_kv_heads=2, head_dim=4,
                             d_ffn=24, block_len=4, prefix_len=3, n_drafts=3)
    wl, Ws, H, pk, pv = _setup(cfg, 2)
    for delta in (0.0, 0.3, 1.0):
        out, fold, _ = oracle.folded_layer(H[0], wl.parents[0], delta, Ws[0], pk[0, 0], pv[0, 0], cfg)
        bout, bfold = oracle.folded_layer_bruteforce(H[0], wl.parents[0], delta, Ws[0],
                                                     pk[0, 0], pv[0, 0], cfg)
        assert np.array_equal(fold, bfold)
        np.testing.assert_allclose(out, bout, rtol=1e-11, atol=1e-13)


def test_zero_prefix_and_no_drafts():
    cfg = CFG.with_(prefix_len=0, n_drafts=0)
    wl, Ws, H, pk, pv = _setup(cfg)
    res = oracle.verify_pass(H, wl.parents, 0.1, lambda l: Ws[l], pk, pv, cfg)
    x = H[0, 0]
    for l in range(cfg.n_layers):
        x = textbook_layer(x, Ws[l], pk[l, 0], pv[l, 0], cfg)
    np.testing.assert_allclose(res["out"][0, 0], x, rtol=1e-10, atol=1e-12)
    assert res["rc_count"].tolist() == [cfg.block_len] * cfg.n_layers
