"""Pins of the oracle's building blocks against hand-derived fixtures, closed
forms and library special cases (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [c.split() for c in line.split("|")]


# ---------------------------------------------------------------- gate

def test_gate_golden():
    n = 0
    for hp, hc, rho, delta, fold in _rows("gate_rho.txt"):
        hp = np.array(hp, float)
        hc = np.array(hc, float)
        want = float(rho[0])
        got = oracle.relative_residual(hc, hp)
        if math.isinf(want):
            assert math.isinf(got)
        else:
            assert got == pytest.approx(want, rel=1e-15, abs=1e-15)
        assert bool(oracle.fold_decision(got, float(delta[0]))) == bool(int(fold[0]))
        n += 1
    assert n >= 10


def test_gate_request_main_branch_never_folds():
    H = np.zeros((3, 4, 8))
    fold, rho = oracle.gate_request(H, [-1, 0, 1], 0.5)
    assert not fold[0].any()
    assert np.isnan(rho[0]).all()
    assert fold[1:].all()          # all-zero rows: rho = 0 <= delta


def test_gate_request_uses_own_parent():
    rng = np.random.default_rng(1)
    H = rng.normal(size=(4, 3, 16))
    parent = [-1, 0, 0, 2]
    _, rho = oracle.gate_request(H, parent, 0.1)
    for i in range(1, 4):
        for n in range(3):
            d = H[i, n] - H[parent[i], n]
            assert rho[i, n] == pytest.approx(np.linalg.norm(d) / np.linalg.norm(H[parent[i], n]))


def test_gate_forced_override():
    H = np.zeros((2, 3, 4))
    forced = -np.ones((2, 3), int)
    forced[1, 1] = 0
    fold, _ = oracle.gate_request(H, [-1, 0], 0.1, forced)
    assert fold[1].tolist() == [True, False, True]


# ---------------------------------------------------------------- compaction / resolution

def test_tree_resolution_golden():
    g = json.load(open(os.path.join(GOLD, "tree_resolution.json")))
    fold = np.array(g["fold"], bool)
    src = oracle.resolve_sources(fold, g["parent"])
    assert src.tolist() == g["src"]
    rc, counts, offsets = oracle.compaction(fold[None])
    assert rc.tolist() == g["rc"]
    assert counts[0].tolist() == g["counts"]
    assert offsets[0].tolist() == g["offsets"]
    L = g["L"]
    slot = {int(r): k for k, r in enumerate(rc)}
    rcslot = [[slot[src[i, n] * L + n] for n in range(L)] for i in range(len(g["parent"]))]
    assert rcslot == g["rcslot"]


def test_resolution_properties_random_trees():
    rng = np.random.default_rng(5)
    for _ in range(50):
        Bp = int(rng.integers(1, 10))
        L = int(rng.integers(1, 12))
        parent = [-1] + [int(rng.integers(0, i)) for i in range(1, Bp)]
        fold = rng.random((Bp, L)) < 0.6
        fold[0] = False
        src = oracle.resolve_sources(fold, parent)
        for i in range(Bp):
            for n in range(L):
                s = src[i, n]
                assert not fold[s, n]                    # the source recomputed n
                j = i
                while j != s:                            # every step on the way folded n
                    assert fold[j, n]
                    j = parent[j]
                    assert j >= 0                        # s is an ancestor-or-self


def test_compaction_multi_request_order():
    fold = np.array([[[0, 1], [1, 0]], [[0, 0], [1, 1]]], bool)   # R=2, Bp=2, L=2
    rc, counts, offsets = oracle.compaction(fold)
    assert rc.tolist() == [0, 3, 4, 5]
    assert counts.tolist() == [[1, 1], [2, 0]]
    assert offsets.tolist() == [[0, 1], [2, 4]]


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_closed_form():
    c, eps, d = -3.0, 1e-6, 10
    out = oracle.rms_norm(np.full(d, c), np.full(d, 2.0), eps)
    np.testing.assert_allclose(out, np.full(d, 2.0 * c / math.sqrt(c * c + eps)), rtol=1e-15)


def test_rms_norm_vs_torch():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(7, 33))
    g = rng.normal(size=33)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (33,), torch.tensor(g), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, g, 1e-5), ref, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- RoPE

def test_rope_golden():
    for pos, x, want in _rows("rope.txt"):
        x = np.array(x, float).reshape(1, 4)
        got = oracle.rope(x, np.array(float(pos[0])), 10000.0)
        np.testing.assert_allclose(got.reshape(4), np.array(want, float), rtol=1e-14, atol=1e-14)


def test_rope_complex_form():
    """Rotate-half RoPE equals multiplication by e^{i a_j} of the complex
    numbers (x_j + i x_{j+hd/2})."""
    rng = np.random.default_rng(3)
    hd, theta = 16, 500.0
    x = rng.normal(size=(5, 3, hd))
    pos = np.array([0, 1, 7, 100, 4095], float)
    z = torch.complex(torch.tensor(x[..., : hd // 2]), torch.tensor(x[..., hd // 2:]))
    freqs = torch.tensor(theta) ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones(5, 1, hd // 2, dtype=torch.float64),
                      torch.tensor(pos)[:, None, None] * freqs)
    zr = z * rot
    ref = torch.cat([zr.real, zr.imag], dim=-1).numpy()
    np.testing.assert_allclose(oracle.rope(x, pos, theta), ref, rtol=1e-12, atol=1e-12)


def test_rope_relative_position_and_norm():
    rng = np.random.default_rng(4)
    hd = 32
    q = rng.normal(size=(1, hd))
    k = rng.normal(size=(1, hd))
    dots = []
    for shift in (0, 3, 50):
        qa = oracle.rope(q, np.array(10.0 + shift), 10000.0)
        kb = oracle.rope(k, np.array(4.0 + shift), 10000.0)
        dots.append(float(qa.ravel() @ kb.ravel()))
        assert np.linalg.norm(qa) == pytest.approx(np.linalg.norm(q), rel=1e-13)
    assert dots[1] == pytest.approx(dots[0], rel=1e-10)
    assert dots[2] == pytest.approx(dots[0], rel=1e-10)


# ---------------------------------------------------------------- FFN

def test_swiglu_golden():
    g = json.load(open(os.path.join(GOLD, "swiglu.json")))
    W = {"ffn_norm": np.ones(2), "w_gate": np.array(g["w_gate"]), "w_up": np.array(g["w_up"]),
         "w_down": np.array(g["w_down"])}
    x = np.array(g["x"])
    # feed a row whose RMSNorm with gain 1 and eps 0 is x itself times 1/rms(x);
    # scale back so the FFN sees x exactly
    class C:
        rms_eps = 0.0
    rms = math.sqrt(np.mean(x * x))
    xn = oracle.rms_norm(x[None], np.ones(2), 0.0)[0]
    np.testing.assert_allclose(xn * rms, x, rtol=1e-15)
    W["ffn_norm"] = np.full(2, rms)
    out = oracle.ffn(x[None], W, C)[0]
    np.testing.assert_allclose(out, np.array(g["expected"]), rtol=1e-14)


# ---------------------------------------------------------------- attention

def test_attention_vs_torch_sdpa_gqa():
    rng = np.random.default_rng(6)
    n, nq, nkv, hd, S = 6, 8, 2, 16, 23
    q = rng.normal(size=(n, nq, hd))
    K = rng.normal(size=(S, nkv, hd))
    V = rng.normal(size=(S, nkv, hd))
    G = nq // nkv
    qt = torch.tensor(q).permute(1, 0, 2)                        # [nq, n, hd]
    Kt = torch.tensor(K).permute(1, 0, 2).repeat_interleave(G, 0)  # [nq, S, hd]
    Vt = torch.tensor(V).permute(1, 0, 2).repeat_interleave(G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)  # [nq, n, hd]
    ref = ref.permute(1, 0, 2).reshape(n, nq * hd).numpy()
    np.testing.assert_allclose(oracle.attention(q, K, V), ref, rtol=1e-12, atol=1e-13)


def test_attention_single_key_returns_value():
    q = np.ones((1, 2, 4))
    K = np.zeros((1, 1, 4))
    V = np.arange(4.0).reshape(1, 1, 4)
    np.testing.assert_allclose(oracle.attention(q, K, V), np.tile(np.arange(4.0), 2)[None])


def test_lse_merge_identity():
    """Prefix partial merged with block partial equals the direct softmax."""
    rng = np.random.default_rng(7)
    nq, nkv, hd, P, L = 6, 2, 8, 11, 5
    q = rng.normal(size=(nq, hd))
    K = rng.normal(size=(P + L, nkv, hd)) * 2
    V = rng.normal(size=(P + L, nkv, hd))
    m, l, acc = oracle.merge_states([oracle.softmax_state(q, K[:P], V[:P]),
                                     oracle.softmax_state(q, K[P:], V[P:])])
    direct = oracle.attention(q[None], K, V)[0]
    np.testing.assert_allclose((acc / l[:, None]).reshape(-1), direct, rtol=1e-12, atol=1e-13)


def test_paper_style_correction_equals_direct():
    """§A.1: parent state minus the parent's changed keys plus the child's."""
    rng = np.random.default_rng(8)
    nq, nkv, hd, S = 4, 2, 8, 20
    q = rng.normal(size=(nq, hd))
    Kp = rng.normal(size=(S, nkv, hd))
    Vp = rng.normal(size=(S, nkv, hd))
    changed = np.zeros(S, bool)
    changed[[3, 11, 12]] = True
    Ko, Vo = Kp.copy(), Vp.copy()
    Ko[changed] = rng.normal(size=(3, nkv, hd)) * 1.5
    Vo[changed] = rng.normal(size=(3, nkv, hd))
    got = oracle.corrected_attention(q, Kp, Vp, Ko, Vo, changed)
    np.testing.assert_allclose(got, oracle.attention(q[None], Ko, Vo)[0], rtol=1e-10, atol=1e-12)
    # nothing changed -> the parent's own attention
    got0 = oracle.corrected_attention(q, Kp, Vp, Kp, Vp, np.zeros(S, bool))
    np.testing.assert_allclose(got0, oracle.attention(q[None], Kp, Vp)[0], rtol=1e-13)


# ---------------------------------------------------------------- verification head

def test_acceptance_golden():
    """Hand-worked draft acceptance on a 6-branch tree (tests/golden/acceptance.json)."""
    import json
    g = json.load(open(os.path.join(GOLD, "acceptance.json")))
    for case in g["cases"]:
        acc, chosen = oracle.accept_drafts(np.array(g["tokens"]), g["parent"], np.array(case["pred"]))
        assert acc.astype(int).tolist() == case["accepted"]
        assert chosen == case["chosen"]


def test_acceptance_invariants():
    """Main always matches; a child equal to its parent matches iff the parent
    does; a child of a rejected draft is rejected whatever it holds."""
    rng = np.random.default_rng(3)
    for _ in range(50):
        Bp, L = 7, 8
        parent = [-1] + [int(rng.integers(0, i)) for i in range(1, Bp)]
        tokens = rng.integers(0, 4, size=(Bp, L))
        pred = rng.integers(0, 4, size=(Bp, L))
        for i in range(1, Bp):                      # some children copy their parent
            if rng.random() < 0.4:
                tokens[i] = tokens[parent[i]]
        acc, chosen = oracle.accept_drafts(tokens, parent, pred)
        assert acc[0] and acc[chosen]
        for i in range(1, Bp):
            if not acc[parent[i]]:
                assert not acc[i]
            if np.array_equal(tokens[i], tokens[parent[i]]):
                assert acc[i] == acc[parent[i]]


def test_greedy_tokens_take_the_first_maximum():
    assert oracle.greedy_tokens(np.array([[1.0, 3.0, 3.0, 0.0], [-2.0, -1.0, -1.5, -1.0]])).tolist() == [1, 1]


def test_lm_head_logits_match_torch():
    """Final RMSNorm + LM head equals torch's rms_norm followed by a matmul."""
    rng = np.random.default_rng(4)
    h = rng.standard_normal((5, 24))
    g = rng.uniform(0.5, 1.5, 24)
    W = rng.standard_normal((24, 40))
    want = torch.nn.functional.rms_norm(torch.tensor(h), (24,), torch.tensor(g), eps=1e-6) @ torch.tensor(W)
    np.testing.assert_allclose(oracle.lm_head_logits(h, g, W, 1e-6), want.numpy(), rtol=1e-12, atol=1e-12)
