"""Verification head (final RMSNorm, LM head, greedy tokens, draft
acceptance) through the C ABI against the oracle (needs a GB300).

The greedy token is an integer decided by floating point: the oracle takes
the decision from the same operands the kernel multiplies (the pass output,
its normalised rows rounded to the context dtype, the weights as stored) in
float64, and a GPU token is accepted when its logit is the row maximum or
within a rounding band of it (a near tie).  Acceptance is integer logic on
the tokens and is compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_reuse_gb300 import build
    build.build()


def _oracle_logits(cfg, hidden, gain, w_lm, rows):
    """fp64 logits of the given rows from the operands the kernel multiplies."""
    h = hidden.reshape(-1, cfg.d_model)[rows].double().cpu().numpy()
    x = oracle.rms_norm(h, gain.double().cpu().numpy(), cfg.rms_eps)
    if cfg.dtype == "bf16":
        x = torch.from_numpy(x).float().to(torch.bfloat16).double().numpy()
    return x @ w_lm.double().cpu().numpy()


def _check_pred(cfg, hidden, gain, w_lm, pred, rows, band):
    logits = _oracle_logits(cfg, hidden, gain, w_lm, rows)
    got = pred.reshape(-1).cpu().numpy()[rows]
    best = logits.max(axis=1)
    mine = logits[np.arange(len(rows)), got]
    scale = np.abs(logits).max(axis=1)
    assert np.all(best - mine <= band * scale), (best - mine)[best - mine > band * scale]
    exact = (got == oracle.greedy_tokens(logits)).mean()
    assert exact >= 0.99, exact
    return got


def _accept_case(sf, cfg, wl, vocab, band, seed=0):
    gain, w_lm = synth.make_head_weights(cfg, vocab, seed, device="cuda")
    gpu = run_gpu(cfg, wl, cfg.delta, debug=False)
    hidden = torch.from_numpy(gpu["out"]).to("cuda").to(wl.hidden.dtype)
    head = sf.Head(d_model=cfg.d_model, vocab=vocab, dtype=cfg.dtype, max_rows=cfg.rows, final_norm=gain, w_lm=w_lm,
                   rms_eps=cfg.rms_eps)
    tok = torch.from_numpy(wl.tokens.astype(np.int32)).to("cuda")
    pred, _, _ = head.verify(hidden, tok, wl.parents)
    torch.cuda.synchronize()
    rows = np.arange(cfg.rows)
    p = _check_pred(cfg, hidden, gain, w_lm, pred, rows, band).reshape(cfg.n_requests, cfg.n_branches, cfg.block_len)
    # drafts built against the predictions: each differs from its parent at
    # one position, holding the parent's prediction there (matches) or not
    rng = np.random.default_rng(seed)
    toks = np.empty_like(wl.tokens, dtype=np.int32)
    for r in range(cfg.n_requests):
        toks[r, 0] = wl.tokens[r, 0]
        for i in range(1, cfg.n_branches):
            par = wl.parents[r, i]
            toks[r, i] = toks[r, par]
            n = int(rng.integers(cfg.block_len))
            toks[r, i, n] = p[r, par, n] if rng.random() < 0.7 else (p[r, par, n] + 1) % vocab
    tok2 = torch.from_numpy(toks).to("cuda")
    pred2, acc, chosen = head.verify(hidden, tok2, wl.parents)
    head.close()
    assert torch.equal(pred2, pred)
    acc = acc.cpu().numpy().astype(bool)
    chosen = chosen.cpu().numpy()
    n_acc = 0
    for r in range(cfg.n_requests):
        want_acc, want_ch = oracle.accept_drafts(toks[r], wl.parents[r], p[r])
        assert np.array_equal(acc[r], want_acc), (r, acc[r], want_acc)
        assert chosen[r] == want_ch
        n_acc += int(want_acc[1:].sum())
    assert 0 < n_acc < cfg.n_requests * cfg.n_drafts     # both outcomes occur


def test_head_fp32_tiny_vocab_not_a_multiple_of_128():
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["tiny"].with_(n_requests=2, n_drafts=5, tree="random", unmask_exact=None)
    wl = synth.make_workload(cfg, seed=21, device="cuda")
    _accept_case(sf, cfg, wl, vocab=1000, band=1e-5)


def test_head_bf16_three_requests():
    import sparse_reuse_gb300 as sf
    cfg = synth.small_config(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=128, d_ffn=320,
                             dtype="bf16", block_len=32, prefix_len=96, n_requests=3, n_drafts=6, delta=0.1)
    wl = synth.make_workload(cfg, seed=22, device="cuda")
    _accept_case(sf, cfg, wl, vocab=5000, band=1e-4)


def test_head_bf16_large_vocab_sampled_rows():
    """1.5B-shaped rows (d = 1536, 288 rows) against the benchmark's 131,072
    entry vocabulary: the LM-head GEMM runs 1,024 vocabulary tiles; 24 rows
    are checked against the oracle."""
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["1.5b"].with_(n_layers=1)
    wl = synth.make_workload(cfg, seed=23, device="cuda")
    gain, w_lm = synth.make_head_weights(cfg, synth.HEAD_VOCAB, 1, device="cuda")
    hidden = (torch.randn(wl.hidden.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(5))
              .to(torch.bfloat16))
    head = sf.Head(d_model=cfg.d_model, vocab=synth.HEAD_VOCAB, dtype="bf16", max_rows=cfg.rows, final_norm=gain,
                   w_lm=w_lm)
    tok = torch.from_numpy(wl.tokens.astype(np.int32)).to("cuda")
    pred, acc, chosen = head.verify(hidden, tok, wl.parents)
    torch.cuda.synchronize()
    head.close()
    rows = np.random.default_rng(0).choice(cfg.rows, 24, replace=False)
    _check_pred(cfg, hidden, gain, w_lm, pred, rows, 1e-4)
    want_acc, want_ch = oracle.accept_drafts(wl.tokens[0], wl.parents[0],
                                             pred.cpu().numpy().reshape(cfg.n_branches, cfg.block_len))
    assert np.array_equal(acc.cpu().numpy()[0].astype(bool), want_acc)
    assert int(chosen.item()) == want_ch


def test_head_argument_errors_launch_nothing():
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["tiny"]
    gain, w_lm = synth.make_head_weights(cfg, 300, 0, device="cuda")
    head = sf.Head(d_model=cfg.d_model, vocab=300, dtype="f32", max_rows=cfg.rows, final_norm=gain, w_lm=w_lm)
    hidden = torch.zeros((1, 3, 32, cfg.d_model), device="cuda")
    tok = torch.zeros((1, 3, 32), dtype=torch.int32, device="cuda")
    pred = torch.zeros((1, 3, 32), dtype=torch.int32, device="cuda")
    for kw, status in [(dict(parent=np.array([[0, 0, 1]])), sf.SF_ERR_TREE),
                       (dict(parent=np.array([[-1, 0, 1, 2]])), sf.SF_ERR_SHAPE),
                       (dict(hidden=hidden.data_ptr() + 4), sf.SF_ERR_INVALID_ARG),
                       (dict(tokens=0), sf.SF_ERR_INVALID_ARG)]:
        par = kw.get("parent", np.array([[-1, 0, 1]]))
        with pytest.raises(sf.SpecFoldError) as e:
            sf.sf_head_verify(head.head, None, kw.get("hidden", hidden.data_ptr()), kw.get("tokens", tok.data_ptr()),
                              par, par.shape[0], par.shape[1] - 1, 32, pred.data_ptr())
        assert e.value.status == status
    head.close()
