"""CUDA path vs the float64 oracle through the C ABI (needs a GB300)."""
import numpy as np
import pytest

import synth
from parity import check_free_running, check_teacher_forced, rel_err_rows, run_gpu, TOL

pytestmark = pytest.mark.gpu

FREE_RUN_BF16 = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_reuse_gb300 import build
    build.build()


def _wl(cfg, seed=0):
    return synth.make_workload(cfg, seed, device="cuda")


def test_tiny_free_running():
    cfg = synth.CONFIGS["tiny"]
    wl = _wl(cfg)
    gpu = run_gpu(cfg, wl, cfg.delta)
    ref, err = check_free_running(cfg, wl, gpu, cfg.delta)
    assert gpu["fold"].any() and (~gpu["fold"][:, :, 1:]).any()


FP32_CASES = {
    "dense_delta0": (dict(), 0.0),
    "no_prefix": (dict(prefix_len=0), 0.1),
    "main_only": (dict(n_drafts=0), 0.1),
    "three_requests": (dict(n_requests=3, n_drafts=5, tree="random"), 0.1),
    "ragged_block_hd128": (dict(block_len=20, head_dim=128, n_q_heads=4, n_kv_heads=1, d_ffn=300), 0.1),
    "long_block": (dict(block_len=64, n_drafts=3, tree="random"), 0.1),
    "fold_everything_but_main": (dict(n_drafts=4, tree="random"), 1e6),
    "siblings": (dict(n_drafts=6, tree="siblings"), 0.1),
}


@pytest.mark.parametrize("name", sorted(FP32_CASES))
def test_fp32_variants_free_running(name):
    kw, delta = FP32_CASES[name]
    cfg = synth.CONFIGS["tiny"].with_(**dict(dict(n_layers=2, prefix_len=37), **kw))
    wl = _wl(cfg, seed=1)
    gpu = run_gpu(cfg, wl, delta)
    check_free_running(cfg, wl, gpu, delta)
    if delta == 0.0:
        assert not gpu["fold"].any()
    if delta >= 1e6:
        assert gpu["fold"][:, :, 1:].all()
        assert gpu["rc_count"].tolist() == [cfg.n_requests * cfg.block_len] * cfg.n_layers


def test_identical_child_reproduces_parent():
    cfg = synth.CONFIGS["tiny"].with_(n_layers=2, n_drafts=3)
    wl = _wl(cfg, seed=2)
    wl.hidden[0, 3] = wl.hidden[0, 2]
    gpu = run_gpu(cfg, wl, 0.1)
    assert gpu["fold"][:, 0, 3].all()
    assert np.array_equal(gpu["out"][0, 3], gpu["out"][0, 2])


def test_graph_replay_is_bitwise_stable():
    import torch
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["tiny"].with_(n_layers=2, n_drafts=4, tree="random")
    wl = _wl(cfg, seed=3)
    ctx = sf.from_config(cfg, wl.weights)
    stream = torch.cuda.Stream()
    out = torch.empty_like(wl.hidden)
    fold = torch.empty((cfg.n_layers, 1, cfg.n_branches, cfg.block_len), dtype=torch.uint8, device="cuda")
    src = torch.empty(fold.shape, dtype=torch.int32, device="cuda")
    rcc = torch.empty((cfg.n_layers,), dtype=torch.int32, device="cuda")
    res = []
    for graphs in (False, True, True, True):
        ctx.set_graphs(graphs)
        ctx.verify(wl.hidden, wl.parents, wl.prefix_k, wl.prefix_v, 0.1, out=out, fold=fold, src=src,
                   rc_count=rcc, stream=stream)
        ctx.sync(stream)
        res.append([t.clone() for t in (out, fold, src, rcc)])
    st = ctx.stats()
    # a different tree recaptures and gives a different result
    p2 = wl.parents.copy()
    p2[0, -1] = 0
    ctx.verify(wl.hidden, p2, wl.prefix_k, wl.prefix_v, 0.1, out=out, fold=fold, src=src, rc_count=rcc,
               stream=stream)
    ctx.sync(stream)
    st2 = ctx.stats()
    ctx.close()
    assert st["graph_replays"] == 3 and st2["graph_replays"] == 4
    for r in res[1:]:
        for a, b in zip(res[0], r):
            assert torch.equal(a, b)
    assert st2["kernel_launches"] - st["kernel_launches"] == st["kernel_launches"] // 4


def test_bf16_small_free_running_dense_and_folded():
    cfg = synth.small_config(n_layers=3, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=128, d_ffn=512,
                             dtype="bf16", block_len=32, prefix_len=96, n_drafts=4)
    wl = _wl(cfg, seed=4)
    for delta in (0.0, 0.1):
        gpu = run_gpu(cfg, wl, delta)
        check_teacher_forced(cfg, wl, gpu, delta, range(cfg.n_layers))
        if delta == 0.0:
            check_free_running(cfg, wl, gpu, delta)


BF16_CASES = {
    "hd64_ragged": dict(head_dim=64, n_q_heads=8, n_kv_heads=2, block_len=20, prefix_len=70, n_drafts=5),
    "no_prefix": dict(prefix_len=0, n_drafts=3),
    "three_requests_gqa7": dict(n_requests=3, n_q_heads=7, n_kv_heads=1, prefix_len=200, n_drafts=4),
    "long_prefix": dict(prefix_len=1000, n_drafts=2, block_len=64),
    # prefixes of 2048+ keys take the tcgen05 prefix kernel (4 splits, ragged
    # last block, several 128-vector query tiles per KV head at delta = 0)
    "tc_prefix_hd64_ragged": dict(head_dim=64, n_q_heads=8, n_kv_heads=2, block_len=20, prefix_len=2100,
                                  n_drafts=5),
    "tc_prefix_three_requests_gqa7": dict(n_requests=3, n_q_heads=7, n_kv_heads=1, prefix_len=2048, n_drafts=4),
    # fused kernel with three splits of the prefix (50 CTAs a split on 152 SMs):
    # each split merges 43, 43 and 42 of a query tile's rows
    "fused_three_splits": dict(head_dim=64, n_q_heads=10, n_kv_heads=10, block_len=8, prefix_len=512,
                               n_drafts=4),
}


@pytest.mark.parametrize("name", sorted(BF16_CASES))
def test_bf16_variants_teacher_forced(name):
    base = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=128, d_ffn=320, dtype="bf16",
                block_len=32, prefix_len=96, n_drafts=4)
    base.update(BF16_CASES[name])
    cfg = synth.small_config(**base)
    wl = _wl(cfg, seed=7)
    for delta in (0.0, 0.1):
        gpu = run_gpu(cfg, wl, delta)
        check_teacher_forced(cfg, wl, gpu, delta, range(cfg.n_layers))


def test_bf16_random_norm_gains_teacher_forced():
    """RMSNorm gains away from 1 (the synthetic weights use unit gains): the
    attention gain goes through the gate's normalised rows, the FFN gain
    through the O epilogue's bf16(h * g2) rows, with the row scale applied in
    the gate/up epilogue."""
    import torch
    cfg = synth.small_config(n_layers=3, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=128, d_ffn=320,
                             dtype="bf16", block_len=32, prefix_len=96, n_drafts=4)
    wl = _wl(cfg, seed=9)
    g = torch.Generator(device="cpu")
    g.manual_seed(2024)
    for W in wl.weights:
        for key in ("attn_norm", "ffn_norm"):
            W[key] = (0.5 + torch.rand(cfg.d_model, generator=g)).to(W[key].device, W[key].dtype)
    for delta in (0.0, 0.1):
        gpu = run_gpu(cfg, wl, delta)
        check_teacher_forced(cfg, wl, gpu, delta, range(cfg.n_layers))


def test_1p5b_all_layers_teacher_forced():
    cfg = synth.CONFIGS["1.5b"]
    wl = _wl(cfg)
    gpu = run_gpu(cfg, wl, cfg.delta)
    worst = check_teacher_forced(cfg, wl, gpu, cfg.delta, range(cfg.n_layers))
    assert worst <= TOL["bf16"]


def test_1p5b_dense_free_running(summary_line):
    """28 bf16 layers run freely from the same input at delta = 0.  bf16
    rounding of the GEMM/attention operands drifts by ~1e-3 per layer and the
    random-init layer map amplifies it: rounding the same activation sites of
    the float64 oracle to bf16 already drifts 2.8e-2 from it over 28 layers.
    The stated 2e-2 bar is held per layer by the teacher-forced tests; here
    the whole stack must stay within FREE_RUN_BF16 and every dense decision
    must match."""
    cfg = synth.CONFIGS["1.5b"]
    wl = _wl(cfg)
    gpu = run_gpu(cfg, wl, 0.0, debug=False)
    assert not gpu["fold"].any()
    _, err = check_free_running(cfg, wl, gpu, 0.0, tol=FREE_RUN_BF16)
    summary_line(f"bf16 free-running drift, 1.5B, 28 layers, delta 0: max row rel err {err:.3e}")


def test_1p5b_folded_free_running(summary_line):
    """The folded pass (delta = 0.1) run freely for 28 bf16 layers.  Free-running
    inputs drift, so a few rho values move across delta: the oracle takes the
    GPU's fold decisions (its own rule's disagreements are counted and must
    all lie near the threshold), and the hidden states must stay within
    FREE_RUN_BF16 of it."""
    import oracle
    from parity import oracle_inputs
    cfg = synth.CONFIGS["1.5b"]
    wl = _wl(cfg)
    gpu = run_gpu(cfg, wl, cfg.delta, debug=False)
    H0, pk, pv = oracle_inputs(wl)
    Ws = {}

    def get_layer(l):
        if l not in Ws:
            Ws[l] = oracle.layer_weights_f64(wl.weights[l])
        return Ws[l]

    ref = oracle.verify_pass(H0, wl.parents, cfg.delta, get_layer, pk, pv, cfg,
                             forced=lambda l: gpu["fold"][l].astype(np.int64))
    assert np.array_equal(ref["fold"], gpu["fold"])
    own = np.zeros_like(gpu["fold"])
    own[:, :, 1:] = oracle.fold_decision(ref["rho"][:, :, 1:], cfg.delta)
    flips = own != gpu["fold"]
    n_dec = flips[:, :, 1:].size
    # the decisions the oracle's rule would take differently are rare
    assert flips.sum() <= 0.02 * n_dec, int(flips.sum())
    far = float(np.max(np.abs(ref["rho"][flips] - cfg.delta)) / cfg.delta) if flips.any() else 0.0
    err = rel_err_rows(gpu["out"], ref["out"])
    assert err <= FREE_RUN_BF16, f"free-running hidden rel err {err:.3e} > {FREE_RUN_BF16}"
    summary_line(f"bf16 free-running drift, 1.5B, 28 layers, delta 0.1: max row rel err {err:.3e}; "
                 f"{int(flips.sum())} of {n_dec} gate decisions differ from the oracle's own rule "
                 f"(|rho - delta| <= {far:.2e} delta)")


@pytest.mark.parametrize("name,delta", [("7b", 0.1), ("7b", 0.0)] +
                         [("8b", d) for d in synth.DELTA_SWEEP_8B])
def test_large_configs_sampled_layers(name, delta):
    cfg = synth.CONFIGS[name]
    wl = _wl(cfg)
    gpu = run_gpu(cfg, wl, delta)
    check_teacher_forced(cfg, wl, gpu, delta, [0, cfg.n_layers // 2, cfg.n_layers - 1])


@pytest.mark.parametrize("B", synth.DRAFT_SWEEP_14B)
def test_14b_batched_draft_sweep_sampled_layers(B):
    cfg = synth.CONFIGS["14b"].with_(n_drafts=B)
    wl = _wl(cfg)
    gpu = run_gpu(cfg, wl, cfg.delta)
    check_teacher_forced(cfg, wl, gpu, cfg.delta, [0, cfg.n_layers - 1])


# ------------------------------------------------------------------ error paths

def test_argument_and_tree_errors_launch_nothing():
    import torch
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["tiny"]
    wl = _wl(cfg)
    ctx = sf.from_config(cfg, wl.weights)
    before = ctx.stats()["kernel_launches"]
    out = torch.empty_like(wl.hidden)
    # a misaligned buffer comes with an invalid tree, which is checked later:
    # the alignment check must be the one that answers, and if it did not the
    # tree check would still refuse the call before any launch
    bad_tree = np.array([[0, 0, 1]])
    bad = [
        (dict(hidden=wl.hidden.data_ptr() + 4, parent=bad_tree), sf.SF_ERR_INVALID_ARG),
        (dict(out=out.data_ptr() + 8, parent=bad_tree), sf.SF_ERR_INVALID_ARG),
        (dict(pk=wl.prefix_k.data_ptr() + 4, parent=bad_tree), sf.SF_ERR_INVALID_ARG),
        (dict(parent=np.array([[0, 0, 1]])), sf.SF_ERR_TREE),
        (dict(parent=np.array([[-1, 1, 1]])), sf.SF_ERR_TREE),
        (dict(parent=np.array([[-1, 0, 3]])), sf.SF_ERR_TREE),
        (dict(delta=-0.1), sf.SF_ERR_INVALID_ARG),
        (dict(delta=float("nan")), sf.SF_ERR_INVALID_ARG),
        (dict(delta=float("inf")), sf.SF_ERR_INVALID_ARG),
        (dict(parent=np.array([[-1, 0, 1, 2]])), sf.SF_ERR_SHAPE),
        (dict(P=cfg.prefix_len + 1), sf.SF_ERR_SHAPE),
        (dict(hidden=0), sf.SF_ERR_INVALID_ARG),
    ]
    for kw, status in bad:
        parent = kw.get("parent", wl.parents)
        with pytest.raises(sf.SpecFoldError) as ei:
            sf.sf_verify(ctx.ctx, None, kw.get("hidden", wl.hidden.data_ptr()), parent,
                         kw.get("pk", wl.prefix_k.data_ptr()), wl.prefix_v.data_ptr(), parent.shape[0],
                         parent.shape[1] - 1, kw.get("P", cfg.prefix_len), kw.get("delta", 0.1),
                         kw.get("out", out.data_ptr()))
        assert ei.value.status == status, (kw, ei.value)
    # the debug capture refuses a misaligned dump buffer (it only records pointers)
    dump = torch.empty((cfg.n_layers + 1) * wl.hidden.numel() + 4, device="cuda")
    with pytest.raises(sf.SpecFoldError) as ei:
        sf.sf_set_debug(ctx.ctx, dump.data_ptr() + 4, None)
    assert ei.value.status == sf.SF_ERR_INVALID_ARG
    assert ctx.stats()["kernel_launches"] == before
    # R = 0 is an empty pass
    sf.sf_verify(ctx.ctx, None, wl.hidden.data_ptr(), np.zeros((0, 3), np.int32), None, None, 0, 2, 0, 0.1,
                 out.data_ptr())
    assert ctx.stats()["kernel_launches"] == before
    ctx.close()


def test_timing_hooks_report_every_family():
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["tiny"]
    wl = _wl(cfg)
    ctx = sf.from_config(cfg, wl.weights)
    sf.sf_timing_begin(ctx.ctx, sf.FAMILIES)
    ctx.verify(wl.hidden, wl.parents, wl.prefix_k, wl.prefix_v, 0.1)
    t = sf.sf_timing_read(ctx.ctx)
    sf.sf_timing_begin(ctx.ctx, [])
    ctx.close()
    for fam in ("gate", "norm", "gemm_qkv", "attn_prefix", "attn_block", "gemm_o", "gemm_gateup",
                "gemm_down", "residual"):
        assert fam in t and t[fam][0] > 0 and t[fam][1] >= 1
