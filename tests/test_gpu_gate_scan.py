"""The fused gate kernel at row counts beyond one wave of resident CTAs, and
its rho diagnostic (needs a GB300).

The gate hands rows out in ascending order by an arrival ticket; a row waits
only for lower rows (prefix look-back, source resolution), so a pass must be
correct whatever fraction of the grid is resident at once.  At 256 threads a
CTA, at most 8 CTAs fit an SM (about 1,216 on 152 SMs), so the shapes here
(2,304 and 8,192 rows) need several waves, and the dense pass makes every row
a recompute row."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_free_running, check_teacher_forced, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_reuse_gb300 import build
    build.build()


def _checked_run(cfg, wl, delta, debug=True):
    """run_gpu, then the device check word must be clean."""
    import sparse_reuse_gb300 as sf
    ctx = sf.from_config(cfg, wl.weights)
    gpu = run_gpu(cfg, wl, delta, debug=debug, ctx=ctx)
    ctx.sync()          # raises SpecFoldError on a bounded wait that ran out
    ctx.close()
    return gpu


@pytest.mark.parametrize("delta", [0.0, 0.1])
def test_fp32_2304_rows_free_running(delta):
    cfg = synth.CONFIGS["tiny"].with_(n_layers=2, n_requests=8, n_drafts=8, tree="random", unmask_exact=None)
    assert cfg.rows == 2304
    wl = synth.make_workload(cfg, seed=11, device="cuda")
    gpu = _checked_run(cfg, wl, delta)
    check_free_running(cfg, wl, gpu, delta)
    if delta == 0.0:
        assert gpu["rc_count"].tolist() == [cfg.rows] * cfg.n_layers
    else:
        assert gpu["fold"].any()


@pytest.mark.parametrize("delta", [0.0, 0.1])
def test_fp32_8192_rows_maximum(delta):
    # the largest pass a context accepts: R * (B+1) * L = 32 * 8 * 32
    cfg = synth.CONFIGS["tiny"].with_(n_layers=1, n_requests=32, n_drafts=7, tree="random", unmask_exact=None,
                                      prefix_len=16)
    assert cfg.rows == 8192
    wl = synth.make_workload(cfg, seed=12, device="cuda")
    gpu = _checked_run(cfg, wl, delta)
    check_free_running(cfg, wl, gpu, delta)


@pytest.mark.parametrize("delta", [0.0, 0.1])
def test_bf16_2304_rows_teacher_forced(delta):
    cfg = synth.small_config(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=128, d_ffn=320,
                             dtype="bf16", block_len=32, prefix_len=96, n_requests=8, n_drafts=8)
    assert cfg.rows == 2304
    wl = synth.make_workload(cfg, seed=13, device="cuda")
    gpu = _checked_run(cfg, wl, delta)
    check_teacher_forced(cfg, wl, gpu, delta, range(cfg.n_layers))
    if delta == 0.0:
        assert gpu["rc_count"].tolist() == [cfg.rows] * cfg.n_layers


def test_rho_dump_matches_oracle_on_gpu_layer_inputs():
    """sf_set_rho_dump: the gate's fp32 rho of every row equals the oracle's
    relative residual of the same layer input (NaN on the main branch)."""
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["tiny"].with_(n_layers=3, n_requests=2, n_drafts=5, tree="random")
    wl = synth.make_workload(cfg, seed=14, device="cuda")
    wl.hidden[1, 4] = wl.hidden[1, wl.parents[1, 4]]   # a child equal to its parent: rho = 0 at layer 0
    ctx = sf.from_config(cfg, wl.weights)
    rho = torch.full((cfg.n_layers, cfg.n_requests, cfg.n_branches, cfg.block_len), -1.0, device="cuda")
    ctx.set_rho_dump(rho)
    gpu = run_gpu(cfg, wl, 0.1, ctx=ctx)
    ctx.set_rho_dump(None)
    ctx.sync()
    ctx.close()
    got = rho.cpu().numpy().astype(np.float64)
    R, Bp, L, d = cfg.n_requests, cfg.n_branches, cfg.block_len, cfg.d_model
    assert np.isnan(got[:, :, 0]).all()
    assert (got[0, 1, 4] == 0.0).all()
    for l in range(cfg.n_layers):
        H_in = gpu["layer_hidden"][l].astype(np.float64).reshape(R, Bp, L, d)
        for r in range(R):
            _, want = oracle.gate_request(H_in[r], wl.parents[r], 0.1)
            np.testing.assert_allclose(got[l, r, 1:], want[1:], rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("delta", [0.0, 0.1])
def test_bf16_wide_rows_2304_teacher_forced(delta):
    """d = 5120 (more than 4 float4 a thread): the two-launch gate, at 2,304
    rows (several waves of its register-heavy first kernel)."""
    cfg = synth.small_config(n_layers=2, d_model=5120, n_q_heads=4, n_kv_heads=2, head_dim=128, d_ffn=256,
                             dtype="bf16", block_len=32, prefix_len=16, n_requests=8, n_drafts=8)
    assert cfg.rows == 2304
    wl = synth.make_workload(cfg, seed=15, device="cuda")
    gpu = _checked_run(cfg, wl, delta)
    assert gpu["stats"]["family_launches"]["gate"] == 2 * cfg.n_layers
    check_teacher_forced(cfg, wl, gpu, delta, range(cfg.n_layers))


def test_fp32_wide_rows_free_running():
    cfg = synth.CONFIGS["tiny"].with_(n_layers=2, d_model=5120, n_q_heads=4, n_kv_heads=2, head_dim=64, d_ffn=256,
                                      n_drafts=4, tree="random", unmask_exact=None)
    wl = synth.make_workload(cfg, seed=16, device="cuda")
    gpu = _checked_run(cfg, wl, 0.1)
    check_free_running(cfg, wl, gpu, 0.1)
