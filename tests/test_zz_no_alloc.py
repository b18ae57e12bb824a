"""The allocation-free gate entry point (sfk_gate_noalloc) against the same
step inside sf_verify.

sfk_gate_noalloc serves callers that cannot allocate device memory (engine
plugins living in a fixed arena, serving loops that ban allocator calls,
code running under stream capture); its scratch is a static device array.
Here two calls in a row, on different workloads, must give exactly the
layer-0 fold mask, resolved sources, recompute list and count that sf_verify
reports for the same input, and the fp32 layer input it records."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sf():
    from sparse_reuse_gb300 import build
    build.build()
    import sparse_reuse_gb300 as m
    return m


def _reference(sf, cfg, wl):
    """Layer-0 gate outputs of a full sf_verify pass (debug capture on)."""
    ctx = sf.from_config(cfg, wl.weights)
    T, d = cfg.rows, cfg.d_model
    dbg = torch.zeros((cfg.n_layers + 1, T, d), dtype=torch.float32, device="cuda")
    rcs = torch.full((cfg.n_layers, T), -1, dtype=torch.int32, device="cuda")
    ctx.set_debug(dbg, rcs)
    _, fold, src, rcc = ctx.verify(wl.hidden, wl.parents, wl.prefix_k, wl.prefix_v, cfg.delta)
    ctx.sync()
    ctx.close()
    n = int(rcc[0].item())
    return {"H": dbg[0].clone(), "fold": fold[0].reshape(-1).clone(), "src": src[0].reshape(-1).clone(),
            "rc": rcs[0, :n].clone(), "count": n}


def _noalloc(sf, cfg, wl, stream):
    T, d = cfg.rows, cfg.d_model
    out = {"H": torch.full((T, d), float("nan"), device="cuda"),
           "fold": torch.full((T,), 7, dtype=torch.uint8, device="cuda"),
           "rc": torch.full((T,), -1, dtype=torch.int32, device="cuda"),
           "rcslot": torch.full((T,), -1, dtype=torch.int32, device="cuda"),
           "src": torch.full((T,), -1, dtype=torch.int32, device="cuda"),
           "count": torch.full((1,), -1, dtype=torch.int32, device="cuda")}
    dtype = sf.SF_BF16 if cfg.dtype == "bf16" else sf.SF_F32
    sf.sfk_gate_noalloc(stream.cuda_stream, wl.hidden.data_ptr(), dtype, wl.parents, cfg.n_requests,
                        cfg.n_drafts, cfg.block_len, cfg.d_model, cfg.delta, out["H"].data_ptr(),
                        out["fold"].data_ptr(), out["rc"].data_ptr(), out["rcslot"].data_ptr(),
                        out["src"].data_ptr(), out["count"].data_ptr())
    return out


def test_noalloc_gate_matches_sf_verify_on_two_calls_in_a_row(sf):
    cases = []
    for cfg, seed in ((synth.CONFIGS["tiny"].with_(n_drafts=4, tree="random", delta=0.3), 5),
                      (synth.small_config(n_layers=1, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                                          d_ffn=256, dtype="bf16", block_len=32, prefix_len=16, n_requests=3,
                                          n_drafts=5, delta=0.1), 6)):
        wl = synth.make_workload(cfg, seed, device="cuda")
        wl.hidden[0, -1] = wl.hidden[0, wl.parents[0, -1]]      # one draft folds everywhere
        cases.append((cfg, wl, _reference(sf, cfg, wl)))
    stream = torch.cuda.Stream()
    outs = [_noalloc(sf, cfg, wl, stream) for cfg, wl, _ in cases]   # two calls back to back
    stream.synchronize()
    for (cfg, wl, ref), got in zip(cases, outs):
        n = ref["count"]
        assert int(got["count"].item()) == n
        assert torch.equal(got["fold"], ref["fold"])
        assert torch.equal(got["src"], ref["src"])
        assert torch.equal(got["rc"][:n], ref["rc"])
        assert torch.equal(got["H"], ref["H"])
        # rcslot points at the recompute row of each row's source
        L, Bp = cfg.block_len, cfg.n_branches
        rows = torch.arange(cfg.rows, device="cuda")
        want_row = ((rows // L) // Bp * Bp + got["src"]) * L + rows % L
        assert torch.equal(got["rc"][got["rcslot"].long()], want_row.int())
        assert got["fold"].any() and not got["fold"].all()


def test_noalloc_gate_rejects_bad_arguments(sf):
    p = np.array([[-1, 0, 1]], np.int32)
    with pytest.raises(sf.SpecFoldError) as e:
        sf.sfk_gate_noalloc(None, 16, 0, np.array([[0, 0, 1]], np.int32), 1, 2, 32, 256, 0.1, 16, 16, 16, 16, 16, 16)
    assert e.value.status == sf.SF_ERR_TREE
    with pytest.raises(sf.SpecFoldError) as e:
        sf.sfk_gate_noalloc(None, 16, 0, np.tile(p, (100, 1)), 100, 2, 32, 256, 0.1, 16, 16, 16, 16, 16, 16)
    assert e.value.status == sf.SF_ERR_SHAPE                   # 9600 rows exceed the static scratch
    with pytest.raises(sf.SpecFoldError) as e:
        sf.sfk_gate_noalloc(None, 16, 0, p, 1, 2, 32, 256, -1.0, 16, 16, 16, 16, 16, 16)
    assert e.value.status == sf.SF_ERR_INVALID_ARG
    # misaligned buffers (with a tree that is refused later, so nothing can
    # launch): fp32 rows need 16 bytes, bf16 rows 8, H_out 16, int32 outputs 4
    bad_tree = np.array([[0, 0, 1]], np.int32)
    for dtype, hidden, h_out, rc in ((0, 24, 16, 16), (1, 20, 16, 16), (0, 16, 24, 16), (0, 16, 16, 18)):
        with pytest.raises(sf.SpecFoldError) as e:
            sf.sfk_gate_noalloc(None, hidden, dtype, bad_tree, 1, 2, 32, 256, 0.1, h_out, 16, rc, 16, 16, 16)
        assert e.value.status == sf.SF_ERR_INVALID_ARG, (dtype, hidden, h_out, rc)
