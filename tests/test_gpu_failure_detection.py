"""Failure detection without a GPU fault (needs a GB300): a wait that nothing
satisfies runs out after its bound, the pass completes, the host reads the
device check word as SF_ERR_DEVICE_ASSERT, and the context then runs a clean
pass with the same result as before."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_recovers():
    import sparse_reuse_gb300 as sf
    cfg = synth.CONFIGS["tiny"]
    wl = synth.make_workload(cfg, 0, device="cuda")
    ctx = sf.from_config(cfg, wl.weights)
    st = torch.cuda.Stream()
    ref, fold_ref, _, _ = ctx.verify(wl.hidden, wl.parents, wl.prefix_k, wl.prefix_v, 0.1, stream=st)
    ctx.sync(st)
    ref = ref.clone()
    fold_ref = fold_ref.clone()

    # layer 0's compaction never signals completion: its recompute rows wait
    # about 2 s, give up and raise the timeout bit
    sf.sf_inject_stall(ctx.ctx, True)
    ctx.verify(wl.hidden, wl.parents, wl.prefix_k, wl.prefix_v, 0.1, stream=st)
    with pytest.raises(sf.SpecFoldError) as e:
        ctx.sync(st)
    assert e.value.status == sf.SF_ERR_DEVICE_ASSERT

    # reported once: the context is usable again and reproduces the clean pass
    sf.sf_inject_stall(ctx.ctx, False)
    out, fold, _, _ = ctx.verify(wl.hidden, wl.parents, wl.prefix_k, wl.prefix_v, 0.1, stream=st)
    ctx.sync(st)
    assert torch.equal(out, ref)
    assert torch.equal(fold, fold_ref)
    ctx.close()
