"""The seeded workload generator produces the draft structure the pages
describe (SpecFold summary §2.2; onedev.kr review, "How it works": drafts
inherit the parent's tokens and unmask at most S_t more positions)."""
import numpy as np

import synth


def test_trees_are_topological_and_shallow():
    cfg = synth.CONFIGS["1.5b"]
    for seed in range(20):
        p = synth.make_tree(cfg, seed)
        assert p[0] == -1 and len(p) == cfg.n_branches
        depth = [0]
        for i in range(1, len(p)):
            assert 0 <= p[i] < i
            depth.append(depth[p[i]] + 1)
        assert max(depth) <= cfg.max_depth


def test_chain_tree_for_tiny():
    assert synth.make_tree(synth.CONFIGS["tiny"]).tolist() == [-1, 0, 1]


def test_children_inherit_and_unmask_few():
    for name in ("tiny", "1.5b", "14b"):
        cfg = synth.CONFIGS[name]
        parents = synth.make_trees(cfg, 3)
        toks = synth.make_all_tokens(cfg, parents, 3)
        for r in range(cfg.n_requests):
            assert (toks[r, 0] == synth.MASK_ID).sum() == cfg.block_len // 2
            for i in range(1, cfg.n_branches):
                par = toks[r, parents[r, i]]
                diff = toks[r, i] != par
                assert (par[diff] == synth.MASK_ID).all()          # only masked slots change
                assert (toks[r, i][diff] != synth.MASK_ID).all()   # and they get real ids
                k = diff.sum()
                if cfg.unmask_exact is not None:
                    assert k == min(cfg.unmask_exact, (par == synth.MASK_ID).sum())
                else:
                    assert 1 <= k <= cfg.unmask_max or (par == synth.MASK_ID).sum() == 0


def test_deterministic():
    cfg = synth.small_config()
    a = synth.make_workload(cfg, 4)
    b = synth.make_workload(cfg, 4)
    assert np.array_equal(a.tokens, b.tokens)
    assert (a.hidden == b.hidden).all() and (a.prefix_k == b.prefix_k).all()
    assert all((a.weights[l][k] == b.weights[l][k]).all() for l in range(cfg.n_layers) for k in a.weights[l])


def test_depth_sweep_trees():
    """Drafting-strategy workload (SpecFold summary §D.2): B = 7 one-token
    drafts, from seven siblings at depth 1 to parent-extending chains at 4."""
    base = synth.CONFIGS["1.5b"]
    for D in synth.DEPTH_SWEEP:
        cfg = synth.depth_config(base, D)
        p = synth.make_tree(cfg)
        assert cfg.n_drafts == 7 and p[0] == -1
        depth = [0]
        for i in range(1, len(p)):
            assert 0 <= p[i] < i
            depth.append(depth[p[i]] + 1)
        assert max(depth) == D
        toks = synth.make_tokens(cfg, p)
        for i in range(1, len(p)):
            assert (toks[i] != toks[p[i]]).sum() == 1      # one more token than the parent
    assert synth.make_tree(synth.depth_config(base, 1)).tolist() == [-1] + [0] * 7


def test_ripple_workload():
    """Residual-ripple workload (SpecFold summary §4.4): the parent has 17 of
    32 positions committed and its only child unmasks one more."""
    cfg = synth.ripple_config(synth.CONFIGS["1.5b"])
    p = synth.make_tree(cfg)
    toks = synth.make_tokens(cfg, p)
    assert p.tolist() == [-1, 0]
    assert (toks[0] != synth.MASK_ID).sum() == 17
    assert (toks[1] != toks[0]).sum() == 1 and (toks[1] != synth.MASK_ID).sum() == 18
