"""Seeded synthetic inputs for the folded multi-branch verification pass.

This module only draws random numbers and arranges them into the shapes the
pass consumes: random-init layer weights, a draft tree, block tokens, the
block's input hidden states and a per-layer prefix K/V cache.  It holds none
of the method's arithmetic; both the CUDA path (through the binding) and the
CPU oracle read the tensors produced here.

Workload shapes follow the draft/verification setup of "SpecFold: Folding
Multi-Branch Redundancy for Faster Speculative Decoding in Diffusion Language
Models" (arXiv 2610.04875v2 summary), §2.2 (drafts inherit the parent's tokens
and unmask a few more positions), §3.1 (block size 32, B = 8 drafts, 28
layers) and §4.1 (the evaluated model sizes), with the S_t <= 4 unmasking
budget from the onedev.kr review of the same paper ("How it works").  No
dataset or checkpoint is used: weights are N(0, 0.02) draws.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

MASK_VOCAB = 1024          # vocabulary size of the synthetic block tokens
MASK_ID = MASK_VOCAB - 1   # token id that marks a still-masked position
W_STD = 0.02               # std of every random-init weight and embedding entry

# tensor ids used in the per-(layer, tensor) weight seed
TENSOR_IDS = {"wq": 0, "wk": 1, "wv": 2, "wo": 3, "w_gate": 4, "w_up": 5, "w_down": 6}


@dataclass(frozen=True)
class Config:
    """One workload: model shape, block/draft shape and gate threshold."""
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    dtype: str                 # "f32" or "bf16": weights, hidden I/O, prefix K/V
    block_len: int = 32        # L
    prefix_len: int = 512      # P
    n_requests: int = 1        # R
    n_drafts: int = 8          # B
    tree: str = "random"       # "random" (depth <= max_depth), "chain", "siblings" or "chains"
    max_depth: int = 3         # "random": depth bound; "chains": length of each chain off the main branch
    unmask_max: int = 4        # S_t upper bound (uniform 1..unmask_max)
    unmask_exact: Optional[int] = None  # if set, every child unmasks exactly this many
    mask_frac: float = 0.5     # fraction of the main block still masked
    delta: float = 0.1
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0

    @property
    def n_branches(self) -> int:
        return self.n_drafts + 1

    @property
    def rows(self) -> int:
        """T = R * (B + 1) * L, all branch-position rows of one pass."""
        return self.n_requests * self.n_branches * self.block_len

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": Config("tiny", 1, 256, 4, 2, 64, 688, "f32", block_len=32, prefix_len=64,
                   n_requests=1, n_drafts=2, tree="chain", unmask_exact=2, delta=0.1),
    "1.5b": Config("1.5b", 28, 1536, 12, 2, 128, 8960, "bf16", prefix_len=512,
                   n_requests=1, n_drafts=8, delta=0.1),
    "7b": Config("7b", 28, 3584, 28, 4, 128, 18944, "bf16", prefix_len=1024,
                 n_requests=1, n_drafts=8, delta=0.1),
    "8b": Config("8b", 32, 4096, 32, 8, 128, 14336, "bf16", prefix_len=2048,
                 n_requests=1, n_drafts=8, delta=0.1),
    "14b": Config("14b", 40, 5120, 40, 8, 128, 13824, "bf16", prefix_len=4096,
                  n_requests=4, n_drafts=8, delta=0.1),
}

DELTA_SWEEP_8B = (0.0, 0.01, 0.1, 0.2, 0.3, 0.7)
DRAFT_SWEEP_14B = (2, 4, 6, 8)
DEPTH_SWEEP = (1, 2, 3, 4)
HEAD_VOCAB = 131072        # synthetic LM-head vocabulary of the benchmark (not a checkpoint's)


def depth_config(base: Config, depth: int) -> Config:
    """Drafting-strategy workload: a budget of B = 7 one-token drafts arranged
    as chains of `depth` off the main branch, from seven siblings (depth 1) to
    parent-extending chains (depth 4), every draft unmasking exactly one more
    position than its parent."""
    return base.with_(name=f"{base.name}-D{depth}", n_drafts=7, tree="chains", max_depth=depth, unmask_exact=1)


def ripple_config(base: Config) -> Config:
    """Residual-ripple workload: a main block with 17 of its 32 positions
    committed (15 still masked) and one child that unmasks one more position."""
    return base.with_(name=f"{base.name}-ripple", n_drafts=1, tree="chain", mask_frac=15 / 32, unmask_exact=1,
                      block_len=32)


def weight_seed(seed: int, layer: int, tensor: str) -> int:
    return seed * 1000003 + layer * 16 + TENSOR_IDS[tensor]


def weight_shapes(cfg: Config):
    """Row-major [in, out] shapes (y = x @ W) of one layer's matrices."""
    d, hq, hkv, F = cfg.d_model, cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.d_ffn
    return {"wq": (d, hq), "wk": (d, hkv), "wv": (d, hkv), "wo": (hq, d),
            "w_gate": (d, F), "w_up": (d, F), "w_down": (F, d)}


def _torch_dtype(cfg: Config):
    import torch
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def make_layer_weights(cfg: Config, layer: int, seed: int = 0, device="cpu"):
    """One layer's weights as torch tensors in cfg.dtype; RMSNorm gains are fp32 ones."""
    import torch
    out = {}
    for name, shape in weight_shapes(cfg).items():
        g = torch.Generator(device=device)
        g.manual_seed(weight_seed(seed, layer, name))
        w = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * W_STD
        out[name] = w.to(_torch_dtype(cfg))
    out["attn_norm"] = torch.ones(cfg.d_model, dtype=torch.float32, device=device)
    out["ffn_norm"] = torch.ones(cfg.d_model, dtype=torch.float32, device=device)
    return out


def make_weights(cfg: Config, seed: int = 0, device="cpu") -> List[dict]:
    return [make_layer_weights(cfg, l, seed, device) for l in range(cfg.n_layers)]


def make_tree(cfg: Config, seed: int = 0, request: int = 0) -> np.ndarray:
    """parent[B+1]: parent[0] = -1, parent[i] < i (topological by index)."""
    Bp = cfg.n_branches
    if cfg.tree == "chain":
        return np.arange(-1, Bp - 1, dtype=np.int32)
    if cfg.tree == "siblings":
        p = np.zeros(Bp, dtype=np.int32)
        p[0] = -1
        return p
    if cfg.tree == "chains":
        # drafts 1..B in chains of max_depth off the main branch, each draft
        # extending the previous one of its chain (the last chain may be
        # shorter): max_depth = 1 gives B siblings, max_depth = B one chain
        p = np.empty(Bp, dtype=np.int32)
        p[0] = -1
        for i in range(1, Bp):
            p[i] = 0 if (i - 1) % cfg.max_depth == 0 else i - 1
        return p
    rng = np.random.default_rng([seed, 7919, request])
    parent = [-1]
    depth = [0]
    for i in range(1, Bp):
        cands = [j for j in range(i) if depth[j] < cfg.max_depth]
        p = int(rng.choice(cands))
        parent.append(p)
        depth.append(depth[p] + 1)
    return np.asarray(parent, dtype=np.int32)


def make_trees(cfg: Config, seed: int = 0) -> np.ndarray:
    return np.stack([make_tree(cfg, seed, r) for r in range(cfg.n_requests)])


def make_tokens(cfg: Config, parent: np.ndarray, seed: int = 0, request: int = 0) -> np.ndarray:
    """tokens[B+1, L]: the main block has mask_frac of its positions masked; each
    draft copies its parent's block and unmasks S_t of the parent's masked positions."""
    rng = np.random.default_rng([seed, 104729, request])
    Bp, L = cfg.n_branches, cfg.block_len
    tok = np.empty((Bp, L), dtype=np.int64)
    tok[0] = rng.integers(0, MASK_ID, size=L)
    n_mask = int(round(cfg.mask_frac * L))
    tok[0, rng.choice(L, size=n_mask, replace=False)] = MASK_ID
    for i in range(1, Bp):
        tok[i] = tok[parent[i]]
        masked = np.flatnonzero(tok[i] == MASK_ID)
        k = cfg.unmask_exact if cfg.unmask_exact is not None else int(rng.integers(1, cfg.unmask_max + 1))
        k = min(k, masked.size)
        if k > 0:
            pos = rng.choice(masked, size=k, replace=False)
            tok[i, pos] = rng.integers(0, MASK_ID, size=k)
    return tok


def make_all_tokens(cfg: Config, parents: np.ndarray, seed: int = 0) -> np.ndarray:
    return np.stack([make_tokens(cfg, parents[r], seed, r) for r in range(cfg.n_requests)])


def make_embedding(cfg: Config, seed: int = 0, device="cpu"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 999_983)
    return torch.randn((MASK_VOCAB, cfg.d_model), generator=g, device=device, dtype=torch.float32) * W_STD


def make_hidden(cfg: Config, tokens: np.ndarray, seed: int = 0, device="cpu"):
    """Block input hidden states [R, B+1, L, d] = embedding rows of the tokens, in cfg.dtype."""
    import torch
    emb = make_embedding(cfg, seed, device)
    idx = torch.as_tensor(tokens, device=device)
    return emb[idx].to(_torch_dtype(cfg)).contiguous()


def make_prefix_kv(cfg: Config, seed: int = 0, device="cpu", n_layers: Optional[int] = None):
    """Committed-context K and V, [n_layers, R, P, n_kv, hd], already rotary-encoded
    (positions 0..P-1), N(0, (0.02 * sqrt(d))^2): the scale of an N(0, 0.02)
    projection of a unit-RMS row."""
    import torch
    nl = cfg.n_layers if n_layers is None else n_layers
    shape = (nl, cfg.n_requests, cfg.prefix_len, cfg.n_kv_heads, cfg.head_dim)
    std = W_STD * float(np.sqrt(cfg.d_model))
    out = []
    for which in (0, 1):
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000003 + 777_767 + which)
        out.append((torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std)
                   .to(_torch_dtype(cfg)).contiguous())
    return out[0], out[1]


def make_head_weights(cfg: Config, vocab: int, seed: int = 0, device="cpu"):
    """Final RMSNorm gain (fp32 ones) and LM head [d, vocab] N(0, 0.02) in cfg.dtype."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 999_979)
    w = (torch.randn((cfg.d_model, vocab), generator=g, device=device, dtype=torch.float32) * W_STD)
    return torch.ones(cfg.d_model, dtype=torch.float32, device=device), w.to(_torch_dtype(cfg)).contiguous()


@dataclass
class Workload:
    cfg: Config
    parents: np.ndarray        # [R, B+1] int32
    tokens: np.ndarray         # [R, B+1, L] int64
    hidden: object             # torch [R, B+1, L, d] cfg.dtype
    prefix_k: object           # torch [n_layers, R, P, n_kv, hd]
    prefix_v: object
    weights: List[dict] = field(default_factory=list)


def make_workload(cfg: Config, seed: int = 0, device="cpu", weights: bool = True) -> Workload:
    parents = make_trees(cfg, seed)
    tokens = make_all_tokens(cfg, parents, seed)
    hidden = make_hidden(cfg, tokens, seed, device)
    pk, pv = make_prefix_kv(cfg, seed, device)
    ws = make_weights(cfg, seed, device) if weights else []
    return Workload(cfg, parents, tokens, hidden, pk, pv, ws)


def small_config(name="small", n_layers=2, d_model=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                 d_ffn=96, dtype="f32", block_len=8, prefix_len=5, n_requests=1, n_drafts=3,
                 **kw) -> Config:
    """A toy shape for CPU tests of the oracle (seconds of fp64 work)."""
    return Config(name, n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn, dtype,
                  block_len=block_len, prefix_len=prefix_len, n_requests=n_requests,
                  n_drafts=n_drafts, **kw)
