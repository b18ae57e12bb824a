"""CPU oracle of the SpecFold folded multi-branch verification pass.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this module; the product path never calls it.  It is
plain numpy in float64 and shares no code with the CUDA library.

What it computes (one verification pass over one denoising block):

* Sources: "SpecFold: Folding Multi-Branch Redundancy for Faster Speculative
  Decoding in Diffusion Language Models" (arXiv 2610.04875v2 summary, cited
  below as [SF]) and the onedev.kr review of the same paper (cited as [KR]).
* The block holds a main branch plus B drafts with parent links, each a full
  block state with bidirectional attention ([SF] §1, §2.2).
* At every layer, every draft position n of branch i is gated by the relative
  residual rho = ||H_i[n] - H_par(i)[n]|| / ||H_par(i)[n]|| of the layer-input
  hidden states ([KR] "What is different"; [SF] §3.1-3.2).  A position with
  rho <= delta is folded; the main branch is never gated ([SF] App. A, App. B).
* A folded position inherits the parent's QKV projection and FFN output; every
  branch keeps its own residual stream and its attention is exact against its
  own keys/values ([SF] §3.2, §A.1, §A.2).  Branches are visited in
  topological order, each inheriting its parent's tables and overwriting the
  positions it recomputes ([SF] App. A, §A.3).

Readings where the pages leave a step open (all restated in the design notes):

* the gate is evaluated on the layer input (the residual stream before the
  attention RMSNorm), once per layer, and governs QKV, the attention query
  and the FFN together;
* fold iff delta > 0 and rho <= delta; delta <= 0 is the dense pass; a parent
  row of zero norm gives rho = 0 if the child row is equal, else +inf;
* pre-norm layer: RMSNorm (unit gains as given), packed Q/K/V without bias,
  rotary embedding in rotate-half form at absolute position P + n with
  inverse frequencies theta^(-2j/hd), softmax scale 1/sqrt(hd), GQA with query
  head h reading KV head h // (nq / nkv), output projection on every row,
  SiLU-gated FFN;
* the prefix K/V is an input, already rotary-encoded, shared by all branches
  of a request and attended by every block row (no causal mask);
* compaction order is ascending in the flattened (request, branch, position)
  row id (r * (B+1) + i) * L + n.
"""
from __future__ import annotations

import math
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------
# Layer primitives ([SF] App. B: RMSNorm, packed QKV with rotary embeddings,
# attention, FFN)
# --------------------------------------------------------------------------

def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis."""
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gain, F64)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    j = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(theta), -2.0 * j / head_dim)


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half pairing (j, j + hd/2).

    x: [..., heads, hd]; pos: [...] (absolute token positions).
    out[j]        = x[j] cos(a_j) - x[j + hd/2] sin(a_j)
    out[j + hd/2] = x[j + hd/2] cos(a_j) + x[j] sin(a_j),  a_j = pos * theta^(-2j/hd)
    """
    x = np.asarray(x, F64)
    hd = x.shape[-1]
    half = hd // 2
    ang = np.asarray(pos, F64)[..., None, None] * rope_inv_freq(hd, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def project_qkv(x_rows: np.ndarray, pos: np.ndarray, W: dict, cfg) -> tuple:
    """RMSNorm1 then Q/K/V projection and rotary encoding of q and k.

    x_rows: [n, d] layer-input rows; pos: [n] absolute positions.
    Returns q [n, nq, hd], k [n, nkv, hd], v [n, nkv, hd].
    """
    nq, nkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    xn = rms_norm(x_rows, W["attn_norm"], cfg.rms_eps)
    q = (xn @ W["wq"]).reshape(-1, nq, hd)
    k = (xn @ W["wk"]).reshape(-1, nkv, hd)
    v = (xn @ W["wv"]).reshape(-1, nkv, hd)
    return rope(q, pos, cfg.rope_theta), rope(k, pos, cfg.rope_theta), v


def ffn(h_rows: np.ndarray, W: dict, cfg) -> np.ndarray:
    """RMSNorm2 then SwiGLU: (silu(x Wg) * (x Wu)) Wd."""
    xn = rms_norm(h_rows, W["ffn_norm"], cfg.rms_eps)
    return (silu(xn @ W["w_gate"]) * (xn @ W["w_up"])) @ W["w_down"]


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Direct softmax attention, no mask, GQA.

    q: [n, nq, hd]; K, V: [S, nkv, hd] (every query row sees all S keys).
    Query head h reads KV head h // (nq / nkv).  Returns [n, nq * hd].
    """
    n, nq, hd = q.shape
    S, nkv, _ = K.shape
    G = nq // nkv
    qg = q.reshape(n, nkv, G, hd)
    s = np.einsum("nkgd,skd->nkgs", qg, K) / math.sqrt(hd)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    o = np.einsum("nkgs,skd->nkgd", p, V)
    return o.reshape(n, nq * hd)


# --------------------------------------------------------------------------
# Gate, compaction, source resolution ([SF] §3.1, §3.2, §A.3, App. B; [KR])
# --------------------------------------------------------------------------

def relative_residual(h_child: np.ndarray, h_parent: np.ndarray) -> np.ndarray:
    """rho = ||h_child - h_parent||_2 / ||h_parent||_2 over the last axis.

    A zero-norm parent row gives 0 when the child row equals it, else +inf."""
    hc = np.asarray(h_child, F64)
    hp = np.asarray(h_parent, F64)
    num = np.sqrt(np.sum((hc - hp) ** 2, axis=-1))
    den = np.sqrt(np.sum(hp * hp, axis=-1))
    with np.errstate(divide="ignore", invalid="ignore"):
        rho = num / den
    rho = np.where(den == 0, np.where(num == 0, 0.0, np.inf), rho)
    return rho


def fold_decision(rho: np.ndarray, delta: float) -> np.ndarray:
    """Fold iff delta > 0 and rho <= delta (ties fold; delta <= 0 never folds)."""
    if not (delta > 0):
        return np.zeros(np.shape(rho), dtype=bool)
    return np.asarray(rho) <= delta


def gate_request(H: np.ndarray, parent: Sequence[int], delta: float,
                 forced: Optional[np.ndarray] = None):
    """Gate every position of one request.

    H: [B+1, L, d] layer input; parent[B+1] with parent[0] = -1.
    forced: optional int array [B+1, L]; entries 0/1 override the rule (used to
    take the other side's decision for rows inside the near-threshold band).
    Returns fold [B+1, L] bool (main branch all False) and rho (main NaN)."""
    Bp, L, _ = H.shape
    fold = np.zeros((Bp, L), dtype=bool)
    rho = np.full((Bp, L), np.nan)
    for i in range(1, Bp):
        rho[i] = relative_residual(H[i], H[parent[i]])
        fold[i] = fold_decision(rho[i], delta)
        if forced is not None:
            sel = forced[i] >= 0
            fold[i, sel] = forced[i, sel].astype(bool)
    return fold, rho


def resolve_sources(fold: np.ndarray, parent: Sequence[int]) -> np.ndarray:
    """src[i, n]: nearest branch on the path i -> root that recomputed n."""
    Bp, L = fold.shape
    src = np.empty((Bp, L), dtype=np.int64)
    for i in range(Bp):
        for n in range(L):
            s = i
            while fold[s, n]:
                s = parent[s]
            src[i, n] = s
    return src


def compaction(fold_all: np.ndarray):
    """Recompute list over all requests, ascending row id (r*(B+1)+i)*L+n.

    fold_all: [R, B+1, L].  Returns (rc [T_rc] int64 row ids, counts [R, B+1],
    offsets [R, B+1] exclusive prefix of counts in the same order)."""
    R, Bp, L = fold_all.shape
    rc = np.flatnonzero(~fold_all.reshape(-1))
    counts = (~fold_all).sum(axis=2)
    offsets = np.concatenate([[0], np.cumsum(counts.reshape(-1))[:-1]]).reshape(R, Bp)
    return rc.astype(np.int64), counts.astype(np.int64), offsets.astype(np.int64)


# --------------------------------------------------------------------------
# One folded layer, literal topological form ([SF] App. A, §A.1-§A.3)
# --------------------------------------------------------------------------

def folded_layer(H: np.ndarray, parent: Sequence[int], delta: float, W: dict,
                 prefix_k: np.ndarray, prefix_v: np.ndarray, cfg,
                 forced: Optional[np.ndarray] = None):
    """One folded layer of one request, branches visited in index order
    (topological since parent[i] < i).

    H: [B+1, L, d] layer input; prefix_k/v: [P, nkv, hd] (rotary-encoded).
    Each branch starts from a copy of its parent's Q/K/V and FFN-output tables
    and overwrites the positions it recomputes; attention for every position
    uses that branch's table (exact against the branch's own keys/values);
    the residual adds always use the branch's own hidden state.
    Returns (out [B+1, L, d], fold [B+1, L], rho [B+1, L])."""
    H = np.asarray(H, F64)
    Bp, L, d = H.shape
    P = prefix_k.shape[0]
    pos = P + np.arange(L)
    fold, rho = gate_request(H, parent, delta, forced)
    nq, nkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    tables: List[dict] = []
    out = np.empty_like(H)
    for i in range(Bp):
        if i == 0:
            tab = {"q": np.zeros((L, nq, hd)), "k": np.zeros((L, nkv, hd)),
                   "v": np.zeros((L, nkv, hd)), "f": np.zeros((L, d))}
        else:
            tab = {key: val.copy() for key, val in tables[parent[i]].items()}
        rec = ~fold[i]
        if rec.any():
            q, k, v = project_qkv(H[i, rec], pos[rec], W, cfg)
            tab["q"][rec], tab["k"][rec], tab["v"][rec] = q, k, v
        K = np.concatenate([np.asarray(prefix_k, F64), tab["k"]], axis=0)
        V = np.concatenate([np.asarray(prefix_v, F64), tab["v"]], axis=0)
        h = H[i] + attention(tab["q"], K, V) @ W["wo"]
        if rec.any():
            tab["f"][rec] = ffn(h[rec], W, cfg)
        out[i] = h + tab["f"]
        tables.append(tab)
    return out, fold, rho


# --------------------------------------------------------------------------
# One folded layer, order-free resolved-source form ([SF] §A.3, App. B)
# --------------------------------------------------------------------------

def folded_layer_resolved(H: np.ndarray, parent: Sequence[int], delta: float, W: dict,
                          prefix_k: np.ndarray, prefix_v: np.ndarray, cfg,
                          forced: Optional[np.ndarray] = None):
    """Same layer evaluated over the compacted recompute set: QKV and FFN run
    once per recomputed row; every (branch, position) reads its query and FFN
    output through its resolved source, and its block keys through the
    sources of the positions of its own branch.
    Returns (out, fold, rho, src)."""
    H = np.asarray(H, F64)
    Bp, L, d = H.shape
    P = prefix_k.shape[0]
    fold, rho = gate_request(H, parent, delta, forced)
    src = resolve_sources(fold, parent)
    rc = np.flatnonzero(~fold.reshape(-1))
    slot = -np.ones(Bp * L, dtype=np.int64)
    slot[rc] = np.arange(rc.size)
    X = H.reshape(Bp * L, d)[rc]
    q, k, v = project_qkv(X, P + rc % L, W, cfg)
    rcslot = slot[src * L + np.arange(L)[None, :]]          # [B+1, L]
    out = np.empty_like(H)
    h_all = np.empty_like(H)
    for i in range(Bp):
        K = np.concatenate([np.asarray(prefix_k, F64), k[rcslot[i]]], axis=0)
        V = np.concatenate([np.asarray(prefix_v, F64), v[rcslot[i]]], axis=0)
        h_all[i] = H[i] + attention(q[rcslot[i]], K, V) @ W["wo"]
    f = ffn(h_all.reshape(Bp * L, d)[rc], W, cfg)
    for i in range(Bp):
        out[i] = h_all[i] + f[rcslot[i]]
    return out, fold, rho, src


# --------------------------------------------------------------------------
# Dense per-branch layer (serialized verification, [SF] App. C)
# --------------------------------------------------------------------------

def dense_layer(H_branch: np.ndarray, W: dict, prefix_k: np.ndarray, prefix_v: np.ndarray, cfg):
    """A plain pre-norm transformer layer over one branch's block [L, d]."""
    H_branch = np.asarray(H_branch, F64)
    L = H_branch.shape[0]
    P = prefix_k.shape[0]
    q, k, v = project_qkv(H_branch, P + np.arange(L), W, cfg)
    K = np.concatenate([np.asarray(prefix_k, F64), k], axis=0)
    V = np.concatenate([np.asarray(prefix_v, F64), v], axis=0)
    h = H_branch + attention(q, K, V) @ W["wo"]
    return h + ffn(h, W, cfg)


# --------------------------------------------------------------------------
# Paper-style incremental attention correction ([SF] §A.1)
# --------------------------------------------------------------------------

def softmax_state(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Streaming-softmax state of one query row over keys K, V: per head the
    running max m, the denominator l = sum exp(s - m) and acc = sum exp(s - m) v.
    q: [nq, hd]; K, V: [S, nkv, hd]."""
    nq, hd = q.shape
    nkv = K.shape[1]
    G = nq // nkv
    s = np.einsum("kgd,skd->kgs", q.reshape(nkv, G, hd), K).reshape(nq, -1) / math.sqrt(hd)
    m = s.max(axis=-1)
    p = np.exp(s - m[:, None])
    Vh = np.repeat(V, G, axis=1)                             # [S, nq, hd]
    acc = np.einsum("hs,shd->hd", p, Vh)
    return m, p.sum(axis=-1), acc


def merge_states(states):
    """Log-sum-exp merge of softmax states over disjoint key sets."""
    m = np.max(np.stack([s[0] for s in states]), axis=0)
    l = sum(s[1] * np.exp(s[0] - m) for s in states)
    acc = sum(s[2] * np.exp(s[0] - m)[:, None] for s in states)
    return m, l, acc


def corrected_attention(q: np.ndarray, K_par: np.ndarray, V_par: np.ndarray,
                        K_own: np.ndarray, V_own: np.ndarray, changed: np.ndarray) -> np.ndarray:
    """Attention of a folded row computed the way §A.1 describes: start from the
    parent's softmax state over the parent's keys, remove the parent's
    contributions at the positions where the child's keys differ, add the
    child's contributions there.  q: [nq, hd]; K_*, V_*: [S, nkv, hd];
    changed: [S] bool.  Returns [nq * hd]."""
    nq, hd = q.shape
    m, l, acc = softmax_state(q, K_par, V_par)
    if changed.any():
        m_old, l_old, acc_old = softmax_state(q, K_par[changed], V_par[changed])
        m_new, l_new, acc_new = softmax_state(q, K_own[changed], V_own[changed])
        mx = np.maximum(m, m_new)
        sc, so, sn = np.exp(m - mx), np.exp(m_old - mx), np.exp(m_new - mx)
        l = l * sc - l_old * so + l_new * sn
        acc = acc * sc[:, None] - acc_old * so[:, None] + acc_new * sn[:, None]
    return (acc / l[:, None]).reshape(nq * hd)


# --------------------------------------------------------------------------
# Verification head: final RMSNorm, LM head, greedy tokens, draft acceptance
# ([SF] §1, §2.2: a draft whose state matches supplies logits that skip later
# denoising passes; App. B: the LM head runs outside the layer kernels)
# --------------------------------------------------------------------------

def lm_head_logits(h_rows: np.ndarray, final_norm: np.ndarray, W_lm: np.ndarray, eps: float) -> np.ndarray:
    """Logits of output rows [..., d]: RMSNorm with the final gain, then the
    LM head W_lm [d, V] (row-major [in, out] like every other weight)."""
    return rms_norm(h_rows, final_norm, eps) @ np.asarray(W_lm, F64)


def greedy_tokens(logits: np.ndarray) -> np.ndarray:
    """Greedy prediction per row: the index of the largest logit, the lowest
    such index on a tie."""
    return np.argmax(np.asarray(logits), axis=-1)


def accept_drafts(tokens: np.ndarray, parent: Sequence[int], pred: np.ndarray):
    """Draft acceptance of one request.

    tokens [B+1, L]: every branch's block tokens; pred [B+1, L]: every
    branch's greedy prediction at every position.  Reading (the pages say only
    that a matching draft can supply logits for later passes): draft i matches
    iff its parent matches and every position where its tokens differ from
    its parent's holds the parent's greedy prediction there.  The main branch
    always matches.  Returns (accepted [B+1] bool, chosen): chosen is the
    deepest matching branch, the lowest index among equally deep ones."""
    tokens = np.asarray(tokens)
    pred = np.asarray(pred)
    Bp = tokens.shape[0]
    accepted = np.zeros(Bp, dtype=bool)
    depth = np.zeros(Bp, dtype=np.int64)
    accepted[0] = True
    for i in range(1, Bp):                      # index order is topological
        p = parent[i]
        depth[i] = depth[p] + 1
        changed = tokens[i] != tokens[p]
        accepted[i] = accepted[p] and bool(np.all(tokens[i][changed] == pred[p][changed]))
    chosen = 0
    for i in range(Bp):
        if accepted[i] and depth[i] > depth[chosen]:
            chosen = i
    return accepted, chosen


# --------------------------------------------------------------------------
# Brute force with scalar loops, for tiny inputs only
# --------------------------------------------------------------------------

def folded_layer_bruteforce(H, parent, delta, W, prefix_k, prefix_v, cfg):
    """Scalar-loop evaluation of one folded layer of one request: every
    position walks its own fold chain, every projection and every attention
    score is an explicit Python sum.  Minutes of work beyond toy sizes."""
    H = np.asarray(H, F64)
    Bp, L, d = H.shape
    P = prefix_k.shape[0]
    nq, nkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    G = nq // nkv
    eps, theta = cfg.rms_eps, cfg.rope_theta
    Wd = {k: np.asarray(v, F64) for k, v in W.items()}

    def rms(row, gain):
        ms = sum(float(x) * float(x) for x in row) / len(row)
        r = 1.0 / math.sqrt(ms + eps)
        return [float(x) * r * float(g) for x, g in zip(row, gain)]

    def matvec(row, M):          # row [in] times M [in, out]
        out = [0.0] * M.shape[1]
        for a, x in enumerate(row):
            if x != 0.0:
                Ma = M[a]
                for b in range(M.shape[1]):
                    out[b] += x * float(Ma[b])
        return out

    def rot(vec, p):             # one head, rotate-half
        half = hd // 2
        res = list(vec)
        for j in range(half):
            a = p * theta ** (-2.0 * j / hd)
            c, s = math.cos(a), math.sin(a)
            res[j] = vec[j] * c - vec[j + half] * s
            res[j + half] = vec[j + half] * c + vec[j] * s
        return res

    # fold decisions from the definition
    fold = [[False] * L for _ in range(Bp)]
    for i in range(1, Bp):
        for n in range(L):
            num = math.sqrt(sum((float(a) - float(b)) ** 2 for a, b in zip(H[i, n], H[parent[i], n])))
            den = math.sqrt(sum(float(b) ** 2 for b in H[parent[i], n]))
            r = (0.0 if num == 0 else math.inf) if den == 0 else num / den
            fold[i][n] = delta > 0 and r <= delta

    def source(i, n):
        while fold[i][n]:
            i = parent[i]
        return i

    qkv_cache = {}

    def qkv(i, n):
        if (i, n) not in qkv_cache:
            xn = rms(H[i, n], Wd["attn_norm"])
            qf, kf, vf = matvec(xn, Wd["wq"]), matvec(xn, Wd["wk"]), matvec(xn, Wd["wv"])
            q = [rot(qf[h * hd:(h + 1) * hd], P + n) for h in range(nq)]
            k = [rot(kf[h * hd:(h + 1) * hd], P + n) for h in range(nkv)]
            v = [vf[h * hd:(h + 1) * hd] for h in range(nkv)]
            qkv_cache[(i, n)] = (q, k, v)
        return qkv_cache[(i, n)]

    h_rows = {}
    for i in range(Bp):
        for n in range(L):
            q = qkv(source(i, n), n)[0]
            attn = []
            for h in range(nq):
                kh = h // G
                scores, vals = [], []
                for m in range(P):
                    scores.append(sum(float(a) * float(b) for a, b in zip(q[h], prefix_k[m, kh])) / math.sqrt(hd))
                    vals.append([float(x) for x in prefix_v[m, kh]])
                for m in range(L):
                    _, km, vm = qkv(source(i, m), m)
                    scores.append(sum(a * b for a, b in zip(q[h], km[kh])) / math.sqrt(hd))
                    vals.append(vm[kh])
                mx = max(scores)
                w = [math.exp(s - mx) for s in scores]
                z = sum(w)
                attn.extend(sum(w[t] * vals[t][j] for t in range(len(w))) / z for j in range(hd))
            o = matvec(attn, Wd["wo"])
            h_rows[(i, n)] = [float(a) + b for a, b in zip(H[i, n], o)]

    f_cache = {}

    def ffn_out(i, n):
        if (i, n) not in f_cache:
            xn = rms(h_rows[(i, n)], Wd["ffn_norm"])
            g, u = matvec(xn, Wd["w_gate"]), matvec(xn, Wd["w_up"])
            act = [a / (1.0 + math.exp(-a)) * b for a, b in zip(g, u)]
            f_cache[(i, n)] = matvec(act, Wd["w_down"])
        return f_cache[(i, n)]

    out = np.empty_like(H)
    for i in range(Bp):
        for n in range(L):
            f = ffn_out(source(i, n), n)
            out[i, n] = [a + b for a, b in zip(h_rows[(i, n)], f)]
    return out, np.asarray(fold)


# --------------------------------------------------------------------------
# Whole pass over all layers and requests
# --------------------------------------------------------------------------

def layer_weights_f64(W: dict) -> dict:
    """Upcast one layer's weights (numpy or torch, any float dtype) to float64 numpy."""
    out = {}
    for k, v in W.items():
        if hasattr(v, "detach"):
            v = v.detach().to("cpu").double().numpy()
        out[k] = np.asarray(v, F64)
    return out


def verify_pass(H0, parents, delta: float, get_layer: Callable[[int], dict],
                prefix_k, prefix_v, cfg, n_layers: Optional[int] = None,
                form: str = "tables", forced: Optional[Callable] = None):
    """Run the folded pass over all layers.

    H0: [R, B+1, L, d]; parents: [R, B+1]; get_layer(l) -> float64 weights;
    prefix_k/v: [n_layers, R, P, nkv, hd].  forced(l) may return an int array
    [R, B+1, L] of decisions to impose (-1 = use the rule).
    Returns dict with out [R,B+1,L,d], fold/src [n_layers,R,B+1,L], rc lists,
    counts per layer and the per-layer inputs."""
    H = np.asarray(H0, F64).copy()
    R, Bp, L, d = H.shape
    nl = cfg.n_layers if n_layers is None else n_layers
    folds = np.zeros((nl, R, Bp, L), dtype=bool)
    srcs = np.zeros((nl, R, Bp, L), dtype=np.int64)
    rhos = np.zeros((nl, R, Bp, L))
    rcs, counts = [], []
    inputs = [H.copy()]
    for l in range(nl):
        W = get_layer(l)
        f_l = forced(l) if forced is not None else None
        out = np.empty_like(H)
        for r in range(R):
            pk = np.asarray(prefix_k[l, r], F64)
            pv = np.asarray(prefix_v[l, r], F64)
            fr = None if f_l is None else f_l[r]
            if form == "tables":
                out[r], fold, rho = folded_layer(H[r], parents[r], delta, W, pk, pv, cfg, fr)
                src = resolve_sources(fold, parents[r])
            else:
                out[r], fold, rho, src = folded_layer_resolved(H[r], parents[r], delta, W, pk, pv, cfg, fr)
            folds[l, r], srcs[l, r], rhos[l, r] = fold, src, rho
        rc, _, _ = compaction(folds[l])
        rcs.append(rc)
        counts.append(rc.size)
        H = out
        inputs.append(H.copy())
    return {"out": H, "fold": folds, "src": srcs, "rho": rhos, "rc": rcs,
            "rc_count": np.asarray(counts), "layer_inputs": inputs}
