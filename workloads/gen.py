"""Seeded generators for draft trees, KV caches and logits.

Everything here is deterministic in its seed (numpy PCG64 streams) and
returns plain numpy arrays.  bf16 tensors are returned as their uint16 bit
patterns, rounded to nearest-even from float32.

Tree conventions used throughout:
  * ``parent[0] == -1`` (node 0 is the token right after the cached prefix),
  * ``0 <= parent[i] < i`` for ``i > 0`` (topological order), and
  * generated trees are relabelled into breadth-first order, children of a
    node keeping their creation order (so "first child" is well defined).

Workload shapes follow the five synthetic configurations of the tree-verify
benchmark: a tiny correctness case, a Llama-3-8B-shaped GOOSE spine tree, a
TALON gated-expansion tree, a ragged batch for stochastic acceptance and a
long-context OPT-Tree-style tree.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np

SEED_BASE = 0x7EE5EED0
MASK64 = (1 << 64) - 1

__all__ = [
    "SEED_BASE", "rng", "splitmix64", "bf16_from_f32", "f32_from_bf16",
    "normal_bf16", "bfs_relabel", "children_of", "depth_of", "random_tree",
    "chain_tree", "star_tree", "spine_tree_60", "opt_tree",
    "distinct_sibling_tokens", "planted_logits", "gumbel_children_tokens",
    "Case", "make_case", "config1", "config2", "config4", "config5",
    "TalonDrafter", "config3_drafter", "config3_verify", "CONFIG3_SIGMAS",
]


# ----------------------------------------------------------------------------
# random plumbing
# ----------------------------------------------------------------------------
def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed) & MASK64))


def splitmix64(x: int) -> int:
    """Vigna's splitmix64 finaliser, used to derive independent seeds."""
    x = (int(x) + 0x9E3779B97F4A7C15) & MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest even.

    Only finite inputs are expected (the generators produce normals)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_b = b.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_b.size, step):
        c = flat_b[s:s + step]
        flat_o[s:s + step] = ((c + np.uint32(0x7FFF) + ((c >> np.uint32(16)) & np.uint32(1)))
                              >> np.uint32(16)).astype(np.uint16)
    return out


def f32_from_bf16(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(r: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat.size, step):
        n = min(step, flat.size - s)
        x = r.standard_normal(n, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        flat[s:s + n] = bf16_from_f32(x)
    return out


# ----------------------------------------------------------------------------
# tree shapes
# ----------------------------------------------------------------------------
def children_of(parent) -> list:
    n = len(parent)
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[int(parent[i])].append(i)
    return kids


def depth_of(parent) -> np.ndarray:
    d = np.zeros(len(parent), dtype=np.int32)
    for i in range(1, len(parent)):
        d[i] = d[int(parent[i])] + 1
    return d


def bfs_relabel(parent):
    """Relabel a rooted tree (root 0, parent[root] = -1) into BFS order.

    Children keep their original relative order. Returns (new_parent, order)
    where order[new_id] = old_id."""
    parent = np.asarray(parent)
    kids = children_of(parent)
    order = [0]
    head = 0
    while head < len(order):
        order.extend(kids[order[head]])
        head += 1
    order = np.asarray(order, dtype=np.int64)
    new_id = np.empty(len(parent), dtype=np.int64)
    new_id[order] = np.arange(len(parent))
    new_parent = np.full(len(parent), -1, dtype=np.int32)
    for new in range(1, len(parent)):
        new_parent[new] = new_id[int(parent[order[new]])]
    return new_parent, order


def random_tree(r: np.random.Generator, n: int, max_depth: int) -> np.ndarray:
    """parent[i] uniform over the earlier nodes of depth < max_depth; BFS order."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int32)
    for i in range(1, n):
        cand = np.nonzero(depth[:i] < max_depth)[0]
        p = int(cand[r.integers(len(cand))])
        parent[i] = p
        depth[i] = depth[p] + 1
    return bfs_relabel(parent)[0]


def chain_tree(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def star_tree(n: int) -> np.ndarray:
    p = np.zeros(n, dtype=np.int32)
    p[0] = -1
    return p


def spine_tree_60():
    """GOOSE-style anisotropic spine tree with 60 nodes.

    A 24-node spine (depth 0..23), depth-1 side branches of widths
    4,4,3,3,2,2,1,1 at spine nodes 0..7 (branch width falling with depth),
    one further child under every branch node of spine nodes 0..3 and under
    the first branch node of spine nodes 4 and 5.  Returns (parent, kind) in
    BFS order with the spine child first; kind 0 = spine, 1 = branch,
    2 = branch child."""
    parent = [-1]
    kind = [0]
    for k in range(1, 24):
        parent.append(k - 1)
        kind.append(0)
    widths = [4, 4, 3, 3, 2, 2, 1, 1]
    branch_ids = []
    for s, w in enumerate(widths):
        ids = []
        for _ in range(w):
            ids.append(len(parent))
            parent.append(s)
            kind.append(1)
        branch_ids.append(ids)
    for s in range(4):
        for b in branch_ids[s]:
            parent.append(b)
            kind.append(2)
    for s in (4, 5):
        parent.append(branch_ids[s][0])
        kind.append(2)
    assert len(parent) == 60
    new_parent, order = bfs_relabel(np.asarray(parent, dtype=np.int32))
    return new_parent, np.asarray(kind, dtype=np.int32)[order]


def opt_tree(seed: int, n: int, V: int, max_depth: int = 16, branch: int = 8,
             sigma: float = 3.0):
    """Best-first tree over synthetic draft distributions (OPT-Tree style).

    Every node gets a draft row N(0, sigma) over V tokens; its `branch` most
    probable tokens are candidate children with path log-probability =
    parent's + log-softmax(row)[token].  Candidates are taken best first
    (ties -> parent, then token ascending) until n nodes exist, with depth
    <= max_depth.  Because path scores only fall along a path, the result is
    the set of n best-scoring reachable nodes.  Returns (parent, tokens) in
    BFS order; siblings have distinct tokens."""
    from scipy.special import log_softmax

    par = [-1]
    tok = [0]
    score = [0.0]
    dep = [0]
    heap: list = []

    def expand(v):
        if dep[v] >= max_depth:
            return
        row = rng(splitmix64(seed ^ (v * 0x9E3779B97F4A7C15 & MASK64))).standard_normal(V)
        row *= sigma
        lp = log_softmax(row)
        top = np.argpartition(-lp, branch)[:branch]
        for t in top:
            heapq.heappush(heap, (-(score[v] + float(lp[t])), v, int(t)))

    expand(0)
    while len(par) < n and heap:
        neg, p, t = heapq.heappop(heap)
        par.append(p)
        tok.append(t)
        score.append(-neg)
        dep.append(dep[p] + 1)
        expand(len(par) - 1)
    parent = np.asarray(par, dtype=np.int32)
    new_parent, order = bfs_relabel(parent)
    tokens = np.asarray(tok, dtype=np.int32)[order]
    return new_parent, tokens


# ----------------------------------------------------------------------------
# tokens and logits
# ----------------------------------------------------------------------------
def distinct_sibling_tokens(r: np.random.Generator, parent, V: int) -> np.ndarray:
    """Tokens for each node; siblings get distinct tokens uniform over V.
    Node 0 (the already-accepted token) gets a uniform token too."""
    n = len(parent)
    tokens = np.zeros(n, dtype=np.int32)
    tokens[0] = r.integers(V)
    for v, kids in enumerate(children_of(parent)):
        if kids:
            tokens[kids] = r.choice(V, size=len(kids), replace=False)
    return tokens


def planted_logits(r: np.random.Generator, parent, tokens, V: int,
                   p_first, p_other: float, boost: float = 10.0):
    """Target logits N(0,1) over V per node, with +boost planted on one child.

    For every node with children: the first child's token gets +boost with
    probability p_first (a float or a callable of the node); otherwise the
    later children are tried in order with probability p_other each, the first
    success winning; if none succeeds nothing is planted.  Row v is the
    distribution over v's children.  Returns (logits float32 [n, V],
    planted int32 [n]) with planted[v] = the planted child or -1."""
    n = len(parent)
    logits = r.standard_normal((n, V), dtype=np.float32)
    planted = np.full(n, -1, dtype=np.int32)
    for v, kids in enumerate(children_of(parent)):
        if not kids:
            continue
        pf = p_first(v) if callable(p_first) else p_first
        chosen = -1
        if r.random() < pf:
            chosen = kids[0]
        else:
            for c in kids[1:]:
                if r.random() < p_other:
                    chosen = c
                    break
        if chosen >= 0:
            logits[v, tokens[chosen]] += np.float32(boost)
            planted[v] = chosen
    return logits, planted


def gumbel_children_tokens(r: np.random.Generator, parent, q_logits: np.ndarray,
                           temperature: float = 1.0) -> np.ndarray:
    """Draft tokens drawn i.i.d. from each parent's draft distribution.

    Uses the Gumbel-max trick (argmax of logits/T plus Gumbel noise), which
    draws from softmax(logits/T) without forming it.  Node 0 gets a uniform
    token."""
    n = len(parent)
    V = q_logits.shape[1]
    tokens = np.zeros(n, dtype=np.int32)
    tokens[0] = r.integers(V)
    for v, kids in enumerate(children_of(parent)):
        if not kids:
            continue
        u = r.random((len(kids), V))
        g = -np.log(-np.log(u))
        tokens[kids] = np.argmax(q_logits[v][None, :].astype(np.float64) / temperature + g, axis=1)
    return tokens


# ----------------------------------------------------------------------------
# verification cases
# ----------------------------------------------------------------------------
@dataclass
class Case:
    name: str
    B: int
    N: int
    Hq: int
    Hkv: int
    D: int
    Lcap: int
    V: int
    kv_len: np.ndarray            # int32 [B]
    parent: np.ndarray            # int32 [B, N]
    tokens: np.ndarray            # int32 [B, N]
    q: Optional[np.ndarray]       # uint16 (bf16 bits) [B, N, Hq, D]
    k: Optional[np.ndarray]       # uint16 [B, Hkv, Lcap, D]
    v: Optional[np.ndarray]       # uint16 [B, Hkv, Lcap, D]
    logits: Optional[np.ndarray] = None     # float32 [B, N, V] (greedy)
    p_logits: Optional[np.ndarray] = None   # float32 [B, N, V] (stochastic)
    q_logits: Optional[np.ndarray] = None   # float32 [B, N, V]
    planted: Optional[np.ndarray] = None    # int32 [B, N]
    temperature: float = 1.0
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def tree_tokens(self) -> int:
        return self.B * self.N


def _attn_arrays(r, B, N, Hq, Hkv, D, Lcap, with_attn=True):
    if not with_attn:
        return None, None, None
    q = normal_bf16(r, (B, N, Hq, D))
    k = normal_bf16(r, (B, Hkv, Lcap, D))
    v = normal_bf16(r, (B, Hkv, Lcap, D))
    return q, k, v


def make_case(seed: int, *, B: int = 1, N: int = 16, L=128, Hq: int = 8, Hkv: int = 8,
              D: int = 64, V: int = 1000, tree: str = "random", max_depth: int = 6,
              mode: str = "greedy", p_first=0.8, p_other: float = 0.15,
              Lcap: Optional[int] = None, with_attn: bool = True,
              q_noise: float = 0.5, temperature: float = 1.0, name: str = "case") -> Case:
    """A generic verification case.

    L is an int (same prefix for every sequence) or a (lo, hi) pair (uniform
    ragged prefix lengths).  tree is 'random', 'chain', 'star', 'spine60' or
    'opt'.  mode 'greedy' makes planted target logits; 'sample' makes target
    logits N(0,1), draft logits = target + N(0, q_noise) and draws every
    node's children i.i.d. from its parent's draft distribution."""
    r = rng(seed)
    if isinstance(L, (tuple, list)):
        kv_len = r.integers(L[0], L[1] + 1, size=B).astype(np.int32)
    else:
        kv_len = np.full(B, int(L), dtype=np.int32)
    if Lcap is None:
        Lcap = int(kv_len.max()) + N
    parents, tokens, planted = [], [], []
    logits = p_log = q_log = None
    if mode == "greedy":
        logits = np.empty((B, N, V), dtype=np.float32)
    else:
        p_log = np.empty((B, N, V), dtype=np.float32)
        q_log = np.empty((B, N, V), dtype=np.float32)
    for b in range(B):
        kind = None
        if tree == "random":
            par = random_tree(r, N, max_depth)
        elif tree == "chain":
            par = chain_tree(N)
        elif tree == "star":
            par = star_tree(N)
        elif tree == "spine60":
            assert N == 60
            par, kind = spine_tree_60()
        elif tree == "opt":
            par, tok_opt = opt_tree(splitmix64(seed + 7919 * b), N, V, max_depth=max_depth)
        else:
            raise ValueError(tree)
        if mode == "greedy":
            tok = tok_opt if tree == "opt" else distinct_sibling_tokens(r, par, V)
            if kind is not None:
                kids = children_of(par)
                pf = (lambda v, kids=kids, kind=kind:
                      p_first if (kids[v] and kind[kids[v][0]] == 0) else p_other)
            else:
                pf = p_first
            lg, pl = planted_logits(r, par, tok, V, pf, p_other)
            logits[b] = lg
            planted.append(pl)
        else:
            lp = r.standard_normal((N, V), dtype=np.float32)
            lq = lp + r.normal(0.0, q_noise, size=(N, V)).astype(np.float32)
            tok = gumbel_children_tokens(r, par, lq, temperature)
            p_log[b] = lp
            q_log[b] = lq
        parents.append(par)
        tokens.append(tok)
    q, k, v = _attn_arrays(r, B, N, Hq, Hkv, D, Lcap, with_attn)
    return Case(name=name, B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, Lcap=Lcap, V=V, kv_len=kv_len,
                parent=np.stack(parents).astype(np.int32),
                tokens=np.stack(tokens).astype(np.int32), q=q, k=k, v=v,
                logits=logits, p_logits=p_log, q_logits=q_log,
                planted=np.stack(planted).astype(np.int32) if planted else None,
                temperature=temperature, seed=seed)


def config1(with_attn: bool = True) -> Case:
    """Tiny reference: 16-node random tree (depth <= 6), prefix 128, 8/8 heads,
    head_dim 64, vocab 1000, planted 0.8 / 0.15."""
    return make_case(SEED_BASE + 1, B=1, N=16, L=128, Hq=8, Hkv=8, D=64, V=1000,
                     tree="random", max_depth=6, p_first=0.8, p_other=0.15,
                     with_attn=with_attn, name="tiny-16node-L128")


def config2(with_attn: bool = True, with_logits: bool = True) -> Case:
    """Llama-3-8B-shaped GOOSE spine tree: 60 nodes, prefix 2048, 32/8 heads,
    head_dim 128, vocab 128256, planted 0.8 on the spine, 0.13 on branches."""
    V = 128256 if with_logits else 8
    return make_case(SEED_BASE + 2, B=1, N=60, L=2048, Hq=32, Hkv=8, D=128, V=V,
                     tree="spine60", p_first=0.8, p_other=0.13, with_attn=with_attn,
                     name="llama3-8b-spine60-L2048")


def config4(B: int = 16, V: int = 128256, with_attn: bool = True) -> Case:
    """Batched ragged stochastic verify: 16 sequences, prefixes uniform in
    [512, 8192], 64-node random trees (depth <= 8), 32/8 heads, head_dim 128,
    vocab 128256, draft = target + N(0, 0.5) noise, temperature 1."""
    return make_case(SEED_BASE + 4, B=B, N=64, L=(512, 8192), Hq=32, Hkv=8, D=128, V=V,
                     tree="random", max_depth=8, mode="sample", q_noise=0.5,
                     with_attn=with_attn, name="batched16-ragged-stochastic")


def config5(n: int = 256, with_attn: bool = True, V: int = 128256) -> Case:
    """Long-context verify: prefix 32768, 32/8 heads, head_dim 128, an
    n-node OPT-Tree-style tree (depth <= 16), vocab 128256, planted 0.8."""
    return make_case(SEED_BASE + 5, B=1, N=n, L=32768, Hq=32, Hkv=8, D=128, V=V,
                     tree="opt", max_depth=16, p_first=0.8, p_other=0.0,
                     with_attn=with_attn, name=f"longctx-L32768-opt{n}")


# ----------------------------------------------------------------------------
# TALON gated-expansion workload (configuration 3)
# ----------------------------------------------------------------------------
CONFIG3_SIGMAS = (1.0, 3.0, 6.0)


class TalonDrafter:
    """Synthetic draft model: node -> logits row N(0, sigma) over V.

    The row depends only on (seed, the token path from the root), so a
    given tree position always gets the same draft row whichever
    implementation grows the tree."""

    def __init__(self, seed: int, V: int, sigma: float):
        self.seed = int(seed) & MASK64
        self.V = int(V)
        self.sigma = float(sigma)

    def child_key(self, parent_key: int, token: int) -> int:
        return splitmix64(parent_key ^ splitmix64(int(token) + 1))

    def root_key(self) -> int:
        return splitmix64(self.seed)

    def row(self, key: int) -> np.ndarray:
        x = rng(key).standard_normal(self.V, dtype=np.float32)
        x *= np.float32(self.sigma)
        return x

    def rows(self, keys) -> np.ndarray:
        out = np.empty((len(keys), self.V), dtype=np.float32)
        for j, kk in enumerate(keys):
            out[j] = self.row(kk)
        return out


def config3_drafter(context: int, V: int = 32000) -> TalonDrafter:
    """One of the three contexts (sigma 1, 3, 6) of the TALON workload."""
    return TalonDrafter(splitmix64(SEED_BASE + 3) ^ context, V, CONFIG3_SIGMAS[context])


def config3_verify(parent: np.ndarray, context: int, *, L: int = 4096, Hq: int = 64,
                   Hkv: int = 8, D: int = 128, V: int = 32000, with_attn: bool = True,
                   tokens: Optional[np.ndarray] = None) -> Case:
    """Verify inputs for an expanded TALON tree: prefix 4096, 64/8 heads,
    head_dim 128, target vocab 32000, +10 planted on the first child with
    probability 0.8."""
    r = rng(splitmix64(SEED_BASE + 33) ^ context)
    N = len(parent)
    if tokens is None:
        tokens = distinct_sibling_tokens(r, parent, V)
    logits, planted = planted_logits(r, parent, tokens, V, 0.8, 0.0)
    Lcap = L + N
    q, k, v = _attn_arrays(r, 1, N, Hq, Hkv, D, Lcap, with_attn)
    return Case(name=f"talon-ctx{context}-N{N}", B=1, N=N, Hq=Hq, Hkv=Hkv, D=D, Lcap=Lcap,
                V=V, kv_len=np.array([L], dtype=np.int32), parent=parent[None].astype(np.int32),
                tokens=np.asarray(tokens, dtype=np.int32)[None], q=q, k=k, v=v,
                logits=logits[None], planted=planted[None], seed=context)
