"""CPU oracle for tree verification -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 statement of every step of the GPU library (tree
encoding, tree-verify attention, greedy and stochastic acceptance, TALON
gated expansion, the commit of the accepted branch into the KV cache, the
expected acceptance length of a tree, the GOOSE spine-tree builder,
OPT-Tree's greedy expansion and subtree selection), in
``oracle.cpp``, loaded here through ctypes.

Only the test suite, ``__graft_entry__.smoke()`` and the bench's CPU
baseline leg may import this package.  The GPU library never does, and the
two share no code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "oracle.cpp")
_LIB = os.path.join(_DIR, "liboracle.so")
_lib = None

ST_OK, ST_INVALID_ARG, ST_INVALID_TREE, ST_INVALID_TOKEN = 0, 1, 2, 6
PURPOSE_ACCEPT, PURPOSE_SAMPLE = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so (plain g++, no GPU)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        fd, tmp = tempfile.mkstemp(suffix=".so", dir=_DIR)
        os.close(fd)
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC", "-o", tmp,
                               _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.or_tree_build.argtypes = [P, I, I, P, P, P]
        lib.or_attn_rows.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, I, P, P]
        lib.or_accept_greedy.argtypes = [P, P, P, I, I, I, P, P, P, P, P, P]
        lib.or_accept_sample.argtypes = [P, P, P, P, I, I, I, ctypes.c_float, ctypes.c_uint64,
                                         ctypes.c_uint64, P, P, P, P, P, P, P, P, P]
        lib.or_set_threads.argtypes = [I]
        lib.or_set_threads.restype = None
        lib.or_expand_gated.argtypes = [P, P, P, I, I, I, I, ctypes.c_float, I, P, P, P, P, P]
        lib.or_expand_topn.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P]
        lib.or_select_topn.argtypes = [P, P, P, P, I, I, I, P, P, P, P, P, P]
        lib.or_commit_path.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P]
        lib.or_expected_accept.argtypes = [P, P, I, I, P, P, P]
        lib.or_build_spine_tree.argtypes = [P, I, P, I, I, I, I, ctypes.c_float, P, P, P]
        lib.or_philox4x64_10.argtypes = [P, P, P]
        lib.or_philox4x64_10.restype = None
        lib.or_draw_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64, I, I, I, ctypes.c_uint32]
        lib.or_draw_word.restype = ctypes.c_uint64
        for f in (lib.or_tree_build, lib.or_attn_rows, lib.or_accept_greedy,
                  lib.or_accept_sample, lib.or_expand_gated, lib.or_commit_path,
                  lib.or_expected_accept, lib.or_build_spine_tree):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def set_threads(n: int) -> None:
    """Threads for the oracle's loops over independent rows (n <= 0: one per
    core, the default)."""
    _load().or_set_threads(int(n))


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _check(rc):
    if rc != ST_OK:
        raise ValueError(f"oracle returned status {rc}")


def tree_build(parent: np.ndarray):
    """parent int32 [B, N] -> (depth int32 [B,N], anc uint64 [B,N,W], status int32 [B])."""
    parent = np.atleast_2d(parent)
    B, N = parent.shape
    W = (N + 63) // 64
    par, pp = _c(parent, np.int32)
    depth = np.zeros((B, N), np.int32)
    anc = np.zeros((B, N, W), np.uint64)
    status = np.zeros(B, np.int32)
    _check(_load().or_tree_build(pp, B, N, depth.ctypes.data, anc.ctypes.data, status.ctypes.data))
    return depth, anc, status


def attn_rows(q, k, v, kv_len, parent, Hq: int, Hkv: int, rows, scale: float = 0.0):
    """fp64 tree attention for the (b, i, h) triples in rows -> (out [n, D], lse [n]).

    q uint16 (bf16 bits) [B,N,Hq,D]; k, v uint16 [B,Hkv,Lcap,D]."""
    B, N, _, D = q.shape
    Lcap = k.shape[2]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = rows.shape[0]
    out = np.zeros((n, D), np.float64)
    lse = np.zeros(n, np.float64)
    qa, qp = _c(q, np.uint16)
    ka, kp = _c(k, np.uint16)
    va, vp = _c(v, np.uint16)
    la, lp = _c(kv_len, np.int32)
    pa, pp = _c(parent, np.int32)
    _check(_load().or_attn_rows(qp, kp, vp, lp, pp, B, N, Hq, Hkv, D, Lcap, float(scale),
                                rows.ctypes.data, n, out.ctypes.data, lse.ctypes.data))
    return out, lse


def attn_all(q, k, v, kv_len, parent, Hq: int, Hkv: int, scale: float = 0.0):
    """fp64 tree attention for every (b, i, h) -> (out [B,N,Hq,D], lse [B,N,Hq])."""
    B, N, _, D = q.shape
    bb, ii, hh = np.meshgrid(np.arange(B), np.arange(N), np.arange(Hq), indexing="ij")
    rows = np.stack([bb.ravel(), ii.ravel(), hh.ravel()], axis=1)
    out, lse = attn_rows(q, k, v, kv_len, parent, Hq, Hkv, rows, scale)
    return out.reshape(B, N, Hq, D), lse.reshape(B, N, Hq)


def accept_greedy(logits, tokens, parent) -> dict:
    logits = np.asarray(logits)
    B, N, V = logits.shape
    la, lp = _c(logits, np.float32)
    ta, tp = _c(tokens, np.int32)
    pa, pp = _c(parent, np.int32)
    r = dict(argmax=np.zeros((B, N), np.int32), accept_len=np.zeros(B, np.int32),
             end_node=np.zeros(B, np.int32), path=np.zeros((B, N), np.int32),
             bonus=np.zeros(B, np.int32), status=np.zeros(B, np.int32))
    _check(_load().or_accept_greedy(lp, tp, pp, B, N, V, r["argmax"].ctypes.data,
                                    r["accept_len"].ctypes.data, r["end_node"].ctypes.data,
                                    r["path"].ctypes.data, r["bonus"].ctypes.data,
                                    r["status"].ctypes.data))
    return r


def accept_sample(p_logits, q_logits, tokens, parent, temperature: float, seed: int,
                  offset: int) -> dict:
    p_logits = np.asarray(p_logits)
    B, N, V = p_logits.shape
    pa, ppl = _c(p_logits, np.float32)
    qa, qpl = _c(q_logits, np.float32)
    ta, tp = _c(tokens, np.int32)
    par, pp = _c(parent, np.int32)
    r = dict(accept_len=np.zeros(B, np.int32), end_node=np.zeros(B, np.int32),
             path=np.zeros((B, N), np.int32), out_token=np.zeros(B, np.int32),
             status=np.zeros(B, np.int32), margin_accept=np.zeros(B, np.float64),
             margin_path=np.zeros((B, N), np.float64), margin_draw=np.zeros(B, np.float64),
             draw_alt=np.zeros(B, np.int32))
    _check(_load().or_accept_sample(ppl, qpl, tp, pp, B, N, V, float(temperature),
                                    int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                    r["accept_len"].ctypes.data, r["end_node"].ctypes.data,
                                    r["path"].ctypes.data, r["out_token"].ctypes.data,
                                    r["status"].ctypes.data, r["margin_accept"].ctypes.data,
                                    r["margin_path"].ctypes.data, r["margin_draw"].ctypes.data,
                                    r["draw_alt"].ctypes.data))
    return r


def expand_gated(draft_logits, frontier_node, frontier_logscore, layer: int, topk: int,
                 alpha: float, budget: int, tree_parent, tree_token, tree_logscore,
                 n_nodes: int):
    """One TALON layer.  tree_* arrays (length >= budget) are updated in place.
    Returns (new n_nodes, margin)."""
    dl = np.ascontiguousarray(draft_logits, dtype=np.float32)
    F, V = dl.shape if dl.ndim == 2 else (0, 1)
    fn, fnp = _c(frontier_node, np.int32)
    fl, flp = _c(frontier_logscore, np.float32)
    assert tree_parent.dtype == np.int32 and tree_token.dtype == np.int32
    assert tree_logscore.dtype == np.float32
    nn = np.array([n_nodes], np.int32)
    margin = np.zeros(1, np.float64)
    _check(_load().or_expand_gated(dl.ctypes.data, fnp, flp, F, V, layer, topk, float(alpha),
                                   budget, tree_parent.ctypes.data, tree_token.ctypes.data,
                                   tree_logscore.ctypes.data, nn.ctypes.data,
                                   margin.ctypes.data))
    return int(nn[0]), float(margin[0])


def expand_tree(drafter, topk: int, alpha: float, budget: int, max_layers: int = 100000):
    """Grow a TALON tree layer by layer until the budget is spent or no
    candidate survives [TALON §5.1: budget-driven iterative growth].

    drafter has root_key(), child_key(key, token) and rows(keys).  Returns
    dict(parent, token, logscore, n, layers, margins)."""
    par = np.full(budget, -1, np.int32)
    tok = np.zeros(budget, np.int32)
    ls = np.zeros(budget, np.float32)
    keys = [drafter.root_key()]
    n = 1
    frontier = [0]
    margins = []
    layer = 1
    while n < budget and frontier and layer <= max_layers:
        rows = drafter.rows([keys[f] for f in frontier])
        n_new, m = expand_gated(rows, np.asarray(frontier, np.int32), ls[frontier], layer, topk,
                                alpha, budget, par, tok, ls, n)
        margins.append(m)
        for j in range(n, n_new):
            keys.append(drafter.child_key(keys[par[j]], tok[j]))
        frontier = list(range(n, n_new))
        n = n_new
        layer += 1
    return dict(parent=par[:n].copy(), token=tok[:n].copy(), logscore=ls[:n].copy(), n=n,
                layers=layer - 1, margins=margins)


def expand_topn(draft_logits, frontier_node, frontier_logscore, width: int, capacity: int,
                tree_parent, tree_token, tree_logscore, n_nodes: int):
    """One OPT-Tree layer: the `width` best children of the frontier are
    appended to the tree_* arrays (length >= capacity, updated in place).
    Returns (new n_nodes, margin)."""
    dl = np.ascontiguousarray(draft_logits, dtype=np.float32)
    F, V = dl.shape
    fn, fnp = _c(frontier_node, np.int32)
    fl, flp = _c(frontier_logscore, np.float32)
    assert tree_parent.dtype == np.int32 and tree_token.dtype == np.int32
    assert tree_logscore.dtype == np.float32 and tree_parent.size >= capacity
    nn = np.array([n_nodes], np.int32)
    margin = np.zeros(1, np.float64)
    _check(_load().or_expand_topn(dl.ctypes.data, fnp, flp, F, V, int(width), int(capacity),
                                  tree_parent.ctypes.data, tree_token.ctypes.data,
                                  tree_logscore.ctypes.data, nn.ctypes.data, margin.ctypes.data))
    return int(nn[0]), float(margin[0])


def select_topn(parent, token, logscore, n_nodes, n: int):
    """OPT-Tree subtree selection over B candidate trees [B, M].
    Returns dict(parent, token, logscore, src [B, n], expected [B], status [B])."""
    parent = np.atleast_2d(np.asarray(parent, np.int32))
    B, M = parent.shape
    pa, pp = _c(parent, np.int32)
    ta, tp = _c(np.atleast_2d(token), np.int32)
    la, lp = _c(np.atleast_2d(logscore), np.float32)
    ma, mp = _c(np.atleast_1d(n_nodes), np.int32)
    out = dict(parent=np.zeros((B, n), np.int32), token=np.zeros((B, n), np.int32),
               logscore=np.zeros((B, n), np.float32), src=np.zeros((B, n), np.int32),
               expected=np.zeros(B, np.float32), status=np.zeros(B, np.int32))
    _check(_load().or_select_topn(pp, tp, lp, mp, B, M, int(n), out["parent"].ctypes.data,
                                  out["token"].ctypes.data, out["logscore"].ctypes.data,
                                  out["src"].ctypes.data, out["expected"].ctypes.data,
                                  out["status"].ctypes.data))
    return out


def opt_tree(drafter, width: int, layers: int, n: int):
    """Grow an OPT-Tree candidate tree for `layers` layers of `width` nodes
    each (the root's layer is 1), then keep its n best nodes [OPT §3].

    drafter has root_key(), child_key(key, token) and rows(keys).  Returns
    dict(parent, token, logscore, n (the candidate tree), margins,
    selected (select_topn's output for the single tree))."""
    cap = 1 + width * layers
    par = np.full(cap, -1, np.int32)
    tok = np.zeros(cap, np.int32)
    ls = np.zeros(cap, np.float32)
    keys = [drafter.root_key()]
    n_nodes = 1
    lo, hi = 0, 1
    margins = []
    for _ in range(layers):
        rows = drafter.rows(keys[lo:hi])
        n_new, m = expand_topn(rows, np.arange(lo, hi, dtype=np.int32), ls[lo:hi], width, cap,
                               par, tok, ls, n_nodes)
        margins.append(m)
        for j in range(n_nodes, n_new):
            keys.append(drafter.child_key(keys[par[j]], tok[j]))
        lo, hi, n_nodes = n_nodes, n_new, n_new
    sel = select_topn(par[None, :n_nodes], tok[None, :n_nodes], ls[None, :n_nodes],
                      [n_nodes], n)
    return dict(parent=par[:n_nodes].copy(), token=tok[:n_nodes].copy(),
                logscore=ls[:n_nodes].copy(), n=n_nodes, margins=margins,
                selected={k: v[0] for k, v in sel.items()})


def commit_path(k, v, kv_len, path, accept_len):
    """Move each sequence's accepted branch to consecutive cache positions.

    k, v uint16 (bf16 bits) [B, Hkv, Lcap, D] are copied, not modified.
    Returns (k', v', new_kv_len int32 [B], status int32 [B])."""
    k2 = np.array(k, dtype=np.uint16, copy=True, order="C")
    v2 = np.array(v, dtype=np.uint16, copy=True, order="C")
    B, Hkv, Lcap, D = k2.shape
    path = np.atleast_2d(np.asarray(path, np.int32))
    N = path.shape[1]
    la, lp = _c(kv_len, np.int32)
    pa, pp = _c(path, np.int32)
    aa, ap = _c(accept_len, np.int32)
    new_len = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    _check(_load().or_commit_path(k2.ctypes.data, v2.ctypes.data, lp, pp, ap, B, N, Hkv, D, Lcap,
                                  new_len.ctypes.data, status.ctypes.data))
    return k2, v2, new_len, status


def expected_accept(parent, prob):
    """Node scores (products of draft probabilities along the path) and the
    expected acceptance length (their sum over draft nodes).
    Returns (score float64 [B, N], expected float64 [B], status int32 [B])."""
    parent = np.atleast_2d(np.asarray(parent, np.int32))
    B, N = parent.shape
    pa, pp = _c(parent, np.int32)
    qa, qp = _c(np.atleast_2d(prob), np.float32)
    score = np.zeros((B, N), np.float64)
    expected = np.zeros(B, np.float64)
    status = np.zeros(B, np.int32)
    _check(_load().or_expected_accept(pp, qp, B, N, score.ctypes.data, expected.ctypes.data,
                                      status.ctypes.data))
    return score, expected, status


def build_spine_tree(spine_tokens, branch_tokens, root_token: int, budget: int,
                     spine_ratio: float):
    """GOOSE spine tree: (parent int32 [n], tokens int32 [n]).

    spine_tokens int32 [S]; branch_tokens int32 [Sb, K] (row j: candidates
    for a branch off spine node j, best first, -1 ends a row)."""
    sp, spp = _c(np.asarray(spine_tokens, np.int32).reshape(-1), np.int32)
    br = np.asarray(branch_tokens, np.int32)
    if br.ndim != 2:
        br = br.reshape(0, 0)
    ba, bp = _c(br, np.int32)
    parent = np.zeros(budget, np.int32)
    tokens = np.zeros(budget, np.int32)
    n = np.zeros(1, np.int32)
    _check(_load().or_build_spine_tree(spp, sp.size, bp, br.shape[0], br.shape[1] if br.ndim == 2 else 0,
                                       int(root_token), int(budget), float(spine_ratio),
                                       parent.ctypes.data, tokens.ctypes.data, n.ctypes.data))
    return parent[:n[0]].copy(), tokens[:n[0]].copy()


def philox4x64_10(ctr, key) -> np.ndarray:
    c, cp = _c(ctr, np.uint64)
    k, kp = _c(key, np.uint64)
    out = np.zeros(4, np.uint64)
    _load().or_philox4x64_10(cp, kp, out.ctypes.data)
    return out


def draw_word(seed: int, offset: int, b: int, node: int, purpose: int, ordinal: int) -> int:
    return int(_load().or_draw_word(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), b, node,
                                    purpose, ordinal))
