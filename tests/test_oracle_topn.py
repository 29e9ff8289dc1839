"""Pins for the oracle's OPT-Tree greedy expansion and subtree selection.

OPT-Tree §3: node scores are products of draft probabilities along the path;
the tree grows by expanding the frontier nodes with the largest scores, and
the n best-scoring nodes are kept as a subtree that contains the root (the
scores never rise along a path, so that set is closed under parents).
Pinned by
  * brute force over every root-containing subtree of n nodes of small
    trees: the selection is the one with the largest sum of scores, and its
    expected length is that sum less the root's,
  * an independent best-first search (a heap over all V children of every
    node, depth-limited) on a synthetic drafter: layers of `width` = n
    followed by the selection give the same n token paths,
  * the one-row case, which is the top-k of a log-softmax (library routines),
    ties to the lower token,
  * exact ties, the capacity cut, and malformed inputs.
"""
import heapq
import itertools

import numpy as np
import pytest
from scipy.special import log_softmax

from workloads import gen


def random_monotone_tree(r, M, tie=False):
    parent = np.full(M, -1, np.int32)
    ls = np.zeros(M, np.float32)
    for i in range(1, M):
        parent[i] = r.integers(0, i)
        step = -float(r.integers(0, 3)) if tie else float(np.log(r.uniform(0.05, 1.0)))
        ls[i] = np.float32(ls[parent[i]] + step)
    return parent, ls


def best_subtree(parent, ls, n):
    """The root-containing, parent-closed set of n nodes with the largest
    sum of exp(score), by enumeration."""
    M = len(parent)
    best, best_val = None, -1.0
    for rest in itertools.combinations(range(1, M), n - 1):
        s = {0, *rest}
        if any(parent[i] not in s for i in rest):
            continue
        val = sum(np.exp(float(ls[i])) for i in s)
        if val > best_val + 1e-12:
            best, best_val = s, val
    return best, best_val


@pytest.mark.parametrize("seed", range(12))
def test_selection_is_the_best_subtree(oracle_mod, seed):
    r = gen.rng(900 + seed)
    M = int(r.integers(2, 10))
    parent, ls = random_monotone_tree(r, M)
    token = r.integers(0, 1000, M).astype(np.int32)
    for n in range(1, M + 1):
        o = oracle_mod.select_topn(parent, token, ls, [M], n)
        assert o["status"][0] == 0
        s, val = best_subtree(parent, ls, n)
        src = o["src"][0]
        assert set(src.tolist()) == s
        assert abs(float(o["expected"][0]) - (val - 1.0)) < 1e-5 * max(1.0, val)
        # renumbering: original order kept, parents mapped, tokens and scores carried
        assert np.all(np.diff(src) > 0) and src[0] == 0
        pos = {int(v): j for j, v in enumerate(src)}
        for j in range(1, n):
            assert o["parent"][0][j] == pos[int(parent[src[j]])] < j
            assert o["token"][0][j] == token[src[j]]
            assert o["logscore"][0][j] == ls[src[j]]
        assert o["parent"][0][0] == -1


def test_selection_ties_go_to_lower_ids(oracle_mod):
    # a star whose leaves all score log(0.5), and a chain of probability one
    parent = np.array([-1, 0, 0, 0, 0, 0], np.int32)
    ls = np.array([0.0] + [np.log(0.5)] * 5, np.float32)
    o = oracle_mod.select_topn(parent, np.arange(6), ls, [6], 3)
    assert o["src"][0].tolist() == [0, 1, 2]
    chain = np.arange(-1, 7, dtype=np.int32)
    o = oracle_mod.select_topn(chain, np.arange(8), np.zeros(8, np.float32), [8], 4)
    assert o["src"][0].tolist() == [0, 1, 2, 3]
    assert o["parent"][0].tolist() == [-1, 0, 1, 2]
    assert o["expected"][0] == 3.0
    # many exact ties in a random tree: still a subtree, still the best sum
    r = gen.rng(77)
    parent, ls = random_monotone_tree(r, 9, tie=True)
    for n in range(1, 10):
        o = oracle_mod.select_topn(parent, np.arange(9), ls, [9], n)
        assert o["status"][0] == 0
        _, val = best_subtree(parent, ls, n)
        assert abs(float(o["expected"][0]) - (val - 1.0)) < 1e-5 * val


def test_selection_ragged_batch_and_bad_inputs(oracle_mod):
    r = gen.rng(5)
    B, M = 6, 12
    par = np.zeros((B, M), np.int32)
    ls = np.zeros((B, M), np.float32)
    for b in range(B):
        par[b], ls[b] = random_monotone_tree(r, M)
    m = np.array([12, 3, 12, 12, 12, 0], np.int32)
    i = int(np.flatnonzero(par[2] > 0)[0])   # a child better than the root, its parent the worst
    ls[2, i] = 0.5
    ls[2, par[2, i]] = -50.0
    par[3, 4] = 9                    # a parent after its child
    ls[4, 2] = np.nan
    tok = np.arange(B * M, dtype=np.int32).reshape(B, M)
    o = oracle_mod.select_topn(par, tok, ls, m, 5)
    assert o["status"].tolist() == [0, 0, 2, 2, 1, 1]
    # fewer nodes than n: all of them, then -1 rows
    assert o["src"][1].tolist() == [0, 1, 2, -1, -1]
    assert o["parent"][1][3:].tolist() == [-1, -1] and o["token"][1][3:].tolist() == [-1, -1]
    for b in (2, 3, 4, 5):
        assert (o["src"][b] == -1).all() and (o["parent"][b] == -1).all()
        assert o["expected"][b] == 0
    # the non-monotone child only breaks the subtree when its parent is cut
    o = oracle_mod.select_topn(par[2:3], tok[2:3], ls[2:3], [12], 12)
    assert o["status"][0] == 0


def best_first(drafter, depth, n):
    """The n best nodes (score = sum of fp64 log-softmax values along the
    path) of the drafter's tree cut at `depth`, by a heap over every child of
    every node taken; returns {token path: score} and the gap at the cut."""
    heap = []
    taken = {(): 0.0}

    def push_children(path, key, score):
        if len(path) >= depth:
            return
        lp = log_softmax(drafter.row(key).astype(np.float64))
        for t in range(drafter.V):
            heapq.heappush(heap, (-(score + lp[t]), path + (t,), key, t))

    push_children((), drafter.root_key(), 0.0)
    while len(taken) < n:
        neg, path, pkey, t = heapq.heappop(heap)
        taken[path] = -neg
        push_children(path, drafter.child_key(pkey, t), -neg)
    gap = (sorted(taken.values())[0] + heap[0][0]) if heap else np.inf
    return taken, gap


def token_paths(parent, token):
    out = []
    for i in range(len(parent)):
        p, path = i, []
        while p > 0:
            path.append(int(token[p]))
            p = parent[p]
        out.append(tuple(reversed(path)))
    return out


@pytest.mark.parametrize("seed,V,sigma,n,depth", [
    (1, 4, 1.0, 12, 4), (2, 6, 2.0, 20, 5), (3, 8, 3.0, 30, 6), (4, 3, 0.5, 15, 8),
    (5, 16, 1.5, 40, 3), (6, 5, 4.0, 25, 10),
])
def test_layers_then_selection_equal_best_first(oracle_mod, seed, V, sigma, n, depth):
    d = gen.TalonDrafter(seed, V, sigma)
    want, gap = best_first(d, depth, n)
    assert gap > 1e-5, "choose a case without a near tie at the cut"
    o = oracle_mod.opt_tree(d, n, depth, n)
    sel = o["selected"]
    assert sel["status"] == 0
    paths = token_paths(sel["parent"], sel["token"])
    assert set(paths) == set(want)
    for j, pth in enumerate(paths):
        assert abs(float(sel["logscore"][j]) - want[pth]) < 1e-5
    want_e = sum(np.exp(v) for pth, v in want.items() if pth)   # the root not counted
    assert abs(float(sel["expected"]) - want_e) < 1e-5 * max(1.0, want_e)
    # every layer keeps `width` nodes while the vocabulary allows it
    depth_of = gen.depth_of(o["parent"])
    for l in range(1, depth + 1):
        assert int((depth_of == l).sum()) == min(n, V ** l)


@pytest.mark.parametrize("V,width", [(50, 7), (300, 300), (9, 20)])
def test_one_row_is_the_top_k_of_log_softmax(oracle_mod, V, width):
    r = gen.rng(V)
    row = np.round(r.standard_normal(V) * 2).astype(np.float32)  # many exact ties
    cap = 1 + width
    par = np.full(cap, -1, np.int32)
    tok = np.zeros(cap, np.int32)
    ls = np.zeros(cap, np.float32)
    n, _ = oracle_mod.expand_topn(row[None], np.array([0], np.int32), np.zeros(1, np.float32),
                                  width, cap, par, tok, ls, 1)
    k = min(width, V)
    assert n == 1 + k
    lp = log_softmax(row.astype(np.float64))
    order = np.lexsort((np.arange(V), -lp))[:k]          # score desc, token asc
    assert tok[1:n].tolist() == order.tolist()
    assert (par[1:n] == 0).all()
    np.testing.assert_allclose(ls[1:n], lp[order].astype(np.float32), rtol=1e-6, atol=1e-6)


def test_layer_over_many_rows_and_the_capacity_cut(oracle_mod):
    r = gen.rng(11)
    F, V, width = 7, 40, 25
    rows = (r.standard_normal((F, V)) * 2).astype(np.float32)
    fl = -np.abs(r.standard_normal(F)).astype(np.float32)
    front = np.arange(3, 3 + F, dtype=np.int32)
    for cap, n0 in ((100, 10), (20, 10)):
        par = np.full(cap, -1, np.int32)
        tok = np.zeros(cap, np.int32)
        ls = np.zeros(cap, np.float32)
        n, margin = oracle_mod.expand_topn(rows, front, fl, width, cap, par, tok, ls, n0)
        k = min(width, cap - n0)
        assert n == n0 + k
        S = fl[:, None].astype(np.float64) + log_softmax(rows.astype(np.float64), axis=1)
        v_idx, c_idx = np.divmod(np.arange(F * V), V)
        best = np.lexsort((c_idx, v_idx, -S.ravel()))[:k]
        want = sorted(zip(front[v_idx[best]].tolist(), (-S.ravel()[best]).tolist(),
                          c_idx[best].tolist()))
        assert list(zip(par[n0:n].tolist(), tok[n0:n].tolist())) == [(p, t) for p, _, t in want]
        assert margin > 0


def test_expand_topn_bad_arguments(oracle_mod):
    z = np.zeros(4, np.int32)
    zl = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        oracle_mod.expand_topn(np.zeros((1, 3), np.float32), [0], [0.0], 0, 4, z, z, zl, 1)
    # a full tree: nothing more is kept
    n, _ = oracle_mod.expand_topn(np.zeros((1, 3), np.float32), [0], [0.0], 2, 4, z, z, zl, 4)
    assert n == 4
