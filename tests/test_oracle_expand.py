"""Pins for the oracle's TALON gated expansion.

TALON §5.1: the tree grows layer by layer until the node budget B is spent.
§5.2.2: layer 1 is the Top-K of the root's draft distribution.  §5.2.1: at
deeper layers every child of every frontier node is a candidate with path
score s(c) = product of draft probabilities along its path; the anchor is
the best candidate; candidates with s >= alpha * s_anchor survive; if more
survive than the remaining budget, the best-scoring ones are kept.

Pinned by
  * exhaustive enumeration over token sequences on tiny vocabularies, with
    path scores recomputed from scratch by a library log-softmax,
  * the invariants the pages fix, checked on the full-size TALON workload
    (vocab 32000, K 10, alpha 0.3, B 512, three entropy levels).
"""
import numpy as np
import pytest
from scipy.special import log_softmax

from workloads import gen


def enumerate_tree(drafter, K, alpha, budget, max_layers=50):
    """Grow the tree over token sequences.  Every sequence's score is the sum of
    library log-softmax terms along its path (no stored partial scores).
    Returns a list of layers, each a list of (sequence, score)."""
    def score(seq):
        key = drafter.root_key()
        tot = 0.0
        for t in seq:
            tot += float(log_softmax(drafter.row(key).astype(np.float64))[t])
            key = drafter.child_key(key, t)
        return tot

    V = drafter.V
    row0 = drafter.row(drafter.root_key())
    order = sorted(range(V), key=lambda t: (-row0[t], t))
    layer1 = [((t,), score((t,))) for t in order[:min(K, budget - 1)]]
    layers = [layer1]
    n = 1 + len(layer1)
    ids = {(): 0}
    for j, (s, _) in enumerate(sorted(layer1, key=lambda x: (-x[1], x[0]))):
        pass
    # number nodes as they are created: (parent asc, score desc, token asc)
    def number(layer_nodes, start):
        layer_nodes.sort(key=lambda x: (ids[x[0][:-1]], -x[1], x[0][-1]))
        for j, (s, _) in enumerate(layer_nodes):
            ids[s] = start + j
    number(layers[0], 1)
    while n < budget and layers[-1] and len(layers) < max_layers:
        cands = [(s + (t,), score(s + (t,))) for s, _ in layers[-1] for t in range(V)]
        anchor = max(c[1] for c in cands)
        keep = [c for c in cands if c[1] >= np.log(np.float32(alpha)) + anchor]
        keep.sort(key=lambda x: (-x[1], ids[x[0][:-1]], x[0][-1]))
        keep = keep[:budget - n]
        number(keep, n)
        n += len(keep)
        layers.append(keep)
    if not layers[-1]:
        layers.pop()
    return layers, ids


class SmallDrafter(gen.TalonDrafter):
    pass


@pytest.mark.parametrize("V,K,alpha,budget,sigma,seed", [
    (8, 3, 0.3, 20, 1.0, 1), (8, 3, 0.3, 20, 3.0, 2), (4, 2, 0.5, 12, 1.0, 3),
    (6, 6, 0.1, 30, 2.0, 4), (5, 1, 0.3, 9, 6.0, 5), (8, 10, 0.3, 20, 1.0, 6),
])
def test_exhaustive_small_vocab(oracle_mod, V, K, alpha, budget, sigma, seed):
    d = SmallDrafter(seed, V, sigma)
    res = oracle_mod.expand_tree(d, K, alpha, budget)
    layers, ids = enumerate_tree(d, K, alpha, budget)
    # rebuild the oracle's tree as token sequences
    seqs = [()]
    for i in range(1, res["n"]):
        seqs.append(seqs[res["parent"][i]] + (int(res["token"][i]),))
    assert res["n"] == 1 + sum(len(l) for l in layers)
    for s, i in ids.items():
        assert seqs[i] == s
    for layer in layers:
        for s, sc in layer:
            assert abs(res["logscore"][ids[s]] - sc) < 1e-5


def check_invariants(tree, drafter, K, alpha, budget):
    n, par, tok, ls = tree["n"], tree["parent"], tree["token"], tree["logscore"]
    V = drafter.V
    assert 1 <= n <= budget
    depth = gen.depth_of(par)
    keys = [drafter.root_key()]
    for i in range(1, n):
        assert 0 <= par[i] < i
        keys.append(drafter.child_key(keys[par[i]], tok[i]))
    # recompute every path score from scratch
    full = np.zeros(n)
    lsm = {}
    for i in range(n):
        if i > 0:
            p = par[i]
            if p not in lsm:
                lsm[p] = log_softmax(drafter.row(keys[p]).astype(np.float64))
            full[i] = full[p] + lsm[p][tok[i]]
    np.testing.assert_allclose(ls[:n], full, atol=2e-4, rtol=1e-5)
    # layer 1 is an exact Top-K of the root row
    l1 = np.nonzero(depth == 1)[0]
    assert len(l1) == min(K, V, budget - 1)
    row0 = drafter.row(keys[0])
    assert sorted(tok[l1].tolist()) == sorted(sorted(range(V), key=lambda t: (-row0[t], t))[:len(l1)])
    # monotone scores, distinct siblings, numbering order
    for i in range(1, n):
        assert full[i] <= full[par[i]] + 1e-12
    for v, kids in enumerate(gen.children_of(par)):
        assert len(set(tok[kids].tolist())) == len(kids)
    for i in range(2, n):
        if depth[i] == depth[i - 1]:
            a, b = i - 1, i
            assert (par[a], -full[a], tok[a]) <= (par[b], -full[b], tok[b]) or \
                (par[a] == par[b] and abs(full[a] - full[b]) < 1e-6)
        else:
            assert depth[i] == depth[i - 1] + 1
    # gate and budget at every layer >= 2
    for l in range(2, depth.max() + 1):
        prev = np.nonzero(depth == l - 1)[0]
        kept = set(np.nonzero(depth == l)[0].tolist())
        cand_scores = np.concatenate([full[v] + lsm.get(v, log_softmax(
            drafter.row(keys[v]).astype(np.float64))) for v in prev])
        anchor = cand_scores.max()
        thr = np.log(np.float32(alpha)) + anchor
        kept_scores = full[list(kept)]
        assert kept_scores.max() == pytest.approx(anchor, abs=1e-6)
        assert (kept_scores >= thr - 1e-6).all()
        n_pass = int((cand_scores >= thr).sum())
        if n_pass > len(kept):
            # truncated to the budget: nothing dropped beats what was kept
            assert depth[:n].tolist().count(l) == len(kept)
            assert n == budget
            dropped = np.sort(cand_scores[cand_scores >= thr])[::-1][len(kept):]
            assert dropped.max() <= kept_scores.min() + 1e-6


@pytest.mark.parametrize("context", [0, 1, 2])
def test_talon_workload_invariants(oracle_mod, context):
    d = gen.config3_drafter(context)
    tree = oracle_mod.expand_tree(d, 10, 0.3, 512)
    check_invariants(tree, d, 10, 0.3, 512)
    assert tree["n"] > 10


def test_invariant_checker_catches_planted_mistake(oracle_mod):
    d = SmallDrafter(7, 8, 1.0)
    tree = oracle_mod.expand_tree(d, 3, 0.3, 20)
    check_invariants(tree, d, 3, 0.3, 20)
    bad = dict(tree)
    bad["logscore"] = tree["logscore"].copy()
    bad["logscore"][-1] += 0.01          # a wrong score
    with pytest.raises(AssertionError):
        check_invariants(bad, d, 3, 0.3, 20)
    bad = dict(tree)
    bad["token"] = tree["token"].copy()
    l1 = np.nonzero(gen.depth_of(tree["parent"]) == 1)[0]
    bad["token"][l1[0]], bad["token"][l1[1]] = bad["token"][l1[1]], bad["token"][l1[0]]
    with pytest.raises(AssertionError):   # numbering order (score desc) broken
        check_invariants(bad, d, 3, 0.3, 20)


def test_layer_arguments(oracle_mod):
    par = np.full(8, -1, np.int32)
    tok = np.zeros(8, np.int32)
    ls = np.zeros(8, np.float32)
    row = np.array([[0.0, 3.0, 3.0, 1.0, 2.0]], np.float32)
    n, _ = oracle_mod.expand_gated(row, np.array([0], np.int32), np.zeros(1, np.float32), 1, 3,
                                   0.3, 8, par, tok, ls, 1)
    assert n == 4 and tok[1:4].tolist() == [1, 2, 4]        # tie 3.0 -> lower token first
    # budget already spent: nothing added
    n2, _ = oracle_mod.expand_gated(row, np.array([1], np.int32), ls[1:2], 2, 3, 0.3, 4, par, tok,
                                    ls, 4)
    assert n2 == 4
    with pytest.raises(ValueError):
        oracle_mod.expand_gated(np.zeros((2, 5), np.float32), np.array([0, 1], np.int32),
                                np.zeros(2, np.float32), 1, 3, 0.3, 8, par, tok, ls, 1)
