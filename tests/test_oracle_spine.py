"""Pins for the oracle's GOOSE spine tree (GOOSE §2A: a deep chain of
context-matched tokens with wide branches of transition tokens forking off
the spine, wide near the root and narrower deeper down; §2B Proposition 2:
the branch allocation decreases linearly with depth; Proposition 3: the
anisotropic tree beats single-source isotropic trees when the sources'
acceptance rates differ).  The pages give the shape, not a formula: the pins
check the rules they state."""
import numpy as np
import pytest

from workloads import gen


def candidates(seed, S, Sb, K, V=50000):
    r = gen.rng(seed)
    spine = r.choice(V, S, replace=False).astype(np.int32)
    br = np.stack([r.choice(V, K, replace=False) for _ in range(Sb)]).astype(np.int32) if Sb else \
        np.zeros((0, K), np.int32)
    return spine, br


def depths(parent):
    return gen.depth_of(parent)


def check_structure(parent, tokens, spine, br, root, budget):
    n = len(parent)
    assert 1 <= n <= budget and parent[0] == -1 and tokens[0] == root
    assert all(0 <= parent[i] < i for i in range(1, n))
    dep = depths(parent)
    assert np.all(np.diff(dep) >= 0)                       # breadth-first numbering
    spine_ids = [0]
    for t in range(1, dep.max() + 1):
        level = np.flatnonzero(dep == t)
        kids_of_spine = [i for i in level if parent[i] == spine_ids[-1]]
        if len(spine_ids) - 1 < len(spine) and t <= len(spine) and tokens[level[0]] == spine[t - 1] \
                and parent[level[0]] == spine_ids[-1]:
            spine_ids.append(int(level[0]))                # the spine child comes first
        assert all(parent[i] in spine_ids for i in level)  # branches hang off the spine
        assert len(set(tokens[kids_of_spine])) == len(kids_of_spine)  # distinct siblings
    return spine_ids


@pytest.mark.parametrize("seed,S,Sb,K,budget,ratio", [
    (1, 24, 24, 8, 60, 0.4), (2, 30, 30, 6, 100, 0.25), (3, 5, 8, 4, 64, 0.5),
    (4, 12, 12, 3, 40, 0.6), (5, 40, 40, 10, 512, 0.1),
])
def test_structure_and_linear_allocation(oracle_mod, seed, S, Sb, K, budget, ratio):
    spine, br = candidates(seed, S, Sb, K)
    parent, tokens = oracle_mod.build_spine_tree(spine, br, 7, budget, ratio)
    spine_ids = check_structure(parent, tokens, spine, br, 7, budget)
    d = len(spine_ids) - 1
    assert d == min(S, int(round(ratio * (budget - 1))))
    assert np.array_equal(tokens[spine_ids[1:]], spine[:d])   # the spine is the PLD chain
    # branch widths: one per spine node, non-increasing with depth while no
    # candidate row runs out, and within one node of a straight line
    w = np.array([sum(1 for i in range(1, len(parent)) if parent[i] == sid and i not in spine_ids)
                  for sid in spine_ids])
    m = min(d + 1, Sb)
    R = budget - 1 - d
    if R <= K * m // 2:   # candidates never limiting in these cases
        assert w.sum() == min(R, K * m)
        assert np.all(np.diff(w[:m]) <= 0)
        line = R * (m - np.arange(m)) / (m * (m + 1) / 2)
        assert np.all(np.abs(w[:m] - line) <= 1.0)


def test_ratio_extremes(oracle_mod):
    spine, br = candidates(9, 20, 20, 5)
    parent, tokens = oracle_mod.build_spine_tree(spine, br, 1, 21, 1.0)   # all to the spine
    assert np.array_equal(parent, np.arange(-1, 20)) and np.array_equal(tokens[1:], spine)
    parent, tokens = oracle_mod.build_spine_tree(spine, br, 1, 30, 0.0)   # no spine: a star
    assert (parent[1:] == 0).all() and len(parent) == 1 + 5
    assert np.array_equal(tokens[1:], br[0])
    parent, tokens = oracle_mod.build_spine_tree(spine, br, 1, 1, 0.5)    # budget of one node
    assert parent.tolist() == [-1]


def test_branches_skip_the_spine_token_and_repeats(oracle_mod):
    spine = np.array([10, 11, 12], np.int32)
    br = np.array([[10, 20, 20, 21, -1, 99], [30, 11, 31, 32, 33, 34], [40, 41, 42, 43, 44, 45]],
                  np.int32)
    parent, tokens = oracle_mod.build_spine_tree(spine, br, 0, 12, 0.3)
    kids0 = tokens[1:][parent[1:] == 0].tolist()
    assert kids0[0] == 10 and kids0[1:] == [20, 21]       # spine child, then row 0 up to -1
    assert 11 not in tokens[parent == 1][1:].tolist()


def test_anisotropic_tree_beats_single_source_trees(oracle_mod):
    """Proposition 3 under a concrete model: the target's next token is the
    spine token with probability ps, else one of the transition candidates,
    the i-th with probability (1 - ps) q (1 - q)^i; a transition-only tree
    sees the candidates with probability q (1 - q)^i.  The spine tree's
    expected acceptance length exceeds the chain's and every balanced
    transition-only tree's of the same size."""
    ps, q, budget, S, K = 0.8, 0.4, 60, 24, 8
    spine, br = candidates(11, S, S, K)
    parent, tokens = oracle_mod.build_spine_tree(spine, br, 0, budget, 0.4)
    spine_ids = check_structure(parent, tokens, spine, br, 0, budget)
    prob = np.zeros(len(parent), np.float32)
    rank = {}
    for i in range(1, len(parent)):
        if i in spine_ids:
            prob[i] = ps
        else:
            k = rank.get(parent[i], 0)
            rank[parent[i]] = k + 1
            prob[i] = (1 - ps) * q * (1 - q) ** k
    _, e_spine, _ = oracle_mod.expected_accept(parent[None], prob[None])
    _, e_chain, _ = oracle_mod.expected_accept(gen.chain_tree(S + 1)[None],
                                               np.full((1, S + 1), ps, np.float32))
    best_tr = 0.0
    for b in range(1, 9):   # balanced b-ary transition-only trees of `budget` nodes
        par = np.array([-1] + [(i - 1) // b for i in range(1, budget)], np.int32)
        pr = np.array([0.0] + [q * (1 - q) ** ((i - 1) % b) for i in range(1, budget)], np.float32)
        _, e, _ = oracle_mod.expected_accept(par[None], pr[None])
        best_tr = max(best_tr, float(e[0]))
    assert e_spine[0] > e_chain[0] and e_spine[0] > best_tr


def test_bad_arguments(oracle_mod):
    spine, br = candidates(3, 4, 4, 2)
    for kw in (dict(budget=0, spine_ratio=0.5), dict(budget=10, spine_ratio=1.5),
               dict(budget=10, spine_ratio=-0.1)):
        with pytest.raises(ValueError):
            oracle_mod.build_spine_tree(spine, br, 0, kw["budget"], kw["spine_ratio"])
