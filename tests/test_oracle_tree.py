"""Pins for the oracle's tree encoding (OPT-Tree §2: the tree attention mask
lets a node see its ancestors and itself).

The outputs are pinned by recursion identities that determine them uniquely
(depth[0] = 0, anc[0] = {0}; depth[i] = depth[parent[i]] + 1,
anc[i] = anc[parent[i]] + {i}), checked over every tree with up to 7 nodes
and on large random trees that cross the 64-bit word boundaries.
"""
import itertools

import numpy as np
import pytest

from workloads import gen


def all_trees(n):
    """Every parent array with parent[0] = -1 and 0 <= parent[i] < i."""
    for choice in itertools.product(*[range(i) for i in range(1, n)]):
        yield np.array((-1,) + choice, dtype=np.int32)


def bits(words, n):
    return {j for j in range(n) if (int(words[j // 64]) >> (j % 64)) & 1}


def check_identities(parent, depth, anc):
    n = len(parent)
    assert depth[0] == 0
    assert bits(anc[0], n) == {0}
    for i in range(1, n):
        p = parent[i]
        assert depth[i] == depth[p] + 1
        assert bits(anc[i], n) == bits(anc[p], n) | {i}
        assert sum(bin(int(w)).count("1") for w in anc[i]) == depth[i] + 1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7])
def test_every_small_tree(oracle_mod, n):
    trees = np.stack(list(all_trees(n)))
    depth, anc, status = oracle_mod.tree_build(trees)
    assert (status == 0).all()
    for t in range(len(trees)):
        check_identities(trees[t], depth[t], anc[t])


@pytest.mark.parametrize("n", [63, 64, 65, 128, 129, 300, 512])
def test_word_boundaries(oracle_mod, n):
    r = gen.rng(n)
    trees = np.stack([gen.random_tree(r, n, 40), gen.chain_tree(n), gen.star_tree(n)])
    depth, anc, status = oracle_mod.tree_build(trees)
    assert anc.shape == (3, n, (n + 63) // 64)
    assert (status == 0).all()
    for t in range(3):
        check_identities(trees[t], depth[t], anc[t])
    assert depth[1, n - 1] == n - 1          # chain
    assert depth[2].max() == 1               # star


def test_invalid_trees_flagged_per_sequence(oracle_mod):
    good = gen.chain_tree(5)
    bad_root = good.copy(); bad_root[0] = 0
    fwd = good.copy(); fwd[2] = 3
    self_loop = good.copy(); self_loop[3] = 3
    second_root = good.copy(); second_root[4] = -1
    neg = good.copy(); neg[1] = -7
    trees = np.stack([good, bad_root, fwd, self_loop, second_root, neg])
    depth, anc, status = oracle_mod.tree_build(trees)
    assert status.tolist() == [0, 2, 2, 2, 2, 2]
    assert (depth[1:] == -1).all() and (anc[1:] == 0).all()


def test_planted_mistake_is_caught():
    """The identity check rejects a plausible bug (off-by-one depth)."""
    parent = gen.chain_tree(4)
    depth = np.array([0, 1, 2, 2], np.int32)
    anc = np.array([[1], [3], [7], [15]], np.uint64)
    with pytest.raises(AssertionError):
        check_identities(parent, depth, anc)
