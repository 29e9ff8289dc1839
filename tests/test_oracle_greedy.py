"""Pins for the oracle's greedy acceptance.

OPT-Tree §2: under greedy sampling the longest branch that matches the
target's highest-probability sequence is accepted (GOOSE §2C: the greedy walk
verifies the whole tree from one pass).  Pinned by
  * top-down enumeration of every branch on small trees (np.argmax for the
    target's choices; the oracle walks upward from every node instead),
  * the planted construction (the generator knows which child it boosted),
  * chains (accept length = number of leading matches),
  * argmax ties, signed zeros and bad inputs.
"""
import itertools

import numpy as np
import pytest

from workloads import gen


def branches_top_down(parent, tokens, logits):
    """All accepted nodes found by walking down from the root: a child c of an
    accepted node v is accepted iff tokens[c] is the target's top token at v."""
    kids = gen.children_of(parent)
    top = np.argmax(logits, axis=1)
    accepted = [0]
    stack = [0]
    while stack:
        v = stack.pop()
        for c in kids[v]:
            if tokens[c] == top[v]:
                accepted.append(c)
                stack.append(c)
    return accepted


def expected_end(parent, tokens, logits):
    depth = gen.depth_of(parent)
    acc = branches_top_down(parent, tokens, logits)
    best = max(depth[a] for a in acc)
    return min(a for a in acc if depth[a] == best)


def path_to(parent, e):
    p = []
    while e >= 0:
        p.append(e)
        e = int(parent[e])
    return p[::-1]


def test_enumeration_small_trees_small_vocab(oracle_mod):
    """Every tree with <= 5 nodes, random tokens over V=3 (so matches and
    duplicate sibling tokens are frequent), random logits."""
    r = gen.rng(21)
    V = 3
    trees = []
    for n in range(1, 6):
        for choice in itertools.product(*[range(i) for i in range(1, n)]):
            trees.append(np.array((-1,) + choice, np.int32))
    for parent in trees:
        n = len(parent)
        for _ in range(4):
            tokens = r.integers(0, V, n).astype(np.int32)
            logits = r.standard_normal((n, V)).astype(np.float32)
            res = oracle_mod.accept_greedy(logits[None], tokens[None], parent[None])
            e = expected_end(parent, tokens, logits)
            assert res["status"][0] == 0
            assert res["end_node"][0] == e
            assert res["accept_len"][0] == gen.depth_of(parent)[e]
            p = path_to(parent, e)
            assert res["path"][0, :len(p)].tolist() == p
            assert (res["path"][0, len(p):] == -1).all()
            assert res["bonus"][0] == np.argmax(logits[e])
            assert res["argmax"][0].tolist() == np.argmax(logits, axis=1).tolist()


def planted_walk(parent, planted):
    v = 0
    while planted[v] >= 0:
        v = int(planted[v])
    return v


@pytest.mark.parametrize("cfg", ["c1", "c2", "c5_64"])
def test_planted_construction(oracle_mod, cfg):
    if cfg == "c1":
        case = gen.config1(with_attn=False)
    elif cfg == "c2":
        case = gen.config2(with_attn=False)
    else:
        case = gen.config5(64, with_attn=False, V=5000)
    res = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    for b in range(case.B):
        parent, tokens, logits = case.parent[b], case.tokens[b], case.logits[b]
        top = np.argmax(logits, axis=1)
        kids = gen.children_of(parent)
        # the construction only fixes the answer when no unplanted row's top
        # token coincides with a child's token
        for v in range(case.N):
            if case.planted[b, v] < 0:
                assert top[v] not in tokens[kids[v]].tolist()
            else:
                assert top[v] == tokens[case.planted[b, v]]
        e = planted_walk(parent, case.planted[b])
        # deepest planted chain node; the oracle's tie rule cannot change it
        # because only one chain of matches exists
        assert res["end_node"][b] == e
        assert res["accept_len"][b] == gen.depth_of(parent)[e]
        assert res["bonus"][b] == top[e]


def test_chain_accepts_leading_matches(oracle_mod):
    r = gen.rng(22)
    N, V = 12, 50
    parent = gen.chain_tree(N)
    for m in range(N):
        logits = r.standard_normal((N, V)).astype(np.float32)
        tokens = r.integers(0, V, N).astype(np.int32)
        top = np.argmax(logits, axis=1)
        for i in range(1, N):
            tokens[i] = top[i - 1] if i <= m else (top[i - 1] + 1) % V
        res = oracle_mod.accept_greedy(logits[None], tokens[None], parent[None])
        assert res["accept_len"][0] == m
        assert res["end_node"][0] == m
        assert res["bonus"][0] == top[m]


def test_ties_lowest_index_and_signed_zero(oracle_mod):
    parent = np.array([-1, 0, 0], np.int32)
    logits = np.zeros((3, 6), np.float32)
    logits[0, [2, 4]] = 5.0          # tie -> token 2
    logits[1] = [-0.0, 0.0, -0.0, 0.0, -1.0, -2.0]   # +-0 compare equal -> 0
    logits[2, 5] = 1.0
    tokens = np.array([0, 4, 2], np.int32)   # child 2 matches
    res = oracle_mod.accept_greedy(logits[None], tokens[None], parent[None])
    assert res["argmax"][0].tolist() == [2, 0, 5]
    assert res["end_node"][0] == 2 and res["accept_len"][0] == 1 and res["bonus"][0] == 5


def test_deepest_tie_goes_to_lowest_node(oracle_mod):
    # two children with the same (matching) token: both valid at depth 1
    parent = np.array([-1, 0, 0], np.int32)
    logits = np.zeros((3, 4), np.float32)
    logits[0, 3] = 1.0
    tokens = np.array([0, 3, 3], np.int32)
    res = oracle_mod.accept_greedy(logits[None], tokens[None], parent[None])
    assert res["end_node"][0] == 1


def test_single_node_and_bad_inputs(oracle_mod):
    logits = np.arange(4, dtype=np.float32)[None, None]
    res = oracle_mod.accept_greedy(logits, np.zeros((1, 1), np.int32),
                                   np.array([[-1]], np.int32))
    assert res["accept_len"][0] == 0 and res["end_node"][0] == 0 and res["bonus"][0] == 3
    parent = np.array([[-1, 0], [-1, 1], [-1, 0]], np.int32)
    tokens = np.array([[0, 1], [0, 1], [0, 9]], np.int32)
    logits = np.zeros((3, 2, 4), np.float32)
    res = oracle_mod.accept_greedy(logits, tokens, parent)
    assert res["status"].tolist() == [0, 2, 6]
    assert res["accept_len"][1:].tolist() == [-1, -1]
    assert (res["path"][1:] == -1).all()
