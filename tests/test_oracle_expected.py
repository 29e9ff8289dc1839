"""Pins for the oracle's expected acceptance length of a draft tree.

OPT-Tree §3: a node's score is the product of the draft probabilities along
its path from the root, and the expected acceptance length is approximated by
the sum of the scores of the tree's nodes.  Pinned by
  * exhaustive enumeration of every accept/reject outcome of the draft nodes
    on small trees (a node counts when every node of its path is accepted),
  * the closed forms of a chain (a geometric series at constant probability)
    and of a star (the sum of the probabilities),
  * greedy acceptance itself: when each node's target argmax falls on child c
    with probability p(c), the mean accepted length that the oracle's greedy
    acceptance returns over many trials converges to the same value,
  * malformed inputs.
"""
import itertools

import numpy as np
import pytest

from workloads import gen


def enumerate_expectation(parent, prob):
    N = len(parent)
    total = 0.0
    for bits in itertools.product((0, 1), repeat=N - 1):
        ok = (1,) + bits
        pr = 1.0
        for i in range(1, N):
            pr *= prob[i] if ok[i] else 1.0 - prob[i]
        count = 0
        for v in range(1, N):
            u = v
            while u > 0 and ok[u]:
                u = parent[u]
            count += (u == 0)
        total += pr * count
    return total


@pytest.mark.parametrize("seed,N", [(1, 2), (2, 5), (3, 8), (4, 10), (5, 11)])
def test_matches_exhaustive_enumeration(oracle_mod, seed, N):
    r = gen.rng(seed)
    par = gen.random_tree(r, N, 6)
    prob = r.random(N).astype(np.float32)
    score, e, st = oracle_mod.expected_accept(par[None], prob[None])
    assert st[0] == 0
    want = enumerate_expectation(par, prob.astype(np.float64))
    assert e[0] == pytest.approx(want, rel=1e-12, abs=1e-12)


def test_chain_and_star_closed_forms(oracle_mod):
    N, p = 40, 0.7
    chain = gen.chain_tree(N)
    _, e, _ = oracle_mod.expected_accept(chain[None], np.full((1, N), p, np.float32))
    pf = float(np.float32(p))
    assert e[0] == pytest.approx(pf * (1 - pf ** (N - 1)) / (1 - pf), rel=1e-12)
    star = gen.star_tree(N)
    r = gen.rng(3)
    prob = r.random(N).astype(np.float32)
    score, e, _ = oracle_mod.expected_accept(star[None], prob[None])
    assert e[0] == pytest.approx(float(prob[1:].astype(np.float64).sum()), rel=1e-12)
    assert np.allclose(score[0, 1:], prob[1:].astype(np.float64), rtol=0, atol=0)


def test_greedy_acceptance_converges_to_it(oracle_mod):
    """Siblings get distinct tokens; each row's argmax lands on child c with
    probability p(c) (or on no child), and accept_len averages to E[A]."""
    r = gen.rng(42)
    N, V, trials = 12, 64, 6000
    par = gen.random_tree(r, N, 5)
    kids = gen.children_of(par)
    prob = np.zeros(N, np.float32)
    for v, ks in enumerate(kids):
        if ks:
            w = r.random(len(ks) + 1)
            prob[ks] = (w[:-1] / w.sum()).astype(np.float32)   # leaves mass for "no child"
    tokens = gen.distinct_sibling_tokens(r, par, V)
    _, e, _ = oracle_mod.expected_accept(par[None], prob[None])
    B = trials
    logits = r.standard_normal((B, N, V)).astype(np.float32)
    for v, ks in enumerate(kids):
        if not ks:
            continue
        cdf = np.cumsum(prob[ks].astype(np.float64))
        u = r.random(B)
        pick = np.searchsorted(cdf, u, side="right")        # len(ks) means no child
        for j, c in enumerate(ks):
            logits[pick == j, v, tokens[c]] += 50.0
    res = oracle_mod.accept_greedy(logits, np.broadcast_to(tokens, (B, N)).copy(),
                                   np.broadcast_to(par, (B, N)).copy())
    mean = res["accept_len"].mean()
    se = res["accept_len"].std() / np.sqrt(B)
    assert abs(mean - e[0]) < 4 * se + 1e-9, (mean, e[0], se)


def test_malformed_inputs(oracle_mod):
    par = np.stack([gen.chain_tree(6)] * 3)
    prob = np.full((3, 6), 0.5, np.float32)
    par[1, 3] = 4
    prob[2, 2] = 1.5
    score, e, st = oracle_mod.expected_accept(par, prob)
    assert st.tolist() == [0, 2, 1]
    assert e[1] == e[2] == 0.0 and (score[1:] == 0).all()
