"""GPU parity: tv_expected_accept against the oracle (OPT-Tree §3: node score
= product of the draft probabilities along the path; expected acceptance
length = sum of the draft nodes' scores).

Tolerance: a score is a product of at most N - 1 fp32 factors, formed in
ceil(log2 N) rounds, so its relative error is below N * 2^-24 (3e-5 at 512
nodes); the sum adds fp32 warp sums of at most 32 scores, within 2e-5."""
import numpy as np
import pytest
import torch

from workloads import gen

from _gpu_util import f32, i32, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


def check(tv, oracle_mod, parent, prob):
    s, e, st = tv.expected_accept(i32(parent), f32(prob))
    torch.cuda.synchronize()
    os_, oe, ost = oracle_mod.expected_accept(parent, prob)
    assert np.array_equal(np_(st), ost)
    np.testing.assert_allclose(np_(s), os_, rtol=4e-5, atol=1e-30)
    np.testing.assert_allclose(np_(e), oe, rtol=2e-5, atol=1e-6)
    return np_(e), oe


@pytest.mark.parametrize("seed,B,N,depth", [(1, 4, 16, 6), (2, 3, 60, 12), (3, 2, 512, 40),
                                             (4, 16, 64, 8), (5, 1, 1, 1), (6, 5, 200, 199)])
def test_random_trees(tv, oracle_mod, seed, B, N, depth):
    r = gen.rng(seed)
    parent = np.stack([gen.random_tree(r, N, depth) for _ in range(B)])
    prob = r.random((B, N)).astype(np.float32)
    check(tv, oracle_mod, parent, prob)


def test_deep_chain_and_wide_star(tv, oracle_mod):
    N = 512
    parent = np.stack([gen.chain_tree(N), gen.star_tree(N)])
    prob = np.full((2, N), 0.98, np.float32)
    e, oe = check(tv, oracle_mod, parent, prob)
    assert oe[1] == pytest.approx(0.98 * (N - 1), rel=1e-6)


def test_talon_tree_from_its_log_scores(tv, oracle_mod):
    """The expanded TALON tree (one context) with each node's draft
    probability exp(logscore - parent's logscore)."""
    t = oracle_mod.expand_tree(gen.config3_drafter(2), 10, 0.3, 512)
    par, ls = t["parent"], t["logscore"].astype(np.float64)
    prob = np.ones(len(par), np.float32)
    # log scores are stored in fp32: a near-certain child can round just above 1
    prob[1:] = np.minimum(1.0, np.exp(ls[1:] - ls[par[1:]])).astype(np.float32)
    check(tv, oracle_mod, par[None], prob[None])


def test_bad_inputs(tv, oracle_mod):
    parent = np.stack([gen.chain_tree(6)] * 3)
    prob = np.full((3, 6), 0.5, np.float32)
    parent[1, 3] = 4
    prob[2, 2] = -0.25
    s, e, st = tv.expected_accept(i32(parent), f32(prob))
    torch.cuda.synchronize()
    assert np_(st).tolist() == [0, 2, 1]
    assert (np_(e)[1:] == 0).all() and (np_(s)[1:] == 0).all()
