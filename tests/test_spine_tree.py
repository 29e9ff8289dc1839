"""The library's GOOSE spine-tree builder (host code) against the oracle: the
same tree, node for node, on randomised candidate lists (duplicates, -1 row
ends, the spine's own token among the branch candidates, short rows), budgets
and spine ratios; and the spine-ratio moving average (GOOSE §2C).  No GPU:
the builder runs on the host."""
import numpy as np
import pytest

from workloads import gen


@pytest.fixture(scope="module")
def tv():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_tree_tv_gb300 as m
    return m


def random_inputs(r, V=300):
    S = int(r.integers(0, 40))
    Sb = int(r.integers(0, 45))
    K = int(r.integers(0, 12))
    spine = r.integers(0, V, S).astype(np.int32)
    br = r.integers(0, V, (Sb, K)).astype(np.int32)
    for j in range(min(S, Sb)):                 # the spine's token among the candidates
        if K and r.random() < 0.3:
            br[j, int(r.integers(0, K))] = spine[j]
    for j in range(Sb):                         # rows ended early
        if K and r.random() < 0.3:
            br[j, int(r.integers(0, K)):] = -1
    budget = int(r.integers(1, 600))
    ratio = float(r.choice([0.0, 1.0, r.random()]))
    return spine, br, int(r.integers(0, V)), budget, ratio


def test_matches_the_oracle(tv, oracle_mod):
    r = gen.rng(2024)
    for _ in range(400):
        spine, br, root, budget, ratio = random_inputs(r)
        gp, gt = tv.build_spine_tree(spine, br, root, budget, ratio)
        op, ot = oracle_mod.build_spine_tree(spine, br, root, budget, ratio)
        assert np.array_equal(gp, op) and np.array_equal(gt, ot), (len(spine), br.shape, budget, ratio)


def test_feeds_the_verify_path(tv, oracle_mod):
    """The built tree is a valid verify tree: the oracle's tree encoding
    accepts it and its depths follow the spine."""
    r = gen.rng(7)
    spine = r.choice(128256, 24, replace=False).astype(np.int32)
    br = np.stack([r.choice(128256, 8, replace=False) for _ in range(24)]).astype(np.int32)
    parent, tokens = tv.build_spine_tree(spine, br, 5, 60, 0.4)
    depth, anc, status = oracle_mod.tree_build(parent[None])
    assert status[0] == 0 and depth[0].max() == 24


def test_spine_ratio_moving_average(tv):
    ratio = 0.5
    for _ in range(200):
        ratio = tv.spine_ratio_update(ratio, 0.8, 0.1)
    assert ratio == pytest.approx(0.8, abs=1e-4)
    assert tv.spine_ratio_update(0.9, 5.0, 1.0) == 1.0
    assert tv.spine_ratio_update(0.1, -3.0, 1.0) == 0.0


def test_bad_arguments(tv):
    with pytest.raises(tv.TVError):
        tv.build_spine_tree(np.arange(4), np.zeros((4, 2)), 0, 0, 0.5)
    with pytest.raises(tv.TVError):
        tv.build_spine_tree(np.arange(4), np.zeros((4, 2)), 0, 10, 1.5)
