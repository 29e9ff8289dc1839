"""GPU parity: tv_expand_gated against the oracle (TALON §5.1, §5.2.1, §5.2.2:
budget-driven growth, root Top-K, anchor/alpha gate, budget truncation).

Both sides grow the tree layer by layer with the same synthetic drafter and
compare scores in fp64.  Trees must be identical (parent and token arrays
bit-exact, log scores within fp32 rounding) up to the first layer whose
oracle margin is below MARGIN; after it the GPU's tree is checked against
TALON's rules (check_valid)."""
import numpy as np
import pytest
import torch

from workloads import gen

from _gpu_util import dev

pytestmark = pytest.mark.gpu

MARGIN = 1e-6


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


def grow_both(tv, oracle_mod, drafter, K, alpha, budget):
    o = oracle_mod.expand_tree(drafter, K, alpha, budget)
    g = tv.expand_tree(drafter.rows, drafter.root_key(), drafter.child_key, K, alpha, budget,
                       dev())
    return g, o


def check_valid(g, K, alpha, budget, V):
    """The GPU's tree obeys TALON's rules whatever its near-threshold
    decisions were: at most B nodes, a root Top-K first layer, every later
    layer gated at log(alpha) below its best score, path scores never above
    the parent's, distinct siblings, and the numbering (parent ascending,
    score descending, token ascending within a layer)."""
    n = g["n"]
    par, tok, ls = g["parent"].numpy()[:n], g["token"].numpy()[:n], g["logscore"].numpy()[:n]
    assert 1 <= n <= budget and par[0] == -1
    depth = gen.depth_of(par)
    assert (np.diff(depth) >= 0).all()                  # layers in order
    assert int((depth == 1).sum()) == min(K, V, budget - 1)
    assert (tok[1:] >= 0).all() and (tok[1:] < V).all()
    assert len(set(zip(par[1:].tolist(), tok[1:].tolist()))) == n - 1
    for i in range(1, n):
        assert par[i] < i and depth[par[i]] == depth[i] - 1
        assert ls[i] <= ls[par[i]] + 1e-6
    for d in range(2, int(depth.max()) + 1):
        lay = np.flatnonzero(depth == d)
        assert (ls[lay] >= np.log(alpha) + ls[lay].max() - 1e-5).all(), d
    for d in range(1, int(depth.max()) + 1):
        lay = np.flatnonzero(depth == d)
        keys = list(zip(par[lay].tolist(), (-ls[lay]).tolist(), tok[lay].tolist()))
        assert keys == sorted(keys), d


def compare_trees(g, o, K, alpha, budget, V):
    depth_o = gen.depth_of(o["parent"])
    # first layer (depth) whose decisions are within rounding of a threshold
    bad_layer = next((l + 1 for l, m in enumerate(o["margins"]) if m < MARGIN), None)
    n_cmp = o["n"] if bad_layer is None else int((depth_o < bad_layer).sum())
    gp, gt, gl = g["parent"].numpy(), g["token"].numpy(), g["logscore"].numpy()
    assert np.array_equal(gp[:n_cmp], o["parent"][:n_cmp])
    assert np.array_equal(gt[:n_cmp], o["token"][:n_cmp])
    np.testing.assert_allclose(gl[:n_cmp], o["logscore"][:n_cmp], rtol=1e-6, atol=1e-5)
    if bad_layer is None:
        assert g["n"] == o["n"]
    check_valid(g, K, alpha, budget, V)
    return bad_layer


@pytest.mark.parametrize("context", [0, 1, 2])
def test_talon_workload(tv, oracle_mod, context):
    d = gen.config3_drafter(context)
    g, o = grow_both(tv, oracle_mod, d, 10, 0.3, 512)
    assert compare_trees(g, o, 10, 0.3, 512, d.V) is None
    assert g["n"] == 512


@pytest.mark.parametrize("V,K,alpha,budget,sigma,seed", [
    (8, 3, 0.3, 20, 1.0, 1), (8, 3, 0.3, 20, 3.0, 2), (4, 2, 0.5, 12, 1.0, 3),
    (6, 6, 0.1, 30, 2.0, 4), (5, 1, 0.3, 9, 6.0, 5), (8, 10, 0.3, 20, 1.0, 6),
    (1000, 10, 0.3, 200, 1.0, 7), (1000, 10, 0.05, 300, 2.0, 8), (8193, 4, 1.0, 64, 3.0, 9),
    (30001, 10, 0.3, 512, 0.5, 10), (3, 3, 0.001, 100, 0.2, 11),
])
def test_expand_fuzz(tv, oracle_mod, V, K, alpha, budget, sigma, seed):
    d = gen.TalonDrafter(seed, V, sigma)
    g, o = grow_both(tv, oracle_mod, d, K, alpha, budget)
    compare_trees(g, o, K, alpha, budget, V)


def test_expand_exact_ties(tv, oracle_mod):
    """Rows with many equal logits: the budget cut and the root Top-K break
    ties by (parent, token) on both sides."""
    class TieDrafter(gen.TalonDrafter):
        def row(self, key):
            x = super().row(key)
            return np.round(x).astype(np.float32)
    d = TieDrafter(12, 64, 1.0)
    g, o = grow_both(tv, oracle_mod, d, 5, 0.3, 150)
    compare_trees(g, o, 5, 0.3, 150, 64)


def test_expand_budget_already_spent(tv):
    par = torch.full((4,), -1, dtype=torch.int32, device=dev())
    tok = torch.zeros(4, dtype=torch.int32, device=dev())
    ls = torch.zeros(4, dtype=torch.float32, device=dev())
    n = torch.tensor([4], dtype=torch.int32, device=dev())
    rows = torch.randn(2, 100, device=dev())
    tv.expand_gated(rows, torch.tensor([1, 2], dtype=torch.int32, device=dev()), ls[1:3].clone(),
                    2, 3, 0.3, 4, par, tok, ls, n)
    assert int(n.item()) == 4
