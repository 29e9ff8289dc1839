"""GPU parity: tv_expand_topn and tv_select_topn against the oracle
(OPT-Tree §3: greedy layer-by-layer expansion keeping the best-scoring
children, then the n best nodes of the candidate tree as a subtree).

The selection compares fp32 scores on both sides and must match bit for bit.
The expansion compares fp64 log scores built from fp32 logits; the two sides
round the row normalisers differently, so a layer whose oracle margin (the
score gap at its cut between children of different parents) is below MARGIN
is ambiguous: trees must be identical up to that layer (parent and token
arrays bit-exact, scores within fp32 rounding) and only valid after it."""
import numpy as np
import pytest
import torch

from workloads import gen

from _gpu_util import dev, f32, i32, np_

pytestmark = pytest.mark.gpu

MARGIN = 1e-6


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


def monotone_trees(r, B, M, m, tie=False):
    par = np.full((B, M), -1, np.int32)
    ls = np.zeros((B, M), np.float32)
    for b in range(B):
        for i in range(1, m[b]):
            par[b, i] = r.integers(max(0, i - 64), i) if r.random() < 0.7 else r.integers(0, i)
            step = -float(r.integers(0, 3)) if tie else float(np.log(r.uniform(0.01, 1.0)))
            ls[b, i] = np.float32(ls[b, par[b, i]] + step)
    tok = r.integers(0, 128256, (B, M)).astype(np.int32)
    return par, tok, ls


def select_both(tv, oracle_mod, par, tok, ls, m, n):
    g = tv.select_topn(i32(par), i32(tok), f32(ls), i32(m), n)
    torch.cuda.synchronize()
    g = {k: np_(v) for k, v in g.items()}
    o = oracle_mod.select_topn(par, tok, ls, m, n)
    assert np.array_equal(g["status"], o["status"])
    for k in ("parent", "token", "src"):
        assert np.array_equal(g[k], o[k]), k
    assert np.array_equal(g["logscore"].view(np.uint32), o["logscore"].view(np.uint32))
    np.testing.assert_allclose(g["expected"], o["expected"], rtol=2e-6, atol=1e-7)
    return g


@pytest.mark.parametrize("B,M,n,tie", [
    (1, 1, 1, False), (4, 9, 3, False), (5, 600, 60, False), (3, 4097, 256, False),
    (2, 16384, 512, False), (6, 700, 100, True), (2, 3000, 1024, True), (3, 50, 200, False),
])
def test_select_matches_oracle(tv, oracle_mod, B, M, n, tie):
    r = gen.rng(M + n)
    m = np.maximum(1, (M * r.uniform(0.5, 1.0, B)).astype(np.int32))
    m[0] = M
    par, tok, ls = monotone_trees(r, B, M, m, tie)
    g = select_both(tv, oracle_mod, par, tok, ls, m, n)
    assert (g["status"] == 0).all()


def test_select_bad_inputs(tv, oracle_mod):
    r = gen.rng(3)
    B, M = 7, 40
    m = np.full(B, M, np.int32)
    par, tok, ls = monotone_trees(r, B, M, m)
    i = int(np.flatnonzero(par[2] > 0)[0])
    ls[2, i] = 0.5                     # better than the root, its parent the worst
    ls[2, par[2, i]] = -50.0
    par[3, 17] = 30                    # a parent after its child
    ls[4, 5] = np.nan
    m[5] = 0
    m[6] = M + 1
    g = select_both(tv, oracle_mod, par, tok, ls, m, 10)
    assert g["status"].tolist() == [0, 0, 2, 2, 1, 1, 1]


def grow_both(tv, oracle_mod, d, width, layers, n):
    o = oracle_mod.opt_tree(d, width, layers, n)
    g = tv.grow_opt_tree(d.rows, d.root_key(), d.child_key, width, layers, n, dev())
    return g, o


def compare_layers(g, o):
    depth_o = gen.depth_of(o["parent"])
    bad = next((l + 1 for l, m in enumerate(o["margins"]) if m < MARGIN), None)
    n_cmp = o["n"] if bad is None else int((depth_o < bad).sum())
    gp, gt, gl = g["parent"].numpy(), g["token"].numpy(), g["logscore"].numpy()
    assert g["n"] == o["n"] == g["n_device"]
    assert np.array_equal(gp[:n_cmp], o["parent"][:n_cmp])
    assert np.array_equal(gt[:n_cmp], o["token"][:n_cmp])
    np.testing.assert_allclose(gl[:n_cmp], o["logscore"][:n_cmp], rtol=1e-6, atol=1e-5)
    # every layer of the GPU's tree is valid: parents in the previous layer,
    # scores never above the parent's, siblings distinct
    for i in range(1, g["n"]):
        assert gp[i] < i and gl[i] <= gl[gp[i]] + 1e-6
    pairs = set(zip(gp.tolist(), gt.tolist()))
    assert len(pairs) == g["n"]
    return bad


@pytest.mark.parametrize("seed,V,sigma,width,layers,n", [
    (1, 4, 1.0, 12, 4, 12), (2, 8, 3.0, 30, 6, 30), (3, 1000, 1.0, 64, 5, 60),
    (4, 2049, 2.0, 100, 4, 150), (5, 30001, 0.5, 256, 3, 256), (6, 3, 0.5, 2048, 8, 512),
    (7, 50, 6.0, 20, 16, 20),
])
def test_opt_tree_matches_oracle(tv, oracle_mod, seed, V, sigma, width, layers, n):
    d = gen.TalonDrafter(seed, V, sigma)
    g, o = grow_both(tv, oracle_mod, d, width, layers, n)
    bad = compare_layers(g, o)
    gs = g["selected"]
    if bad is None:
        os_ = o["selected"]
        for k in ("parent", "token", "src", "status"):
            assert np.array_equal(gs[k].numpy(), np.asarray(os_[k])), k
        np.testing.assert_allclose(float(gs["expected"]), float(os_["expected"]), rtol=1e-5)
    assert int(gs["status"]) == 0


def test_opt_tree_llama3_vocabulary(tv, oracle_mod):
    """The long-context workload's shape: vocabulary 128,256, width 256, N(0, 3)
    draft rows; three layers (the third expands 256 rows) on both sides."""
    d = gen.TalonDrafter(gen.splitmix64(99), 128256, 3.0)
    g, o = grow_both(tv, oracle_mod, d, 256, 3, 256)
    assert compare_layers(g, o) is None
    assert g["n"] == 1 + 256 * 3


def test_exact_ties_across_rows(tv, oracle_mod):
    """Every node gets the same row of integer logits: the best children of
    each layer form one group of exact ties across many rows (about 15,000 at
    the second layer), more than the select sorts, so the cut inside the group
    is taken one tie at a time, by the lower (parent, token), on both sides.
    Both sides round a row's normaliser their own way but every row alike,
    so the trees must agree exactly."""
    class Same(gen.TalonDrafter):
        def row(self, key):
            return np.round(super().row(self.root_key()) * 0.2).astype(np.float32)
    d = Same(8, 20000, 1.0)
    g, o = grow_both(tv, oracle_mod, d, 300, 3, 300)
    assert g["n"] == o["n"] == 901
    assert np.array_equal(g["parent"].numpy(), o["parent"])
    assert np.array_equal(g["token"].numpy(), o["token"])
    np.testing.assert_allclose(g["logscore"].numpy(), o["logscore"], rtol=1e-6, atol=1e-5)


def test_capacity_cut_and_shared_workspace(tv, oracle_mod):
    """A layer that meets the end of the tree arrays keeps what fits; the
    workspace it leaves behind serves a TALON expansion unchanged."""
    d = gen.TalonDrafter(5, 700, 2.0)
    rows = f32(d.rows([d.root_key()]))
    cap = 8
    par = torch.full((cap,), -1, dtype=torch.int32, device=dev())
    tok = torch.zeros(cap, dtype=torch.int32, device=dev())
    ls = torch.zeros(cap, dtype=torch.float32, device=dev())
    n = torch.tensor([3], dtype=torch.int32, device=dev())
    tv.expand_topn(rows, torch.zeros(1, dtype=torch.int32, device=dev()),
                   torch.zeros(1, dtype=torch.float32, device=dev()), 50, cap, par, tok, ls, n)
    assert int(n.item()) == cap
    op = np.full(cap, -1, np.int32)
    ot = np.zeros(cap, np.int32)
    ol = np.zeros(cap, np.float32)
    on, _ = oracle_mod.expand_topn(np_(rows), [0], [0.0], 50, cap, op, ot, ol, 3)
    assert on == cap
    assert np.array_equal(np_(tok)[3:], ot[3:]) and np.array_equal(np_(par)[3:], op[3:])
    # a full tree: nothing is appended
    tv.expand_topn(rows, torch.zeros(1, dtype=torch.int32, device=dev()),
                   torch.zeros(1, dtype=torch.float32, device=dev()), 50, cap, par, tok, ls, n)
    assert int(n.item()) == cap
    t = gen.config3_drafter(0, V=5000)
    gt = tv.expand_tree(t.rows, t.root_key(), t.child_key, 10, 0.3, 200, dev())
    ot_ = oracle_mod.expand_tree(t, 10, 0.3, 200)
    k = int((gen.depth_of(ot_["parent"]) < 3).sum())
    assert np.array_equal(gt["parent"].numpy()[:k], ot_["parent"][:k])
    assert np.array_equal(gt["token"].numpy()[:k], ot_["token"][:k])
