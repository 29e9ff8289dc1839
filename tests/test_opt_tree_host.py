"""Host logic of the OPT-Tree growth (no GPU): the layer sizes the host
derives without reading the device, and the binding's growth loop (frontier
ranges, drafter keys, the final selection) run with oracle-backed stand-ins for
the two device calls, against the oracle's own growth (OPT-Tree §3)."""
import numpy as np
import pytest
import torch

from workloads import gen


@pytest.fixture(scope="module")
def api():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_tree_tv_gb300.api as m
    return m


@pytest.mark.parametrize("seed,V,width,layers", [
    (1, 4, 12, 4), (2, 3, 20, 6), (3, 50, 7, 3), (4, 2, 100, 9),
])
def test_layer_sizes_match_the_oracle_growth(api, oracle_mod, seed, V, width, layers):
    d = gen.TalonDrafter(seed, V, 1.5)
    o = oracle_mod.opt_tree(d, width, layers, width)
    depth = gen.depth_of(o["parent"])
    sizes = api.opt_tree_layer_sizes(width, layers, V, 1 + width * layers)
    assert len(sizes) == layers
    lo = 0
    for l, (a, f) in enumerate(sizes):
        assert a == lo and f == int((depth == l).sum())
        lo += f
    assert lo + int((depth == layers).sum()) == o["n"]


def test_layer_sizes_capacity_and_empty(api):
    assert api.opt_tree_layer_sizes(256, 16, 128256, 4097)[-1] == (3585, 256)
    assert api.opt_tree_layer_sizes(4, 5, 10, 7) == [(0, 1), (1, 4)]   # 1 + 4 + 2 nodes
    assert api.opt_tree_layer_sizes(4, 5, 10, 1) == []


def test_growth_loop_with_oracle_device_calls(api, oracle_mod, monkeypatch):
    def fake_expand(rows, fnode, fls, width, cap, par, tok, ls, n_dev, ws=None):
        n_new, _ = oracle_mod.expand_topn(rows.numpy(), fnode.numpy(), fls.numpy(), width, cap,
                                          par.numpy(), tok.numpy(), ls.numpy(), int(n_dev[0]))
        n_dev[0] = n_new

    def fake_select(parent, token, logscore, n_nodes, n, out=None):
        o = oracle_mod.select_topn(parent.numpy(), token.numpy(), logscore.numpy(),
                                   n_nodes.numpy(), n)
        return {k: torch.from_numpy(np.asarray(v)) for k, v in o.items()}

    monkeypatch.setattr(api, "expand_topn", fake_expand)
    monkeypatch.setattr(api, "select_topn", fake_select)
    for seed, V, width, layers, n in ((3, 7, 10, 5, 10), (4, 2, 9, 6, 12), (5, 40, 16, 3, 30)):
        d = gen.TalonDrafter(seed, V, 2.0)
        g = api.grow_opt_tree(d.rows, d.root_key(), d.child_key, width, layers, n, "cpu")
        o = oracle_mod.opt_tree(d, width, layers, n)
        assert g["n"] == g["n_device"] == o["n"]
        assert np.array_equal(g["parent"].numpy(), o["parent"])
        assert np.array_equal(g["token"].numpy(), o["token"])
        for k in ("parent", "token", "src"):
            assert np.array_equal(g["selected"][k].numpy(), np.asarray(o["selected"][k])), k
