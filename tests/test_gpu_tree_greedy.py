"""GPU parity: tv_tree_build and tv_accept_greedy against the oracle, bit-exact
(OPT-Tree §2: tree attention mask; longest branch matching the target's
greedy sequence)."""
import numpy as np
import pytest
import torch

from workloads import gen

from _gpu_util import case_tensors, dev, i32, f32, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


# ------------------------------------------------------------------ tree build
@pytest.mark.parametrize("N", [1, 2, 7, 63, 64, 65, 128, 300, 511, 512])
def test_tree_build_matches_oracle(tv, oracle_mod, N):
    r = gen.rng(100 + N)
    trees = np.stack([gen.random_tree(r, N, 40), gen.chain_tree(N), gen.star_tree(N),
                      gen.random_tree(r, N, 3)])
    depth, anc, status = tv.tree_build(i32(trees))
    od, oa, os_ = oracle_mod.tree_build(trees)
    assert np_(status).tolist() == os_.tolist()
    assert np.array_equal(np_(depth), od)
    assert np.array_equal(np_(anc).view(np.uint64), oa)


def test_tree_build_flags_bad_trees(tv, oracle_mod):
    good = gen.chain_tree(6)
    bad = [good.copy() for _ in range(5)]
    bad[0][0] = 0
    bad[1][3] = 4
    bad[2][2] = 2
    bad[3][5] = -1
    bad[4][1] = -3
    trees = np.stack([good] + bad + [good])
    depth, anc, status = tv.tree_build(i32(trees))
    od, oa, os_ = oracle_mod.tree_build(trees)
    assert np_(status).tolist() == os_.tolist() == [0, 2, 2, 2, 2, 2, 0]
    assert np.array_equal(np_(depth), od)
    assert np.array_equal(np_(anc).view(np.uint64), oa)


# ---------------------------------------------------------------------- greedy
def run_greedy(tv, case):
    t = case_tensors(case)
    depth, anc, st = tv.tree_build(t["parent"])
    res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
    torch.cuda.synchronize()
    return {k: np_(v) for k, v in res.items()}


def compare_greedy(g, o):
    for k in ("argmax", "accept_len", "end_node", "path", "bonus", "status"):
        assert np.array_equal(g[k], o[k]), k


@pytest.mark.parametrize("which", ["c1", "c2", "c5"])
def test_greedy_configs(tv, oracle_mod, which):
    case = {"c1": lambda: gen.config1(with_attn=False),
            "c2": lambda: gen.config2(with_attn=False),
            "c5": lambda: gen.config5(256, with_attn=False)}[which]()
    g = run_greedy(tv, case)
    o = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    compare_greedy(g, o)
    assert (g["status"] == 0).all()


def test_greedy_batched_ragged_shapes(tv, oracle_mod):
    case = gen.make_case(201, B=16, N=64, L=4, V=128256, tree="random", max_depth=8,
                         with_attn=False)
    compare_greedy(run_greedy(tv, case), oracle_mod.accept_greedy(case.logits, case.tokens,
                                                                  case.parent))


@pytest.mark.parametrize("seed,B,N,V,tree", [
    (1, 1, 1, 2, "chain"), (2, 3, 5, 3, "random"), (3, 2, 17, 257, "random"),
    (4, 4, 64, 300, "random"), (5, 1, 40, 8193, "chain"), (6, 2, 33, 16384, "star"),
    (7, 5, 12, 1001, "random"), (8, 1, 512, 50, "random"), (9, 2, 100, 24577, "random"),
    (10, 1, 3, 262148, "chain"),  # 1 MB rows: many staged chunks per row
])
def test_greedy_fuzz(tv, oracle_mod, seed, B, N, V, tree):
    r = gen.rng(seed)
    case = gen.make_case(seed, B=B, N=N, L=4, V=max(V, N), tree=tree, max_depth=12,
                         with_attn=False)
    logits = case.logits
    if seed % 2 == 0:
        # many exact ties and signed zeros
        logits = np.round(logits * 2).astype(np.float32) * np.float32(0.5)
        logits[logits == 0] = np.where(r.random((logits == 0).sum()) < 0.5, -0.0, 0.0)
    # random tokens so that matches and non-matches both occur
    tokens = case.tokens.copy()
    top = logits.argmax(axis=2)
    for b in range(B):
        for i in range(1, N):
            p = case.parent[b, i]
            tokens[b, i] = top[b, p] if r.random() < 0.6 else r.integers(case.V)
    case.logits, case.tokens = logits, tokens
    compare_greedy(run_greedy(tv, case), oracle_mod.accept_greedy(logits, tokens, case.parent))


def test_greedy_bad_inputs_per_sequence(tv, oracle_mod):
    case = gen.make_case(210, B=4, N=10, L=4, V=100, with_attn=False)
    case.tokens[1, 3] = 100          # out of range
    case.parent[2, 4] = 7            # forward edge
    t = case_tensors(case)
    depth, anc, st = tv.tree_build(t["parent"])
    res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
    g = {k: np_(v) for k, v in res.items()}
    o = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    assert g["status"].tolist() == o["status"].tolist() == [0, 6, 2, 0]
    for k in ("accept_len", "end_node", "path", "bonus"):
        assert np.array_equal(g[k], o[k]), k
    assert np.array_equal(g["argmax"], o["argmax"])


def test_greedy_repeated_calls_reuse_workspace(tv, oracle_mod):
    """The arrival counters and row keys return to zero after every call."""
    case = gen.make_case(211, B=2, N=30, L=4, V=20000, with_attn=False)
    o = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    for _ in range(5):
        compare_greedy(run_greedy(tv, case), o)
    ws = tv.workspace("greedy", 0, dev())
    assert int(ws.count_nonzero()) == 0


@pytest.mark.parametrize("N", [10, 64, 65, 100])
def test_greedy_bad_inputs_both_scan_paths(tv, oracle_mod, N):
    """Trees of up to 64 nodes are scanned by one warp, larger ones by the
    whole CTA; both flag a bad token, a forward edge and a depth that does
    not match the parents, sequence by sequence."""
    case = gen.make_case(220 + N, B=5, N=N, L=4, V=300, with_attn=False)
    case.tokens[1, N - 1] = 300       # out of range
    case.parent[2, N // 2] = N - 1    # forward edge
    t = case_tensors(case)
    depth, anc, st = tv.tree_build(t["parent"])
    depth[3, N - 1] += 1              # depth inconsistent with the parents
    res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
    g = {k: np_(v) for k, v in res.items()}
    o = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    assert g["status"].tolist() == [0, 6, 2, 2, 0]
    for b in (0, 4):
        for k in ("accept_len", "end_node", "path", "bonus"):
            assert np.array_equal(g[k][b], o[k][b]), (k, b)
    for b in (1, 2, 3):
        assert g["accept_len"][b] == g["end_node"][b] == g["bonus"][b] == -1
        assert (g["path"][b] == -1).all()
    assert np.array_equal(g["argmax"], o["argmax"])
