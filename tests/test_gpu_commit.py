"""GPU parity: tv_commit_path against the oracle (Speculative Decoding concept
page, "The protocol" step 4; OPT-Tree §2: the accepted branch's K/V rows move
from their tree slots to consecutive prefix positions).  The copy is exact,
so the caches must agree bit for bit."""
import numpy as np
import pytest
import torch

from workloads import gen

from _gpu_util import bf16, case_tensors, dev, i32, np_

from test_oracle_commit import branch_to, random_commit_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


def run_commit(tv, k, v, kv_len, path, alen):
    kt, vt = bf16(k), bf16(v)
    new_len, status = tv.commit_path(kt, vt, i32(kv_len), i32(path), i32(alen))
    torch.cuda.synchronize()
    to_bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    return to_bits(kt), to_bits(vt), np_(new_len), np_(status)


@pytest.mark.parametrize("seed,B,N,Hkv,D,L", [
    (1, 3, 16, 2, 64, 40), (2, 4, 60, 8, 128, (0, 7, 300, 64)), (3, 2, 200, 1, 64, 5),
    (4, 1, 512, 2, 128, 17), (5, 16, 64, 8, 128, 1000),
])
def test_commit_matches_oracle(tv, oracle_mod, seed, B, N, Hkv, D, L):
    k, v, kv_len, parents, path, alen, Lcap = random_commit_case(seed, B, N, Hkv, D, L)
    gk, gv, glen, gst = run_commit(tv, k, v, kv_len, path, alen)
    ok, ov, olen, ost = oracle_mod.commit_path(k, v, kv_len, path, alen)
    assert np.array_equal(gst, ost) and np.array_equal(glen, olen)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_long_branches_take_several_batches(tv, oracle_mod):
    """512 nodes: even nodes form a chain (i -> i - 2), odd ones hang off it
    (i -> i - 1).  The branch to node 510 has 256 nodes at path[d] = 2d, so
    every row moves, 32 rows per batch; a second sequence takes its first 100."""
    N, Hkv, D = 512, 2, 128
    r = gen.rng(12)
    parent = np.array([-1] + [i - 1 if i % 2 else i - 2 for i in range(1, N)], np.int32)
    br = branch_to(parent, 510)
    assert br == list(range(0, 511, 2))
    path = np.full((2, N), -1, np.int32)
    path[0, :len(br)] = br
    path[1, :100] = br[:100]
    alen = np.array([len(br) - 1, 99], np.int32)
    Lcap = 40 + N
    k = gen.normal_bf16(r, (2, Hkv, Lcap, D))
    v = gen.normal_bf16(r, (2, Hkv, Lcap, D))
    kv_len = np.array([40, 12], np.int32)
    gk, gv, glen, gst = run_commit(tv, k, v, kv_len, path, alen)
    ok, ov, olen, ost = oracle_mod.commit_path(k, v, kv_len, path, alen)
    assert gst.tolist() == [0, 0] and np.array_equal(glen, olen)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


@pytest.mark.parametrize("bad", ["first", "order", "outside", "cache", "negative"])
def test_malformed_paths_are_flagged(tv, oracle_mod, bad):
    k, v, kv_len, parents, path, alen, Lcap = random_commit_case(21, 2, 30, 2, 64, 10, slack=0)
    b, a = 1, 3
    path[b, :a + 1] = [0, 4, 9, 17]
    alen[b] = a
    if bad == "first":
        path[b, 0] = 2
    elif bad == "order":
        path[b, 2] = 4
    elif bad == "outside":
        path[b, 3] = 30
    elif bad == "cache":
        kv_len[b] = Lcap - 17
    else:
        alen[b] = -1
    gk, gv, glen, gst = run_commit(tv, k, v, kv_len, path, alen)
    ok, ov, olen, ost = oracle_mod.commit_path(k, v, kv_len, path, alen)
    assert gst.tolist() == ost.tolist() == [0, 1]
    assert np.array_equal(glen, olen)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_greedy_step_then_commit_on_the_spine_shape(tv, oracle_mod):
    """The Llama-3-8B-shaped step at full size: tree, greedy acceptance, then
    the commit of the accepted spine prefix, against the oracle."""
    case = gen.config2()
    t = case_tensors(case)
    depth, anc, _ = tv.tree_build(t["parent"])
    res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
    path, alen = np_(res["path"]), np_(res["accept_len"])
    o = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    assert np.array_equal(path, o["path"]) and np.array_equal(alen, o["accept_len"])
    new_len, status = tv.commit_path(t["k"], t["v"], t["kv_len"], res["path"], res["accept_len"])
    torch.cuda.synchronize()
    ok, ov, olen, ost = oracle_mod.commit_path(case.k, case.v, case.kv_len, path, alen)
    to_bits = lambda x: x.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np_(status).tolist() == [0] and np.array_equal(np_(new_len), olen)
    assert np.array_equal(to_bits(t["k"]), ok) and np.array_equal(to_bits(t["v"]), ov)
