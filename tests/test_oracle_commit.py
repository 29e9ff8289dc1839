"""Pins for the oracle's commit of the accepted branch into the KV cache.

Speculative Decoding concept page, "The protocol" step 4: the accepted
tokens (and the correction) become part of the prefix; OPT-Tree §2: the
accepted tokens form one root-to-node branch of the draft tree, whose K/V
rows the verify pass wrote at the tree slots kv_len + node.  The oracle moves
them in place, row by row; it is pinned against
  * an out-of-place gather of the same rows from the untouched cache (numpy),
  * attention: after the commit, a single query at the end of the new prefix
    sees exactly the keys the end node saw in the tree, so its output equals
    the end node's tree attention (both from the oracle's fp64 attention),
  * the chain tree with every node accepted, which needs no move at all,
  * malformed paths, which leave the cache alone.
"""
import numpy as np
import pytest

from workloads import gen


def branch_to(parent, end):
    p = []
    x = int(end)
    while x >= 0:
        p.append(x)
        x = int(parent[x])
    return p[::-1]


def random_commit_case(seed, B, N, Hkv, D, L, slack=3):
    r = gen.rng(seed)
    Lb = np.asarray(L if isinstance(L, (list, tuple)) else [L] * B, np.int32)
    Lcap = int(Lb.max()) + N + slack
    k = gen.normal_bf16(r, (B, Hkv, Lcap, D))
    v = gen.normal_bf16(r, (B, Hkv, Lcap, D))
    parents, paths, alen = [], np.full((B, N), -1, np.int32), np.zeros(B, np.int32)
    for b in range(B):
        par = gen.random_tree(r, N, 10)
        parents.append(par)
        br = branch_to(par, int(r.integers(0, N)))
        paths[b, :len(br)] = br
        alen[b] = len(br) - 1
    return k, v, Lb, np.stack(parents), paths, alen, Lcap


def gather_reference(k, v, kv_len, path, alen):
    k2, v2 = k.copy(), v.copy()
    for b in range(k.shape[0]):
        L, a = int(kv_len[b]), int(alen[b])
        src = L + path[b, :a + 1]
        dst = L + np.arange(a + 1)
        k2[b][:, dst] = k[b][:, src]
        v2[b][:, dst] = v[b][:, src]
    return k2, v2


@pytest.mark.parametrize("seed,B,N,Hkv,D,L", [
    (1, 3, 16, 2, 64, 40), (2, 4, 60, 8, 128, (0, 7, 300, 64)), (3, 2, 200, 1, 64, 5),
    (4, 1, 512, 2, 128, 17),
])
def test_commit_matches_out_of_place_gather(oracle_mod, seed, B, N, Hkv, D, L):
    k, v, kv_len, parents, path, alen, Lcap = random_commit_case(seed, B, N, Hkv, D, L)
    k2, v2, new_len, status = oracle_mod.commit_path(k, v, kv_len, path, alen)
    rk, rv = gather_reference(k, v, kv_len, path, alen)
    assert (status == 0).all()
    assert np.array_equal(new_len, kv_len + alen + 1)
    assert np.array_equal(k2, rk) and np.array_equal(v2, rv)
    # nothing outside [kv_len, kv_len + a] changes
    for b in range(B):
        L, a = int(kv_len[b]), int(alen[b])
        assert np.array_equal(k2[b][:, :L], k[b][:, :L])
        assert np.array_equal(k2[b][:, L + a + 1:], k[b][:, L + a + 1:])


def test_commit_then_attention_sees_the_branch(oracle_mod):
    """The end node's tree attention (prefix + its ancestors) equals plain
    decode attention of the same query at the end of the committed prefix."""
    case = gen.make_case(11, B=2, N=40, L=(50, 90), Hq=8, Hkv=2, D=64, V=64, tree="random",
                         max_depth=9)
    r = gen.rng(5)
    for b in range(case.B):
        depth = gen.depth_of(case.parent[b])
        end = int(np.argmax(depth)) if b == 0 else int(r.integers(1, case.N))
        br = branch_to(case.parent[b], end)
        path = np.full((1, case.N), -1, np.int32)
        path[0, :len(br)] = br
        a = len(br) - 1
        kb, vb = case.k[b:b + 1], case.v[b:b + 1]
        k2, v2, new_len, status = oracle_mod.commit_path(kb, vb, case.kv_len[b:b + 1], path,
                                                         np.array([a], np.int32))
        assert status[0] == 0 and new_len[0] == case.kv_len[b] + a + 1
        rows = np.array([(b, end, h) for h in range(case.Hq)], np.int32)
        tree_out, tree_lse = oracle_mod.attn_rows(case.q, case.k, case.v, case.kv_len,
                                                  case.parent, case.Hq, case.Hkv, rows)
        # one node (parent -1) whose own slot is kv_len' + 0 = kv_len + a: the end node's row
        q1 = case.q[b:b + 1, end:end + 1]
        one = np.array([[-1]], np.int32)
        rows1 = np.array([(0, 0, h) for h in range(case.Hq)], np.int32)
        dec_out, dec_lse = oracle_mod.attn_rows(q1, k2, v2, np.array([case.kv_len[b] + a], np.int32),
                                                one, case.Hq, case.Hkv, rows1)
        np.testing.assert_allclose(dec_out, tree_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dec_lse, tree_lse, rtol=0, atol=1e-12)


def test_chain_fully_accepted_moves_nothing(oracle_mod):
    r = gen.rng(9)
    N, L = 24, 30
    k = gen.normal_bf16(r, (1, 3, L + N, 64))
    v = gen.normal_bf16(r, (1, 3, L + N, 64))
    path = np.arange(N, dtype=np.int32)[None]
    k2, v2, new_len, status = oracle_mod.commit_path(k, v, np.array([L], np.int32), path,
                                                     np.array([N - 1], np.int32))
    assert status[0] == 0 and new_len[0] == L + N
    assert np.array_equal(k2, k) and np.array_equal(v2, v)


def test_nothing_accepted_keeps_node_zero_only(oracle_mod):
    r = gen.rng(10)
    k = gen.normal_bf16(r, (2, 2, 20, 64))
    v = gen.normal_bf16(r, (2, 2, 20, 64))
    path = np.full((2, 8), -1, np.int32)
    path[:, 0] = 0
    k2, v2, new_len, status = oracle_mod.commit_path(k, v, np.array([5, 12], np.int32), path,
                                                     np.zeros(2, np.int32))
    assert status.tolist() == [0, 0] and new_len.tolist() == [6, 13]
    assert np.array_equal(k2, k) and np.array_equal(v2, v)


@pytest.mark.parametrize("bad", ["first", "order", "outside", "cache", "negative"])
def test_malformed_paths_leave_the_cache_alone(oracle_mod, bad):
    k, v, kv_len, parents, path, alen, Lcap = random_commit_case(21, 2, 30, 2, 64, 10, slack=0)
    b = 1
    a = 3
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
    k2, v2, new_len, status = oracle_mod.commit_path(k, v, kv_len, path, alen)
    assert status[b] == 1 and new_len[b] == kv_len[b]
    assert np.array_equal(k2[b], k[b]) and np.array_equal(v2[b], v[b])
    assert status[0] == 0
