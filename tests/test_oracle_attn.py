"""Pins for the oracle's tree-verify attention.

OPT-Tree §2: the target verifies every tree token in one pass under a tree
attention mask; each node sees the cached prefix, its ancestors and itself.
Pinned against cases that reduce to textbook attention computed by a library
routine (torch's scaled_dot_product_attention in fp64 on CPU):
  * a single node is ordinary decode attention over prefix + 1 keys,
  * a chain tree is causal attention of N new tokens after the prefix,
  * every root-to-leaf path equals causal attention over prefix + path,
  * K = 0 with one-hot V rows gives exactly the indicator of the visible set.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from workloads import gen


def f64(bits):
    return torch.from_numpy(gen.f32_from_bf16(bits).astype(np.float64))


def sdpa_sequence(case, b, nodes, scale=None):
    """Attention of the given node sequence (a root path, in order) as an
    ordinary causal sequence after the prefix: query t sees the prefix and
    nodes[0..t].  Returns (out [len, Hq, D], lse [len, Hq])."""
    L = int(case.kv_len[b])
    slots = list(range(L)) + [L + j for j in nodes]
    q = f64(case.q[b, nodes]).permute(1, 0, 2)[None]              # [1, Hq, T, D]
    k = f64(case.k[b][:, slots])[None]                             # [1, Hkv, S, D]
    v = f64(case.v[b][:, slots])[None]
    T, S = len(nodes), len(slots)
    mask = torch.arange(S)[None, :] <= (L + torch.arange(T))[:, None]
    out = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale,
                                         enable_gqa=True)[0].permute(1, 0, 2)
    G = case.Hq // case.Hkv
    kk = k[0].repeat_interleave(G, dim=0)
    sc = scale if scale is not None else 1.0 / np.sqrt(case.D)
    s = torch.einsum("htd,hsd->hts", q[0], kk) * sc
    s = s.masked_fill(~mask[None], float("-inf"))
    lse = torch.logsumexp(s, dim=-1).T
    return out.numpy(), lse.numpy()


def root_paths(parent):
    kids = gen.children_of(parent)
    leaves = [i for i in range(len(parent)) if not kids[i]]
    paths = []
    for leaf in leaves:
        p = []
        x = leaf
        while x >= 0:
            p.append(x)
            x = int(parent[x])
        paths.append(p[::-1])
    return paths


@pytest.mark.parametrize("Hq,Hkv,D,L", [(8, 8, 64, 128), (8, 2, 128, 37), (4, 1, 64, 0)])
def test_single_node_is_decode_attention(oracle_mod, Hq, Hkv, D, L):
    case = gen.make_case(11, B=2, N=1, L=L, Hq=Hq, Hkv=Hkv, D=D, V=10, tree="chain")
    out, lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, Hq, Hkv)
    for b in range(2):
        ref, ref_lse = sdpa_sequence(case, b, [0])
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-12, atol=1e-12)


def test_chain_tree_is_causal_attention(oracle_mod):
    case = gen.make_case(12, B=1, N=24, L=50, Hq=8, Hkv=4, D=64, V=10, tree="chain")
    out, lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, 8, 4)
    ref, ref_lse = sdpa_sequence(case, 0, list(range(24)))
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("tree,seed", [("random", 1), ("random", 2), ("spine60", 3), ("star", 4)])
def test_every_root_path_is_a_causal_sequence(oracle_mod, tree, seed):
    N = 60 if tree == "spine60" else 30
    case = gen.make_case(seed, B=2, N=N, L=(0, 70), Hq=4, Hkv=2, D=64, V=100, tree=tree,
                         max_depth=5)
    out, lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, 4, 2)
    for b in range(2):
        for path in root_paths(case.parent[b]):
            ref, ref_lse = sdpa_sequence(case, b, path)
            np.testing.assert_allclose(out[b, path], ref, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lse[b, path], ref_lse, rtol=1e-11, atol=1e-12)


def test_explicit_scale(oracle_mod):
    case = gen.make_case(13, B=1, N=9, L=17, Hq=2, Hkv=1, D=64, V=10, tree="random")
    out, lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, 2, 1,
                                   scale=0.3)
    for path in root_paths(case.parent[0]):
        ref, ref_lse = sdpa_sequence(case, 0, path, scale=0.3)
        np.testing.assert_allclose(out[0, path], ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[0, path], ref_lse, rtol=1e-11, atol=1e-12)


def test_zero_keys_one_hot_values_expose_the_mask(oracle_mod):
    """K = 0 makes every visible key weigh the same; V[slot] = e_slot turns the
    output into (indicator of the visible slots) / (their count)."""
    L, N, D = 20, 40, 64
    case = gen.make_case(14, B=1, N=N, L=L, Hq=2, Hkv=2, D=D, V=10, tree="random",
                         max_depth=7)
    k = np.zeros_like(case.k)
    v = np.zeros_like(case.v)
    one = gen.bf16_from_f32(np.float32([1.0]))[0]
    for s in range(L + N):
        v[0, :, s, s] = one
    out, lse = oracle_mod.attn_all(case.q, k, v, case.kv_len, case.parent, 2, 2)
    depth = gen.depth_of(case.parent[0])
    for i in range(N):
        vis = set(range(L))
        x = i
        while x >= 0:
            vis.add(L + x)
            x = int(case.parent[0, x])
        expect = np.array([1.0 / len(vis) if d in vis else 0.0 for d in range(D)])
        assert len(vis) == L + depth[i] + 1
        for h in range(2):
            np.testing.assert_allclose(out[0, i, h], expect, rtol=0, atol=1e-15)
            np.testing.assert_allclose(lse[0, i, h], np.log(len(vis)), rtol=1e-14)


def test_rejects_bad_arguments(oracle_mod):
    case = gen.make_case(15, B=1, N=4, L=8, Hq=4, Hkv=2, D=64, V=10)
    bad_len = np.array([case.Lcap], np.int32)        # L + N > Lcap
    with pytest.raises(ValueError):
        oracle_mod.attn_all(case.q, case.k, case.v, bad_len, case.parent, 4, 2)
    with pytest.raises(ValueError):
        oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, 4, 3)
