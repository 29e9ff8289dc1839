"""GPU parity: tv_attn_verify against the fp64 oracle (OPT-Tree §2: one target
pass over the whole tree under the tree attention mask; GQA kv head h / G).

Tolerance: bf16 inputs with fp32 accumulation and a bf16 output, compared with
fp64: max-abs <= 3e-2 and relative L2 <= 1e-2 per case; the natural-log
normaliser (fp32 output) within 2e-3 absolute."""
import numpy as np
import pytest
import torch

from workloads import gen

from _gpu_util import bf16, bf16_np, case_tensors, check_attn, dev, i32, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


def run_attn(tv, case, scale=0.0, k=None, v=None):
    t = case_tensors(case)
    depth, anc, _ = tv.tree_build(t["parent"])
    out, lse, status = tv.attn_verify(t["q"], t["k"] if k is None else k,
                                      t["v"] if v is None else v, t["kv_len"], anc, scale)
    torch.cuda.synchronize()
    return bf16_np(out), np_(lse), np_(status)


def full_check(tv, oracle_mod, case, what, scale=0.0):
    out, lse, status = run_attn(tv, case, scale)
    ref, ref_lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, case.Hq,
                                       case.Hkv, scale)
    assert (status == 0).all()
    check_attn(out, ref, what)
    np.testing.assert_allclose(lse, ref_lse, atol=2e-3, rtol=0)


def sampled_check(tv, oracle_mod, case, n_rows, seed, what):
    out, lse, status = run_attn(tv, case)
    r = gen.rng(seed)
    rows = np.stack([r.integers(0, case.B, n_rows), r.integers(0, case.N, n_rows),
                     r.integers(0, case.Hq, n_rows)], axis=1)
    # always include the deepest node and the root of sequence 0
    depth = gen.depth_of(case.parent[0])
    rows[0] = (0, int(np.argmax(depth)), 0)
    rows[1] = (0, 0, case.Hq - 1)
    ref, ref_lse = oracle_mod.attn_rows(case.q, case.k, case.v, case.kv_len, case.parent, case.Hq,
                                        case.Hkv, rows)
    assert (status == 0).all()
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    check_attn(got, ref, what)
    np.testing.assert_allclose(lse[rows[:, 0], rows[:, 1], rows[:, 2]], ref_lse, atol=2e-3)


def test_config1_tiny(tv, oracle_mod):
    full_check(tv, oracle_mod, gen.config1(), "config1")


@pytest.mark.parametrize("seed,B,N,L,Hq,Hkv,D,tree", [
    (1, 1, 1, 0, 8, 8, 64, "chain"),          # a single node with no prefix
    (2, 1, 37, 300, 8, 2, 128, "random"),     # ragged prefix tail, GQA 4
    (3, 2, 64, (1, 700), 16, 2, 64, "random"),  # ragged batch, GQA 8
    (4, 1, 65, 129, 4, 4, 128, "chain"),      # chain tree crossing a mask word
    (5, 3, 20, (0, 260), 32, 8, 128, "star"),
    (6, 1, 130, 1000, 4, 1, 64, "random"),
    (7, 1, 60, 2048, 32, 8, 128, "spine60"),  # the Llama-3-8B spine case, full size
    (8, 2, 50, (90, 400), 12, 4, 64, "random"),  # GQA 3: a row block holds 42 nodes (126 rows)
    (9, 1, 100, 500, 6, 1, 128, "random"),     # GQA 6: 21 nodes (126 rows), three node tiles
])
def test_attention_full(tv, oracle_mod, seed, B, N, L, Hq, Hkv, D, tree):
    case = gen.make_case(seed, B=B, N=N, L=L, Hq=Hq, Hkv=Hkv, D=D, V=max(64, N), tree=tree,
                         max_depth=12)
    full_check(tv, oracle_mod, case, f"case{seed}")


@pytest.mark.parametrize("plan", ["128,1", "128,4", "256,1", "256,3"])
@pytest.mark.parametrize("seed,B,N,L,Hq,Hkv,D,tree", [
    (31, 1, 60, 700, 32, 8, 128, "spine60"),    # two row blocks of 32 nodes each
    (32, 2, 20, (100, 900), 8, 2, 64, "random"),  # 256-row CTAs with an empty second block
    (33, 1, 130, 300, 4, 1, 64, "random"),      # three node tiles, the last one ragged
])
def test_attention_every_plan_kind(tv, oracle_mod, monkeypatch, plan, seed, B, N, L, Hq, Hkv, D,
                                   tree):
    """Both CTA heights, with and without a split key range (and so with and
    without the merge kernel), forced through TV_ATTN_PLAN and compared row by
    row with the oracle."""
    monkeypatch.setenv("TV_ATTN_PLAN", plan)
    case = gen.make_case(seed, B=B, N=N, L=L, Hq=Hq, Hkv=Hkv, D=D, V=64, tree=tree, max_depth=12)
    rows, splits = (int(x) for x in plan.split(","))
    got = tv.attn_plan(B, N, Hq, Hkv, D, case.Lcap)
    assert (got["rows_per_cta"], got["splits"]) == (rows, splits)
    full_check(tv, oracle_mod, case, f"case{seed}-plan{plan}")


def test_explicit_scale(tv, oracle_mod):
    case = gen.make_case(20, B=1, N=24, L=200, Hq=8, Hkv=4, D=64, V=64)
    full_check(tv, oracle_mod, case, "scale", scale=0.05)


def test_unused_cache_slots_may_hold_nan(tv, oracle_mod):
    """Slots at and beyond kv_len + N are never part of a result."""
    case = gen.make_case(21, B=2, N=30, L=(100, 180), Hq=8, Hkv=2, D=128, V=64,
                         Lcap=400)
    k = case.k.copy()
    v = case.v.copy()
    for b in range(case.B):
        end = case.kv_len[b] + case.N
        k[b, :, end:] = 0x7FC0   # bf16 NaN
        v[b, :, end:] = 0x7FC0
    out, lse, status = run_attn(tv, case, k=bf16(k), v=bf16(v))
    ref, ref_lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, 8, 2)
    check_attn(out, ref, "nan-tail")


def test_bad_kv_len_is_flagged(tv):
    case = gen.make_case(22, B=3, N=8, L=16, Hq=4, Hkv=4, D=64, V=64)
    case.kv_len = np.array([16, case.Lcap, -1], np.int32)
    out, lse, status = run_attn(tv, case)
    assert status.tolist() == [0, 1, 1]
    assert (out[1:] == 0).all()


def unit_rows(tv, case, seqs):
    """Every (node, head) row of the first and the last node tile of the
    sequences `seqs` under the plan the call takes: whole CTA units, so every
    split of the key range, both row blocks of a 256-row CTA and every kv head
    of those nodes are compared."""
    plan = tv.attn_plan(case.B, case.N, case.Hq, case.Hkv, case.D, case.Lcap)
    G = case.Hq // case.Hkv
    per_tile = (plan["rows_per_cta"] // 128) * (128 // G)
    last0 = (plan["node_tiles"] - 1) * per_tile
    nodes = sorted(set(range(0, min(per_tile, case.N))) | set(range(last0, case.N)))
    rows = np.array([(b, n, h) for b in seqs for n in nodes for h in range(case.Hq)], np.int64)
    return rows, plan


def unit_check(tv, oracle_mod, case, seqs, what):
    out, lse, status = run_attn(tv, case)
    assert (status == 0).all()
    rows, plan = unit_rows(tv, case, seqs)
    ref, ref_lse = oracle_mod.attn_rows(case.q, case.k, case.v, case.kv_len, case.parent, case.Hq,
                                        case.Hkv, rows)
    check_attn(out[rows[:, 0], rows[:, 1], rows[:, 2]], ref, what)
    np.testing.assert_allclose(lse[rows[:, 0], rows[:, 1], rows[:, 2]], ref_lse, atol=2e-3)
    return out, plan


def test_config4_ragged_batch_units(tv, oracle_mod):
    """Batched ragged workload: whole node tiles of the first sequence and of
    the one with the longest prefix (every head, every key)."""
    case = gen.config4(V=8)
    longest = int(np.argmax(case.kv_len))
    unit_check(tv, oracle_mod, case, sorted({0, longest}), "config4")
    sampled_check(tv, oracle_mod, case, 48, 5, "config4-sampled")


def test_config5_long_context_units(tv, oracle_mod):
    """Long context, 256 nodes: the first and last node tiles in full (a plan
    of 256-row CTAs over several key splits: both row blocks, every split)."""
    case = gen.config5(256, V=5000)
    _, plan = unit_check(tv, oracle_mod, case, [0], "config5")
    assert plan["splits"] > 1


@pytest.mark.parametrize("n", [16, 64, 512])
def test_config5_long_context_sweep(tv, oracle_mod, n):
    """The long-context workload's node-count sweep (16, 64 and 512 nodes over
    the 32,768-key prefix; 256 is the case above): every row at 16 nodes, the
    first and last node tiles in full at 64 and 512."""
    case = gen.config5(n, V=64)
    if n == 16:
        full_check(tv, oracle_mod, case, "config5-n16")
    else:
        unit_check(tv, oracle_mod, case, [0], f"config5-n{n}")


def test_config3_talon_chain(tv, oracle_mod):
    """The TALON workload end to end on the GPU -- gated expansion, tree
    encoding, attention, greedy acceptance -- against the same chain on the
    oracle: the tree and the acceptance result bit-exact, the attention rows
    of the first and last node tiles in full within the attention tolerance."""
    d = gen.config3_drafter(1)
    g = tv.expand_tree(d.rows, d.root_key(), d.child_key, 10, 0.3, 512, dev())
    o = oracle_mod.expand_tree(d, 10, 0.3, 512)
    assert g["n"] == o["n"] == 512
    gpar, gtok = g["parent"].numpy()[:512], g["token"].numpy()[:512]
    assert np.array_equal(gpar, o["parent"]) and np.array_equal(gtok, o["token"])
    case = gen.config3_verify(gpar, 1, tokens=gtok)
    t = case_tensors(case)
    depth, anc, tstat = tv.tree_build(t["parent"])
    out, lse, astat = tv.attn_verify(t["q"], t["k"], t["v"], t["kv_len"], anc)
    res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
    torch.cuda.synchronize()
    od, oa, ost = oracle_mod.tree_build(case.parent)
    assert np.array_equal(np_(depth), od) and np.array_equal(np_(anc).view(np.uint64), oa)
    assert (np_(tstat) == 0).all() and (np_(astat) == 0).all()
    rows, _ = unit_rows(tv, case, [0])
    ref, _ = oracle_mod.attn_rows(case.q, case.k, case.v, case.kv_len, case.parent, case.Hq,
                                  case.Hkv, rows)
    check_attn(bf16_np(out)[rows[:, 0], rows[:, 1], rows[:, 2]], ref, "config3-chain")
    og = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    for k in ("argmax", "accept_len", "end_node", "path", "bonus", "status"):
        assert np.array_equal(np_(res[k]), og[k]), k


def test_split_partials_keep_the_range(tv, oracle_mod, monkeypatch):
    """Split plans hold partial rows in bf16, which keeps the fp32 exponent
    range: values of v of magnitude 1e5 and more (beyond fp16) survive the
    merge.  The output is bf16, so the comparison is relative to the values'
    scale: max-abs within 3e-2 of the largest |v| and rel-L2 within 1e-2."""
    case = gen.make_case(41, B=1, N=60, L=1500, Hq=32, Hkv=8, D=128, V=64, tree="spine60")
    big = case.v.copy()
    f = gen.f32_from_bf16(big) * np.float32(3e5)
    big = gen.bf16_from_f32(f)
    case.v = big
    for plan in ("128,4", "256,3", "128,1"):
        monkeypatch.setenv("TV_ATTN_PLAN", plan)
        out, lse, status = run_attn(tv, case)
        assert (status == 0).all()
        ref, ref_lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent,
                                           case.Hq, case.Hkv)
        scale = float(np.abs(gen.f32_from_bf16(case.v)).max())
        assert np.isfinite(out).all(), plan
        err = np.abs(out - ref)
        assert err.max() <= 3e-2 * scale, (plan, err.max() / scale)
        assert np.linalg.norm(out - ref) <= 1e-2 * np.linalg.norm(ref), plan


def test_merge_kernel_path_large_batch(tv, oracle_mod):
    """96 (sequence, kv head) pairs over 6,000 prefix keys: the plan takes
    128-row CTAs in several splits and more than one wave of CTAs, whose
    partials a separate kernel merges."""
    case = gen.make_case(23, B=24, N=60, L=6000, Hq=16, Hkv=4, D=64, V=64)
    assert tv.attn_workspace_size(24, 60, 16, 4, 64, case.Lcap) > 0
    sampled_check(tv, oracle_mod, case, 48, 8, "merge-kernel")


@pytest.mark.parametrize("B,L", [(1, 1500), (1, 6000)])
def test_split_plans_single_wave(tv, oracle_mod, B, L):
    """One sequence, 60 nodes: 1,500 keys split 256-row CTAs, 6,000 keys
    split 128-row CTAs with a two-stage K/V ring; every row is compared."""
    case = gen.make_case(24 + L, B=B, N=60, L=L, Hq=16, Hkv=4, D=64, V=64)
    assert tv.attn_workspace_size(B, 60, 16, 4, 64, case.Lcap) > 0
    out, lse, status = run_attn(tv, case)
    assert (status == 0).all()
    ref, ref_lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, 16, 4)
    check_attn(out, ref, f"split-L{L}")


def test_split_plan_repeats_bitwise(tv, oracle_mod):
    """A split plan on a reused workspace: repeated calls agree bit for bit
    (the merge order is fixed) and match the oracle."""
    case = gen.make_case(24, B=1, N=60, L=1500, Hq=32, Hkv=8, D=128, V=64, tree="spine60")
    assert tv.attn_workspace_size(1, 60, 32, 8, 128, case.Lcap) > 0
    first = run_attn(tv, case)
    for _ in range(3):
        again = run_attn(tv, case)
        assert np.array_equal(first[0], again[0])
        assert np.array_equal(first[1], again[1])
    ref, ref_lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, case.Hq,
                                       case.Hkv)
    check_attn(first[0], ref, "coop")


def test_bad_kv_len_in_a_split_plan(tv, oracle_mod):
    """A sequence whose kv_len does not fit the cache is flagged and zeroed
    while the others of the batch, split across CTAs, are still right."""
    case = gen.make_case(25, B=3, N=40, L=900, Hq=8, Hkv=2, D=64, V=64)
    assert tv.attn_workspace_size(3, 40, 8, 2, 64, case.Lcap) > 0
    good = case.kv_len.copy()
    case.kv_len = np.array([good[0], case.Lcap, -1], np.int32)
    out, lse, status = run_attn(tv, case)
    assert status.tolist() == [0, 1, 1]
    assert (out[1:] == 0).all()
    rows = np.array([(0, n, h) for n in range(0, 40, 3) for h in range(8)], np.int64)
    ref, ref_lse = oracle_mod.attn_rows(case.q, case.k, case.v, good, case.parent, 8, 2, rows)
    check_attn(out[rows[:, 0], rows[:, 1], rows[:, 2]], ref, "split-bad-kv")


@pytest.mark.parametrize("seed,B,N,L,Hq,Hkv,D,tree,plan", [
    (61, 1, 60, 2048, 32, 8, 128, "spine60", None),   # the Llama-3-8B spine step (split plan)
    (62, 3, 64, (10, 700), 16, 4, 64, "random", None),
    (63, 2, 33, 300, 8, 8, 128, "chain", "256,1"),
    (64, 1, 1, 0, 8, 2, 64, "chain", None),
    (65, 2, 50, 900, 32, 8, 128, "random", "128,4"),
    (66, 1, 100, 500, 8, 2, 64, "random", None),       # more than 64 nodes: two launches
])
def test_attn_verify_tree_equals_two_calls(tv, oracle_mod, monkeypatch, seed, B, N, L, Hq, Hkv,
                                           D, tree, plan):
    """tv_attn_verify_tree (the tree encoding inside the attention launch for
    trees of up to 64 nodes) gives, bit for bit, what tv_tree_build followed by
    tv_attn_verify gives, and matches the oracle."""
    if plan:
        monkeypatch.setenv("TV_ATTN_PLAN", plan)
    case = gen.make_case(seed, B=B, N=N, L=L, Hq=Hq, Hkv=Hkv, D=D, V=64, tree=tree, max_depth=12)
    t = case_tensors(case)
    depth, anc, tst = tv.tree_build(t["parent"])
    out, lse, ast = tv.attn_verify(t["q"], t["k"], t["v"], t["kv_len"], anc)
    f_out, f_lse, f_ast, f_depth, f_anc, f_tst = tv.attn_verify_tree(
        t["q"], t["k"], t["v"], t["kv_len"], t["parent"])
    torch.cuda.synchronize()
    for a, b_, what in ((out.view(torch.int16), f_out.view(torch.int16), "out"),
                        (lse.view(torch.int32), f_lse.view(torch.int32), "lse"),
                        (ast, f_ast, "status"), (depth, f_depth, "depth"), (anc, f_anc, "anc"),
                        (tst, f_tst, "tree_status")):
        assert torch.equal(a, b_), what
    ref, ref_lse = oracle_mod.attn_all(case.q, case.k, case.v, case.kv_len, case.parent, Hq, Hkv)
    check_attn(bf16_np(f_out), ref, f"fused-{seed}")


def test_attn_verify_tree_invalid_tree(tv):
    """An invalid parent array: the fused call reports it in tree_status with
    depth -1 and empty masks, exactly as tv_tree_build does, and the attention
    runs on the empty masks as the two calls would."""
    case = gen.make_case(67, B=3, N=20, L=100, Hq=8, Hkv=2, D=64, V=64)
    case.parent[1, 7] = 9          # a parent after its child
    case.parent[2, 0] = 0          # the root has a parent
    t = case_tensors(case)
    depth, anc, tst = tv.tree_build(t["parent"])
    out, lse, ast = tv.attn_verify(t["q"], t["k"], t["v"], t["kv_len"], anc)
    f = tv.attn_verify_tree(t["q"], t["k"], t["v"], t["kv_len"], t["parent"])
    torch.cuda.synchronize()
    assert np_(f[5]).tolist() == np_(tst).tolist() == [0, 2, 2]
    assert torch.equal(f[3], depth) and torch.equal(f[4], anc)
    assert torch.equal(f[0].view(torch.int16), out.view(torch.int16))
