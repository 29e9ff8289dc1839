"""GPU parity: tv_accept_sample against the oracle (Speculative Decoding
concept page, "The protocol" step 3: min(1, p/q) acceptance with (p - q)+
residual resampling).

Both sides draw the same Philox4x64-10 words and take every decision in fp64;
they can only disagree where a decision sits within rounding distance of its
threshold.  The oracle reports, per tree, the smallest relative distance of an
accept test from its threshold (|u - r/q| / (r/q)) and the distance of the
final draw from the nearest cumulative-mass boundary (as a fraction of the
total mass).  The GPU holds each probability in fp32 (about 1e-6 relative
error) and sums them in fp64 or compensated fp32, so accept tests closer than
1e-5 and draws closer than 1e-7 are "ambiguous": those trees are checked for
validity only (and counted); all other trees must match bit for bit."""
import numpy as np
import pytest
import torch
from scipy.special import softmax
from scipy.stats import chi2

from workloads import gen

from _gpu_util import case_tensors, i32, f32, np_

pytestmark = pytest.mark.gpu

MARGIN_ACCEPT = 1e-5
MARGIN_DRAW = 1e-7


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


def run_sample(tv, case, seed, offset, T=1.0):
    t = case_tensors(case)
    depth, _, _ = tv.tree_build(t["parent"])
    res = tv.accept_sample(t["p_logits"], t["q_logits"], t["tokens"], t["parent"], depth, T,
                           seed, offset)
    torch.cuda.synchronize()
    return {k: np_(v) for k, v in res.items()}


def compare(g, o, parent):
    ambiguous = 0
    for b in range(len(o["status"])):
        assert g["status"][b] == o["status"][b]
        if o["margin_accept"][b] < MARGIN_ACCEPT or o["margin_draw"][b] < MARGIN_DRAW:
            ambiguous += 1
            e = g["end_node"][b]
            assert 0 <= e < parent.shape[1]
            assert g["accept_len"][b] == gen.depth_of(parent[b])[e]
            continue
        for k in ("accept_len", "end_node", "path", "out_token"):
            assert np.array_equal(g[k][b], o[k][b]), (k, b)
    return ambiguous


def test_config4_batched_ragged(tv, oracle_mod):
    case = gen.config4(with_attn=False)
    for offset in (0, 1):
        g = run_sample(tv, case, 0x5EED, offset)
        o = oracle_mod.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, 1.0,
                                     0x5EED, offset)
        assert compare(g, o, case.parent) <= 2


@pytest.mark.parametrize("seed,B,N,V,T,noise", [
    (1, 4, 9, 16, 1.0, 1.0), (2, 8, 33, 1000, 1.0, 0.5), (3, 3, 64, 8191, 0.7, 0.5),
    (4, 2, 5, 3, 1.3, 2.0), (5, 6, 20, 40000, 1.0, 0.1), (6, 1, 1, 77, 1.0, 0.5),
    (7, 2, 128, 500, 2.0, 1.0),
])
def test_sample_fuzz(tv, oracle_mod, seed, B, N, V, T, noise):
    case = gen.make_case(seed, B=B, N=N, L=4, V=V, mode="sample", tree="random", max_depth=8,
                         q_noise=noise, temperature=T, with_attn=False)
    total_amb = 0
    for offset in range(3):
        g = run_sample(tv, case, seed * 1000 + 1, offset, T)
        o = oracle_mod.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, T,
                                     seed * 1000 + 1, offset)
        total_amb += compare(g, o, case.parent)
    assert total_amb <= max(2, (3 * B) // 5)


def test_q_equals_p_and_one_hot(tv, oracle_mod):
    case = gen.make_case(20, B=8, N=40, L=4, V=300, mode="sample", tree="random", max_depth=6,
                         with_attn=False)
    case.q_logits = case.p_logits.copy()
    g = run_sample(tv, case, 3, 0)
    o = oracle_mod.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, 1.0, 3, 0)
    compare(g, o, case.parent)
    for b in range(case.B):     # every first child accepted down to a leaf
        kids = gen.children_of(case.parent[b])
        v = 0
        while kids[v]:
            v = kids[v][0]
        assert g["end_node"][b] == v


def test_gpu_lossless_chi_square(tv):
    """The GPU walk itself reproduces p: first emitted token over 2^19 trials."""
    V, N = 16, 10
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)
    r = gen.rng(77)
    lp = r.standard_normal((N, V)).astype(np.float32)
    lq = (lp + r.normal(0, 1.0, (N, V))).astype(np.float32)
    qr = softmax(lq.astype(np.float64), axis=1)
    kids = gen.children_of(parent)
    trials = 1 << 16
    counts = np.zeros(V, np.int64)
    P = f32(np.broadcast_to(lp, (trials, N, V)))
    Q = f32(np.broadcast_to(lq, (trials, N, V)))
    par = i32(np.broadcast_to(parent, (trials, N)))
    depth, _, _ = tv.tree_build(par)
    for rep in range(8):
        tok = np.zeros((trials, N), np.int32)
        for v, ks in enumerate(kids):
            if ks:
                cdf = np.cumsum(qr[v])
                tok[:, ks] = np.minimum(np.searchsorted(cdf, r.random((trials, len(ks))) * cdf[-1],
                                                        side="right"), V - 1)
        res = tv.accept_sample(P, Q, i32(tok), par, depth, 1.0, 4242, rep)
        al, path, out = np_(res["accept_len"]), np_(res["path"]), np_(res["out_token"])
        first = np.where(al >= 1, tok[np.arange(trials), np.maximum(path[:, 1], 0)], out)
        counts += np.bincount(first, minlength=V)
    p = softmax(lp.astype(np.float64), axis=1)[0]
    stat = (((counts - p * counts.sum()) ** 2) / (p * counts.sum())).sum()
    assert stat < chi2.ppf(1 - 1e-3, V - 1)


def test_sample_bad_inputs(tv, oracle_mod):
    case = gen.make_case(30, B=3, N=8, L=4, V=50, mode="sample", with_attn=False)
    case.tokens[1, 2] = -1
    case.parent[2, 5] = 6
    g = run_sample(tv, case, 1, 0)
    o = oracle_mod.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, 1.0, 1, 0)
    assert g["status"].tolist() == o["status"].tolist() == [0, 6, 2]
    assert g["end_node"][1:].tolist() == [-1, -1]
