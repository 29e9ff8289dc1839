"""GPU parity: tv_accept_sample against the oracle (Speculative Decoding
concept page, "The protocol" step 3: min(1, p/q) acceptance with (p - q)+
residual resampling).

Both sides draw the same Philox4x64-10 words.  The oracle takes every decision
in fp64; the GPU holds each probability in fp32, made with the special-function
unit's 2^x (about 2^-22 relative error) and fp32 products, so each probability
is within about 5e-7 of its fp64 value, relative.  Two kinds of decision can
therefore go either way, and only those:
  * an accept test u < r(x)/q(x) whose ratio lies within 1e-5 of u, relative
    to the ratio (5e-7 per probability, amplified by the cancellation in a
    residual (r - q)+ up to twenty-fold);
  * the final draw, when u times the total mass lies within 1e-6 of the total
    from a cumulative boundary (cumulative masses and the target each within
    5e-7 of the total).
With a 128,256-token vocabulary each token holds about 8e-6 of the mass, so a
uniform target falls that close to a boundary in roughly one draw in eight;
at the batched configuration's seeds no accept test is closer than 2e-2 to its
threshold and five of the 32 draws are inside the draw margin.
The oracle reports the margin of every decision along its walk.  A tree whose
decisions all clear their margins must match bit for bit.  Otherwise the GPU's
walk must agree with the oracle's on every node reached before the first
near-threshold decision, its path must be the root chain of its end node, and
a draw-only ambiguity must give the oracle's token or the one across the
nearest boundary."""
import numpy as np
import pytest
import torch
from scipy.special import softmax
from scipy.stats import chi2

from workloads import gen

from _gpu_util import case_tensors, i32, f32, np_

pytestmark = pytest.mark.gpu

MARGIN_ACCEPT = 1e-5   # relative to r(x)/q(x)
MARGIN_DRAW = 1e-6     # fraction of the total mass


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


def compare(g, o, parent, V):
    """Check every tree; return the indices of the trees with a decision
    inside its rounding margin."""
    ambiguous = []
    for b in range(len(o["status"])):
        assert g["status"][b] == o["status"][b], b
        if o["status"][b] != 0:
            assert g["end_node"][b] == -1 and g["out_token"][b] == -1, b
            continue
        od = int(o["accept_len"][b])
        amb_depth = np.nonzero(o["margin_path"][b, :od + 1] < MARGIN_ACCEPT)[0]
        draw_amb = o["margin_draw"][b] < MARGIN_DRAW
        if len(amb_depth) == 0 and not draw_amb:
            for k in ("accept_len", "end_node", "path", "out_token"):
                assert np.array_equal(g[k][b], o[k][b]), (k, b)
            continue
        ambiguous.append(b)
        # the GPU's result is a valid walk: its path is the root chain of its
        # end node, padded with -1, and its token lies in the vocabulary
        e = int(g["end_node"][b])
        assert 0 <= e < parent.shape[1]
        chain = [e]
        while parent[b][chain[-1]] >= 0:
            chain.append(int(parent[b][chain[-1]]))
        chain = chain[::-1]
        assert g["accept_len"][b] == len(chain) - 1
        assert g["path"][b][:len(chain)].tolist() == chain
        assert (g["path"][b][len(chain):] == -1).all()
        assert 0 <= g["out_token"][b] < V
        if len(amb_depth):
            # every decision before the first near-threshold accept test is
            # exact: both walks reach the node that makes it
            d0 = int(amb_depth[0])
            assert g["accept_len"][b] >= d0
            assert np.array_equal(g["path"][b][:d0 + 1], o["path"][b][:d0 + 1]), b
        else:
            # only the final draw is near a boundary: same walk, and the token
            # is the oracle's or the one across that boundary
            for k in ("accept_len", "end_node", "path"):
                assert np.array_equal(g[k][b], o[k][b]), (k, b)
            assert g["out_token"][b] in (o["out_token"][b], o["draw_alt"][b]), b
    return ambiguous


def test_config4_batched_ragged(tv, oracle_mod):
    case = gen.config4(with_attn=False)
    for offset in (0, 1):
        g = run_sample(tv, case, 0x5EED, offset)
        o = oracle_mod.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, 1.0,
                                     0x5EED, offset)
        amb = compare(g, o, case.parent, case.V)
        # the ambiguous trees are the ones the oracle's margins mark: here only
        # final draws (no accept test of these seeds is within 2e-2 of its threshold)
        assert all(o["margin_path"][b].min() > 1e-2 for b in range(case.B)), offset
        print(f"offset {offset}: draws inside the margin in trees {amb}, margins "
              f"{[float(o['margin_draw'][b]) for b in amb]}")


@pytest.mark.parametrize("seed,B,N,V,T,noise", [
    (1, 4, 9, 16, 1.0, 1.0), (2, 8, 33, 1000, 1.0, 0.5), (3, 3, 64, 8191, 0.7, 0.5),
    (4, 2, 5, 3, 1.3, 2.0), (5, 6, 20, 40000, 1.0, 0.1), (6, 1, 1, 77, 1.0, 0.5),
    (7, 2, 128, 500, 2.0, 1.0),
])
def test_sample_fuzz(tv, oracle_mod, seed, B, N, V, T, noise):
    case = gen.make_case(seed, B=B, N=N, L=4, V=V, mode="sample", tree="random", max_depth=8,
                         q_noise=noise, temperature=T, with_attn=False)
    for offset in range(3):
        g = run_sample(tv, case, seed * 1000 + 1, offset, T)
        o = oracle_mod.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, T,
                                     seed * 1000 + 1, offset)
        compare(g, o, case.parent, V)


def test_q_equals_p_and_one_hot(tv, oracle_mod):
    case = gen.make_case(20, B=8, N=40, L=4, V=300, mode="sample", tree="random", max_depth=6,
                         with_attn=False)
    case.q_logits = case.p_logits.copy()
    g = run_sample(tv, case, 3, 0)
    o = oracle_mod.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, 1.0, 3, 0)
    compare(g, o, case.parent, case.V)
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
