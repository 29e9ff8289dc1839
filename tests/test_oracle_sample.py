"""Pins for the oracle's stochastic acceptance and its random numbers.

Speculative Decoding concept page, "The protocol" step 3: accept a draft
token with probability min(1, p/q), on rejection resample from (p - q)+;
the accepted sequence is distributed exactly as p (lossless).  On a tree the
children of a node are tested in turn against the running residual.

Pinned by
  * Philox4x64-10 against numpy's own Philox bit generator (a library
    implementation of the same published generator),
  * a chi-square test of losslessness over 10^6 trials on a 16-token vocab:
    the first emitted token follows p_root, and given that child c was
    accepted, the next emitted token follows p_c,
  * special cases: q = p accepts every first child; a one-hot target reduces
    to greedy acceptance; a zero draft probability always accepts.
"""
import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chi2

from workloads import gen

M64 = 2**64 - 1


def numpy_philox_block(ctr, key):
    """Philox4x64-10 of (ctr, key) through numpy (which increments its counter
    before producing a block, so start it one below)."""
    c = [int(x) for x in ctr]
    v = (c[0] | (c[1] << 64) | (c[2] << 128) | (c[3] << 192)) - 1
    v %= 2**256
    prev = np.array([(v >> (64 * i)) & M64 for i in range(4)], dtype=np.uint64)
    bg = np.random.Philox(counter=prev, key=np.array(key, dtype=np.uint64))
    return bg.random_raw(4)


def test_philox_matches_numpy(oracle_mod):
    r = gen.rng(31)
    cases = [([1, 0, 0, 0], [0, 0]), ([M64, M64, M64, M64], [M64, M64]),
             ([0, 1, 0, 0], [5, 0])]
    for _ in range(300):
        cases.append(([int(x) for x in r.integers(0, M64, 4, dtype=np.uint64, endpoint=True)],
                      [int(x) for x in r.integers(0, M64, 2, dtype=np.uint64, endpoint=True)]))
    for ctr, key in cases:
        assert oracle_mod.philox4x64_10(ctr, key).tolist() == \
            numpy_philox_block(ctr, key).tolist()


def test_draw_word_counter_layout(oracle_mod):
    seed, offset, b, node, purpose, ordinal = 0xDEADBEEF12345678, 77, 5, 13, 1, 3
    w = oracle_mod.draw_word(seed, offset, b, node, purpose, ordinal)
    expect = numpy_philox_block([offset, b, node, (purpose << 32) | ordinal], [seed, 0])[0]
    assert w == int(expect)


def test_uniformity_of_draw_words(oracle_mod):
    """Chi-square of the top 4 bits over 2^16 words (df 15)."""
    words = [oracle_mod.draw_word(1234, 0, b, 0, 0, 0) for b in range(1 << 16)]
    top = np.array([w >> 60 for w in words])
    counts = np.bincount(top, minlength=16)
    stat = ((counts - len(words) / 16) ** 2 / (len(words) / 16)).sum()
    assert stat < chi2.ppf(1 - 1e-3, 15)


# ---------------------------------------------------------------------------
# losslessness
# ---------------------------------------------------------------------------
V16 = 16
PARENT10 = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)   # 3 children, 2 each


def _draft_tokens(r, q_rows, parent, trials):
    """Children of node v drawn i.i.d. from q_v for every trial."""
    kids = gen.children_of(parent)
    tok = np.zeros((trials, len(parent)), np.int32)
    for v, ks in enumerate(kids):
        if not ks:
            continue
        cdf = np.cumsum(q_rows[v])
        u = r.random((trials, len(ks))) * cdf[-1]
        tok[:, ks] = np.minimum(np.searchsorted(cdf, u, side="right"), V16 - 1)
    return tok


def _chi2(counts, probs):
    expect = probs * counts.sum()
    return float(((counts - expect) ** 2 / expect).sum())


def run_trials(oracle_mod, lp, lq, parent, trials, seed, chunk=125000):
    N = len(parent)
    r = gen.rng(seed)
    q_rows = softmax(lq.astype(np.float64), axis=1)
    first, second_given_1 = [], []
    for start in range(0, trials, chunk):
        t = min(chunk, trials - start)
        tok = _draft_tokens(r, q_rows, parent, t)
        P = np.broadcast_to(lp, (t, N, V16)).copy()
        Q = np.broadcast_to(lq, (t, N, V16)).copy()
        res = oracle_mod.accept_sample(P, Q, tok, np.broadcast_to(parent, (t, N)).copy(), 1.0,
                                       seed, start)
        assert (res["status"] == 0).all()
        al, path, out = res["accept_len"], res["path"], res["out_token"]
        rows = np.arange(t)
        emitted1 = np.where(al >= 1, tok[rows, np.maximum(path[:, 1], 0)], out)
        first.append(emitted1)
        sel = path[:, 1] == 1
        e2 = np.where(al >= 2, tok[rows, np.maximum(path[:, 2], 0)], out)
        second_given_1.append(e2[sel])
    return np.concatenate(first), np.concatenate(second_given_1)


def test_lossless_chi_square_1e6(oracle_mod):
    r = gen.rng(32)
    lp = r.standard_normal((10, V16)).astype(np.float32)
    lq = (lp + r.normal(0, 1.0, (10, V16))).astype(np.float32)
    first, second = run_trials(oracle_mod, lp, lq, PARENT10, 1_000_000, seed=99)
    p = softmax(lp.astype(np.float64), axis=1)
    q = softmax(lq.astype(np.float64), axis=1)
    thr = chi2.ppf(1 - 1e-3, V16 - 1)
    c1 = np.bincount(first, minlength=V16)
    c2 = np.bincount(second, minlength=V16)
    assert _chi2(c1, p[0]) < thr
    assert len(second) > 100000
    assert _chi2(c2, p[1]) < thr
    # power: the same statistic rejects the draft distribution outright
    assert _chi2(c1, q[0]) > 100 * thr


def test_single_child_chain_lossless(oracle_mod):
    """A chain with one draft per step is the textbook Leviathan case."""
    r = gen.rng(33)
    parent = gen.chain_tree(4)
    lp = r.standard_normal((4, V16)).astype(np.float32)
    lq = (lp + r.normal(0, 1.5, (4, V16))).astype(np.float32)
    q_rows = softmax(lq.astype(np.float64), axis=1)
    trials = 400000
    tok = _draft_tokens(r, q_rows, parent, trials)
    res = oracle_mod.accept_sample(np.broadcast_to(lp, (trials, 4, V16)).copy(),
                                   np.broadcast_to(lq, (trials, 4, V16)).copy(), tok,
                                   np.broadcast_to(parent, (trials, 4)).copy(), 1.0, 7, 0)
    al, out = res["accept_len"], res["out_token"]
    first = np.where(al >= 1, tok[:, 1], out)
    p = softmax(lp.astype(np.float64), axis=1)
    assert _chi2(np.bincount(first, minlength=V16), p[0]) < chi2.ppf(1 - 1e-3, V16 - 1)


def test_temperature_scales_both_distributions(oracle_mod):
    r = gen.rng(34)
    T = 0.7
    lp = r.standard_normal((10, V16)).astype(np.float32)
    lq = (lp + r.normal(0, 1.0, (10, V16))).astype(np.float32)
    # softmax(l / T) is what must come out
    first, _ = run_trials(oracle_mod, (lp / np.float32(T)).astype(np.float32),
                          (lq / np.float32(T)).astype(np.float32), PARENT10, 200000, seed=5)
    p = softmax((lp / np.float32(T)).astype(np.float64), axis=1)
    assert _chi2(np.bincount(first, minlength=V16), p[0]) < chi2.ppf(1 - 1e-3, V16 - 1)
    # and the oracle's own temperature argument agrees decision for decision
    tok = _draft_tokens(r, softmax((lq / T).astype(np.float64), axis=1), PARENT10, 2000)
    P = np.broadcast_to(lp, (2000, 10, V16)).copy()
    Q = np.broadcast_to(lq, (2000, 10, V16)).copy()
    a = oracle_mod.accept_sample(P, Q, tok, np.broadcast_to(PARENT10, (2000, 10)).copy(), T, 3, 0)
    b = oracle_mod.accept_sample((P / np.float32(T)).astype(np.float32),
                                 (Q / np.float32(T)).astype(np.float32), tok,
                                 np.broadcast_to(PARENT10, (2000, 10)).copy(), 1.0, 3, 0)
    agree = (a["out_token"] == b["out_token"]) & (a["end_node"] == b["end_node"])
    assert agree.mean() > 0.999


# ---------------------------------------------------------------------------
# special cases
# ---------------------------------------------------------------------------
def test_q_equals_p_accepts_first_children(oracle_mod):
    case = gen.make_case(35, B=8, N=40, L=4, V=300, mode="sample", tree="random", max_depth=6,
                         with_attn=False)
    res = oracle_mod.accept_sample(case.p_logits, case.p_logits, case.tokens, case.parent, 1.0,
                                   11, 0)
    for b in range(case.B):
        kids = gen.children_of(case.parent[b])
        v = 0
        while kids[v]:
            v = kids[v][0]
        assert res["end_node"][b] == v


def test_one_hot_target_equals_greedy(oracle_mod):
    case = gen.make_case(36, B=6, N=30, L=4, V=200, mode="greedy", tree="random", max_depth=5,
                         with_attn=False)
    logits = case.logits.copy()
    top = logits.argmax(axis=2)
    onehot = np.full_like(logits, -30.0)
    np.put_along_axis(onehot, top[..., None], 30.0, axis=2)
    g = oracle_mod.accept_greedy(onehot, case.tokens, case.parent)
    s = oracle_mod.accept_sample(onehot, np.zeros_like(onehot), case.tokens, case.parent, 1.0,
                                 4, 0)
    assert s["end_node"].tolist() == g["end_node"].tolist()
    assert s["out_token"].tolist() == g["bonus"].tolist()
    assert s["path"].tolist() == g["path"].tolist()


def test_zero_draft_probability_accepts(oracle_mod):
    parent = np.array([[-1, 0]], np.int32)
    lp = np.zeros((1, 2, 8), np.float32)
    lq = np.zeros((1, 2, 8), np.float32)
    lq[0, 0, 5] = -2000.0          # q_root(5) underflows to 0
    tokens = np.array([[0, 5]], np.int32)
    for seed in range(20):
        res = oracle_mod.accept_sample(lp, lq, tokens, parent, 1.0, seed, 0)
        assert res["end_node"][0] == 1


def test_bad_inputs(oracle_mod):
    parent = np.array([[-1, 0], [-1, 5], [-1, 0]], np.int32)
    tokens = np.array([[0, 1], [0, 1], [0, 8]], np.int32)
    lp = np.zeros((3, 2, 8), np.float32)
    res = oracle_mod.accept_sample(lp, lp, tokens, parent, 1.0, 0, 0)
    assert res["status"].tolist() == [0, 2, 6]
    with pytest.raises(ValueError):
        oracle_mod.accept_sample(lp, lp, tokens, parent, 0.0, 0, 0)


def test_draw_margin_and_alternative_token(oracle_mod):
    """The final draw (concept page, "The protocol" step 3; inverse CDF in
    ascending token order) recomputed with numpy for root-only trees, where
    the draw is from p_root: the drawn token, its distance from the nearest
    cumulative boundary and the token on the other side of that boundary."""
    r = gen.rng(91)
    for trial in range(40):
        V = int(r.integers(2, 300))
        lp = r.standard_normal((1, 1, V)).astype(np.float32) * 2
        lp[0, 0, r.integers(0, V, 3)] = -np.inf if trial % 5 == 0 else lp[0, 0, 0]
        lq = lp.copy()
        o = oracle_mod.accept_sample(lp, lq, np.zeros((1, 1), np.int32),
                                     np.array([[-1]], np.int32), 1.0, 500 + trial, 0)
        p = np.exp(lp[0, 0].astype(np.float64) - np.logaddexp.reduce(lp[0, 0].astype(np.float64)))
        w = oracle_mod.draw_word(500 + trial, 0, 0, 0, oracle_mod.PURPOSE_SAMPLE, 0)
        u = (w >> 11) * 2.0 ** -53
        cum = np.cumsum(p)
        target = u * cum[-1]
        k = int(np.searchsorted(cum, target, side="right"))
        assert o["out_token"][0] == k
        lo = cum[k - 1] if k > 0 else 0.0
        margin = min(cum[k] - target, target - lo) / cum[-1]
        assert abs(o["margin_draw"][0] - margin) <= 1e-12
        pos = np.nonzero(p > 0)[0]
        if target - lo <= cum[k] - target:
            below = pos[pos < k]
            alt = int(below[-1]) if len(below) else -1
        else:
            above = pos[pos > k]
            alt = int(above[0]) if len(above) else -1
        assert o["draw_alt"][0] == alt


def test_margin_path_locates_each_accept_test(oracle_mod):
    """margin_path[b, d] is the smallest |u - r/q| / (r/q) over the accept
    tests made at the walk's node of depth d: recomputed for a chain, where
    each node has one child and r = p at every test."""
    r = gen.rng(92)
    N, V = 6, 40
    parent = np.arange(-1, N - 1, dtype=np.int32)[None]
    lp = r.standard_normal((1, N, V)).astype(np.float32)
    lq = (lp + r.normal(0, 1.0, (1, N, V))).astype(np.float32)
    tok = r.integers(0, V, (1, N)).astype(np.int32)
    o = oracle_mod.accept_sample(lp, lq, tok, parent, 1.0, 77, 3)
    sm = lambda x: np.exp(x - np.logaddexp.reduce(x))
    end = o["accept_len"][0]
    for d in range(N):
        if d > end or d == N - 1:
            assert np.isinf(o["margin_path"][0, d])
            continue
        p = sm(lp[0, d].astype(np.float64))
        q = sm(lq[0, d].astype(np.float64))
        x = tok[0, d + 1]
        u = (oracle_mod.draw_word(77, 3, 0, d, oracle_mod.PURPOSE_ACCEPT, 0) >> 11) * 2.0 ** -53
        ratio = p[x] / q[x]
        assert abs(o["margin_path"][0, d] - abs(u - ratio) / ratio) <= 1e-9 * max(1.0, ratio)
        assert (u < ratio) == (d < end)
