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
