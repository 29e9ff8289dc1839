"""The bench's algorithmic work (the numerators of its roofline fractions)
against the per-configuration figures derived independently in the
measurement plan: attention bytes 4·D·Hkv·Σ(L_b + N) + Q/O + mask, attention
flops 4·Hq·D per visible (query, key) pair, acceptance bytes 4·B·N·V + 12·B·N.
The expected values are that plan's printed figures (MB, GFLOP, rounded to
the digits shown), not recomputed here."""
import pytest

import bench
from workloads import gen

# config -> (attention MB, attention GFLOP, acceptance MB), as printed
PLAN = {
    "tiny": (lambda: gen.config1(), ("0.33", "0.0043", "0.064")),
    "llama3-8b spine": (lambda: gen.config2(), ("9.62", "2.021", "30.78")),
    "long context 16": (lambda: gen.config5(16, with_attn=False), ("134.5", "8.6", "8.2")),
    "long context 64": (lambda: gen.config5(64, with_attn=False), ("135.5", "34.4", "32.8")),
    "long context 256": (lambda: gen.config5(256, with_attn=False), ("139.5", "137.5", "131.3")),
    "long context 512": (lambda: gen.config5(512, with_attn=False), ("144.7", "274.9", "262.7")),
}


def close(got, printed):
    """got rounds to the printed figure: within half a unit of its last digit."""
    decimals = len(printed.split(".")[1]) if "." in printed else 0
    return abs(got - float(printed)) <= 0.5 * 10 ** -decimals + 1e-12


@pytest.mark.parametrize("name", sorted(PLAN))
def test_algorithmic_work_matches_the_plan(name):
    make, (attn_mb, gflop, acc_mb) = PLAN[name]
    case = make()
    nb = bench.algorithmic_bytes(case)
    assert close(nb["attn"] / 1e6, attn_mb), (nb["attn"], attn_mb)
    assert close(bench.attention_flops(case) / 1e9, gflop), (bench.attention_flops(case), gflop)
    assert close(nb["greedy"] / 1e6, acc_mb), (nb["greedy"], acc_mb)


def test_spine_visible_key_count():
    # the plan's count of visible (query, key) pairs at the spine shape
    case = gen.config2()
    assert bench.attention_flops(case) == 4 * 32 * 128 * 123346
