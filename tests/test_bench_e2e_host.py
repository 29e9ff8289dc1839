"""The end-to-end leg's packed host path (bench.py), on CPU: the step's inputs
packed in one host buffer must come out of the device buffer's views exactly
as the workload generated them (tree, tokens, kv_len, queries, the tree's
own K/V slots placed in the cache, target logits), and the acceptance
results must be read back in one contiguous copy.  Pinned memory, the CUDA
graph and the library calls need a GPU: here the "device" is the CPU, pinning
is the identity, the timed loop runs two steps, and the step is a stand-in
that checks what the API would be handed and writes known results."""
import numpy as np
import pytest
import torch

import bench
from workloads import gen


@pytest.mark.parametrize("make", [gen.config1, gen.config2], ids=["tiny", "llama3-8b-spine"])
def test_packed_inputs_reach_the_api_views_unchanged(monkeypatch, make):
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    case = make()
    B, N = case.B, case.N
    L = int(case.kv_len[0])
    dev = torch.device("cpu")
    sets, _ = bench.make_sets(case, torch, dev, 1 << 20)
    # the known results the stand-in step writes, as the library would
    gouts = dict(accept_len=torch.full((B,), 3, dtype=torch.int32),
                 end_node=torch.full((B,), 5, dtype=torch.int32),
                 path=torch.arange(B * N, dtype=torch.int32).view(B, N),
                 bonus=torch.full((B,), 77, dtype=torch.int32),
                 argmax=torch.zeros((B, N), dtype=torch.int32),
                 status=torch.zeros(B, dtype=torch.int32))
    steps_seen = []

    def step(es, outs):
        assert np.array_equal(es["parent"].numpy(), case.parent)
        assert np.array_equal(es["tokens"].numpy(), case.tokens)
        assert np.array_equal(es["kv_len"].numpy(), case.kv_len)
        assert es["q"].dtype == torch.bfloat16 and tuple(es["q"].shape) == tuple(case.q.shape)
        assert np.array_equal(es["q"].view(torch.int16).numpy(), case.q.view(np.int16))
        assert np.array_equal(es["logits"].numpy(), case.logits)
        for name, src in (("k", case.k), ("v", case.v)):
            got = es[name].view(torch.int16).numpy()[0, :, L:L + N]
            assert np.array_equal(got, src[0, :, L:L + N].view(np.int16)), name
        # each segment starts 256 bytes into the buffer's storage, which a
        # device allocation aligns at least that far
        for t in (es["parent"], es["tokens"], es["kv_len"], es["q"], es["logits"]):
            assert t.is_contiguous() and (t.storage_offset() * t.element_size()) % 256 == 0
        for k, v in gouts.items():
            outs[k].copy_(v)
        steps_seen.append(1)

    def two_steps(torch_, stream, e2e_step, M, steps):
        e2e_step(0)
        e2e_step(M - 1)
        return 1.0, 2, "cpu"

    monkeypatch.setattr(bench, "e2e_timed", two_steps)

    class Args:
        steps = 20

    r = bench.measure_e2e_packed(Args, torch, None, case, sets, step, gouts, None, dev)
    assert len(steps_seen) == 2
    inputs = (case.parent.nbytes + case.tokens.nbytes + case.kv_len.nbytes + case.q.nbytes
              + 2 * case.k[0, :, L:L + N].nbytes + case.logits.nbytes)
    assert inputs <= r["h2d_bytes_per_step"] < inputs + 7 * 256   # segment padding only
    assert r["d2h_bytes_per_step"] == 4 * (3 * B + B * N)
    assert r["copies_per_step"] == {"h2d": 1, "d2h": 1, "device_to_device": 2}
