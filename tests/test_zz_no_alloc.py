"""The allocation-free greedy acceptance entry point.

tv_accept_greedy_noalloc serves callers that cannot allocate device memory
where they run acceptance -- a serving loop whose memory was planned once at
start-up, a plug-in that is handed no allocator, a real-time path that must
not allocate.  It keeps its scratch in a fixed array inside the library
instead of a caller workspace.  This test calls it directly through the C ABI
three times in a row (different tree batches, so each call runs on whatever
the previous one left in the array; the third has 200-node trees and an odd
vocabulary, which take the shared-memory tree scan and the scalar-load
kernel) and checks every output against the workspace-taking
tv_accept_greedy on the same inputs and against the CPU oracle: acceptance
results are integers, so they must be identical.  It lives in a file of its
own that is collected last, and it needs nothing from the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import gen

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import speculative_decoding_tree_tv_gb300 as tv
    fn = tv.lib.tv_accept_greedy_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, P, I, I, I, P, P, P, P, P, P, P]
    fn.restype = ctypes.c_int
    return tv, fn


def _inputs(case, dev):
    t = dict(logits=torch.from_numpy(case.logits).to(dev),
             tokens=torch.from_numpy(case.tokens).to(dev),
             parent=torch.from_numpy(case.parent).to(dev))
    return t


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(oracle_mod):
    tv, fn = _noalloc_fn()
    dev = torch.device("cuda:0")
    cases = [gen.make_case(901, B=3, N=40, L=4, V=20000, tree="random", max_depth=9,
                           with_attn=False),
             gen.make_case(902, B=8, N=64, L=4, V=128256, tree="random", max_depth=8,
                           with_attn=False),
             gen.make_case(903, B=2, N=200, L=4, V=1001, tree="random", max_depth=20,
                           with_attn=False)]
    for case in cases:
        t = _inputs(case, dev)
        depth, _, _ = tv.tree_build(t["parent"])
        ref = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
        B, N, V = case.logits.shape
        out = {k: torch.full_like(v, -7) for k, v in ref.items()}
        stream = torch.cuda.current_stream(dev).cuda_stream
        rc = fn(t["logits"].data_ptr(), t["tokens"].data_ptr(), t["parent"].data_ptr(),
                depth.data_ptr(), B, N, V, out["argmax"].data_ptr(), out["accept_len"].data_ptr(),
                out["end_node"].data_ptr(), out["path"].data_ptr(), out["bonus"].data_ptr(),
                out["status"].data_ptr(), stream)
        assert rc == tv.TV_OK, tv.status_string(rc)
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(out[k], ref[k]), k
        assert int(ref["status"].abs().sum()) == 0
        og = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
        for k in ("argmax", "accept_len", "end_node", "path", "bonus", "status"):
            assert np.array_equal(out[k].cpu().numpy(), og[k]), k


def test_noalloc_rejects_sizes_beyond_its_array():
    tv, fn = _noalloc_fn()
    dummy = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first
    rc = fn(dummy, dummy, dummy, dummy, 200, 512, 1000, dummy, dummy, dummy, dummy, dummy, dummy,
            None)
    assert rc == tv.TV_ERR_UNSUPPORTED
