"""Failure detection on the GPU without a fault: every wait in the kernels is
bounded, and a wait that runs out is reported as TV_ERR_TIMEOUT in status[b]
while the kernel leaves with no copy in flight.  A test hook shortens the
reporting limit of tv_accept_greedy's chunk-copy waits to a single
non-blocking test, so the copies (just issued) are never found complete: every
sequence must report the timeout with its outputs cleared, and the workspace
must come back zero-filled, so that the next call with the regular limit is
exact again."""
import numpy as np
import pytest
import torch

from workloads import gen

from _gpu_util import case_tensors, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


# (B, N): one wave of CTAs with the warp scan (1 x 60: 600 items), and several
# waves with the warp scan (3 x 40) and the block scan (3 x 200)
@pytest.mark.parametrize("B,N", [(1, 60), (3, 40), (3, 200)])
def test_greedy_copy_wait_runs_out(tv, oracle_mod, B, N):
    case = gen.make_case(950 + N, B=B, N=N, L=4, V=128256, tree="random", max_depth=12,
                         with_attn=False)
    t = case_tensors(case)
    depth, _, _ = tv.tree_build(t["parent"])
    try:
        assert tv.lib.tv_debug_set_wait_limit(0) == tv.TV_OK
        res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
        torch.cuda.synchronize()
    finally:
        assert tv.lib.tv_debug_set_wait_limit(tv.TV_WAIT_LIMIT_DEFAULT) == tv.TV_OK
    assert (np_(res["status"]) == tv.TV_ERR_TIMEOUT).all()
    for k in ("accept_len", "end_node", "bonus"):
        assert (np_(res[k]) == -1).all(), k
    assert (np_(res["path"]) == -1).all()
    # regular limit again: the same workspace, an exact result
    res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
    torch.cuda.synchronize()
    og = oracle_mod.accept_greedy(case.logits, case.tokens, case.parent)
    for k in ("argmax", "accept_len", "end_node", "path", "bonus", "status"):
        assert np.array_equal(np_(res[k]), og[k]), k
