"""The C ABI: libtreeverify.so loads without a GPU, exports every function
declared in include/treeverify.h, and rejects bad host-side arguments before
launching anything (these calls never reach the GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treeverify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def tvlib():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_tree_tv_gb300 as tv
    return tv


def test_header_declares_the_five_steps():
    names = declared_functions()
    for f in ("tv_tree_build", "tv_attn_verify", "tv_accept_greedy", "tv_accept_sample",
              "tv_expand_gated"):
        assert f in names


def test_every_declared_symbol_is_exported(tvlib):
    lib = ctypes.CDLL(tvlib.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(tvlib):
    assert tvlib.status_string(0) == "TV_OK"
    assert tvlib.status_string(2) == "TV_ERR_INVALID_TREE"
    assert tvlib.status_string(99) == "TV_ERR_UNKNOWN"
    assert tvlib.version() >= 100


def test_workspace_sizes(tvlib):
    assert tvlib.greedy_workspace_size(1, 60, 128256) >= 60 * 8
    assert tvlib.sample_workspace_size(16, 64, 128256) == 0  # the walk keeps its state on chip
    assert tvlib.expand_workspace_size(511, 32000) >= 511 * 32000 * 8
    # a 2108-slot cache over 16 row tiles is split across CTAs: partials + stats
    ws = tvlib.attn_workspace_size(1, 60, 32, 8, 128, 2108)
    assert ws >= 2 * 16 * 128 * (128 * 2 + 8)
    # one 128-key tile cannot be split: no workspace
    assert tvlib.attn_workspace_size(1, 60, 32, 8, 128, 128) == 0


def test_host_side_argument_errors_launch_nothing(tvlib):
    lib = tvlib.lib
    dummy = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its checks first
    # N = 0, N > 512
    assert lib.tv_tree_build(dummy, 1, 0, dummy, dummy, dummy, None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_tree_build(dummy, 1, 513, dummy, dummy, dummy, None) == tvlib.TV_ERR_INVALID_ARG
    # B = 0 is a no-op
    assert lib.tv_tree_build(dummy, 0, 4, dummy, dummy, dummy, None) == tvlib.TV_OK
    # unsupported head_dim, Hq % Hkv != 0, negative scale
    args = [dummy] * 5
    assert lib.tv_attn_verify(*args, 1, 4, 8, 8, 96, 64, 0.0, dummy, None, None, dummy, 256,
                              None) == tvlib.TV_ERR_UNSUPPORTED
    assert lib.tv_attn_verify(*args, 1, 4, 8, 3, 64, 64, 0.0, dummy, None, None, dummy, 256,
                              None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_attn_verify(*args, 1, 4, 8, 8, 64, 64, -1.0, dummy, None, None, dummy, 256,
                              None) == tvlib.TV_ERR_INVALID_ARG
    # attention: a split key range needs the partials workspace
    assert lib.tv_attn_verify(*args, 1, 60, 32, 8, 128, 2108, 0.0, dummy, None, None, None, 0,
                              None) == tvlib.TV_ERR_WORKSPACE
    # greedy: workspace too small
    assert lib.tv_accept_greedy(dummy, dummy, dummy, dummy, 2, 8, 100, dummy, dummy, dummy,
                                dummy, dummy, dummy, dummy, 8, None) == tvlib.TV_ERR_WORKSPACE
    # sample: temperature 0
    assert lib.tv_accept_sample(dummy, dummy, dummy, dummy, dummy, 1, 4, 10, 0.0, 1, 0, dummy,
                                dummy, dummy, dummy, dummy, dummy, 1 << 20,
                                None) == tvlib.TV_ERR_INVALID_ARG
    # expand: layer 1 needs exactly one frontier row; alpha out of range
    assert lib.tv_expand_gated(dummy, dummy, dummy, 2, 10, 1, 3, 0.3, 20, dummy, dummy, dummy,
                               dummy, dummy, 1 << 20, None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_expand_gated(dummy, dummy, dummy, 2, 10, 2, 3, 1.5, 20, dummy, dummy, dummy,
                               dummy, dummy, 1 << 20, None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_expand_gated(dummy, dummy, dummy, 1, 10, 1, 3, 0.3, 5000, dummy, dummy, dummy,
                               dummy, dummy, 1 << 20, None) == tvlib.TV_ERR_UNSUPPORTED
    # commit: head_dim not a multiple of 8, N = 0, new_kv_len aliasing kv_len, misaligned cache
    other = ctypes.c_void_p(0x2000)
    assert lib.tv_commit_path(dummy, dummy, dummy, dummy, dummy, 1, 8, 2, 12, 64, other, dummy,
                              None) == tvlib.TV_ERR_UNSUPPORTED
    assert lib.tv_commit_path(dummy, dummy, dummy, dummy, dummy, 1, 0, 2, 64, 64, other, dummy,
                              None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_commit_path(dummy, dummy, dummy, dummy, dummy, 1, 8, 2, 64, 64, dummy, dummy,
                              None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_commit_path(ctypes.c_void_p(0x1008), dummy, dummy, dummy, dummy, 1, 8, 2, 64,
                              64, other, dummy, None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_commit_path(dummy, dummy, dummy, dummy, dummy, 0, 8, 2, 64, 64, other, dummy,
                              None) == tvlib.TV_OK


def test_opt_tree_host_side_errors(tvlib):
    lib = tvlib.lib
    d = ctypes.c_void_p(0x1000)
    ws = 1 << 30
    # width 0, capacity 0, width above 2048, F above 2048, F = 0, workspace too small
    assert lib.tv_expand_topn(d, d, d, 1, 10, 0, 8, d, d, d, d, d, ws, None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_expand_topn(d, d, d, 1, 10, 4, 0, d, d, d, d, d, ws, None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_expand_topn(d, d, d, 1, 10, 3000, 8, d, d, d, d, d, ws, None) == tvlib.TV_ERR_UNSUPPORTED
    assert lib.tv_expand_topn(d, d, d, 3000, 10, 4, 8, d, d, d, d, d, ws, None) == tvlib.TV_ERR_UNSUPPORTED
    assert lib.tv_expand_topn(d, d, d, 0, 10, 4, 8, d, d, d, d, d, ws, None) == tvlib.TV_OK
    assert lib.tv_expand_topn(d, d, d, 4, 1000, 4, 8, d, d, d, d, d, 64, None) == tvlib.TV_ERR_WORKSPACE
    # selection: M above 16384, n = 0, B = 0, a missing output
    assert lib.tv_select_topn(d, d, d, d, 1, 16385, 8, d, d, d, d, d, d, None) == tvlib.TV_ERR_UNSUPPORTED
    assert lib.tv_select_topn(d, d, d, d, 1, 100, 0, d, d, d, d, d, d, None) == tvlib.TV_ERR_INVALID_ARG
    assert lib.tv_select_topn(d, d, d, d, 0, 100, 8, d, d, d, d, d, d, None) == tvlib.TV_OK
    assert lib.tv_select_topn(d, d, d, d, 1, 100, 8, d, d, d, d, None, d, None) == tvlib.TV_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(tvlib):
    import torch
    parent = torch.tensor([[-1, 0]], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        tvlib.tree_build(parent)
    i32 = torch.zeros(4, dtype=torch.int32)
    f32 = torch.zeros(4, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        tvlib.expand_topn(torch.zeros((1, 8)), i32[:1], f32[:1], 2, 4, i32, i32, f32, i32[:1])
    with pytest.raises(ValueError, match="CUDA"):
        tvlib.select_topn(parent, parent, torch.zeros((1, 2)), i32[:1], 2)


# --------------------------------------------------------------- attention plan
# Host-only: the plan tv_attn_verify takes for the benchmark shapes (152 SMs,
# the GB300 count, which is also the fallback when no GPU can be queried).
PLAN_CASES = {
    # name: (B, N, Hq, Hkv, D, Lcap) -> (rows per CTA, node tiles, splits)
    "tiny": ((1, 16, 8, 8, 64, 144), (128, 1, 1)),
    "llama3-8b spine, 60 nodes": ((1, 60, 32, 8, 128, 2108), (128, 2, 9)),
    "TALON verify, 512 nodes": ((1, 512, 64, 8, 128, 4608), (256, 16, 1)),
    "ragged batch of 16": ((16, 64, 32, 8, 128, 8256), (128, 2, 1)),
    "long context, 256 nodes": ((1, 256, 32, 8, 128, 33024), (256, 4, 9)),
}


@pytest.mark.parametrize("name", sorted(PLAN_CASES))
def test_attention_plan_of_the_benchmark_shapes(tvlib, monkeypatch, name):
    monkeypatch.delenv("TV_ATTN_PLAN", raising=False)
    shape, (rows, tiles, splits) = PLAN_CASES[name]
    plan = tvlib.attn_plan(*shape)
    assert (plan["rows_per_cta"], plan["node_tiles"], plan["splits"]) == (rows, tiles, splits)
    B, N, Hq, Hkv, D, Lcap = shape
    assert plan["ctas"] == B * Hkv * tiles * splits
    # a workspace exactly when the key range is split
    assert (tvlib.attn_workspace_size(*shape) > 0) == (splits > 1)


def test_attention_plan_override(tvlib, monkeypatch):
    shape = (1, 60, 32, 8, 128, 2108)  # 17 key tiles
    monkeypatch.setenv("TV_ATTN_PLAN", "256,3")
    assert tvlib.attn_plan(*shape) == {"rows_per_cta": 256, "node_tiles": 1, "splits": 3,
                                       "ctas": 24}
    assert tvlib.attn_workspace_size(*shape) == 3 * 8 * 256 * 128 * 2 + 3 * 8 * 256 * 8
    for bad in ("256,18", "64,2", "128,0", "junk", "128"):  # ignored: the model decides
        monkeypatch.setenv("TV_ATTN_PLAN", bad)
        assert tvlib.attn_plan(*shape)["splits"] == 9
    monkeypatch.delenv("TV_ATTN_PLAN")
    with pytest.raises(tvlib.TVError):
        tvlib.attn_plan(0, 60, 32, 8, 128, 2108)
    with pytest.raises(tvlib.TVError):
        tvlib.attn_plan(1, 60, 32, 8, 96, 2108)


def test_wait_limit_hook_rejects_bad_values(tvlib):
    """Other negative limits are refused on the host, before any device access."""
    assert tvlib.lib.tv_debug_set_wait_limit(-5) == tvlib.TV_ERR_INVALID_ARG


def test_checked_build_exports_every_symbol(tvlib):
    """The bounds-checked twin exports the same entry points and says which
    build it is; its debug calls refuse bad arguments on the host."""
    from speculative_decoding_tree_tv_gb300._build import CHECKED_LIB_PATH, LIB_PATH
    checked = ctypes.CDLL(CHECKED_LIB_PATH)
    regular = ctypes.CDLL(LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(checked, n)]
    assert not missing, missing
    assert checked.tv_checked_build() == 1
    assert regular.tv_checked_build() == 0
    for lib in (checked, regular):
        lib.tv_debug_check_take.argtypes = [ctypes.c_void_p]
        assert lib.tv_debug_check_take(None) == tvlib.TV_ERR_INVALID_ARG
        lib.tv_debug_check_selftest.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_void_p]
        assert lib.tv_debug_check_selftest(None, 4, 2, None) == tvlib.TV_ERR_INVALID_ARG
        assert lib.tv_debug_check_selftest(ctypes.c_void_p(0x1000), -1, 2, None) == \
            tvlib.TV_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    """A copy of the binding without its built library refuses to import, with
    the build command in the message: there is no fallback to run instead."""
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "speculative_decoding_tree_tv_gb300")
    shutil.copytree(pkg, tmp_path / "speculative_decoding_tree_tv_gb300",
                    ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__", "csrc"))
    r = subprocess.run([sys.executable, "-c", "import speculative_decoding_tree_tv_gb300"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=300,
                       env={**os.environ, "PYTHONPATH": str(tmp_path), "TV_CHECKED": "0"})
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libtreeverify.so not found" in r.stderr
