"""Loading libtreeverify.so and declaring its C signatures for ctypes."""
from __future__ import annotations

import ctypes
import os

from ._build import CHECKED_LIB_PATH, LIB_PATH

# TV_CHECKED=1 in the environment loads the bounds-checked build instead (same
# entry points; a failed index check is recorded, see tv_debug_check_take).
CHECKED = os.environ.get("TV_CHECKED", "0") not in ("", "0")
_PATH = CHECKED_LIB_PATH if CHECKED else LIB_PATH

TV_OK = 0
TV_ERR_INVALID_ARG = 1
TV_ERR_INVALID_TREE = 2
TV_ERR_UNSUPPORTED = 3
TV_ERR_CUDA = 4
TV_ERR_TIMEOUT = 5
TV_ERR_INVALID_TOKEN = 6
TV_ERR_WORKSPACE = 7
TV_MAX_NODES = 512
TV_WAIT_LIMIT_DEFAULT = -1


class TVError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


def library_path() -> str:
    return _PATH


if not os.path.exists(_PATH):
    raise ImportError(
        f"{os.path.basename(_PATH)} not found at {_PATH}; build it first "
        "(python -c 'import __graft_entry__ as g; g.build()' or "
        "python speculative_decoding_tree_tv_gb300/_build.py)")

lib = ctypes.CDLL(_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64

_SIGS = {
    "tv_status_string": (ctypes.c_char_p, [_I]),
    "tv_version": (_I, []),
    "tv_workspace_clear": (_I, [_P, _SZ, _P]),
    "tv_tree_build": (_I, [_P, _I, _I, _P, _P, _P, _P]),
    "tv_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "tv_attn_plan": (_I, [_I, _I, _I, _I, _I, _I, _P]),
    "tv_attn_verify": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _SZ,
                            _P]),
    "tv_accept_greedy_workspace_size": (_SZ, [_I, _I, _I]),
    "tv_accept_greedy": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tv_accept_sample_workspace_size": (_SZ, [_I, _I, _I]),
    "tv_accept_sample": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _F, _U64, _U64, _P, _P, _P, _P, _P,
                              _P, _SZ, _P]),
    "tv_expand_workspace_size": (_SZ, [_I, _I]),
    "tv_commit_path": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "tv_expected_accept": (_I, [_P, _P, _I, _I, _P, _P, _P, _P]),
    "tv_build_spine_tree": (_I, [_P, _I, _P, _I, _I, _I, _I, _F, _P, _P, _P]),
    "tv_spine_ratio_update": (_F, [_F, _F, _F]),
    "tv_expand_gated": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "tv_expand_topn": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "tv_select_topn": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "tv_debug_set_wait_limit": (_I, [ctypes.c_longlong]),
    "tv_checked_build": (_I, []),
    "tv_debug_check_take": (_I, [_P]),
    "tv_debug_check_selftest": (_I, [_P, _I, _I, _P]),
    "tv_attn_verify_tree": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P,
                                 _P, _P, _SZ, _P]),
}

for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def status_string(code: int) -> str:
    return lib.tv_status_string(int(code)).decode()


def version() -> int:
    return int(lib.tv_version())


def check(fn: str, code: int) -> None:
    if code != TV_OK:
        raise TVError(fn, code)


def check_take() -> int:
    """The first failed index check since the last call (checked build), as
    (source unit << 16) | line, or 0; clears it.  Synchronises the device."""
    site = ctypes.c_int32(0)
    rc = lib.tv_debug_check_take(ctypes.byref(site))
    if rc != TV_OK:
        raise TVError("tv_debug_check_take", rc)
    return int(site.value)
