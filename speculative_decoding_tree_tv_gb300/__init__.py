"""speculative_decoding_tree_tv_gb300 -- Python binding of libtreeverify.

Thin ctypes wrappers over the C ABI declared in ``include/treeverify.h``.
Every function takes CUDA torch tensors, checks dtypes/shapes/devices,
allocates outputs and workspaces with torch, and calls the library on the
current CUDA stream.  All arithmetic runs in the library's kernels; there is
no CPU path.  Import fails loudly when the compiled library is missing.
"""
from ._lib import (  # noqa: F401
    TV_OK, TV_ERR_INVALID_ARG, TV_ERR_INVALID_TREE, TV_ERR_UNSUPPORTED, TV_ERR_CUDA,
    TV_ERR_TIMEOUT, TV_ERR_INVALID_TOKEN, TV_ERR_WORKSPACE, TV_MAX_NODES, TV_WAIT_LIMIT_DEFAULT,
    TVError, CHECKED,
    lib, library_path, status_string, version, check_take,
)
from .api import (  # noqa: F401
    tree_build, attn_verify, attn_verify_tree, accept_greedy, accept_sample, expand_gated, expand_tree, expand_topn, select_topn, grow_opt_tree, opt_tree_layer_sizes, commit_path, expected_accept, build_spine_tree, spine_ratio_update,
    workspace, attn_workspace_size, attn_plan, greedy_workspace_size, sample_workspace_size,
    expand_workspace_size,
)
