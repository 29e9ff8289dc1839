"""Torch-tensor front end of libtreeverify (argument marshalling only)."""
from __future__ import annotations

from typing import Callable, Optional

import torch

from ._lib import TV_MAX_NODES, check, lib

__all__ = ["tree_build", "attn_verify", "accept_greedy", "accept_sample", "expand_gated",
           "expand_tree", "commit_path", "expected_accept", "build_spine_tree", "spine_ratio_update", "workspace", "attn_workspace_size", "attn_plan", "greedy_workspace_size",
           "sample_workspace_size", "expand_workspace_size"]

_workspaces: dict = {}


def workspace(name: str, nbytes: int, device: torch.device) -> torch.Tensor:
    """A zero-filled scratch buffer cached per (device, name), grown on demand.

    The library returns zero-filled workspaces zero-filled, so a cached buffer
    can be reused by the next call on the same stream."""
    key = (torch.device(device), name)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def attn_workspace_size(B, N, Hq, Hkv, D, Lcap) -> int:
    return int(lib.tv_attn_workspace_size(B, N, Hq, Hkv, D, Lcap))


def attn_plan(B, N, Hq, Hkv, D, Lcap) -> dict:
    """The launch plan tv_attn_verify takes for this shape on the current device."""
    import ctypes
    info = (ctypes.c_int32 * 4)()
    check("tv_attn_plan", lib.tv_attn_plan(B, N, Hq, Hkv, D, Lcap, info))
    return {"rows_per_cta": info[0], "node_tiles": info[1], "splits": info[2], "ctas": info[3]}


def greedy_workspace_size(B, N, V) -> int:
    return int(lib.tv_accept_greedy_workspace_size(B, N, V))


def sample_workspace_size(B, N, V) -> int:
    return int(lib.tv_accept_sample_workspace_size(B, N, V))


def expand_workspace_size(F, V) -> int:
    return int(lib.tv_expand_workspace_size(F, V))


# ---------------------------------------------------------------------------
def tree_build(parent: torch.Tensor, depth=None, anc_mask=None, status=None):
    """parent int32 [B, N] -> (depth int32 [B,N], anc_mask int64 [B,N,W], status int32 [B]).

    anc_mask holds the uint64 ancestor-or-self bitmasks (torch has no uint64;
    the bits are the same)."""
    _need(parent, "parent", torch.int32)
    B, N = parent.shape
    dev = parent.device
    W = (N + 63) // 64
    depth = torch.empty((B, N), dtype=torch.int32, device=dev) if depth is None else depth
    anc_mask = (torch.empty((B, N, W), dtype=torch.int64, device=dev)
                if anc_mask is None else anc_mask)
    status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
    _need(depth, "depth", torch.int32, (B, N), dev)
    _need(anc_mask, "anc_mask", torch.int64, (B, N, W), dev)
    _need(status, "status", torch.int32, (B,), dev)
    check("tv_tree_build", lib.tv_tree_build(parent.data_ptr(), B, N, depth.data_ptr(),
                                             anc_mask.data_ptr(), status.data_ptr(),
                                             _stream(dev)))
    return depth, anc_mask, status


def attn_verify(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kv_len: torch.Tensor,
                anc_mask: torch.Tensor, scale: float = 0.0, out=None, lse=None, status=None,
                want_lse: bool = True, ws: Optional[torch.Tensor] = None):
    """Tree-verify attention.  q bf16 [B,N,Hq,D]; k, v bf16 [B,Hkv,Lcap,D];
    kv_len int32 [B]; anc_mask int64 [B,N,W].  Returns (out, lse, status)."""
    _need(q, "q", torch.bfloat16)
    B, N, Hq, D = q.shape
    dev = q.device
    _need(k, "k", torch.bfloat16, device=dev)
    _, Hkv, Lcap, Dk = k.shape
    if k.shape[0] != B or Dk != D:
        raise ValueError("k must be [B, Hkv, Lcap, D]")
    _need(v, "v", torch.bfloat16, tuple(k.shape), dev)
    _need(kv_len, "kv_len", torch.int32, (B,), dev)
    _need(anc_mask, "anc_mask", torch.int64, (B, N, (N + 63) // 64), dev)
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if want_lse and lse is None:
        lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, N, Hq), dev)
    status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
    _need(status, "status", torch.int32, (B,), dev)
    need = attn_workspace_size(B, N, Hq, Hkv, D, Lcap)
    ws = workspace("attn", need, dev) if ws is None else ws
    check("tv_attn_verify", lib.tv_attn_verify(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), kv_len.data_ptr(), anc_mask.data_ptr(), B, N,
        Hq, Hkv, D, Lcap, float(scale), out.data_ptr(), _ptr(lse), status.data_ptr(),
        ws.data_ptr(), ws.numel(), _stream(dev)))
    return out, lse, status


def attn_verify_tree(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kv_len: torch.Tensor,
                     parent: torch.Tensor, scale: float = 0.0, out=None, lse=None, status=None,
                     depth=None, anc_mask=None, tree_status=None, want_lse: bool = True,
                     ws: Optional[torch.Tensor] = None):
    """Tree encoding and tree-verify attention in one call (one launch for
    trees of up to 64 nodes).  parent int32 [B,N]; q, k, v, kv_len as for
    attn_verify.  Returns (out, lse, status, depth, anc_mask, tree_status)."""
    _need(q, "q", torch.bfloat16)
    B, N, Hq, D = q.shape
    dev = q.device
    _need(k, "k", torch.bfloat16, device=dev)
    _, Hkv, Lcap, Dk = k.shape
    if k.shape[0] != B or Dk != D:
        raise ValueError("k must be [B, Hkv, Lcap, D]")
    _need(v, "v", torch.bfloat16, tuple(k.shape), dev)
    _need(kv_len, "kv_len", torch.int32, (B,), dev)
    _need(parent, "parent", torch.int32, (B, N), dev)
    W = (N + 63) // 64
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if want_lse and lse is None:
        lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, N, Hq), dev)
    status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
    depth = torch.empty((B, N), dtype=torch.int32, device=dev) if depth is None else depth
    anc_mask = (torch.empty((B, N, W), dtype=torch.int64, device=dev)
                if anc_mask is None else anc_mask)
    tree_status = torch.empty(B, dtype=torch.int32, device=dev) if tree_status is None else tree_status
    _need(status, "status", torch.int32, (B,), dev)
    _need(depth, "depth", torch.int32, (B, N), dev)
    _need(anc_mask, "anc_mask", torch.int64, (B, N, W), dev)
    _need(tree_status, "tree_status", torch.int32, (B,), dev)
    need = attn_workspace_size(B, N, Hq, Hkv, D, Lcap)
    ws = workspace("attn", need, dev) if ws is None else ws
    check("tv_attn_verify_tree", lib.tv_attn_verify_tree(
        parent.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), kv_len.data_ptr(), B, N,
        Hq, Hkv, D, Lcap, float(scale), out.data_ptr(), _ptr(lse), status.data_ptr(),
        depth.data_ptr(), anc_mask.data_ptr(), tree_status.data_ptr(), ws.data_ptr(), ws.numel(),
        _stream(dev)))
    return out, lse, status, depth, anc_mask, tree_status


def accept_greedy(logits: torch.Tensor, tokens: torch.Tensor, parent: torch.Tensor,
                  depth: torch.Tensor, outs: Optional[dict] = None,
                  ws: Optional[torch.Tensor] = None) -> dict:
    """Greedy acceptance.  logits float32 [B,N,V]; tokens, parent, depth int32 [B,N].
    Returns dict(argmax, accept_len, end_node, path, bonus, status)."""
    _need(logits, "logits", torch.float32)
    B, N, V = logits.shape
    dev = logits.device
    for name, t in (("tokens", tokens), ("parent", parent), ("depth", depth)):
        _need(t, name, torch.int32, (B, N), dev)
    if outs is None:
        outs = dict(argmax=torch.empty((B, N), dtype=torch.int32, device=dev),
                    accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                    end_node=torch.empty(B, dtype=torch.int32, device=dev),
                    path=torch.empty((B, N), dtype=torch.int32, device=dev),
                    bonus=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    ws = workspace("greedy", greedy_workspace_size(B, N, V), dev) if ws is None else ws
    check("tv_accept_greedy", lib.tv_accept_greedy(
        logits.data_ptr(), tokens.data_ptr(), parent.data_ptr(), depth.data_ptr(), B, N, V,
        outs["argmax"].data_ptr(), outs["accept_len"].data_ptr(), outs["end_node"].data_ptr(),
        outs["path"].data_ptr(), outs["bonus"].data_ptr(), outs["status"].data_ptr(),
        ws.data_ptr(), ws.numel(), _stream(dev)))
    return outs


def commit_path(k: torch.Tensor, v: torch.Tensor, kv_len: torch.Tensor, path: torch.Tensor,
                accept_len: torch.Tensor, new_kv_len: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None):
    """Move each sequence's accepted branch to consecutive cache slots, in place.

    k, v bf16 [B, Hkv, Lcap, D]; kv_len, accept_len int32 [B]; path int32 [B, N].
    Returns (new_kv_len int32 [B], status int32 [B])."""
    _need(k, "k", torch.bfloat16)
    B, Hkv, Lcap, D = k.shape
    dev = k.device
    _need(v, "v", torch.bfloat16, (B, Hkv, Lcap, D), dev)
    _need(path, "path", torch.int32, None, dev)
    if path.dim() != 2 or path.shape[0] != B:
        raise ValueError(f"path must have shape [B, N] with B = {B}")
    N = path.shape[1]
    _need(kv_len, "kv_len", torch.int32, (B,), dev)
    _need(accept_len, "accept_len", torch.int32, (B,), dev)
    new_kv_len = torch.empty(B, dtype=torch.int32, device=dev) if new_kv_len is None else new_kv_len
    status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
    check("tv_commit_path", lib.tv_commit_path(
        k.data_ptr(), v.data_ptr(), kv_len.data_ptr(), path.data_ptr(), accept_len.data_ptr(), B,
        N, Hkv, D, Lcap, new_kv_len.data_ptr(), status.data_ptr(), _stream(dev)))
    return new_kv_len, status


def expected_accept(parent: torch.Tensor, prob: torch.Tensor, score: Optional[torch.Tensor] = None,
                    expected: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """Node scores (products of draft probabilities along the path) and the
    expected acceptance length of each tree.  parent int32 [B, N]; prob float32
    [B, N].  Returns (score float32 [B, N], expected float32 [B], status int32 [B])."""
    _need(parent, "parent", torch.int32)
    B, N = parent.shape
    dev = parent.device
    _need(prob, "prob", torch.float32, (B, N), dev)
    score = torch.empty((B, N), dtype=torch.float32, device=dev) if score is None else score
    expected = torch.empty(B, dtype=torch.float32, device=dev) if expected is None else expected
    status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
    check("tv_expected_accept", lib.tv_expected_accept(
        parent.data_ptr(), prob.data_ptr(), B, N, score.data_ptr(), expected.data_ptr(),
        status.data_ptr(), _stream(dev)))
    return score, expected, status


def build_spine_tree(spine_tokens, branch_tokens, root_token: int, budget: int,
                     spine_ratio: float):
    """GOOSE spine tree on the host.  spine_tokens int32 [S]; branch_tokens
    int32 [Sb, K] (row j: branch candidates off spine node j, best first, -1
    ends a row).  Returns (parent, tokens) as int32 numpy arrays."""
    import numpy as np
    sp = np.ascontiguousarray(np.asarray(spine_tokens, dtype=np.int32).reshape(-1))
    br = np.asarray(branch_tokens, dtype=np.int32)
    br = np.ascontiguousarray(br if br.ndim == 2 else br.reshape(0, 0))
    parent = np.zeros(max(int(budget), 1), np.int32)
    tokens = np.zeros(max(int(budget), 1), np.int32)
    n = np.zeros(1, np.int32)
    check("tv_build_spine_tree", lib.tv_build_spine_tree(
        sp.ctypes.data if sp.size else None, sp.size, br.ctypes.data if br.size else None,
        br.shape[0], br.shape[1], int(root_token), int(budget), float(spine_ratio),
        parent.ctypes.data, tokens.ctypes.data, n.ctypes.data))
    return parent[:n[0]].copy(), tokens[:n[0]].copy()


def spine_ratio_update(ratio: float, observed_accept_rate: float, beta: float) -> float:
    """GOOSE's spine ratio: an exponential moving average of the observed
    acceptance rate of the spine, clamped to [0, 1]."""
    return float(lib.tv_spine_ratio_update(float(ratio), float(observed_accept_rate), float(beta)))


def accept_sample(p_logits: torch.Tensor, q_logits: torch.Tensor, tokens: torch.Tensor,
                  parent: torch.Tensor, depth: torch.Tensor, temperature: float, seed: int,
                  offset: int, outs: Optional[dict] = None,
                  ws: Optional[torch.Tensor] = None) -> dict:
    """Stochastic acceptance.  Returns dict(accept_len, end_node, path, out_token, status)."""
    _need(p_logits, "p_logits", torch.float32)
    B, N, V = p_logits.shape
    dev = p_logits.device
    _need(q_logits, "q_logits", torch.float32, (B, N, V), dev)
    for name, t in (("tokens", tokens), ("parent", parent), ("depth", depth)):
        _need(t, name, torch.int32, (B, N), dev)
    if outs is None:
        outs = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                    end_node=torch.empty(B, dtype=torch.int32, device=dev),
                    path=torch.empty((B, N), dtype=torch.int32, device=dev),
                    out_token=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    ws = workspace("sample", sample_workspace_size(B, N, V), dev) if ws is None else ws
    check("tv_accept_sample", lib.tv_accept_sample(
        p_logits.data_ptr(), q_logits.data_ptr(), tokens.data_ptr(), parent.data_ptr(),
        depth.data_ptr(), B, N, V, float(temperature), int(seed) & (2**64 - 1),
        int(offset) & (2**64 - 1), outs["accept_len"].data_ptr(), outs["end_node"].data_ptr(),
        outs["path"].data_ptr(), outs["out_token"].data_ptr(), outs["status"].data_ptr(),
        ws.data_ptr(), ws.numel(), _stream(dev)))
    return outs


def expand_gated(draft_logits: torch.Tensor, frontier_node: torch.Tensor,
                 frontier_logscore: torch.Tensor, layer: int, topk: int, alpha: float,
                 budget: int, tree_parent: torch.Tensor, tree_token: torch.Tensor,
                 tree_logscore: torch.Tensor, n_nodes: torch.Tensor,
                 ws: Optional[torch.Tensor] = None) -> None:
    """One TALON layer; appends to the tree_* tensors and bumps n_nodes (device int32[1])."""
    _need(draft_logits, "draft_logits", torch.float32)
    F, V = draft_logits.shape
    dev = draft_logits.device
    _need(frontier_node, "frontier_node", torch.int32, (F,), dev)
    _need(frontier_logscore, "frontier_logscore", torch.float32, (F,), dev)
    _need(tree_parent, "tree_parent", torch.int32, device=dev)
    _need(tree_token, "tree_token", torch.int32, device=dev)
    _need(tree_logscore, "tree_logscore", torch.float32, device=dev)
    _need(n_nodes, "n_nodes", torch.int32, (1,), dev)
    if min(tree_parent.numel(), tree_token.numel(), tree_logscore.numel()) < budget:
        raise ValueError("tree arrays must hold `budget` nodes")
    ws = workspace("expand", expand_workspace_size(F, V), dev) if ws is None else ws
    check("tv_expand_gated", lib.tv_expand_gated(
        draft_logits.data_ptr(), frontier_node.data_ptr(), frontier_logscore.data_ptr(), F, V,
        int(layer), int(topk), float(alpha), int(budget), tree_parent.data_ptr(),
        tree_token.data_ptr(), tree_logscore.data_ptr(), n_nodes.data_ptr(), ws.data_ptr(),
        ws.numel(), _stream(dev)))


def expand_topn(draft_logits: torch.Tensor, frontier_node: torch.Tensor,
                frontier_logscore: torch.Tensor, width: int, capacity: int,
                tree_parent: torch.Tensor, tree_token: torch.Tensor, tree_logscore: torch.Tensor,
                n_nodes: torch.Tensor, ws: Optional[torch.Tensor] = None) -> None:
    """One OPT-Tree layer: appends the `width` best children of the frontier
    to the tree_* tensors (length >= capacity) and bumps n_nodes (device int32[1])."""
    _need(draft_logits, "draft_logits", torch.float32)
    F, V = draft_logits.shape
    dev = draft_logits.device
    _need(frontier_node, "frontier_node", torch.int32, (F,), dev)
    _need(frontier_logscore, "frontier_logscore", torch.float32, (F,), dev)
    _need(tree_parent, "tree_parent", torch.int32, device=dev)
    _need(tree_token, "tree_token", torch.int32, device=dev)
    _need(tree_logscore, "tree_logscore", torch.float32, device=dev)
    _need(n_nodes, "n_nodes", torch.int32, (1,), dev)
    if min(tree_parent.numel(), tree_token.numel(), tree_logscore.numel()) < capacity:
        raise ValueError("tree arrays must hold `capacity` nodes")
    ws = workspace("expand", expand_workspace_size(F, V), dev) if ws is None else ws
    check("tv_expand_topn", lib.tv_expand_topn(
        draft_logits.data_ptr(), frontier_node.data_ptr(), frontier_logscore.data_ptr(), F, V,
        int(width), int(capacity), tree_parent.data_ptr(), tree_token.data_ptr(),
        tree_logscore.data_ptr(), n_nodes.data_ptr(), ws.data_ptr(), ws.numel(), _stream(dev)))


def select_topn(parent: torch.Tensor, token: torch.Tensor, logscore: torch.Tensor,
                n_nodes: torch.Tensor, n: int, out: Optional[dict] = None) -> dict:
    """OPT-Tree subtree selection over B candidate trees [B, M]: the n best
    nodes, renumbered.  Returns dict(parent, token, logscore, src [B, n],
    expected [B], status [B]) of device tensors (or fills `out`)."""
    _need(parent, "parent", torch.int32)
    B, M = parent.shape
    dev = parent.device
    _need(token, "token", torch.int32, (B, M), dev)
    _need(logscore, "logscore", torch.float32, (B, M), dev)
    _need(n_nodes, "n_nodes", torch.int32, (B,), dev)
    if out is None:
        out = dict(parent=torch.empty((B, n), dtype=torch.int32, device=dev),
                   token=torch.empty((B, n), dtype=torch.int32, device=dev),
                   logscore=torch.empty((B, n), dtype=torch.float32, device=dev),
                   src=torch.empty((B, n), dtype=torch.int32, device=dev),
                   expected=torch.empty(B, dtype=torch.float32, device=dev),
                   status=torch.empty(B, dtype=torch.int32, device=dev))
    check("tv_select_topn", lib.tv_select_topn(
        parent.data_ptr(), token.data_ptr(), logscore.data_ptr(), n_nodes.data_ptr(), B, M,
        int(n), out["parent"].data_ptr(), out["token"].data_ptr(), out["logscore"].data_ptr(),
        out["src"].data_ptr(), out["expected"].data_ptr(), out["status"].data_ptr(),
        _stream(dev)))
    return out


def opt_tree_layer_sizes(width: int, layers: int, V: int, capacity: int) -> list:
    """Frontier id ranges (lo, F) of an OPT-Tree growth from the root: layer l
    expands the nodes layer l - 1 added, and a layer adds min(width, F x V,
    capacity - nodes so far) nodes (tv_expand_topn).  Stops early when a layer
    would add nothing.  Host arithmetic only: no device value is read."""
    out = []
    lo, hi = 0, 1
    for _ in range(layers):
        k = min(width, (hi - lo) * V, capacity - hi)
        if k <= 0:
            break
        out.append((lo, hi - lo))
        lo, hi = hi, hi + k
    return out


def grow_opt_tree(draft_rows: Callable, root_key, child_key: Callable, width: int, layers: int,
                  n: int, device) -> dict:
    """Grow an OPT-Tree candidate tree of `layers` layers (the root's is
    layer 1) of `width` nodes each, calling the drafter between layers, then
    keep its n best nodes (OPT-Tree §3).  Layer sizes follow from width, V and
    the capacity, so the layers are enqueued without reading the device; the
    drafter's keys for the new nodes are read back once per layer.  Returns
    dict(parent, token, logscore, n (the candidate tree, cpu), selected
    (select_topn's output for the one tree, cpu))."""
    dev = torch.device(device)
    cap = 1 + width * layers
    par = torch.full((cap,), -1, dtype=torch.int32, device=dev)
    tok = torch.zeros(cap, dtype=torch.int32, device=dev)
    ls = torch.zeros(cap, dtype=torch.float32, device=dev)
    node_ids = torch.arange(cap, dtype=torch.int32, device=dev)
    n_dev = torch.ones(1, dtype=torch.int32, device=dev)
    keys = [root_key]
    m = 1
    sizes = None
    for li in range(layers):
        lo, F = (0, 1) if sizes is None else sizes[li]
        rows = torch.as_tensor(draft_rows(keys[lo:lo + F]), dtype=torch.float32).to(dev)
        rows = rows.contiguous()
        if sizes is None:   # the vocabulary is known once the drafter has answered
            sizes = opt_tree_layer_sizes(width, layers, rows.shape[1], cap)
            if not sizes:
                break
        expand_topn(rows, node_ids[lo:lo + F], ls[lo:lo + F], width, cap, par, tok, ls, n_dev)
        k = min(width, F * rows.shape[1], cap - m)
        new_par = par[m:m + k].cpu().tolist()
        new_tok = tok[m:m + k].cpu().tolist()
        for p, t in zip(new_par, new_tok):
            keys.append(child_key(keys[p], t))
        m += k
        if li + 1 >= len(sizes):
            break
    sel = select_topn(par[None, :m].contiguous(), tok[None, :m].contiguous(),
                      ls[None, :m].contiguous(), torch.tensor([m], dtype=torch.int32, device=dev),
                      n)
    return dict(parent=par[:m].cpu(), token=tok[:m].cpu(), logscore=ls[:m].cpu(), n=m,
                n_device=int(n_dev.item()), selected={k: v[0].cpu() for k, v in sel.items()})


def expand_tree(draft_rows: Callable, root_key, child_key: Callable, topk: int, alpha: float,
                budget: int, device, max_layers: int = 100000) -> dict:
    """Grow a TALON tree until the budget is spent (TALON §5.1), calling the
    drafter between layers.  draft_rows(keys) -> float32 [F, V] (host numpy or
    torch); root_key / child_key(key, token) name tree positions for the
    drafter.  One host round trip per layer (the new node count sizes the next
    frontier).  Returns dict(parent, token, logscore (cpu tensors), n, layers)."""
    dev = torch.device(device)
    par = torch.full((budget,), -1, dtype=torch.int32, device=dev)
    tok = torch.zeros(budget, dtype=torch.int32, device=dev)
    ls = torch.zeros(budget, dtype=torch.float32, device=dev)
    node_ids = torch.arange(budget, dtype=torch.int32, device=dev)
    n_dev = torch.ones(1, dtype=torch.int32, device=dev)
    keys = [root_key]
    n = 1
    lo, hi = 0, 1          # the frontier is always the id range [lo, hi)
    layer = 1
    while n < budget and hi > lo and layer <= max_layers:
        rows = draft_rows(keys[lo:hi])
        rows = torch.as_tensor(rows, dtype=torch.float32).to(dev).contiguous()
        expand_gated(rows, node_ids[lo:hi], ls[lo:hi], layer, topk, alpha, budget, par, tok, ls,
                     n_dev)
        n_new = int(n_dev.item())
        new_par = par[n:n_new].cpu().tolist()
        new_tok = tok[n:n_new].cpu().tolist()
        for p, t in zip(new_par, new_tok):
            keys.append(child_key(keys[p], t))
        lo, hi = n, n_new
        n = n_new
        layer += 1
    return dict(parent=par[:n].cpu(), token=tok[:n].cpu(), logscore=ls[:n].cpu(), n=n,
                layers=layer - 1)
