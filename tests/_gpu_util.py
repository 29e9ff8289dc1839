"""Helpers shared by the GPU parity tests: numpy <-> CUDA tensors and the
attention tolerance (bf16 inputs, fp32 accumulation, bf16 output against the
fp64 oracle: max-abs 3e-2 and relative L2 1e-2)."""
import numpy as np
import torch

from workloads import gen

ATTN_MAX_ABS = 3e-2
ATTN_REL_L2 = 1e-2


def dev():
    return torch.device("cuda:0")


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16, dtype=np.uint16).view(np.int16)).to(
        dev()).view(torch.bfloat16)


def bf16_np(t):
    """bf16 CUDA tensor -> float64 numpy."""
    u = t.view(torch.int16).cpu().numpy().view(np.uint16)
    return gen.f32_from_bf16(u).astype(np.float64)


def np_(t):
    return t.cpu().numpy()


def check_attn(out_gpu, ref, what=""):
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(out_gpu).all(), f"{what}: non-finite output"
    err = np.abs(out_gpu - ref)
    max_abs = float(err.max()) if err.size else 0.0
    rel_l2 = float(np.linalg.norm(out_gpu - ref) / max(np.linalg.norm(ref), 1e-30))
    assert max_abs <= ATTN_MAX_ABS, f"{what}: max-abs {max_abs:.3g}"
    assert rel_l2 <= ATTN_REL_L2, f"{what}: rel-L2 {rel_l2:.3g}"
    return max_abs, rel_l2


def case_tensors(case):
    """Upload a workloads.Case to the GPU."""
    t = dict(parent=i32(case.parent), tokens=i32(case.tokens), kv_len=i32(case.kv_len))
    if case.q is not None:
        t.update(q=bf16(case.q), k=bf16(case.k), v=bf16(case.v))
    if case.logits is not None:
        t["logits"] = f32(case.logits)
    if case.p_logits is not None:
        t["p_logits"] = f32(case.p_logits)
        t["q_logits"] = f32(case.q_logits)
    return t
