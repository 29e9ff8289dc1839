#!/usr/bin/env python
"""Tree-verify step throughput on GB300.

One step = one pass of the verify hot path over one synthetic draft tree:
the tree encoding and one attention layer over the KV prefix plus the tree
(tv_attn_verify_tree: tv_tree_build and tv_attn_verify in one launch for
trees of up to 64 nodes) -> tv_accept_greedy (argmax over every node's
vocabulary row and the longest matching branch).  Workload: Llama-3-8B-shaped GOOSE spine tree
(batch 1, KV prefix 2048, 32 query / 8 KV heads, head_dim 128, 60 nodes,
vocab 128256).

Timing: W warm-up steps, then exactly K steps replayed from CUDA graphs,
bracketed by a barrier and cudaDeviceSynchronize, timed with CUDA events on
the launching stream.  Steps rotate over input sets whose total size is at
least 3x the L2 cache, so every step reads HBM.  Under torchrun each rank runs
an independent replica (the path needs no exchange between GPUs) and the
slowest rank's time is reported.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tree-verify steps/s & achieved HBM GB/s (Llama-3-8B shape, 60-node tree)"
UNIT = "steps/s"
WORKLOAD = ("llama3-8b-spine60-L2048: batch 1, KV prefix 2048, 32 q / 8 kv heads, head_dim 128, "
            "bf16 Q/K/V; 60-node GOOSE spine tree; fp32 target logits over vocab 128256; "
            "greedy acceptance")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100000)
    p.add_argument("--warmup", type=int, default=1000)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--graph-steps", type=int, default=200)
    p.add_argument("--no-configs", action="store_true",
                   help="skip the secondary measurements on the other configurations")
    p.add_argument("--ncu-steps", type=int, default=0,
                   help="profiling driver: run this many eager steps of the workload on "
                        "one input set (no graphs, no timing) and exit; for ncu captures")
    p.add_argument("--ncu-workload", default="verify",
                   choices=["verify", "opt_tree", "talon_verify", "long_context", "batched_small",
                            "talon_expand"],
                   help="what --ncu-steps runs: the verify step (Llama-3-8B spine), one OPT-Tree "
                        "growth (16 layers of width 256 over vocab 128256, then the selection), "
                        "the TALON verify step (512 nodes, 64/8 heads, prefix 4096), the "
                        "long-context step (256 nodes, prefix 32768), the batched stochastic "
                        "step on its first 4 sequences, or one TALON growth (vocab 32000)")
    return p.parse_args()


# ----------------------------------------------------------------------------
# environment helpers
# ----------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# entry point, from the ncu captures summarised under profiles/.  A figure is
# reported only while the kernel sources hash to the value recorded when the
# counters were taken; after any change to them it is null until re-captured.
KERNEL_SOURCES = {
    "tv_tree_build": ["tv_tree.cu", "tv_common.cuh"],
    "tv_attn_verify": ["tv_attn.cu", "tv_sm100.cuh", "tv_common.cuh"],
    "tv_attn_verify_tree": ["tv_attn.cu", "tv_sm100.cuh", "tv_common.cuh"],
    "tv_accept_greedy": ["tv_greedy.cu", "tv_sm100.cuh", "tv_common.cuh"],
}
NCU_TRAFFIC = {
    # attention kernel with the tree encoding, cold (9,198,848) + merge kernel
    # with the L2 as the step leaves it (0 + 165,376)
    "tv_attn_verify_tree": {"sha256": "0316274025701df97e9f535d1f7d7a65c7f1603c3b4a8860453db587d5c455be", "bytes": 9364224,
                            "profile": "profiles/attn_verify_tree_llama3-8b-spine60.md"},
    "tv_accept_greedy": {"sha256": "76c77e809430f25b2b72d1ee6af89e42c4c43d851e632172ac898ffa9450de7b", "bytes": 30825216,
                         "profile": "profiles/greedy_bulk_kernel_llama3-8b-spine60.md"},
}


def slowest_rank_ms(elapsed_ms, dist, device):
    """The job's time: the maximum of the replicas' times (every rank gets it)."""
    if dist is None:
        return float(elapsed_ms)
    import torch
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(steps_per_rank, world, slowest_ms):
    """Whole-job steps/s: each of the `world` replicas runs its own steps, and
    the job lasts as long as the slowest one (weak scaling)."""
    return steps_per_rank * world / (slowest_ms / 1e3)


def sources_sha256(name):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[name]:
        with open(os.path.join(ROOT, "speculative_decoding_tree_tv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_traffic(name):
    rec = NCU_TRAFFIC.get(name)
    if rec is None or rec["sha256"] != sources_sha256(name):
        return None
    return rec["bytes"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background (200 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), util=float(parts[4]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["util"] > 0] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_busy": len(busy)}


# ----------------------------------------------------------------------------
# workload
# ----------------------------------------------------------------------------
def algorithmic_bytes(case):
    """Bytes each kernel must move at minimum (one launch), per the step's
    definition: K and V of every visible key once, Q and O once, the mask
    once; every logit once plus the small per-node integer arrays."""
    B, N, Hq, Hkv, D, V = case.B, case.N, case.Hq, case.Hkv, case.D, case.V
    W = (N + 63) // 64
    keys = int(np.sum(case.kv_len.astype(np.int64) + N))
    attn = 4 * D * Hkv * keys + 4 * B * N * Hq * D + 8 * B * N * W
    greedy = 4 * B * N * V + 12 * B * N
    tree = 4 * B * N + 4 * B * N + 8 * B * N * W
    return dict(tree=tree, attn=attn, greedy=greedy)


def attention_flops(case):
    """4 * Hq * D per visible (query, key) pair: prefix plus ancestors-or-self."""
    from workloads import gen
    tot = 0
    for b in range(case.B):
        d = gen.depth_of(case.parent[b])
        tot += int(np.sum(case.kv_len[b] + d + 1))
    return 4 * case.Hq * case.D * tot


def make_sets(case, torch, device, l2_bytes):
    def bf16(u):
        return torch.from_numpy(np.ascontiguousarray(u).view(np.int16)).to(device).view(
            torch.bfloat16)

    base = dict(
        parent=torch.from_numpy(case.parent).to(device),
        tokens=torch.from_numpy(case.tokens).to(device),
        kv_len=torch.from_numpy(case.kv_len).to(device),
        q=bf16(case.q), k=bf16(case.k), v=bf16(case.v),
        logits=torch.from_numpy(case.logits).to(device))
    set_bytes = sum(t.numel() * t.element_size() for t in base.values())
    M = max(2, int(np.ceil(3 * l2_bytes / set_bytes)))
    sets = [base] + [{k: t.clone() for k, t in base.items()} for _ in range(M - 1)]
    return sets, set_bytes


# ----------------------------------------------------------------------------
# the other configurations: every hot-path row measured on its own workload
# ----------------------------------------------------------------------------
def graph_time_us(torch, stream, fn, glen, reps):
    """Average time of one fn() call: a CUDA graph of glen calls, replayed
    reps times after one warm replay, CUDA events on the launching stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(glen):
            fn()
    with torch.cuda.stream(stream):
        g.replay()
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        z.record(stream)
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(z) * 1e3 / (reps * glen)


def measure_commit(torch, tv, stream, k, v, kv_len, path, accept_len, hbm):
    """tv_commit_path after the step's acceptance, on a copy of the cache:
    per-launch time and the bytes it must move (K and V of every accepted
    node that is not already in place, read and written, every kv head)."""
    kc, vc = k.clone(), v.clone()
    B, Hkv, Lcap, D = kc.shape
    new_len = torch.empty(B, dtype=torch.int32, device=kc.device)
    st = torch.empty_like(new_len)

    def f_commit():
        tv.commit_path(kc, vc, kv_len, path, accept_len, new_len, st)

    with torch.cuda.stream(stream):
        f_commit()
    torch.cuda.synchronize()
    assert int(st.max()) == 0
    pth, al = path.cpu().numpy(), accept_len.cpu().numpy()
    moved = int(sum(int(np.sum(pth[b, 1:al[b] + 1] != np.arange(1, al[b] + 1))) for b in range(B)))
    nbytes = 2 * 2 * D * 2 * Hkv * moved
    us = graph_time_us(torch, stream, f_commit, 20, 5)
    del kc, vc
    return {"us_per_launch": us, "moved_rows": moved, "bytes": nbytes,
            "roofline_us": nbytes / (hbm * 1e9) * 1e6, "frac": nbytes / (hbm * 1e9) * 1e6 / us,
            "bound": "latency (a few KB per launch)"}


def measure_verify_config(name, case, accept, torch, tv, device, stream, hbm, tflops, l2,
                          oracle_budget_s=0.0):
    """One verify step of a configuration: tree -> attention -> acceptance.
    The timed graphs cycle over enough copies of the inputs that the steps
    in flight read at least three times the L2 size, so every step reads HBM
    (one copy when a single step's inputs already exceed that)."""
    def bf16(u):
        return torch.from_numpy(np.ascontiguousarray(u).view(np.int16)).to(device).view(
            torch.bfloat16)

    B, N, V = case.B, case.N, case.V
    t = dict(parent=torch.from_numpy(case.parent).to(device),
             tokens=torch.from_numpy(case.tokens).to(device),
             kv_len=torch.from_numpy(case.kv_len).to(device),
             q=bf16(case.q), k=bf16(case.k), v=bf16(case.v))
    if accept == "greedy":
        t["logits"] = torch.from_numpy(case.logits).to(device)
    else:
        t["p"] = torch.from_numpy(case.p_logits).to(device)
        t["q_l"] = torch.from_numpy(case.q_logits).to(device)
    set_bytes = sum(x.numel() * x.element_size() for x in t.values())
    # enough copies to read 3x the L2 per cycle, at most 64 (a tiny workload
    # then stays in the L2, which its line says)
    M = min(64, max(1, int(np.ceil(3 * l2 / set_bytes))))
    sets = [t] + [{k: x.clone() for k, x in t.items()} for _ in range(M - 1)]
    cur = [0]   # the set the next call uses; advanced by each whole step

    def s_():
        return sets[cur[0] % M]
    W = (N + 63) // 64
    depth = torch.empty((B, N), dtype=torch.int32, device=device)
    anc = torch.empty((B, N, W), dtype=torch.int64, device=device)
    tst = torch.empty(B, dtype=torch.int32, device=device)
    out = torch.empty_like(t["q"])
    lse = torch.empty((B, N, case.Hq), dtype=torch.float32, device=device)
    ast = torch.empty(B, dtype=torch.int32, device=device)
    if accept == "greedy":
        aouts = dict(argmax=torch.empty((B, N), dtype=torch.int32, device=device),
                     accept_len=torch.empty(B, dtype=torch.int32, device=device),
                     end_node=torch.empty(B, dtype=torch.int32, device=device),
                     path=torch.empty((B, N), dtype=torch.int32, device=device),
                     bonus=torch.empty(B, dtype=torch.int32, device=device),
                     status=torch.empty(B, dtype=torch.int32, device=device))
    else:
        aouts = dict(accept_len=torch.empty(B, dtype=torch.int32, device=device),
                     end_node=torch.empty(B, dtype=torch.int32, device=device),
                     path=torch.empty((B, N), dtype=torch.int32, device=device),
                     out_token=torch.empty(B, dtype=torch.int32, device=device),
                     status=torch.empty(B, dtype=torch.int32, device=device))

    def f_tree(advance=True):
        tv.tree_build(s_()["parent"], depth, anc, tst)
        cur[0] += advance

    def f_attn(advance=True):
        x = s_()
        tv.attn_verify(x["q"], x["k"], x["v"], x["kv_len"], anc, out=out, lse=lse, status=ast)
        cur[0] += advance

    def f_acc(advance=True):
        x = s_()
        if accept == "greedy":
            tv.accept_greedy(x["logits"], x["tokens"], x["parent"], depth, outs=aouts)
        else:
            tv.accept_sample(x["p"], x["q_l"], x["tokens"], x["parent"], depth, 1.0, 1234, 0,
                             outs=aouts)
        cur[0] += advance

    def f_attn_tree(advance=True):
        x = s_()
        tv.attn_verify_tree(x["q"], x["k"], x["v"], x["kv_len"], x["parent"], out=out, lse=lse,
                            status=ast, depth=depth, anc_mask=anc, tree_status=tst)
        cur[0] += advance

    def f_step():
        f_attn_tree(False)
        f_acc(False)
        cur[0] += 1

    with torch.cuda.stream(stream):
        for _ in range(3):
            f_step()
    torch.cuda.synchronize()
    assert int(tst.max()) == 0 and int(ast.max()) == 0 and int(aouts["status"].max()) == 0
    glen = M * max(1, -(-20 // M))
    us = {k: graph_time_us(torch, stream, f, glen, 5)
          for k, f in (("step", f_step), ("tv_attn_verify_tree", f_attn_tree),
                       ("tv_tree_build", f_tree), ("tv_attn_verify", f_attn),
                       ("tv_accept_" + accept, f_acc))}
    commit = measure_commit(torch, tv, stream, t["k"], t["v"], t["kv_len"], aouts["path"],
                            aouts["accept_len"], hbm)
    nb = algorithmic_bytes(case)
    if accept == "greedy":
        acc_bytes = nb["greedy"]
    else:
        # the walk reads the p and q rows of the nodes it visits (the accepted
        # path, root included) and nothing else; rejections reuse the cached
        # rows, so the method's minimum is 8 V bytes per visited node
        visited = int((aouts["accept_len"].to(torch.int64) + 1).sum())
        acc_bytes = 8 * V * visited + 12 * B * N
    flops = attention_flops(case)
    t_attn = max(nb["attn"] / (hbm * 1e9), flops / (tflops * 1e12)) * 1e6
    t_acc = acc_bytes / (hbm * 1e9) * 1e6
    t_tree = nb["tree"] / (hbm * 1e9) * 1e6
    resident = set_bytes
    oracle_line = None
    if oracle_budget_s > 0:
        cores = os.cpu_count() or 1
        v_all, what = oracle_rate(case, accept, oracle_budget_s, cores)
        v_one, _ = oracle_rate(case, accept, oracle_budget_s, 1)
        oracle_line = {"steps_per_s": v_all, "cores": cores, "steps_per_s_1_thread": v_one,
                       "sample": what}
    return {
        "workload": name, "us_per_step": us["step"],
        "oracle": oracle_line,
        "us_per_launch": {k: v for k, v in us.items() if k != "step"},
        "roofline_step_us": t_attn + t_acc + t_tree,
        "roofline_step_frac": (t_attn + t_acc + t_tree) / us["step"],
        "attn": {"bound": "tensor" if flops / (tflops * 1e12) > nb["attn"] / (hbm * 1e9)
                 else "hbm", "bytes": nb["attn"], "flops": flops, "roofline_us": t_attn,
                 "frac": t_attn / us["tv_attn_verify"]},
        "accept": {"bound": "hbm", "bytes": acc_bytes, "roofline_us": t_acc,
                   **({} if accept == "greedy" else {"visited_nodes": visited}),
                   "frac": t_acc / us["tv_accept_" + accept]},
        "commit": commit,
        "inputs_resident_mb": resident / 1e6,
        "l2": (f"{M} rotating input sets of {resident / 1e6:.1f} MB" if M > 1 else
               f"one input set of {resident / 1e6:.0f} MB") +
              (f" (>= 3x the {l2 / 1e6:.0f} MB L2 per cycle of the timed graph)"
               if M * resident >= 3 * l2 else
               f" (L2-resident: {M * resident / 1e6:.1f} MB against the {l2 / 1e6:.0f} MB L2)"),
    }


def measure_talon_expansion(torch, tv, device, stream, hbm):
    """TALON workload (context 0): grow the tree once with the host drafter,
    recording each layer's draft rows, then time the whole device expansion
    (every layer's tv_expand_gated, from the root) replayed in one graph."""
    from workloads import gen
    K, alpha, budget = 10, 0.3, 512
    drafter = gen.config3_drafter(0)
    rec = []

    def rows_of(keys):
        r = drafter.rows(keys)
        rec.append(r)
        return r

    tree = tv.expand_tree(rows_of, drafter.root_key(), drafter.child_key, K, alpha, budget,
                          device)
    V = drafter.V
    dev_rows = [torch.from_numpy(r).to(device) for r in rec]
    F = [r.shape[0] for r in rec]
    par = torch.full((budget,), -1, dtype=torch.int32, device=device)
    tok = torch.zeros(budget, dtype=torch.int32, device=device)
    ls = torch.zeros(budget, dtype=torch.float32, device=device)
    ids = torch.arange(budget, dtype=torch.int32, device=device)
    n_dev = torch.ones(1, dtype=torch.int32, device=device)
    tv.workspace("expand", tv.expand_workspace_size(max(F), V), device)
    lo = [0]
    for f in F[:-1]:
        lo.append(lo[-1] + f)

    def f_expand():
        n_dev.fill_(1)
        for layer, (rows, l0, f) in enumerate(zip(dev_rows, lo, F), start=1):
            tv.expand_gated(rows, ids[l0:l0 + f], ls[l0:l0 + f], layer, K, alpha, budget, par,
                            tok, ls, n_dev)

    with torch.cuda.stream(stream):
        f_expand()
    torch.cuda.synchronize()
    assert int(n_dev.item()) == tree["n"]
    assert torch.equal(par[:tree["n"]].cpu(), tree["parent"])
    us = graph_time_us(torch, stream, f_expand, 5, 5)
    # the expanded tree's expected acceptance length (OPT-Tree's objective),
    # each node's draft probability exp(logscore - parent's logscore)
    n = tree["n"]
    par_d = par[:n].clone()[None]
    prob_d = torch.ones((1, n), dtype=torch.float32, device=device)
    prob_d[0, 1:] = torch.exp(ls[1:n] - ls[par[1:n].long()]).clamp(max=1.0)
    ex_out = tv.expected_accept(par_d, prob_d)
    torch.cuda.synchronize()
    us_ex = graph_time_us(torch, stream, lambda: tv.expected_accept(par_d, prob_d, *ex_out),
                          20, 5)
    # the method reads every frontier row's draft logits once (4 V bytes a row);
    # the kernels' second (filter) pass over a layer's rows hits the L2
    nbytes = sum(4 * f * V for f in F)
    return tree, {
        "workload": f"TALON context 0: K {K}, alpha {alpha}, budget {budget}, vocab {V}; "
                    f"{len(F)} layers, {tree['n']} nodes",
        "us_per_expansion": us, "layers": len(F), "frontier_rows": int(sum(F)),
        "bytes": nbytes, "roofline_us": nbytes / (hbm * 1e9) * 1e6,
        "frac": nbytes / (hbm * 1e9) * 1e6 / us,
        "expected_accept": {"us_per_launch": us_ex, "nodes": n,
                            "expected_accept_len": float(ex_out[1][0]),
                            "bound": "latency (one CTA, a few KB)"},
    }


def opt_tree_setup(torch, tv, device):
    """OPT-Tree growth at the long-context workload's shape: 16 layers of
    width 256 over a 128,256-token vocabulary (N(0, 3) draft rows, drawn once
    per layer and resident), then the 256 best nodes of the 4,097-node
    candidate tree.  The layer sizes follow from width, vocabulary and
    capacity, so nothing is read back between layers.  Returns the build and
    select closures and the state they work on."""
    width, layers, n_keep, V = 256, 16, 256, 128256
    cap = 1 + width * layers
    gen_t = torch.Generator(device=device)
    gen_t.manual_seed(5)
    sizes = tv.opt_tree_layer_sizes(width, layers, V, cap)
    lo, F = [a for a, _ in sizes], [f for _, f in sizes]
    rows = [torch.randn((f, V), generator=gen_t, device=device) * 3.0 for f in F]
    st = dict(width=width, layers=layers, n_keep=n_keep, V=V, cap=cap, F=F, rows=rows,
              par=torch.full((cap,), -1, dtype=torch.int32, device=device),
              tok=torch.zeros(cap, dtype=torch.int32, device=device),
              ls=torch.zeros(cap, dtype=torch.float32, device=device),
              ids=torch.arange(cap, dtype=torch.int32, device=device),
              n_dev=torch.ones(1, dtype=torch.int32, device=device),
              m_dev=torch.full((1,), cap, dtype=torch.int32, device=device))
    tv.workspace("expand", tv.expand_workspace_size(max(F), V), device)
    st["sel"] = tv.select_topn(st["par"][None], st["tok"][None], st["ls"][None], st["m_dev"],
                               n_keep)

    def f_select():
        tv.select_topn(st["par"][None], st["tok"][None], st["ls"][None], st["m_dev"], n_keep,
                       st["sel"])

    def f_build():
        st["n_dev"].fill_(1)
        for r_, l0, f in zip(rows, lo, F):
            tv.expand_topn(r_, st["ids"][l0:l0 + f], st["ls"][l0:l0 + f], width, cap, st["par"],
                           st["tok"], st["ls"], st["n_dev"])
        f_select()

    return f_build, f_select, st


def check_opt_tree(st):
    par, ls, ids = st["par"], st["ls"], st["ids"]
    assert int(st["n_dev"].item()) == st["cap"] and int(st["sel"]["status"][0]) == 0
    assert bool((par[1:] < ids[1:]).all()) and bool((ls[1:] <= ls[par[1:].long()]).all())


def measure_opt_tree(torch, tv, device, stream, hbm):
    """Times opt_tree_setup's growth, every launch from the root replayed in
    one graph, and the selection alone."""
    f_build, f_select, st = opt_tree_setup(torch, tv, device)
    with torch.cuda.stream(stream):
        f_build()
    torch.cuda.synchronize()
    check_opt_tree(st)
    us = graph_time_us(torch, stream, f_build, 5, 3)
    us_sel = graph_time_us(torch, stream, f_select, 20, 5)
    # the method reads every frontier row's draft logits once (4 V bytes a row)
    V, F = st["V"], st["F"]
    nbytes = sum(4 * f * V for f in F)
    out = {
        "workload": f"OPT-Tree growth: {st['layers']} layers of width {st['width']}, vocab {V}, "
                    f"N(0, 3) draft rows, then the {st['n_keep']} best of {st['cap']} nodes",
        "us_per_build": us, "layers": st["layers"], "frontier_rows": int(sum(F)),
        "bytes": nbytes, "roofline_us": nbytes / (hbm * 1e9) * 1e6,
        "frac": nbytes / (hbm * 1e9) * 1e6 / us,
        "select_topn": {"us_per_launch": us_sel, "nodes": st["cap"], "kept": st["n_keep"],
                        "expected_accept_len": float(st["sel"]["expected"][0]),
                        "bound": "latency (one CTA, 16 KB of keys)"},
    }
    del st
    return out


def measure_other_configs(torch, tv, device, hbm, tflops, oracle_budget_s=0.0):
    """Tiny, long context (greedy), batched stochastic acceptance, TALON
    expansion and its 512-node verify; with oracle_budget_s > 0 the oracle is
    timed beside each verify configuration."""
    from workloads import gen
    stream = torch.cuda.Stream(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    res = {}
    # GOOSE spine tree on the host (a 24-token context-matched spine, 8
    # transition candidates per position, 60 nodes), as a decode step builds it
    r = np.random.default_rng(3)
    spine = r.choice(case_vocab := 128256, 24, replace=False).astype(np.int32)
    branch = np.stack([r.choice(case_vocab, 8, replace=False) for _ in range(24)]).astype(np.int32)
    tv.build_spine_tree(spine, branch, 0, 60, 0.4)
    t0 = time.perf_counter()
    for _ in range(2000):
        sp_par, _ = tv.build_spine_tree(spine, branch, 0, 60, 0.4)
    res["spine_tree_build"] = {"workload": "GOOSE spine tree on the host: 24-token spine, 8 "
                               "candidates per position, budget 60, ratio 0.4",
                               "us_per_call": (time.perf_counter() - t0) / 2000 * 1e6,
                               "nodes": int(len(sp_par)), "where": "host CPU (Python call included)"}
    case = gen.config2()
    t = make_sets(case, torch, device, 0)[0][0]
    depth, _, _ = tv.tree_build(t["parent"])
    g = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
    res["spine_commit"] = dict(workload="tv_commit_path after greedy acceptance on the "
                               "Llama-3-8B spine step (8 kv heads, head_dim 128)",
                               **measure_commit(torch, tv, stream, t["k"], t["v"], t["kv_len"],
                                                g["path"], g["accept_len"], hbm))
    del t, g
    case = gen.config1()
    res["tiny"] = measure_verify_config(
        "tiny: prefix 128, 8/8 heads, head_dim 64, 16-node random tree, vocab 1000, greedy",
        case, "greedy", torch, tv, device, stream, hbm, tflops, l2, oracle_budget_s)
    del case
    case = gen.config5(256)
    res["long_context"] = measure_verify_config(
        "long context: prefix 32768, 32/8 heads, head_dim 128, 256-node OPT-Tree-style tree, "
        "vocab 128256, greedy", case, "greedy", torch, tv, device, stream, hbm, tflops, l2,
        oracle_budget_s)
    del case
    # the same workload's node-count sweep (16, 64 and 512 nodes; 256 is above)
    sweep = {}
    for n in (16, 64, 512):
        case = None
        try:
            case = gen.config5(n)
            r5 = measure_verify_config(
                f"long context, {n}-node tree", case, "greedy", torch, tv, device, stream, hbm,
                tflops, l2)
            sweep[str(n)] = {k: r5[k] for k in ("us_per_step", "us_per_launch",
                                                "roofline_step_us", "roofline_step_frac", "attn")}
        except Exception as e:  # recorded in the line rather than ending the run
            sweep[str(n)] = {"error": repr(e)[:200]}
        del case
    res["long_context_sweep"] = sweep
    case = gen.config4()
    res["batched_stochastic"] = measure_verify_config(
        "batched stochastic: 16 sequences, prefixes in [512, 8192], 64-node trees, 32/8 heads, "
        "head_dim 128, vocab 128256, p/q acceptance at T = 1", case, "sample", torch, tv, device,
        stream, hbm, tflops, l2, oracle_budget_s)
    del case
    res["opt_tree_growth"] = measure_opt_tree(torch, tv, device, stream, hbm)
    tree, res["talon_expansion"] = measure_talon_expansion(torch, tv, device, stream, hbm)
    case = gen.config3_verify(tree["parent"].numpy().astype(np.int32), 0,
                              tokens=tree["token"].numpy().astype(np.int32))
    res["talon_verify"] = measure_verify_config(
        f"TALON verify: prefix 4096, 64/8 heads, head_dim 128, the {case.N}-node expanded tree, "
        "vocab 32000, greedy", case, "greedy", torch, tv, device, stream, hbm, tflops, l2,
        oracle_budget_s)
    torch.cuda.synchronize()
    return res


# ----------------------------------------------------------------------------
# our implementation
# ----------------------------------------------------------------------------
def run_ncu_steps(args):
    """K eager steps (tree encoding + attention, then acceptance) on one input set, for ncu:
    each launch is a separate, serialised kernel there, so the per-launch
    counters of the same kernels as in the timed run can be read."""
    import torch
    import speculative_decoding_tree_tv_gb300 as tv
    from workloads import gen

    device = torch.device("cuda", 0)
    if args.ncu_workload in ("talon_verify", "long_context", "batched_small"):
        if args.ncu_workload == "talon_verify":
            d = gen.config3_drafter(0)
            tree = tv.expand_tree(d.rows, d.root_key(), d.child_key, 10, 0.3, 512, device)
            case = gen.config3_verify(tree["parent"].numpy().astype(np.int32), 0,
                                      tokens=tree["token"].numpy().astype(np.int32))
            accept = "greedy"
        elif args.ncu_workload == "long_context":
            case, accept = gen.config5(256), "greedy"
        else:
            case, accept = gen.config4(B=4), "sample"
        t = {"parent": torch.from_numpy(case.parent).to(device),
             "tokens": torch.from_numpy(case.tokens).to(device),
             "kv_len": torch.from_numpy(case.kv_len).to(device)}
        for k in ("q", "k", "v"):
            t[k] = torch.from_numpy(np.ascontiguousarray(getattr(case, k)).view(np.int16)).to(
                device).view(torch.bfloat16)
        for k in ("logits", "p_logits", "q_logits"):
            if getattr(case, k) is not None:
                t[k] = torch.from_numpy(getattr(case, k)).to(device)
        for _ in range(args.ncu_steps):
            out, lse, astat, depth, anc, tstat = tv.attn_verify_tree(
                t["q"], t["k"], t["v"], t["kv_len"], t["parent"])
            if accept == "greedy":
                res = tv.accept_greedy(t["logits"], t["tokens"], t["parent"], depth)
            else:
                res = tv.accept_sample(t["p_logits"], t["q_logits"], t["tokens"], t["parent"],
                                       depth, 1.0, 1234, 0)
        torch.cuda.synchronize()
        assert int(tstat.max()) == 0 and int(astat.max()) == 0 and int(res["status"].max()) == 0
        print(json.dumps({"ncu_steps": args.ncu_steps, "workload": args.ncu_workload}), flush=True)
        return
    if args.ncu_workload == "talon_expand":
        d = gen.config3_drafter(0)
        for _ in range(args.ncu_steps):
            tree = tv.expand_tree(d.rows, d.root_key(), d.child_key, 10, 0.3, 512, device)
        torch.cuda.synchronize()
        assert tree["n"] == 512
        print(json.dumps({"ncu_steps": args.ncu_steps, "workload": args.ncu_workload}), flush=True)
        return
    if args.ncu_workload == "opt_tree":
        f_build, _, st = opt_tree_setup(torch, tv, device)
        for _ in range(args.ncu_steps):
            f_build()
        torch.cuda.synchronize()
        check_opt_tree(st)
        print(json.dumps({"ncu_steps": args.ncu_steps, "workload": "opt_tree"}), flush=True)
        return
    case = gen.config2()
    s = make_sets(case, torch, device, 0)[0][0]
    for _ in range(args.ncu_steps):
        out, lse, astat, depth, anc, tstat = tv.attn_verify_tree(
            s["q"], s["k"], s["v"], s["kv_len"], s["parent"])
        res = tv.accept_greedy(s["logits"], s["tokens"], s["parent"], depth)
    torch.cuda.synchronize()
    assert int(tstat[0]) == 0 and int(astat[0]) == 0 and int(res["status"][0]) == 0
    print(json.dumps({"ncu_steps": args.ncu_steps, "workload": WORKLOAD}), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import speculative_decoding_tree_tv_gb300 as tv
    from workloads import gen

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    case = gen.config2()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    sets, set_bytes = make_sets(case, torch, device, l2)
    M = len(sets)
    B, N, Hq = case.B, case.N, case.Hq
    W = (N + 63) // 64
    depth = torch.empty((B, N), dtype=torch.int32, device=device)
    anc = torch.empty((B, N, W), dtype=torch.int64, device=device)
    tstat = torch.empty(B, dtype=torch.int32, device=device)
    out = torch.empty_like(sets[0]["q"])
    lse = torch.empty((B, N, Hq), dtype=torch.float32, device=device)
    astat = torch.empty(B, dtype=torch.int32, device=device)
    gouts = dict(argmax=torch.empty((B, N), dtype=torch.int32, device=device),
                 accept_len=torch.empty(B, dtype=torch.int32, device=device),
                 end_node=torch.empty(B, dtype=torch.int32, device=device),
                 path=torch.empty((B, N), dtype=torch.int32, device=device),
                 bonus=torch.empty(B, dtype=torch.int32, device=device),
                 status=torch.empty(B, dtype=torch.int32, device=device))

    def k_tree(s):
        tv.tree_build(s["parent"], depth, anc, tstat)

    def k_attn(s):
        tv.attn_verify(s["q"], s["k"], s["v"], s["kv_len"], anc, out=out, lse=lse, status=astat)

    def k_attn_tree(s):
        tv.attn_verify_tree(s["q"], s["k"], s["v"], s["kv_len"], s["parent"], out=out, lse=lse,
                            status=astat, depth=depth, anc_mask=anc, tree_status=tstat)

    def k_greedy(s, outs=None):
        tv.accept_greedy(s["logits"], s["tokens"], s["parent"], depth,
                         outs=gouts if outs is None else outs)

    def step(s, outs=None):
        k_attn_tree(s)
        k_greedy(s, outs)

    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(min(args.warmup, 3 * M)):     # eager warm-up: workspaces, sanity
            step(sets[i % M])
    torch.cuda.synchronize()
    assert int(gouts["status"][0]) == 0 and int(astat[0]) == 0

    def capture(fn, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(count):
                fn(sets[j % M])
        return g

    C = max(M, (args.graph_steps // M) * M)
    full_reps = args.steps // C
    rem = args.steps % C
    g_full = capture(step, C) if full_reps else None
    g_rem = capture(step, rem) if rem else None
    timed = [g for g in (g_rem, g_full) if g is not None]

    # warm-up: every graph the timed region replays is replayed here first (its
    # upload and first execution stay outside the timed region), then more
    # untimed replays until at least W steps ran through the graphs
    warm = 0
    with torch.cuda.stream(stream):
        for g in timed:
            g.replay()
            warm += C if g is g_full else rem
        while warm < args.warmup:
            timed[0].replay()
            warm += C if timed[0] is g_full else rem
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        # one more untimed replay ahead of the start event, so the timed graphs
        # are already queued behind busy work when the clock starts
        timed[0].replay()
        e0.record(stream)
        if g_rem is not None:
            g_rem.replay()
        for _ in range(full_reps):
            g_full.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    elapsed_ms = e0.elapsed_time(e1)
    clocks = sampler.stop()
    assert int(gouts["status"][0]) == 0
    elapsed_ms = slowest_rank_ms(elapsed_ms, dist, device)

    # per-kernel average launch time, each kernel replayed alone over the same rotation
    per_kernel = {}
    nk = min(args.steps, 20000)
    for name, fn in (("tv_attn_verify_tree", k_attn_tree), ("tv_accept_greedy", k_greedy),
                     ("tv_tree_build", k_tree), ("tv_attn_verify", k_attn)):
        g = capture(fn, C)
        with torch.cuda.stream(stream):
            g.replay()
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(max(1, nk // C)):
                g.replay()
            z.record(stream)
        torch.cuda.synchronize()
        per_kernel[name] = a.elapsed_time(z) * 1e3 / (max(1, nk // C) * C)   # us per launch
        del g

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, torch, tv, case, sets, step, gouts, stream, device)

    # tree encoding and attention (one launch up to 64 nodes; + the split-KV
    # merge when the plan splits), greedy
    launches = (2 + int(case.N > 64) +
                int(tv.attn_workspace_size(case.B, case.N, case.Hq, case.Hkv, case.D,
                                           case.Lcap) > 0))
    return dict(case=case, elapsed_ms=elapsed_ms, per_kernel=per_kernel, clocks=clocks, M=M,
                set_bytes=set_bytes, l2=l2, e2e=e2e, launches_per_step=launches)


def measure_e2e(args, torch, tv, case, sets, step, gouts, stream, device):
    """The e2e figure: packed host buffers (one copy in, one copy out per step);
    should that path fail, the per-tensor copies below, with the reason."""
    try:
        return measure_e2e_packed(args, torch, tv, case, sets, step, gouts, stream, device)
    except Exception as ex:  # pragma: no cover - reported in the JSON line
        torch.cuda.synchronize()
        r = measure_e2e_per_tensor(args, torch, tv, case, sets, step, gouts, stream, device)
        r["packed_error"] = f"{type(ex).__name__}: {ex}"[:200]
        return r


def e2e_timed(torch, stream, e2e_step, M, steps):
    """Steps of e2e_step(j) over the M input sets, replayed from a CUDA graph
    (eager if capture fails); returns (ms, steps, mode)."""
    mode = "graph"
    try:
        C = M * max(1, 50 // M)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(C):
                e2e_step(j % M)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // C)
        steps = reps * C
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                g.replay()
            z.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(z)
        del g
    except Exception:
        mode = "eager"
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for j in range(3):
                e2e_step(j % M)
            a.record(stream)
            for j in range(steps):
                e2e_step(j % M)
            z.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(z)
    return ms, steps, mode


def measure_e2e_packed(args, torch, tv, case, sets, step, gouts, stream, device):
    """Same step through the public API, its inputs packed in one pinned host
    buffer (tree, tokens, kv_len, queries, the tree's own K/V slots, target
    logits, each segment 256-byte aligned): every step copies that buffer
    host->device in one copy into a device buffer the API reads through views,
    places the tree's K/V slots in the cache (two device-side copies), runs the
    step, and reads the acceptance result (accept_len, end_node, bonus, path,
    contiguous) back in one copy.  The KV prefix stays resident in HBM."""
    B, N = case.B, case.N
    L = int(case.kv_len[0])
    segs = [("parent", np.ascontiguousarray(case.parent), torch.int32),
            ("tokens", np.ascontiguousarray(case.tokens), torch.int32),
            ("kv_len", np.ascontiguousarray(case.kv_len), torch.int32),
            ("q", np.ascontiguousarray(case.q).view(np.int16), torch.int16),
            ("ktree", np.ascontiguousarray(case.k[0, :, L:L + N]).view(np.int16), torch.int16),
            ("vtree", np.ascontiguousarray(case.v[0, :, L:L + N]).view(np.int16), torch.int16),
            ("logits", np.ascontiguousarray(case.logits), torch.float32)]
    offs, o = {}, 0
    for name, a, _ in segs:
        offs[name] = o
        o = (o + a.nbytes + 255) // 256 * 256
    total = o
    hbuf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    hnp = hbuf.numpy()
    for name, a, _ in segs:
        hnp[offs[name]:offs[name] + a.nbytes] = a.reshape(-1).view(np.uint8)

    def views(buf):
        return {name: buf[offs[name]:offs[name] + a.nbytes].view(dt).view(a.shape)
                for name, a, dt in segs}

    M = len(sets)
    dbufs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(M)]
    dviews = [views(b) for b in dbufs]
    esets = [dict(parent=dv["parent"], tokens=dv["tokens"], kv_len=dv["kv_len"],
                  q=dv["q"].view(torch.bfloat16), k=s["k"], v=s["v"], logits=dv["logits"])
             for s, dv in zip(sets, dviews)]
    # results first, in the order they are read back, then what stays on the device
    res = torch.empty(3 * B + 2 * B * N + B, dtype=torch.int32, device=device)
    nres = 3 * B + B * N
    outs = dict(accept_len=res[0:B], end_node=res[B:2 * B], bonus=res[2 * B:3 * B],
                path=res[3 * B:nres].view(B, N), argmax=res[nres:nres + B * N].view(B, N),
                status=res[nres + B * N:])
    hres = torch.empty(nres, dtype=torch.int32).pin_memory()

    def e2e_step(j):
        dbufs[j].copy_(hbuf, non_blocking=True)
        es = esets[j]
        es["k"].view(torch.int16)[0, :, L:L + N].copy_(dviews[j]["ktree"], non_blocking=True)
        es["v"].view(torch.int16)[0, :, L:L + N].copy_(dviews[j]["vtree"], non_blocking=True)
        step(es, outs)
        hres.copy_(res[:nres], non_blocking=True)

    ms, steps, mode = e2e_timed(torch, stream, e2e_step, M, min(args.steps, 2000))
    got = hres.clone()
    assert int(got[0]) == int(gouts["accept_len"][0]) and int(got[2 * B]) == int(gouts["bonus"][0])
    assert torch.equal(got[3 * B:nres].view(B, N), gouts["path"].cpu())
    return {"value": steps / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(total),
            "d2h_bytes_per_step": int(nres * 4), "steps": steps, "mode": mode,
            "copies_per_step": {"h2d": 1, "d2h": 1, "device_to_device": 2}}


def measure_e2e_per_tensor(args, torch, tv, case, sets, step, gouts, stream, device):
    """Same step through the public API from pinned host buffers: every step
    copies its inputs host->device (tree, tokens, queries, the tree's own K/V
    slots, target logits) and reads the acceptance result back."""
    B, N, Hkv = case.B, case.N, case.Hkv
    L = int(case.kv_len[0])
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h = dict(parent=pin(case.parent), tokens=pin(case.tokens), kv_len=pin(case.kv_len),
             q=pin(case.q.view(np.int16)), logits=pin(case.logits),
             ktree=pin(case.k[0, :, L:L + N].view(np.int16)),
             vtree=pin(case.v[0, :, L:L + N].view(np.int16)))
    hout = {k: torch.empty_like(gouts[k], device="cpu").pin_memory()
            for k in ("accept_len", "end_node", "path", "bonus")}
    M = len(sets)
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in hout.values())

    def e2e_step(s):
        s["parent"].copy_(h["parent"], non_blocking=True)
        s["tokens"].copy_(h["tokens"], non_blocking=True)
        s["kv_len"].copy_(h["kv_len"], non_blocking=True)
        s["q"].view(torch.int16).copy_(h["q"], non_blocking=True)
        s["logits"].copy_(h["logits"], non_blocking=True)
        kv16 = s["k"].view(torch.int16)
        vv16 = s["v"].view(torch.int16)
        for kvh in range(Hkv):
            kv16[0, kvh, L:L + N].copy_(h["ktree"][kvh], non_blocking=True)
            vv16[0, kvh, L:L + N].copy_(h["vtree"][kvh], non_blocking=True)
        step(s)
        for k in hout:
            hout[k].copy_(gouts[k], non_blocking=True)

    ms, steps, mode = e2e_timed(torch, stream, lambda j: e2e_step(sets[j]), M,
                                min(args.steps, 2000))
    assert int(hout["accept_len"][0]) == int(gouts["accept_len"][0])
    return {"value": steps / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "mode": mode}


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------
def oracle_step_sample(case, rows_attn, rows_greedy, rng):
    """One bounded sample of a step on the oracle: the tree encoding, the
    attention rows `rows_attn` of the (node, head) grid and the greedy
    acceptance over `rows_greedy` node rows (a whole tree when equal to N)."""
    import oracle
    oracle.tree_build(case.parent)
    if rows_attn:
        idx = rng.choice(case.N * case.Hq, size=rows_attn, replace=False)
        rows = np.stack([np.zeros(rows_attn, np.int64), idx // case.Hq, idx % case.Hq], axis=1)
        oracle.attn_rows(case.q, case.k, case.v, case.kv_len, case.parent, case.Hq, case.Hkv, rows)
    if rows_greedy >= case.N:
        oracle.accept_greedy(case.logits, case.tokens, case.parent)
    elif rows_greedy:
        # argmax rows only (the tree scan needs every row)
        oracle.accept_greedy(case.logits[:, :rows_greedy], case.tokens[:, :rows_greedy],
                             np.ascontiguousarray(case.parent[:, :rows_greedy]))


def cpu_model():
    """The host CPU's model name (lscpu), for the baseline's record."""
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                             text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def oracle_rate(case, accept, budget_s, threads, seed=0):
    """Oracle verify steps/s of a workload on `threads` host threads: tree
    encoding, attention rows, acceptance.  Whole steps when they fit the
    budget; otherwise a random sample of the attention rows, scaled to the
    whole step (the tree encoding and the acceptance are always whole).
    Returns (steps/s, description of the sample)."""
    import oracle
    oracle.build()
    oracle.set_threads(threads)
    rng = np.random.default_rng(seed)
    total_rows = case.B * case.N * case.Hq

    def accept_once():
        if accept == "greedy":
            oracle.accept_greedy(case.logits, case.tokens, case.parent)
        else:
            oracle.accept_sample(case.p_logits, case.q_logits, case.tokens, case.parent, 1.0,
                                 1234, 0)

    t0 = time.perf_counter()
    oracle.tree_build(case.parent)
    accept_once()
    t_fixed = time.perf_counter() - t0
    # probe the cost of a row, then size the sample to the budget
    probe = min(total_rows, max(threads, 8))

    def rows_time(k):
        idx = rng.choice(total_rows, size=k, replace=False)
        rows = np.stack([idx // (case.N * case.Hq), (idx // case.Hq) % case.N, idx % case.Hq],
                        axis=1)
        t1 = time.perf_counter()
        oracle.attn_rows(case.q, case.k, case.v, case.kv_len, case.parent, case.Hq, case.Hkv,
                         rows)
        return time.perf_counter() - t1

    t_probe = rows_time(probe) / probe
    k = int(min(total_rows, max(probe, (budget_s - t_fixed) / max(t_probe, 1e-9))))
    t_rows = rows_time(k)
    step_s = t_fixed + t_rows * total_rows / k
    what = ("whole step" if k == total_rows else
            f"{k} of {total_rows} attention rows scaled to the step") + \
        f", tree encoding and {accept} acceptance whole"
    oracle.set_threads(0)
    return 1.0 / step_s, what


def cpu_baseline(case, budget_s=8.0):
    """The oracle on the headline workload: all host cores (OpenMP over
    independent rows, the arithmetic unchanged) and one core."""
    cores = os.cpu_count() or 1
    v_all, what_all = oracle_rate(case, "greedy", budget_s, cores)
    v_one, what_one = oracle_rate(case, "greedy", budget_s, 1)
    return {"value": v_all, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{what_all} ({cores} threads); one thread: {v_one:.3g} steps/s "
                      f"({what_one}); CPU: {cpu_model()}",
            "single_thread": {"value": v_one, "cores": 1}, "cpu_model": cpu_model()}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each timed step is a bounded sample of
    the workload, scaled to whole steps in the reported rate."""
    from workloads import gen
    import oracle
    if rank != 0:
        return None
    oracle.build()
    oracle.set_threads(0)   # every host core (independent rows in parallel)
    cores = os.cpu_count() or 1
    case = gen.config2()
    rng = np.random.default_rng(1)
    # size the per-step sample so the whole run takes about 90 s
    t0 = time.perf_counter()
    oracle_step_sample(case, 8, 1, rng)
    t_probe = (time.perf_counter() - t0) / 8
    total = max(1, args.steps + args.warmup)
    per_step_s = 90.0 / total
    rows = int(min(case.N * case.Hq, max(1, per_step_s / max(t_probe, 1e-6))))
    g_rows = max(1, min(case.N, rows * case.N // (case.N * case.Hq) or 1))
    for _ in range(args.warmup):
        oracle_step_sample(case, rows, g_rows, rng)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step_sample(case, rows, g_rows, rng)
    dt = time.perf_counter() - t0
    frac = rows / (case.N * case.Hq)
    value = args.steps * frac / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_per_step": f"{rows} of {case.N * case.Hq} "
                       f"attention rows + {g_rows} greedy rows, scaled to whole steps"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{rows} attention rows per step, {cores} threads; "
                                       f"CPU: {cpu_model()}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


# ----------------------------------------------------------------------------
def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if args.ncu_steps > 0:
        run_ncu_steps(args)
        return
    r = run_ours(args, rank, world, local_rank)
    if rank != 0:
        return
    case = r["case"]
    hbm, tflops, peak_src = load_peaks()
    nbytes = algorithmic_bytes(case)
    flops = attention_flops(case)
    value = job_rate(args.steps, world, r["elapsed_ms"])
    ms_per_step = r["elapsed_ms"] / args.steps
    step_bytes = sum(nbytes.values())
    pk = r["per_kernel"]
    g_us = pk["tv_accept_greedy"]
    a_us = pk["tv_attn_verify"]
    at_us = pk["tv_attn_verify_tree"]
    greedy_gbs = nbytes["greedy"] / (g_us * 1e-6) / 1e9
    attn_gbs = nbytes["attn"] / (a_us * 1e-6) / 1e9
    t_roof_us = sum(max(nbytes[k] / (hbm * 1e9), (flops if k == "attn" else 0) / (tflops * 1e12))
                    for k in nbytes) * 1e6
    # roofline of the dominant entry point (largest measured time per launch).
    # Attention: its algorithmic bytes take longer at the HBM peak than its
    # flops at the bf16 tensor peak, so it is HBM-bound too.
    # the step's two entry points: the fused tree encoding + attention, and greedy
    step_bytes_of = {"tv_attn_verify_tree": nbytes["attn"] + nbytes["tree"],
                     "tv_accept_greedy": nbytes["greedy"]}
    key = {"tv_attn_verify_tree": "attn", "tv_accept_greedy": "greedy"}
    dom = max(step_bytes_of, key=lambda k: pk[k])
    dom_gbs = step_bytes_of[dom] / (pk[dom] * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": hbm, "unit": "GB/s",
                "frac": dom_gbs / hbm, "traffic": ncu_traffic(dom),
                "peak_source": f"{peak_src} hbm_gbs", "bytes_per_launch": step_bytes_of[dom],
                "us_per_launch": pk[dom]}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16/f32", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "l2": f"{r['M']} rotating input sets of {r['set_bytes'] / 1e6:.1f} MB "
                         f"(>= 3x the {r['l2'] / 1e6:.0f} MB L2)",
                   "timing": "CUDA graphs of whole steps, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "tree_tokens_per_s": value * case.B * case.N,
        "achieved_hbm_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
        "roofline_step_us": t_roof_us,
        "roofline_step_frac": t_roof_us / (ms_per_step * 1e3),
        "roofline": roofline,
        "kernels": {k: {"us_per_launch": v} for k, v in pk.items()},
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
    }
    line["kernels"]["tv_attn_verify"].update(
        {"algorithmic_bytes": nbytes["attn"], "flops": flops, "achieved_gbs": attn_gbs,
         "achieved_tflops": flops / (a_us * 1e-6) / 1e12, "hbm_frac": attn_gbs / hbm,
         "traffic": ncu_traffic("tv_attn_verify")})
    line["kernels"]["tv_accept_greedy"].update(
        {"algorithmic_bytes": nbytes["greedy"], "achieved_gbs": greedy_gbs,
         "hbm_frac": greedy_gbs / hbm, "traffic": ncu_traffic("tv_accept_greedy")})
    line["kernels"]["tv_tree_build"].update({"algorithmic_bytes": nbytes["tree"],
                                             "traffic": ncu_traffic("tv_tree_build")})
    at_bytes = nbytes["attn"] + nbytes["tree"]
    line["kernels"]["tv_attn_verify_tree"].update(
        {"algorithmic_bytes": at_bytes, "flops": flops,
         "achieved_gbs": at_bytes / (at_us * 1e-6) / 1e9,
         "hbm_frac": at_bytes / (at_us * 1e-6) / 1e9 / hbm,
         "traffic": ncu_traffic("tv_attn_verify_tree"),
         "note": "the step's tree encoding and attention in one launch (plus the split merge)"})
    if r["e2e"] is not None:
        line["e2e"] = r["e2e"]
    if world == 1 and not args.no_configs:
        import torch
        import speculative_decoding_tree_tv_gb300 as tv
        line["other_configs"] = measure_other_configs(
            torch, tv, torch.device("cuda", local_rank), hbm, tflops,
            0.0 if args.no_cpu_baseline else 4.0)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
