"""Benchmark of the Prism block-sparse attention hot path (forward + backward).

One step = the whole path on one batch of the seeded synthetic 2K-like grid
(21 x 90 x 160 latent tokens, 24 heads, d = 128, bf16, 3 x 16 x 16 zones,
128-token blocks, Top-k floor 8, Top-p 0.9), every stage through the C ABI:
zone statistics -> shapes + permutation + pooling -> block selection ->
sparse attention forward -> inverse permutation of O -> permutation of dO ->
sparse attention backward -> inverse permutation of dQ, dK, dV.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`value` is effective TFLOP/s: the attention flops of the selected
(query block, key block) pairs, 4 S^2 d forward + 10 S^2 d backward per pair,
divided by the whole step time.  Multi-GPU runs are independent replicas
(every head of every batch is independent; no data-path collective).
`--impl reference` times the CPU oracle (fp64 numpy) on a bounded sample of
the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from content_adaptive_block_02_b300 import build, prism, synth  # noqa: E402

METRIC = "sparse-attn fwd+bwd ms & effective TFLOP/s at 2K grid; % of bf16 tensor peak"
# kernels one step launches: statistics, assign, permute_pool, score digits,
# score product, select fast / fallback, 2 scans, CSR fill, CSC count and fill,
# forward, unpermute (O), permute (dO), bwd_pre, dK/dV, dQ, unpermute (dQ, dK, dV)
KERNELS_PER_STEP = 21


def pair_flops(w):
    """Flops per selected (query block, key block) pair of S-token blocks:
    forward 4 S^2 d, backward 10 S^2 d (algorithmic), and what the dK/dV
    (8 S^2 d) and dQ (6 S^2 d, S and dP recomputed) kernels compute."""
    u = w.block * w.block * w.d
    return {"fwd": 4 * u, "bwd": 10 * u, "attn_fwd": 4 * u, "attn_dkdv": 8 * u, "attn_dq": 6 * u}
# DRAM bytes (read + written) per launch of the attention kernels on the 2K-like
# workload, from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum,
# 1 pass) of the kernel code whose digest (source_digest) is given, with the
# plan's number of key ranges; reported only for that workload and range count,
# and as null once the kernel's code has changed since.
TRAFFIC_2K = {
    "attn_fwd_tc_kernel": ("attn_tc.cu", "e62fc53d1541ffef", 3, 24.24e9 + 5.50e9),
    "attn_dkdv_tc_kernel": ("attn_tc_dkdv.cu", "779df76c79c99244", 3, 20.39e9 + 11.89e9),
    "attn_dq_tc_kernel": ("attn_tc_dq.cu", "667fec371cf742e6", 3, 32.88e9 + 4.98e9),
}


def source_digest(name: str) -> str:
    """SHA-256 prefix of a kernel source file's code lines (comments and blank
    lines dropped, so that a comment edit keeps a capture valid)."""
    import hashlib
    import re
    path = os.path.join(ROOT, "content_adaptive_block_02_b300", "csrc", name)
    with open(path) as f:
        code = [re.sub(r"//.*$", "", line).strip() for line in f]
    return hashlib.sha256("\n".join(c for c in code if c).encode()).hexdigest()[:16]


def measured_traffic(kernel: str, key_ranges: int):
    """DRAM bytes per launch of `kernel` if its code and the plan's key ranges
    are still the captured ones."""
    ent = TRAFFIC_2K.get(kernel)
    if ent is None or ent[1] is None or ent[2] != key_ranges:
        return None
    return ent[3] if source_digest(ent[0]) == ent[1] else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return dict(bf16=m["bf16_tflops"], bf16_sus=m["bf16_tflops_sustained"],
                    hbm=m["hbm_gbs"], src="measured")
    except Exception:
        return dict(bf16=1800.0, bf16_sus=1400.0, hbm=6400.0, src="fallback")


class Clocks:
    """nvidia-smi samples (200 ms) taken while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.idx = dev_index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p is not None:
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "out", "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_workload(w, rank: int):
    """The problem of replica `rank`: the same workload with its own seeds, so
    that N replicas process N independent problems (every head of every batch
    is independent through all steps; no data-path exchange)."""
    return w.with_(seed_base=w.seed_base + 100 * rank)


def max_over_ranks(x: float, device) -> float:
    """Slowest rank's value (timings are bracketed by barriers on every rank)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device) -> float:
    """Whole-job total of a per-rank count (the units all ranks processed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t)
    return float(t.item())


# ----------------------------------------------------------------- ours ----

CALLS = ("a2v_norms", "zone_stats", "assign_permute", "block_select", "attn_fwd_call",
         "unpermute_O", "permute_dO", "attn_bwd_call", "unpermute_dQ", "unpermute_dK",
         "unpermute_dV")


def call_bytes(w, plan, fused: bool):
    """Algorithmic HBM bytes of the memory-bound calls: every tensor read or
    written once at its stored size (a [B, N, H, d] bf16 tensor is
    B*N*H*d*2 bytes; block-order tensors hold Np rows, padding included)."""
    B, N, H, d, Np, nb = w.B, w.N, w.H, w.d, plan.Np, plan.nb
    tok = B * N * H * d * 2                 # one model-side bf16 tensor
    ptok = B * H * Np * d * 2               # one block-order bf16 tensor
    out = {
        "zone_stats": tok + (B * N * 4 if fused else B * N * w.Ca * 2),
        "assign_permute": 3 * tok + 3 * ptok + 4 * B * H * nb * d * 4 + B * H * (Np + N) * 4
                          + B * H * nb * 4,
        "permute_dO": tok + ptok + B * H * Np * 4,
        "unpermute_O": 2 * tok + B * H * N * 4,
        "bwd_pre": 2 * ptok + B * H * Np * 4 * 3,
    }
    for k in ("unpermute_dQ", "unpermute_dK", "unpermute_dV"):
        out[k] = out["unpermute_O"]
    if fused:
        out["a2v_norms"] = B * N * w.Ca * 2 + B * N * 4
    return out


class Runner:
    """One Prism attention layer (forward + backward) on the device through
    the C ABI, with optional CUDA events around every call."""

    def __init__(self, w, dev, key_chunk_blocks=0, fused=True, x=None, shape_id=None):
        self.w, self.dev, self.fused = w, dev, fused
        self.shape_id = shape_id   # [B, H, Z] uint8: given shapes (Table 9 baselines)
        self.x = synth.generate(w, dev) if x is None else x
        self.att = prism.PrismAttention(w, dev, key_chunk_blocks=key_chunk_blocks)
        self.stream = torch.cuda.current_stream()
        self.nrm = torch.empty(w.B, w.N, dtype=torch.float32, device=dev)

    def step(self, ev=None, trace=None, xin=None):
        att, p, st = self.att, self.att.plan, self.stream
        xi = self.x if xin is None else xin
        if trace is not None:
            p.set_trace_events(trace)

        def mark(k):
            if ev is not None:
                ev[k].record(st)
        o = att.perm_out
        mark(0)
        if self.shape_id is not None:
            mark(1)
            mark(2)
            p.permute_shapes(self.shape_id, xi["Q"], xi["K"], xi["V"], att.ws, o)
        else:
            if self.fused:
                p.a2v_norms(xi["qa"], xi["audio"], xi["audio"], att.ws, self.nrm)
                mark(1)
                p.zone_stats_norms(xi["V"], self.nrm, att.stats)
            else:
                mark(1)
                p.zone_stats(xi["V"], xi["a2v"], att.stats)
            mark(2)
            p.assign_and_permute(att.stats, xi["Q"], xi["K"], xi["V"], o)
        mark(3)
        p.block_select(o["shape_id"], o["Qbar"], o["Qbar_lo"], o["Kbar"], o["Kbar_lo"],
                       o["n_valid"], att.ws, att.lists)
        mark(4)
        p.sparse_attn_fwd(o["Qp"], o["Kp"], o["Vp"], o["n_valid"], att.lists["row_ptr"],
                          att.lists["col_idx"], att.scale, att.ws, att.Op, att.lse)
        mark(5)
        p.unpermute(o["inv"], att.Op, att.O)
        mark(6)
        p.permute(o["perm"], xi["dO"], att.dOp)
        mark(7)
        p.sparse_attn_bwd(o["Qp"], o["Kp"], o["Vp"], att.Op, att.dOp, att.lse, o["n_valid"],
                          att.lists, att.scale, att.ws, att.dQp, att.dKp, att.dVp)
        mark(8)
        p.unpermute(o["inv"], att.dQp, att.dQ)
        mark(9)
        p.unpermute(o["inv"], att.dKp, att.dK)
        mark(10)
        p.unpermute(o["inv"], att.dVp, att.dV)
        mark(11)

    def selection_summary(self):
        att, w = self.att, self.w
        nb = att.plan.nb
        rp = att.lists["row_ptr"]
        pairs = int(rp[-1].item())
        counts = (rp[1:] - rp[:-1]).long()
        nv = att.perm_out["n_valid"].reshape(-1).long()
        rows = torch.repeat_interleave(torch.arange(counts.numel(), device=rp.device), counts)
        cols = att.lists["col_idx"][:pairs].long()
        # token pairs actually attended (real query rows x real key rows)
        tok_pairs = int((nv[rows] * nv[(rows // nb) * nb + cols]).sum().item())
        lens = counts[nv > 0].cpu().numpy()
        sid = att.perm_out["shape_id"].reshape(-1).cpu().numpy().astype(np.int64)
        hist = np.bincount(sid, minlength=len(w.menu))
        return dict(
            pairs=pairs, tok_pairs=tok_pairs,
            lengths={"min": int(lens.min()), "p50": int(np.median(lens)),
                     "p99": int(np.percentile(lens, 99)), "max": int(lens.max()),
                     "mean": round(float(lens.mean()), 1)},
            shapes={"x".join(str(e) for e in w.menu[k]): int(hist[k])
                    for k in range(len(w.menu)) if hist[k] > 0},
            ties={"zone_shapes": int(att.perm_out["shape_tie"].sum().item()),
                  "selection_rows": int(att.lists["sel_tie"].sum().item())},
            amb=int(att.ws[4:8].view(torch.int32).item()))

    def measure(self, steps, warmup, barrier=lambda: None, clock_dev=None):
        """W untimed steps, then K steps between events; per-call and
        per-kernel times from events recorded on the launching stream."""
        ev = lambda: torch.cuda.Event(enable_timing=True)
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        st = self.att.status()
        if st != 0:
            raise RuntimeError(f"device status {st} after warm-up")
        calls = [[ev() for _ in range(len(CALLS) + 1)] for _ in range(steps)]
        # per-kernel marks recorded by the library around each attention
        # kernel; every event is recorded once here so that its handle exists
        traces = [{s: (ev(), ev()) for s in prism.Plan.TRACE_SLOTS} for _ in range(steps)]
        for tr in traces:
            for pair in tr.values():
                for e in pair:
                    e.record(self.stream)
        barrier()
        torch.cuda.synchronize()
        t0, t1 = ev(), ev()
        clk = Clocks(clock_dev) if clock_dev is not None else None
        if clk is not None:
            clk.__enter__()
        t0.record(self.stream)
        for k in range(steps):
            self.step(calls[k], traces[k])
        t1.record(self.stream)
        torch.cuda.synchronize()
        if clk is not None:
            clk.__exit__(None, None, None)
        self.att.plan.set_trace_events(None)
        mean = lambda f: statistics.mean(f(k) for k in range(steps))
        call_ms = {c: mean(lambda k, i=i: calls[k][i].elapsed_time(calls[k][i + 1]))
                   for i, c in enumerate(CALLS)}
        kern_ms = {s: mean(lambda k, s=s: traces[k][s][0].elapsed_time(traces[k][s][1]))
                   for s in prism.Plan.TRACE_SLOTS}
        return dict(ms=t0.elapsed_time(t1) / steps, call_ms=call_ms, kern_ms=kern_ms,
                    clocks=clk.summary() if clk is not None else None,
                    status=self.att.status())


def hbm_summary(w, plan, fused, call_ms, kern_ms, pk):
    """GB/s of the memory-bound kernels from their algorithmic bytes, timed by
    the library's own events around each kernel where it has a slot (zone
    statistics, permutation + pooling, bwd_pre), else around the call."""
    by = call_bytes(w, plan, fused)
    t = dict(call_ms)
    t["bwd_pre"] = kern_ms["bwd_pre"]
    t["zone_stats"] = kern_ms.get("zone_stats", t["zone_stats"])
    by["permute_pool"] = by.pop("assign_permute")
    t["permute_pool"] = kern_ms.get("permute_pool", t["assign_permute"])
    out = {}
    for k, b in by.items():
        ms = t[k]
        if ms > 0:
            gbs = b / (ms * 1e-3) / 1e9
            out[k] = {"ms": round(ms, 3), "bytes": b, "gbs": round(gbs, 1),
                      "frac": round(gbs / pk["hbm"], 3)}
    return out


def workload_desc(w):
    return (f"{w.name}: {w.T}x{w.Hg}x{w.W} grid, {w.H} heads, d={w.d}, zones {w.zone}, "
            f"{w.block}-token blocks, top-k {w.topk_floor}, top-p {w.topp}")


def run_ours(args, w):
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    build.build()
    fused = not args.a2v_input
    wr = replica_workload(w, rank)     # an independent problem per replica
    R = Runner(wr, dev, args.key_chunk_blocks, fused)
    att, stream = R.att, R.stream
    ev = lambda: torch.cuda.Event(enable_timing=True)
    barrier = (lambda: torch.distributed.barrier()) if ws > 1 else (lambda: None)
    for _ in range(args.warmup):
        R.step()
    torch.cuda.synchronize()
    sel = R.selection_summary()
    pairs = sel["pairs"]
    PF = pair_flops(wr)
    flop = pairs * (PF["fwd"] + PF["bwd"])
    real_flop = sel["tok_pairs"] * 14 * wr.d           # 4 d forward + 10 d backward per token pair
    m = R.measure(args.steps, 0, barrier, clock_dev=local)
    ms = max_over_ranks(m["ms"], dev)
    flop_all = sum_over_ranks(flop, dev)
    real_all = sum_over_ranks(real_flop, dev)
    kern_ms, call_ms = m["kern_ms"], m["call_ms"]
    fwd_ms, bwd_ms = call_ms["attn_fwd_call"], call_ms["attn_bwd_call"]

    # ---- end to end through host buffers (pinned): every step's inputs are
    # copied host -> device and its outputs device -> host inside the timed
    # region, pipelined over two device buffer sets on two copy streams, so
    # the copies of one step overlap the compute of its neighbours ----
    x = R.x
    names_in = ["Q", "K", "V", "dO"] + (["qa", "audio"] if fused else ["a2v"])
    names_out = ("O", "dQ", "dK", "dV")
    host_in = {k: x[k].cpu().pin_memory() for k in names_in}
    host_out = {k: torch.empty(x["Q"].shape, dtype=torch.bfloat16).pin_memory()
                for k in names_out}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    xb = [x, {k: torch.empty_like(x[k]) for k in names_in}]
    ob = [{k: torch.empty_like(att.O) for k in names_out} for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    e_steps = max(1, args.steps)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(stream)
    s_h2d.wait_stream(stream)
    s_d2h.wait_stream(stream)
    for k in range(e_steps):
        b = k % 2
        with torch.cuda.stream(s_h2d):
            if k >= 2:
                s_h2d.wait_event(comp_done[b])  # step k-2 has finished reading buffer b
            for n in names_in:
                xb[b][n].copy_(host_in[n], non_blocking=True)
            in_ready[b].record(s_h2d)
        stream.wait_event(in_ready[b])
        if k >= 2:
            stream.wait_event(out_free[b])  # step k-2's outputs have left buffer b
        R.step(xin=xb[b])
        for n, src in zip(names_out, (att.O, att.dQ, att.dK, att.dV)):
            ob[b][n].copy_(src, non_blocking=True)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(comp_done[b])
            for n in names_out:
                host_out[n].copy_(ob[b][n], non_blocking=True)
            out_free[b].record(s_d2h)
    stream.wait_stream(s_d2h)
    stream.wait_stream(s_h2d)
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dev)

    pk = peaks()
    clk_sum = m["clocks"]
    kern_flop = {k: PF[k] for k in ("attn_fwd", "attn_dkdv", "attn_dq")}
    kern_tf = {s: round(pairs * f / (kern_ms[s] * 1e-3) / 1e12, 1) for s, f in kern_flop.items()}
    dom = max(kern_flop, key=lambda s: kern_ms[s])     # the longest attention kernel
    dom_name = {"attn_fwd": "attn_fwd_tc_kernel", "attn_dkdv": "attn_dkdv_tc_kernel",
                "attn_dq": "attn_dq_tc_kernel"}[dom]
    line = {
        "metric": METRIC,
        "value": round(flop_all / (ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "real_token_tflops": round(real_all / (ms * 1e-3) / 1e12, 2),
        "config": {"workload": workload_desc(w),
                   "global_batch": w.B * ws, "tokens": w.N, "parallelism": f"replicas x{ws}",
                   "a2v": ("norms computed on the device from the A2V queries and the "
                           f"{w.Na} audio tokens" if fused else "A2V output given"),
                   "l2": "inputs larger than L2 (no flush needed)",
                   "selected_pairs": pairs,
                   "real_token_pairs": sel["tok_pairs"],
                   "block_density": round(pairs / (w.B * w.H * att.plan.nb ** 2), 4),
                   "rows_decided_exactly": sel["amb"],
                   "selected_per_query_block": sel["lengths"],
                   "shapes_chosen": sel["shapes"],
                   "near_ties": sel["ties"],
                   "key_ranges": att.plan.sz.key_chunks},
        "attn_ms": {"fwd": round(fwd_ms, 3), "bwd": round(bwd_ms, 3),
                    "other": round(ms - fwd_ms - bwd_ms, 3)},
        "attn_tflops": {"fwd": round(pairs * PF["fwd"] / (fwd_ms * 1e-3) / 1e12, 1),
                        "bwd": round(pairs * PF["bwd"] / (bwd_ms * 1e-3) / 1e12, 1)},
        "dense_equiv_tflops": round(w.B * w.H * (att.plan.nb ** 2) *
                                    (PF["fwd"] + PF["bwd"]) / (ms * 1e-3) / 1e12 * ws, 1),
        "call_ms": {c: round(v, 3) for c, v in call_ms.items()},
        "kernel_ms": {s: round(v, 3) for s, v in kern_ms.items()},
        "kernel_tflops": kern_tf,
        "hbm_kernels": hbm_summary(wr, att.plan, fused, call_ms, kern_ms, pk),
        "roofline": {"bound": "tensor",
                     "kernel": f"{dom_name} (library-recorded events around the launch)",
                     "achieved": kern_tf[dom], "peak": pk["bf16"],
                     "peak_kind": f"bf16 dense burst ({pk['src']})", "unit": "TFLOP/s",
                     "frac": round(kern_tf[dom] / pk["bf16"], 4),
                     "frac_sustained": round(kern_tf[dom] / pk["bf16_sus"], 4),
                     # the burst peak scaled to the SM clock sampled in the timed
                     # region (the burst GEMM taken to run at the maximum clock)
                     "frac_at_run_clock": (round(kern_tf[dom] / (pk["bf16"] * clk_sum["sm_mhz"] /
                                                                 clk_sum["sm_max_mhz"]), 4)
                                           if clk_sum.get("sm_mhz") else None),
                     "flop_per_launch": pairs * kern_flop[dom],
                     "traffic": (measured_traffic(dom_name, att.plan.sz.key_chunks)
                                 if w.name == "2k" else None)},
        "e2e": {"value": round(flop_all / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e_steps,
                "copies": "pinned host buffers, two device buffer sets, copy streams "
                          "overlapped with the neighbouring steps' compute"},
        "gpu_launches": (KERNELS_PER_STEP + (1 if fused else 0) +
                         (4 if att.plan.sz.key_chunks > 1 else 0) +
                         (2 if att.plan.sz.multi_tile else 0) +
                         (2 if att.plan.sz.half_tile else 0)) * args.steps,
        "clocks": clk_sum,
        "device_status": m["status"],
    }
    del xb, ob, host_in, host_out
    if rank == 0 and ws == 1 and not args.no_dense:
        line["dense"] = dense_run(wr, dev, args, R.x, fused)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, R.x, fused)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return line if rank == 0 else None


def dense_run(w, dev, args, x, fused, steps=2, warmup=1):
    """The same kernels with every valid key block selected (Top-p = 1), on
    the same inputs: the dense-attention reference timed next to the sparse
    step (fewer steps: a dense 2K step is several seconds)."""
    wd = w.with_(topp=1.0, name=w.name + "-dense")
    R = Runner(wd, dev, args.key_chunk_blocks, fused, x=x)
    for _ in range(warmup):
        R.step()
    torch.cuda.synchronize()
    pairs = int(R.att.lists["row_ptr"][-1].item())
    m = R.measure(steps, 0)
    out = {"steps": steps, "warmup": warmup, "ms_per_step": round(m["ms"], 1),
           "selected_pairs": pairs,
           "value": round(pairs * (pair_flops(w)["fwd"] + pair_flops(w)["bwd"]) /
                          (m["ms"] * 1e-3) / 1e12, 1),
           "unit": "TFLOP/s",
           "kernel_ms": {s: round(v, 2) for s, v in m["kern_ms"].items()},
           "device_status": m["status"]}
    del R
    torch.cuda.empty_cache()
    return out


def sweep(args):
    """One line per workload of the measurement plan: the 720p, 1080p and 2K
    grids, the 41-frame grid, the 2K grid with 128- and 256-token blocks mixed
    (3 x 16 x 16 and 4 x 16 x 16 zones), the 2K stress inputs (white field,
    one dominant source, skewed noise) at Top-p 0.5 / 0.9 / 0.99, and the
    block-shape baselines of Table 9 on the 2K grid."""
    cases = [(synth.WORKLOADS[n], None) for n in ("720p", "1080p", "2k", "2k_long", "2k_mc",
                                                  "2k_mc4")]
    for v in ("white", "onesrc", "skew"):
        for p in (0.5, 0.9, 0.99):
            cases.append((synth.stress("2k", v, p), None))
    # the block-shape baselines of Table 9 on the 2K grid, shapes given to
    # every zone: Random (seeded, over the admissible 128-token shapes), Fixed
    # (1,8,16), Fixed 8^3 (8x16x16 zones, 512-token blocks), Only C256
    # (4x16x16 zones, the 256-token menu through Eq. 7)
    w2 = synth.WORKLOADS["2k"]
    rng = np.random.default_rng(9)
    Zc = w2.n_zones
    cases.append((w2.with_(name="2k_random_shapes"),
                  rng.choice([0, 1], size=(w2.B, w2.H, Zc)).astype(np.uint8)))
    cases.append((w2.with_(name="2k_fixed_1x8x16"), np.zeros((w2.B, w2.H, Zc), np.uint8)))
    w8 = w2.with_(name="2k_fixed_8cubed", zone=(8, 16, 16), menu=((8, 8, 8),))
    cases.append((w8, np.zeros((w8.B, w8.H, w8.n_zones), np.uint8)))
    cases.append((w2.with_(name="2k_only_c256", zone=(4, 16, 16), menu=synth.MENU_256), None))
    # the 64-token baselines (Only C64, Fixed 4^3) share 128-row tiles between
    # two blocks, which needs zones without padding: a 2K-wide grid of 24 x 96
    # x 160 tokens (4 x 16 x 16 zones, 24 heads), with the 128-token menu on
    # the same grid beside them
    w96 = w2.with_(name="2k96_c128", T=24, Hg=96, zone=(4, 16, 16))
    cases.append((w96, None))
    cases.append((w96.with_(name="2k96_only_c64", menu=synth.MENU_64, class_tau=()), None))
    w4 = w96.with_(name="2k96_fixed_4cubed", menu=((4, 4, 4),), class_tau=())
    cases.append((w4, np.zeros((w4.B, w4.H, w4.n_zones), np.uint8)))
    if args.sweep_filter:
        cases = [(w, sid) for w, sid in cases if args.sweep_filter in w.name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    pk = peaks()
    for w, sid in cases:
        # the one-source stress input scales the A2V output itself: it runs
        # with the A2V output given
        fused = not args.a2v_input and w.src_mass is None
        sid_t = None if sid is None else torch.as_tensor(sid).to(dev)
        R = Runner(w, dev, args.key_chunk_blocks, fused, shape_id=sid_t)
        for _ in range(args.warmup):
            R.step()
        torch.cuda.synchronize()
        sel = R.selection_summary()
        m = R.measure(args.steps, 0, clock_dev=0)
        pairs = sel["pairs"]
        PF = pair_flops(w)
        kern_tf = {s: round(pairs * PF[s] / (m["kern_ms"][s] * 1e-3) / 1e12, 1)
                   for s in ("attn_fwd", "attn_dkdv", "attn_dq")}
        print(json.dumps({
            "workload": workload_desc(w), "a2v_on_device": fused and sid is None,
            "shapes": "given" if sid is not None else "Eq. 7", "ms_per_step": round(m["ms"], 2),
            "value": round(pairs * (PF["fwd"] + PF["bwd"]) / (m["ms"] * 1e-3) / 1e12, 1),
            "unit": "TFLOP/s", "real_token_tflops":
                round(sel["tok_pairs"] * 14 * w.d / (m["ms"] * 1e-3) / 1e12, 1),
            "block_density": round(pairs / (w.B * w.H * R.att.plan.nb ** 2), 4),
            "selected_per_query_block": sel["lengths"], "near_ties": sel["ties"],
            "kernel_tflops": kern_tf, "frac_burst_dkdv": round(kern_tf["attn_dkdv"] / pk["bf16"], 3),
            "hbm_kernels": {k: v["gbs"] for k, v in
                            hbm_summary(w, R.att.plan, fused, m["call_ms"], m["kern_ms"], pk).items()
                            if sid is None or k not in ("zone_stats", "a2v_norms")},
            "key_ranges": R.att.plan.sz.key_chunks, "clocks": m["clocks"],
            "device_status": m["status"]}), flush=True)
        del R
        torch.cuda.empty_cache()


# ------------------------------------------------------------ oracle leg ----
# The oracle is timed as it stands, one process per head with one BLAS thread
# each (every head is independent through every step), started with `spawn`
# (never forked from a process that holds a CUDA context).

_ONE_THREAD = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def _bits(t):
    """bf16 tensor -> its uint16 bit patterns as a numpy array (exact)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle_head(job):
    """One head of the oracle (runs in a spawned worker): steps 1-4 in full,
    attention forward + backward on `rows` sampled query blocks.  Returns
    (seconds of steps 1-4, selected pairs of the head, pairs sampled,
    seconds of the sampled attention)."""
    shared, own, w, rows_sample, fused, seed = job
    from oracle import prism_oracle as orc
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    S_, O_ = np.load(shared), np.load(own)
    X = {k: f(O_[k]) for k in O_.files}
    A = {k: f(S_[k]) for k in S_.files}
    w1 = w.with_(H=1)
    t0 = time.perf_counter()
    if fused:
        n = orc.a2v_norms(A["qa"], A["audio"], A["audio"])
        st = orc.zone_stats_from_norms(w1, X["V"], n)
    else:
        st = orc.zone_stats(w1, X["V"], A["a2v"])
    sid, _ = orc.assign_shapes(w1, st)
    perm, inv, nval = orc.build_permutation(w1, sid)
    Qp, Kp, Vp = orc.permute(X["Q"], perm), orc.permute(X["K"], perm), orc.permute(X["V"], perm)
    Qb, Kb = orc.pool(Qp, nval, w.block), orc.pool(Kp, nval, w.block)
    lists, _ = orc.select_blocks(w1, Qb, Kb, nval)
    t1 = time.perf_counter()
    L = lists[(0, 0)]
    pairs = sum(len(s) for s in L if s is not None)
    rng = np.random.default_rng(seed)
    cand = [i for i in range(len(L)) if L[i] is not None and len(L[i]) > 0]
    rows = rng.choice(cand, size=min(rows_sample, len(cand)), replace=False)
    dOp = orc.permute(X["dO"], perm)
    scale = 1.0 / math.sqrt(w.d)
    t2 = time.perf_counter()
    sp = 0
    for i in rows:
        orc.attn_fwd_row(Qp[0, 0], Kp[0, 0], Vp[0, 0], nval[0, 0], int(i), L[i], w.block, scale)
        orc.attn_bwd_row(Qp[0, 0], Kp[0, 0], Vp[0, 0], dOp[0, 0], nval[0, 0], int(i), L[i],
                         w.block, scale)
        sp += len(L[i])
    return t1 - t0, pairs, sp, time.perf_counter() - t2


class OracleSampler:
    """The oracle on the host cores: P = min(heads, cores) heads at once,
    one spawned process (one thread) per head."""

    def __init__(self, w, x, fused):
        import multiprocessing as mp
        import tempfile
        self.w, self.fused = w, fused
        self.cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (
            os.cpu_count() or 1)
        self.P = max(1, min(w.H * w.B, self.cores))
        self.dir = tempfile.mkdtemp(prefix="prism_oracle_")
        self.shared = os.path.join(self.dir, "shared.npz")
        if fused:
            np.savez(self.shared, qa=_bits(x["qa"]), audio=_bits(x["audio"]))
        else:
            np.savez(self.shared, a2v=_bits(x["a2v"]))
        self.own = []
        for h in range(self.P):
            path = os.path.join(self.dir, f"head{h}.npz")
            np.savez(path, **{k: _bits(x[k][:, :, h:h + 1]) for k in ("Q", "K", "V", "dO")})
            self.own.append(path)
        saved = {k: os.environ.get(k) for k in _ONE_THREAD}
        os.environ.update(_ONE_THREAD)
        try:
            self.pool = mp.get_context("spawn").Pool(self.P)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def sample(self, rows_sample, seed=0):
        """Seconds the oracle needs for one whole step of the workload,
        extrapolated from one wave of P heads; and the description."""
        w = self.w
        jobs = [(self.shared, self.own[h], w, rows_sample, self.fused, seed + h)
                for h in range(self.P)]
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_head, jobs)
        wall = time.perf_counter() - t0
        t14 = max(r[0] for r in res)
        per_pair = sum(r[3] for r in res) / max(1, sum(r[2] for r in res))
        pairs_head = statistics.mean(r[1] for r in res)
        heads = w.H * w.B
        waves = -(-heads // self.P)
        pairs_all = pairs_head * heads
        total = waves * t14 + per_pair * pairs_all / self.P
        desc = (f"oracle, one process and thread per head, {self.P} heads at once on "
                f"{self.cores} host cores: steps 1-4 timed in full on {self.P} heads (slowest "
                f"{t14:.1f} s, {waves} wave(s) for {heads} heads); attention fwd+bwd timed on "
                f"{rows_sample} query block(s) per head ({sum(r[2] for r in res)} pairs, "
                f"{per_pair * 1e3:.2f} ms per pair per thread), extrapolated to "
                f"{pairs_all:.0f} pairs over {self.P} threads")
        return total, pairs_all * 14 * w.block * w.block * w.d, desc, wall

    def close(self):
        import shutil
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)


def cpu_baseline(w, x, fused, rows_sample=3):
    smp = OracleSampler(w, x, fused)
    try:
        total, flop, desc, wall = smp.sample(rows_sample)
    finally:
        smp.close()
    return {"value": round(flop / total / 1e12, 6), "unit": "TFLOP/s", "cores": smp.P,
            "host_cores": smp.cores, "kind": "oracle", "sample": desc,
            "seconds_spent": round(wall, 1), "extrapolated_s_per_step": round(total, 1)}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    # the seeded inputs (untimed setup): made by the generator's torch ops on the
    # device when there is one, then held in host memory for the oracle
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    x = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in synth.generate(w, gen).items()}
    fused = not args.a2v_input
    smp = OracleSampler(w, x, fused)
    try:
        for k in range(args.warmup):
            smp.sample(1, seed=1000 * (k + 1))
        vals, descs, spent = [], [], 0.0
        for k in range(args.steps):
            total, flop, desc, wall = smp.sample(1, seed=k)
            vals.append(total)
            descs.append(desc)
            spent += wall
    finally:
        smp.close()
    total = statistics.mean(vals)
    v = flop / total / 1e12
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total * 1e3, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w), "global_batch": w.B, "tokens": w.N,
                       "a2v": ("norms computed from the A2V queries and the audio tokens"
                               if fused else "A2V output given")},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": smp.P,
                             "host_cores": smp.cores, "kind": "oracle", "sample": descs[-1]},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "seconds_spent": round(spent, 1)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="2k", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dense", action="store_true",
                    help="Top-p = 1: every valid key block (the dense comparison)")
    ap.add_argument("--key-chunk-blocks", type=int, default=0,
                    help="key / query range size of the attention kernels (0: automatic)")
    ap.add_argument("--stress", choices=["white", "onesrc", "skew"], default=None,
                    help="stress inputs: white field / one dominant audio source / skewed noise")
    ap.add_argument("--a2v-input", action="store_true",
                    help="take the A2V output as an input instead of computing its norms")
    ap.add_argument("--no-dense", action="store_true",
                    help="skip the all-blocks dense run timed next to the sparse step")
    ap.add_argument("--heads", type=int, default=0,
                    help="override the workload's head count (smaller cases for profiling)")
    ap.add_argument("--sweep", action="store_true",
                    help="one line per workload of the measurement plan (not the contract line)")
    ap.add_argument("--sweep-filter", default="",
                    help="with --sweep: only the workloads whose name contains this text")
    args = ap.parse_args()
    if args.sweep:
        sweep(args)
        return
    w = synth.WORKLOADS[args.workload]
    if args.heads > 0:
        w = w.with_(H=args.heads, name=f"{w.name}-h{args.heads}")
    if args.stress is not None:
        w = synth.stress(args.workload, args.stress, w.topp)
    if args.dense:
        w = w.with_(topp=1.0, name=w.name + "-dense")
    if args.stress == "onesrc":
        args.a2v_input = True   # this input scales the A2V output itself
    line = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
