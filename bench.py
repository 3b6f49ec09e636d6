#!/usr/bin/env python
"""Packed-tree KDA forward + backward throughput on one GB300 (or N, weak scaling).

A step is one pass of the whole hot path over one synthetic rollout forest: the
forward (one packed call per round), the backward state pass (rounds in reverse,
gradients through the state handoffs) and the per-chunk gradient pass with the
replay-row fold.  The metric is compact tokens per second, C / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own forest (weak scaling, no collective on the data
path); the timed region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "wide256k_bf16"
METRIC = "packed-tree KDA fwd+bwd compact tokens/s"
UNIT = "compact tokens/s"
NOMINAL_HBM_GBS = 8000.0          # nominal HBM rate of one GB300 (8 TB/s)
NOMINAL_BF16_TFLOPS = 2250.0      # nominal dense bf16 tensor peak of one GB300


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-expanded", action="store_true",
                    help="skip the leg that times the same kernels on the trajectory-expanded input")
    ap.add_argument("--fidelity", action="store_true",
                    help="also compare the forward outputs of the tree plans with the "
                         "per-trajectory run, by handoff depth")
    ap.add_argument("--logprob", action="store_true",
                    help="also time the compact-to-semantic log-probabilities (64K-token forest, "
                         "V = 157,184)")
    ap.add_argument("--conv", action="store_true",
                    help="also time the short convolution (fwd, bwd) on the forest's q")
    ap.add_argument("--attn", action="store_true",
                    help="also time the branch attention (forward) on the forest's q, k, v")
    ap.add_argument("--nodewise", action="store_true",
                    help="also time the same kernels on the node-wise plan of the forest")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def forest_for_rank(workload, rank):
    """Each rank runs its own seeded forest of the workload (weak scaling: the per-GPU
    work stays fixed as ranks are added; no data crosses ranks)."""
    from prefix_shared_chunkwise_gb300.synth import WORKLOAD_ORDER, make_tree
    seed = WORKLOAD_ORDER.index(workload) + 1000 * rank
    parent, seg_len = make_tree(workload, seed=seed)
    return parent, seg_len, seed


def reduce_across_ranks(C_local, ms_local, device):
    """Whole-job compact tokens (sum over ranks) and the slowest rank's step time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return int(C_local), float(ms_local)
    c = torch.tensor([float(C_local)], dtype=torch.float64, device=device)
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return int(round(c.item())), float(t.item())


# ---- algorithmic cost model (per step) ---------------------------------------------------

def cost_model(info, H, D, B):
    """Algorithmic bytes and flops of the path (bf16 tensors, fp32 states).

    Per compact or replay token-head: fwd reads q, k, v, g (2 B each per channel) and
    beta (2 B), writes o for own rows; bwd reads the same plus dO for own rows and writes
    dq, dk, dv, dg, dbeta; a replay row's dk, dv, dg, dbeta are read-modified-written.
    Handoffs: 4 dk dv H bytes per slot write/read and per consumer gradient write/read.
    Flops: 2B(3dk + 2dv) + 6 dk dv per token-head forward, backward twice that."""
    C, R, Nst, Ncons = info["C"], info["R"], info["n_states"], info["n_cons"]
    tok_in = 4 * 2 * D + 2
    fwd_b = (C + R) * H * tok_in + C * H * 2 * D + 4 * D * D * H * (Nst + Ncons)
    bwd_b = ((C + R) * H * tok_in + C * H * 2 * D + C * H * tok_in
             + R * H * 2 * (3 * 2 * D + 2) + 4 * D * D * H * (Nst + 2 * Ncons))
    f_tok = 2 * B * (3 * D + 2 * D) + 6 * D * D
    fwd_f = (C + R) * H * f_tok
    bwd_f = 2 * fwd_f
    return dict(fwd_bytes=fwd_b, bwd_bytes=bwd_b, fwd_flops=fwd_f, bwd_flops=bwd_f)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def traffic_from_profiles(kernel):
    """DRAM bytes per launch for `kernel` from the committed ncu summary, if present."""
    p = os.path.join(ROOT, "profiles", "traffic_per_launch.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 2 and parts[0] == kernel:
            try:
                return float(parts[1])
            except ValueError:
                return None
    return None


# ---- clocks ------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        import torch
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        uuid = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd[1:1] = ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), hw=f[5], hwt=f[6], swt=f[7], pc=f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        sms = sorted(r["sm"] for r in rows)
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pc", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=sms[len(sms) // 2], sm_max_mhz=max(r["smax"] for r in rows),
                    reasons=sorted(reasons), samples=len(rows))


# ---- oracle baseline on host cores -------------------------------------------------------

def pick_sample_tree(parent, seg_len, target_S):
    """Split the forest into trees; return the segment ids of the tree whose expanded
    size is closest to target_S."""
    import numpy as np
    n = len(parent)
    root = np.zeros(n, np.int64)
    for i in range(n):
        root[i] = i if parent[i] < 0 else root[parent[i]]
    from prefix_shared_chunkwise_gb300.synth import tree_stats
    best, best_d = None, None
    for r in np.unique(root):
        ids = np.nonzero(root == r)[0]
        remap = {int(v): j for j, v in enumerate(ids)}
        sub_parent = np.array([-1 if parent[v] < 0 else remap[int(parent[v])] for v in ids], np.int32)
        st = tree_stats(sub_parent, seg_len[ids])
        d = abs(st["S"] - target_S)
        if best is None or d < best_d:
            best, best_d = (ids, sub_parent, st), d
    return best


def oracle_sample(parent, seg_len, seg_offset, inputs, H_sample, B, target_S):
    """Run the fp64 oracle forward + backward over one tree of the forest (heads
    [0, H_sample)); returns (compact tokens of the tree, heads, seconds, threads, stats)."""
    import numpy as np
    import oracle
    ids, sub_parent, st = pick_sample_tree(parent, seg_len, target_S)
    rows = np.concatenate([np.arange(seg_offset[v], seg_offset[v] + seg_len[v]) for v in ids])
    sub_off = np.zeros(len(ids), np.int64)
    acc = 0
    for j, v in enumerate(ids):
        sub_off[j] = acc
        acc += int(seg_len[v])
    import torch
    idx = torch.as_tensor(rows, device=inputs["q"].device)
    host = {k: inputs[k].index_select(0, idx)[:, :H_sample].float().cpu().double().numpy()
            for k in ("q", "k", "v", "g", "beta", "W")}
    threads = len(os.sched_getaffinity(0))
    t0 = time.time()
    oracle.kda_forest(sub_parent, seg_len[ids], sub_off, host["q"], host["k"], host["v"],
                      host["g"], host["beta"], chunk=B, W=host["W"], n_threads=threads)
    dt = time.time() - t0
    return st["C"], H_sample, dt, min(threads, H_sample), st


def oracle_rate(step, budget_s=4.0, max_units=10_000):
    """Call `step()` (which runs the oracle on one sampled unit and returns the units it
    processed) until `budget_s` seconds have passed; returns (units, seconds)."""
    units, t0 = 0, time.time()
    while time.time() - t0 < budget_s and units < max_units:
        units += step()
    return units, time.time() - t0


# ---- our arm -----------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from prefix_shared_chunkwise_gb300 import _lib, build
    from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
    from prefix_shared_chunkwise_gb300.synth import WORKLOADS, make_inputs

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        build.build()
    if ws > 1:
        dist.barrier()
    wl = WORKLOADS[args.workload]
    H, D, B = wl.H, wl.dk, wl.chunk
    parent, seg_len, seed = forest_for_rank(args.workload, rank)
    # planning (host) and plan upload, reported apart from the kernels' time
    t_pl = time.perf_counter()
    pl = Plan(parent, seg_len, B)
    plan_ms = (time.perf_counter() - t_pl) * 1e3
    torch.cuda.synchronize()
    t_up = time.perf_counter()
    pl.upload()
    torch.cuda.synchronize()
    upload_ms = (time.perf_counter() - t_up) * 1e3
    info = pl.info
    C = info["C"]
    x = make_inputs(C, H, D, D, wl.dtype, seed=3 + rank, device="cuda")
    dev = torch.device("cuda", local)
    dtc = 1 if wl.dtype == "bf16" else 0
    esz = 2 if wl.dtype == "bf16" else 4
    o = torch.empty((C, H, D), dtype=x["q"].dtype, device=dev)
    states = torch.empty((max(info["n_states"], 1), H, D, D), dtype=torch.float32, device=dev)
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, dtc) // esz, dtype=x["q"].dtype, device=dev)
    grads = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]), dv=torch.empty_like(x["v"]),
                 dg=torch.empty_like(x["g"]), dbeta=torch.empty_like(x["beta"]))
    wsb = torch.empty(max(pl.bwd_workspace_bytes(H, D, D), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fwd(inp):
        kda_fwd(pl, inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], o=o, states=states,
                chunk_states=cs)

    def bwd(inp, phase):
        kda_bwd(pl, inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["W"], states=states,
                chunk_states=cs, grads=grads, workspace=wsb, phase=phase)

    for _ in range(max(args.warmup, 3)):
        fwd(x); bwd(x, "state"); bwd(x, "grad")
    torch.cuda.synchronize()
    if pl.device_error() != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        fwd(x)
        ev[i][1].record(stream)
        bwd(x, "state")
        ev[i][2].record(stream)
        bwd(x, "grad")
        ev[i][3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    ph = np.array([[ev[i][0].elapsed_time(ev[i][1]), ev[i][1].elapsed_time(ev[i][2]),
                    ev[i][2].elapsed_time(ev[i][3])] for i in range(K)]).mean(0)
    if pl.device_error() != 0:
        raise RuntimeError("device error during the timed steps")
    C_all, ms = reduce_across_ranks(C, total_ms / K, dev)
    value = C_all / (ms / 1e3)

    # ---- end to end through the public API with host buffers --------------------------
    # Every step copies its inputs (q, k, v, g, beta and the loss weight W) from pinned
    # host memory, runs the forward and backward, and reads back the step's product: the
    # gradients dq, dk, dv, dg, dbeta and the loss L = sum W o.  Copies overlap compute:
    # step i + 1's inputs go up on one stream while step i computes, and step i's
    # gradients come down on another while step i + 1 computes (inputs and gradients are
    # double-buffered on the device).  `all_outputs` times the plain serial variant that
    # also reads o back and overlaps nothing.
    e2e = None
    if not args.no_e2e:
        host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in x.items()}
        for k in host_in:
            host_in[k].copy_(x[k])
        bufs = [{k: torch.empty_like(v) for k, v in x.items()} for _ in range(2)]
        gbufs = [grads] + [{k: torch.empty_like(v) for k, v in grads.items()}]
        host_g = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in grads.items()}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        K2 = max(2, K)
        loss_dev = torch.empty((), dtype=o.dtype, device=dev)
        loss_host = torch.empty((K2 + 1,), dtype=o.dtype, pin_memory=True)
        d2h = sum(t.numel() * t.element_size() for t in host_g.values()) + loss_dev.element_size()
        copy_s = torch.cuda.Stream(device=dev)
        down_s = torch.cuda.Stream(device=dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        buf_free = [torch.cuda.Event() for _ in range(2)]
        g_ready = [torch.cuda.Event() for _ in range(2)]
        g_free = [torch.cuda.Event() for _ in range(2)]

        def issue_copy(i):
            b_ = i & 1
            if i >= 2:
                copy_s.wait_event(buf_free[b_])
            with torch.cuda.stream(copy_s):
                for k in host_in:
                    bufs[b_][k].copy_(host_in[k], non_blocking=True)
            in_ready[b_].record(copy_s)

        def compute(i):
            b_ = i & 1
            stream.wait_event(in_ready[b_])
            if i >= 2:
                stream.wait_event(g_free[b_])
            inp = bufs[b_]
            fwd(inp)
            kda_bwd(pl, inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["W"], states=states,
                    chunk_states=cs, grads=gbufs[b_], workspace=wsb, phase="state")
            kda_bwd(pl, inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["W"], states=states,
                    chunk_states=cs, grads=gbufs[b_], workspace=wsb, phase="grad")
            torch.dot(inp["W"].view(-1), o.view(-1), out=loss_dev)
            buf_free[b_].record(stream)
            loss_host[i].copy_(loss_dev, non_blocking=True)
            g_ready[b_].record(stream)
            down_s.wait_event(g_ready[b_])
            with torch.cuda.stream(down_s):
                for k in host_g:
                    host_g[k].copy_(gbufs[b_][k], non_blocking=True)
            g_free[b_].record(down_s)

        issue_copy(0); compute(0)                       # warm the pipeline once
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        a0 = torch.cuda.Event(enable_timing=True); a1 = torch.cuda.Event(enable_timing=True)
        a0.record(copy_s)
        issue_copy(0)
        for i in range(K2):
            if i + 1 < K2:
                issue_copy(i + 1)
            compute(i)
        stream.wait_stream(down_s)
        a1.record(stream)
        torch.cuda.synchronize()
        _, ems = reduce_across_ranks(C, a0.elapsed_time(a1) / K2, dev)
        e2e = dict(value=round(C_all / (ems / 1e3), 1), unit=UNIT, h2d_bytes_per_step=int(h2d),
                   d2h_bytes_per_step=int(d2h), ms_per_step=round(ems, 3),
                   loss=float(loss_host[K2 - 1]), returns="dq, dk, dv, dg, dbeta and the loss",
                   overlap="step i+1's inputs copied up and step i's gradients copied down during compute")
        # serial variant: copy in, compute, read the output and every gradient back
        outs = dict(o=o, **grads)
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
        d2h_all = sum(t.numel() * t.element_size() for t in host_out.values())
        b0 = torch.cuda.Event(enable_timing=True); b1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        b0.record(stream)
        for _ in range(2):
            for k in host_in:
                bufs[0][k].copy_(host_in[k], non_blocking=True)
            fwd(bufs[0]); bwd(bufs[0], "state"); bwd(bufs[0], "grad")
            for k in host_out:
                host_out[k].copy_(outs[k], non_blocking=True)
        b1.record(stream)
        torch.cuda.synchronize()
        _, ams = reduce_across_ranks(C, b0.elapsed_time(b1) / 2, dev)
        e2e["all_outputs"] = dict(value=round(C_all / (ams / 1e3), 1), ms_per_step=round(ams, 3),
                                  h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h_all))
        del host_in, host_out, host_g, bufs, gbufs
        torch.cuda.empty_cache()

    # ---- roofline ----------------------------------------------------------------------
    cm = cost_model(info, H, D, B)
    hbm, tf_burst, tf_sus, src = peaks()
    phase_ms = dict(fwd=float(ph[0]), bwd_state=float(ph[1]), bwd_grad=float(ph[2]))
    # bytes / flops attributed to each phase: the state pass reads its inputs and the
    # handoff gradients; the gradient pass does the rest of the backward
    phase_bytes = dict(fwd=cm["fwd_bytes"],
                       bwd_state=(info["C"] + info["R"]) * H * (3 * 2 * D + 2) + info["C"] * H * 2 * D
                       + 4 * D * D * H * 2 * info["n_cons"],
                       bwd_grad=cm["bwd_bytes"])
    phase_bytes["bwd_grad"] -= phase_bytes["bwd_state"]
    dom = max(phase_ms, key=phase_ms.get)
    kernel_name = {"fwd": "kda_fwd_tc2", "bwd_state": "kda_bwd_state_tc2", "bwd_grad": "kda_bwd_grad_tc2"}[dom]
    achieved = phase_bytes[dom] / (phase_ms[dom] / 1e3) / 1e9
    traffic = traffic_from_profiles(kernel_name)
    step_bytes = cm["fwd_bytes"] + cm["bwd_bytes"]
    step_flops = cm["fwd_flops"] + cm["bwd_flops"]
    t_mem, t_math = step_bytes / (hbm * 1e9), step_flops / (tf_sus * 1e12)
    t_star = max(t_mem, t_math)
    # nominal roofline, beside the measured-peak one: the slower of 8 TB/s HBM and the
    # nominal dense bf16 tensor peak (2.25 PFLOP/s) of one GB300
    ns_mem, ns_math = step_bytes / (NOMINAL_HBM_GBS * 1e9), step_flops / (NOMINAL_BF16_TFLOPS * 1e12)
    ns_t = max(ns_mem, ns_math)
    roofline = dict(bound="hbm" if t_mem >= t_math else "tensor", kernel=kernel_name,
                    achieved=round(achieved, 1), peak=hbm, unit="GB/s", frac=round(achieved / hbm, 4),
                    traffic=traffic, peak_source=f"{src} hbm_gbs",
                    step=dict(algorithmic_bytes=int(step_bytes), algorithmic_flops=int(step_flops),
                              bound="hbm" if t_mem >= t_math else "tensor",
                              t_star_ms=round(t_star * 1e3, 3), frac=round(t_star * 1e3 / ms, 4),
                              frac_of="measured peaks (MEASURED_PEAKS.json: copy GB/s, sustained bf16)"),
                    nominal=dict(hbm_gbs=NOMINAL_HBM_GBS, bf16_tflops=NOMINAL_BF16_TFLOPS,
                                 bound="hbm" if ns_mem >= ns_math else "tensor",
                                 t_star_ms=round(ns_t * 1e3, 3), frac=round(ns_t * 1e3 / ms, 4),
                                 kernel_frac=round(achieved / NOMINAL_HBM_GBS, 4)))

    expanded = None
    if not args.no_expanded:
        expanded = run_expanded(parent, seg_len, pl, x, wl, ms)
    nodewise = None
    if args.nodewise:
        nodewise = run_nodewise(parent, seg_len, pl, x, wl, ms)
    conv = None
    if args.conv:
        conv = run_conv(pl, x, wl, hbm)
    lp = None
    if args.logprob:
        lp = run_logprob(hbm)
    attn = None
    if args.attn:
        attn = run_attn(parent, seg_len, pl, x, tf_burst)
    fidelity = None
    if args.fidelity:
        fidelity = run_fidelity(parent, seg_len, pl, x, wl)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        c_s, h_s, dt, thr, st = oracle_sample(parent, seg_len, pl.arrays()["seg_offset"], x, H, B,
                                              target_S=12000)
        cpu = dict(value=round(c_s / dt, 2), unit=UNIT, cores=thr, kind="oracle", arch=platform.machine(),
                   sample=f"one tree of the forest ({c_s} compact / {st['S']} expanded tokens, "
                          f"all {h_s} heads), fp64 token recurrence fwd+bwd, {dt:.1f} s")

    if rank == 0:
        line = dict(metric=METRIC, value=round(value, 1), unit=UNIT, n_gpus=ws, steps=K,
                    warmup=max(args.warmup, 3), ms_per_step=round(ms, 3), higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype=wl.dtype, data="synthetic",
                    config=dict(workload=args.workload, trees=wl.n_trees, C=C, S=info["S"],
                                R=info["R"], calls=info["n_rounds"], sequences=info["n_seq"],
                                states=info["n_states"], H=H, dk=D, dv=D, chunk=B,
                                parallelism=f"dp{ws} (one forest per GPU)",
                                l2=f"inputs larger than L2 (each input tensor {C * H * D * 2 / 1e9:.2f} GB)"),
                    phases_ms={k: round(v, 3) for k, v in phase_ms.items()},
                    host_ms=dict(plan=round(plan_ms, 3), upload=round(upload_ms, 3)),
                    gpu_launches=K * (2 * info["n_rounds"] + 1 + (1 if info["n_fold_rows"] else 0)),
                    roofline=roofline, cpu_baseline=cpu, e2e=e2e, clocks=clk)
        if expanded:
            line["expanded"] = expanded
        if nodewise:
            line["nodewise"] = nodewise
        if fidelity:
            line["fidelity"] = fidelity
        if conv:
            line["conv"] = conv
        if lp:
            line["logprob"] = lp
        if attn:
            line["attn"] = attn
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_expanded(parent, seg_len, pl_tree, x, wl, tree_ms):
    """Same kernels on the trajectory-expanded input: every root-to-leaf trajectory is
    its own root sequence (S rows, one round)."""
    import numpy as np
    import torch
    from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
    from prefix_shared_chunkwise_gb300.synth import expand_rows
    rows, ptr, _ = expand_rows(parent, seg_len, pl_tree.arrays()["seg_offset"])
    n_traj = len(ptr) - 1
    e_parent = -np.ones(n_traj, np.int32)
    e_len = np.diff(ptr).astype(np.int64)
    pl = Plan(e_parent, e_len, wl.chunk).upload()
    H, D = wl.H, wl.dk
    idx = torch.as_tensor(rows, device=x["q"].device)
    xe = {k: v.index_select(0, idx) for k, v in x.items()}
    dev = x["q"].device
    o = torch.empty_like(xe["v"])
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, 1) // 2, dtype=torch.bfloat16, device=dev)
    grads = dict(dq=torch.empty_like(xe["q"]), dk=torch.empty_like(xe["k"]), dv=torch.empty_like(xe["v"]),
                 dg=torch.empty_like(xe["g"]), dbeta=torch.empty_like(xe["beta"]))
    wsb = torch.empty(max(pl.bwd_workspace_bytes(H, D, D), 256), dtype=torch.uint8, device=dev)

    def step():
        kda_fwd(pl, xe["q"], xe["k"], xe["v"], xe["g"], xe["beta"], o=o, chunk_states=cs)
        kda_bwd(pl, xe["q"], xe["k"], xe["v"], xe["g"], xe["beta"], xe["W"], states=None,
                chunk_states=cs, grads=grads, workspace=wsb)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        step()
    e1.record()
    torch.cuda.synchronize()
    ems = e0.elapsed_time(e1) / 3
    return dict(rows=int(pl.info["C"]), trajectories=n_traj, ms_per_step=round(ems, 3),
                speedup_tree_vs_expanded=round(ems / tree_ms, 3))


def run_nodewise(parent, seg_len, pl_tree, x, wl, tree_ms):
    """Same kernels on the node-wise plan of the same forest (one sequence per segment,
    one call per tree level, handoffs at segment ends): the pages' "Node-wise LA"
    comparison.  The inputs are moved into that plan's row layout first (untimed)."""
    import numpy as np
    import torch
    from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
    pl = Plan(parent, seg_len, wl.chunk, nodewise=True).upload()
    so_t = pl_tree.arrays()["seg_offset"]
    so_n = pl.arrays()["seg_offset"]
    C = int(pl.info["C"])
    rows = np.empty(C, np.int64)
    for v in range(len(parent)):
        rows[so_n[v]:so_n[v] + seg_len[v]] = so_t[v] + np.arange(seg_len[v])
    H, D = wl.H, wl.dk
    dev = x["q"].device
    idx = torch.as_tensor(rows, device=dev)
    xn = {k: t.index_select(0, idx) for k, t in x.items()}
    o = torch.empty_like(xn["v"])
    st = torch.empty((max(pl.info["n_states"], 1), H, D, D), dtype=torch.float32, device=dev)
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, 1) // 2, dtype=torch.bfloat16, device=dev)
    grads = dict(dq=torch.empty_like(xn["q"]), dk=torch.empty_like(xn["k"]), dv=torch.empty_like(xn["v"]),
                 dg=torch.empty_like(xn["g"]), dbeta=torch.empty_like(xn["beta"]))
    wsb = torch.empty(max(pl.bwd_workspace_bytes(H, D, D), 256), dtype=torch.uint8, device=dev)

    def step():
        kda_fwd(pl, xn["q"], xn["k"], xn["v"], xn["g"], xn["beta"], o=o, states=st, chunk_states=cs)
        kda_bwd(pl, xn["q"], xn["k"], xn["v"], xn["g"], xn["beta"], xn["W"], states=st,
                chunk_states=cs, grads=grads, workspace=wsb)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        step()
    e1.record()
    torch.cuda.synchronize()
    nms = e0.elapsed_time(e1) / 5
    return dict(calls=int(pl.info["n_rounds"]), sequences=int(pl.info["n_seq"]),
                states=int(pl.info["n_states"]), chunks=int(pl.info["n_chunks"]),
                ms_per_step=round(nms, 3), speedup_tree_vs_nodewise=round(nms / tree_ms, 3))


def run_logprob(hbm):
    """Compact-to-semantic log-probabilities on the 64K-token forest (fb64k_bf16) at the
    pages' vocabulary (157,184), bf16 logits: CUDA-event times of harts_logprob_fwd and
    _bwd, algorithmic bytes (fwd reads the C x V logits; bwd reads them and writes the
    gradient) against the HBM peak, and S / C, the factor of vocabulary work that the
    compact rows save over S x V expanded logits."""
    import torch
    from prefix_shared_chunkwise_gb300.api import Plan, logprob_bwd, logprob_fwd, semantic_map
    from prefix_shared_chunkwise_gb300.synth import make_tree
    parent, seg_len = make_tree("fb64k_bf16")
    pl = Plan(parent, seg_len, 64)
    sem_row, row_ptr, row_sem = semantic_map(pl)
    C, S, V = int(pl.info["C"]), len(sem_row), 157_184
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(21)
    z = (torch.randn((C, V), generator=g, device=dev) * 3).to(torch.bfloat16)
    target = torch.randint(0, V, (S,), generator=g, device=dev, dtype=torch.int32)
    dl = torch.randn(S, generator=g, device=dev)
    rp, rs = torch.as_tensor(row_ptr, device=dev), torch.as_tensor(row_sem, device=dev)
    logp = torch.empty(S, device=dev)
    lse = torch.empty(C, device=dev)
    dz = torch.empty_like(z)

    def timed(fn, reps=5):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    tf = timed(lambda: logprob_fwd(z, rp, rs, target, lse=lse, logp=logp))
    tb = timed(lambda: logprob_bwd(z, rp, rs, target, lse, dl, dlogits=dz))
    fb, bb = C * V * 2, 2 * C * V * 2
    # the oracle beside it: forward + backward on sampled compact rows with their positions
    import numpy as np
    from oracle import logprob as olp
    rng = np.random.default_rng(0)
    tg, dlh = target.cpu().numpy(), dl.cpu().numpy()

    def some_rows():
        cs = rng.integers(0, C, size=8)
        zc = z[torch.as_tensor(cs, device=dev)].double().cpu().numpy()
        pos = [row_sem[row_ptr[c]:row_ptr[c + 1]] for c in cs]
        sr = np.concatenate([np.full(len(pp), j) for j, pp in enumerate(pos)]).astype(np.int64)
        pp = np.concatenate(pos).astype(np.int64)
        olp.logprob_fwd(zc, sr, tg[pp])
        olp.logprob_bwd(zc, sr, tg[pp], dlh[pp])
        return len(cs)

    n_o, t_o = oracle_rate(some_rows)
    oracle_leg = dict(value=round(n_o / t_o, 2), unit="compact rows/s (fwd + bwd, V = 157,184)",
                      gpu=round(C / ((tf + tb) / 1e3), 1), cores=len(os.sched_getaffinity(0)), kind="oracle",
                      sample=f"{n_o} uniformly drawn rows with their semantic positions, {t_o:.1f} s")
    out = dict(C=C, S=S, V=V, vocab_work_saved=round(S / C, 3), oracle=oracle_leg,
               fwd=dict(ms=round(tf, 3), gb_s=round(fb / tf / 1e6, 1), frac=round(fb / tf / 1e6 / hbm, 3)),
               bwd=dict(ms=round(tb, 3), gb_s=round(bb / tb / 1e6, 1), frac=round(bb / tb / 1e6 / hbm, 3)),
               peak_gb_s=hbm)
    del z, dz
    torch.cuda.empty_cache()
    return out


def run_attn(parent, seg_len, pl, x, tf_peak):
    """Branch attention over the compact layout on the forest's q, k, v ([C, H, 128] bf16):
    CUDA-event times of harts_attn_fwd and harts_attn_bwd, algorithmic FLOPs (per head and
    visible (query, key) pair: 4 d forward, Q K^T and P V; 10 d backward, S, dP, dV, dQ,
    dK) against the bf16 tensor peak, the FLOPs of
    the 128 x 128 tiles the kernel issues (masked entries included), and the pairs the
    per-trajectory execution would compute instead (every trajectory causally over its
    own tokens)."""
    import numpy as np
    import torch
    from prefix_shared_chunkwise_gb300.api import attn_bwd, attn_fwd
    C, H, d = x["q"].shape
    a = pl.arrays()
    pos, ln = a["seg_pos"].astype(np.float64), np.asarray(seg_len, np.float64)
    pairs = float((ln * pos + ln * (ln + 1) / 2).sum())
    # the kernel's tiles: per sequence and 128-query tile, keys up to the tile's last query
    cu, fs = a["cu_seqlens"], a["seq_first_seg"]
    tiles = 0
    for i in range(len(fs)):
        own, h = int(cu[i + 1] - cu[i]), int(a["seg_pos"][fs[i]])
        for t in range((own + 127) // 128):
            tiles += (h + min(own, (t + 1) * 128) - 1) // 128 + 1
    # per-trajectory pairs: sum over leaves of L (L + 1) / 2
    parent = np.asarray(parent)
    depth_len = np.zeros(len(parent))
    for v in range(len(parent)):
        depth_len[v] = ln[v] + (depth_len[parent[v]] if parent[v] >= 0 else 0)
    leaf = np.ones(len(parent), bool)
    leaf[parent[parent >= 0]] = False
    traj_pairs = float((depth_len[leaf] * (depth_len[leaf] + 1) / 2).sum())
    o = torch.empty_like(x["q"])
    lse = torch.empty((C, H), dtype=torch.float32, device=o.device)

    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    do = x["v"]                                      # any [C, H, d] bf16 tensor serves as dL/do
    from prefix_shared_chunkwise_gb300 import _lib
    ws = torch.empty(max(int(_lib.lib().harts_attn_bwd_workspace_bytes(pl.handle, H)), 256), dtype=torch.uint8,
                     device=o.device)

    def fwd():
        attn_fwd(pl, x["q"], x["k"], x["v"], o=o, lse=lse)

    def bwd():
        attn_bwd(pl, x["q"], x["k"], x["v"], o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws)

    def timed(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    ms = timed(fwd)
    ms_b = timed(bwd)
    if pl.device_error() != 0:                       # a wait ran out: the times mean nothing
        raise RuntimeError("branch attention reported a device error")
    flops = 4.0 * d * H * pairs
    flops_b = 10.0 * d * H * pairs                   # S, dP, dV, dQ, dK: 2 d each per pair
    tile_flops = 4.0 * d * H * tiles * 128 * 128
    # the oracle beside it: forward + backward of uniformly sampled compact rows over their
    # trajectory prefixes (all heads), fp64 on the host
    from oracle import attn as oattn
    rng = np.random.default_rng(0)
    so = a["seg_offset"]

    def one_row():
        r = int(rng.integers(0, C))
        view = oattn.trajectory_prefix(parent, seg_len, so, r)
        idx = torch.as_tensor(view, device=o.device)
        qq = x["q"][r].double().cpu().numpy()
        kk, vv = x["k"][idx].double().cpu().numpy(), x["v"][idx].double().cpu().numpy()
        oattn.attn_query(qq, kk, vv, d ** -0.5)
        oattn.attn_query_bwd(qq, kk, vv, do[r].double().cpu().numpy(), d ** -0.5)
        return 1

    n_o, t_o = oracle_rate(one_row)
    oracle_leg = dict(value=round(n_o / t_o, 2), unit="compact query rows/s (fwd + bwd, all heads)",
                      gpu=round(C / ((ms + ms_b) / 1e3), 1), cores=len(os.sched_getaffinity(0)), kind="oracle",
                      sample=f"{n_o} uniformly drawn rows of the forest, {t_o:.1f} s")
    return dict(shape=[C, H, d], ms=round(ms, 3), visible_pairs=int(pairs), oracle=oracle_leg,
                tflops=round(flops / ms / 1e9, 1), frac=round(flops / ms / 1e9 / tf_peak, 4),
                tile_tflops=round(tile_flops / ms / 1e9, 1), tile_util=round(pairs * H / (tiles * 128 * 128 * H), 3),
                bwd=dict(ms=round(ms_b, 3), tflops=round(flops_b / ms_b / 1e9, 1),
                         frac=round(flops_b / ms_b / 1e9 / tf_peak, 4)),
                per_trajectory_pairs=int(traj_pairs), work_saved=round(traj_pairs / pairs, 3),
                peak_tflops=tf_peak, peak_source="bf16_tflops (burst, kernel timed alone)")


def run_conv(pl, x, wl, hbm):
    """Short convolution over the compact layout on the forest's q ([C, H*dk] bf16), width
    4, SiLU, with bias: CUDA-event times of harts_conv_fwd and harts_conv_bwd, and their
    algorithmic bytes (fwd: read x, write y; bwd: read x and dy, write dx; weights are
    negligible) against the HBM peak.  Inputs are larger than L2."""
    import torch
    from prefix_shared_chunkwise_gb300.api import conv_bwd, conv_fwd
    C = int(pl.info["C"])
    xx = x["q"].reshape(C, -1)
    ch = xx.shape[1]
    g = torch.Generator(device=xx.device).manual_seed(11)
    W = torch.randn((ch, 4), generator=g, device=xx.device) * 0.5
    b = torch.randn(ch, generator=g, device=xx.device)
    dy = x["v"].reshape(C, -1)
    y = torch.empty_like(xx)
    dx = torch.empty_like(xx)
    dW = torch.empty_like(W)
    db = torch.empty_like(b)

    def timed(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    tf = timed(lambda: conv_fwd(pl, xx, W, b, activation="silu", y=y))
    tb = timed(lambda: conv_bwd(pl, xx, W, b, dy, activation="silu", dx=dx, dweight=dW, dbias=db))
    elem = C * ch * xx.element_size()
    fb, bb = 2 * elem, 3 * elem
    # the oracle beside it: forward + backward over one tree of the forest, 256 channels at
    # a time until the time budget is spent
    import numpy as np
    from oracle import conv as oconv
    from prefix_shared_chunkwise_gb300.synth import make_tree
    parent, seg_len = make_tree(wl.name)
    ids, sub_parent, st = pick_sample_tree(parent, seg_len, 4000)
    so = pl.arrays()["seg_offset"]
    rows = np.concatenate([np.arange(so[v], so[v] + seg_len[v]) for v in ids])
    sub_off = np.concatenate([[0], np.cumsum(seg_len[ids])[:-1]]).astype(np.int64)
    idx = torch.as_tensor(rows, device=xx.device)
    xs_all, dys_all = xx.index_select(0, idx), dy.index_select(0, idx)
    blk = [0]

    def one_block():
        c0 = (blk[0] * 256) % ch
        blk[0] += 1
        xs = xs_all[:, c0:c0 + 256].double().cpu().numpy()
        dys = dys_all[:, c0:c0 + 256].double().cpu().numpy()
        Ws, bs = W[c0:c0 + 256].double().cpu().numpy(), b[c0:c0 + 256].double().cpu().numpy()
        oconv.conv_forest(sub_parent, seg_len[ids], sub_off, xs, Ws, bs, act="silu")
        oconv.conv_forest_bwd(sub_parent, seg_len[ids], sub_off, xs, Ws, bs, "silu", dys)
        return len(rows) * 256

    n_o, t_o = oracle_rate(one_block, budget_s=3.0, max_units=10 ** 12)
    oracle_leg = dict(value=round(n_o / t_o, 1), unit="row-channels/s (fwd + bwd)",
                      gpu=round(C * ch / ((tf + tb) / 1e3), 1), cores=1, kind="oracle",
                      sample=f"one tree ({len(rows)} compact rows) x {n_o // len(rows)} channels, {t_o:.1f} s")
    return dict(shape=[C, ch], width=4, activation="silu", oracle=oracle_leg,
                fwd=dict(ms=round(tf, 3), gb_s=round(fb / tf / 1e6, 1), frac=round(fb / tf / 1e6 / hbm, 3)),
                bwd=dict(ms=round(tb, 3), gb_s=round(bb / tb / 1e6, 1), frac=round(bb / tb / 1e6 / hbm, 3)),
                peak_gb_s=hbm)


def run_fidelity(parent, seg_len, pl_tree, x, wl):
    """Forward outputs of the tree plans against the per-trajectory run of the same
    kernels (every root-to-leaf trajectory its own sequence, chunk grid from its start):
    the pages' replay-vs-no-replay fidelity comparison (section 5.3, Fig. 5), with the
    per-trajectory run as the baseline.  Per handoff depth (sequence boundaries on the
    path from the root to a row's segment, in each plan): rows, rel. L2 and max |diff|
    of o, and the fraction of rows bit-identical to the baseline."""
    import numpy as np
    import torch
    from prefix_shared_chunkwise_gb300.api import Plan, kda_fwd
    from prefix_shared_chunkwise_gb300.synth import expand_rows
    n = len(parent)
    so_t = pl_tree.arrays()["seg_offset"]
    rows, ptr, _ = expand_rows(parent, seg_len, so_t)
    dev = x["q"].device
    keys = ("q", "k", "v", "g", "beta")

    def fwd(pl, xx):
        o = torch.empty_like(xx["v"])
        st = torch.empty((max(pl.info["n_states"], 1), wl.H, wl.dk, wl.dv), dtype=torch.float32, device=dev)
        kda_fwd(pl, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], o=o, states=st)
        torch.cuda.synchronize()
        return o

    # baseline: one root sequence per trajectory
    idx = torch.as_tensor(rows, device=dev)
    n_traj = len(ptr) - 1
    pl_e = Plan(-np.ones(n_traj, np.int32), np.diff(ptr).astype(np.int64), wl.chunk).upload()
    o_base = fwd(pl_e, {k: x[k].index_select(0, idx) for k in keys})
    # segment of every compact row of the tree layout
    seg_of_row = np.empty(int(pl_tree.info["C"]), np.int64)
    for v in range(n):
        seg_of_row[so_t[v]:so_t[v] + seg_len[v]] = v
    seg_of_exp = seg_of_row[rows]

    def depth_of(pl):
        ss = pl.arrays()["seg_seq"]
        d = np.zeros(n, np.int64)
        for v in range(n):
            d[v] = 0 if parent[v] < 0 else d[parent[v]] + (ss[v] != ss[parent[v]])
        return d

    # the baseline's own spread: a shared row computed in several trajectories (with
    # different chunk-mates where the trajectories fork) against its first occurrence
    _, first = np.unique(rows, return_index=True)
    first_of = np.empty(int(pl_tree.info["C"]), np.int64)
    first_of[rows[first]] = first
    o_first = o_base.index_select(0, torch.as_tensor(first_of[rows], device=dev))
    out = {}
    d_row = depth_of(pl_tree)[seg_of_exp]
    spread = {}
    for dd in range(int(d_row.max()) + 1):
        sel = torch.as_tensor(np.nonzero(d_row == dd)[0], device=dev)
        if sel.numel() == 0:
            continue
        a_, b_ = o_first.index_select(0, sel), o_base.index_select(0, sel)
        spread[str(dd)] = dict(rel_l2=float((a_.float() - b_.float()).norm() / b_.float().norm()),
                               bit_identical=round(float((a_ == b_).all(dim=2).all(dim=1).float().mean()), 6))
    out["baseline_spread"] = dict(by_handoff_depth=spread)
    for name, kw in (("harts", {}), ("noreplay", {"noreplay": True})):
        pl = pl_tree if not kw else Plan(parent, seg_len, wl.chunk, **kw).upload()
        so = pl.arrays()["seg_offset"]
        t2p = np.empty(int(pl.info["C"]), np.int64)     # tree-layout row -> this plan's row
        for v in range(n):
            t2p[so_t[v]:so_t[v] + seg_len[v]] = so[v] + np.arange(seg_len[v])
        p2t = np.empty_like(t2p)
        p2t[t2p] = np.arange(len(t2p))
        xp = {k: x[k].index_select(0, torch.as_tensor(p2t, device=dev)) for k in keys}
        o_p = fwd(pl, xp).index_select(0, torch.as_tensor(t2p[rows], device=dev))
        d_row = depth_of(pl)[seg_of_exp]
        per = {}
        for dd in range(int(d_row.max()) + 1):
            sel = torch.as_tensor(np.nonzero(d_row == dd)[0], device=dev)
            if sel.numel() == 0:
                continue
            op, ob = o_p.index_select(0, sel), o_base.index_select(0, sel)
            df = op.float() - ob.float()
            same = (op == ob).all(dim=2).all(dim=1)
            ob = ob.float()
            per[str(dd)] = dict(rows=int(sel.numel()),
                                rel_l2=float(df.norm() / ob.norm()),
                                max_abs=float(df.abs().max()),
                                bit_identical=round(float(same.float().mean()), 6))
        out[name] = dict(calls=int(pl.info["n_rounds"]), by_handoff_depth=per)
    return out


# ---- reference arm: the oracle on host cores ---------------------------------------------

def run_reference(args):
    import numpy as np
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import torch
    from prefix_shared_chunkwise_gb300.synth import WORKLOAD_ORDER, WORKLOADS, make_inputs, make_tree
    wl = WORKLOADS[args.workload]
    H, D, B = wl.H, wl.dk, wl.chunk
    seed = WORKLOAD_ORDER.index(args.workload)
    parent, seg_len = make_tree(args.workload, seed=seed)
    ids, sub_parent, st = pick_sample_tree(parent, seg_len, target_S=6000)
    # seeded inputs of the workload's distributions for the sampled tree only
    h_s = min(H, 8)
    sub = make_inputs(st["C"], h_s, D, D, wl.dtype, seed=3, device="cpu")
    host = {k: v.float().double().numpy() for k, v in sub.items()}
    sub_off = np.cumsum([0] + [int(seg_len[v]) for v in ids[:-1]]).astype(np.int64)
    import oracle
    threads = len(os.sched_getaffinity(0))

    def step():
        oracle.kda_forest(sub_parent, seg_len[ids], sub_off, host["q"], host["k"], host["v"],
                          host["g"], host["beta"], chunk=B, W=host["W"], n_threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.time()
    for _ in range(args.steps):
        step()
    dt = (time.time() - t0) / args.steps
    # the sample covers st["C"] compact tokens on h_s of H heads
    value = st["C"] * (h_s / H) / dt
    sample = (f"one tree ({st['C']} compact / {st['S']} expanded tokens), {h_s} of {H} heads, "
              f"fp64 token recurrence fwd+bwd per step")
    line = dict(metric=METRIC, value=round(value, 2), unit=UNIT, n_gpus=ws, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(dt * 1e3, 1), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=dict(workload=args.workload, trees=wl.n_trees, H=H, dk=D, dv=D, chunk=B),
                cpu_baseline=dict(value=round(value, 2), unit=UNIT, kind="oracle",
                                  cores=min(threads, h_s), sample=sample),
                e2e=dict(value=round(value, 2), unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
