"""Benchmark of the tree-masked attention hot path on GB300.

One step = the whole path over one tree: plan (host node pass + device kernels), RoPE at
depth positions, attention forward, the g_t/K loss weights on the upstream gradient, and
the backward (delta, dK/dV with on-chip reduction and the dQ accumulator, dQ finalize).
Inputs are resident in HBM before the timed region; the L2 (129 MB) is flushed by writing a
256 MiB buffer between steps, outside the CUDA-event brackets.

Metric: visible-pair TFLOP/s = 14 d Hq N_pairs / step time (forward 4 d, backward 10 d flops
per visible query-key pair per q head; N_pairs = sum_t (pos_t + 1)), plus tokens/s.
  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]
Under torchrun each rank runs its own tree (weak scaling, no data-path collective); rank 0
prints one JSON line with the max-over-ranks time.

Other single-GPU lines on the same tree: --partition (the tree as gateway partitions), --conv
(hybrid-layer causal convolution forward + backward, algorithmic GB/s), --ce (next-token
cross-entropy fused with the vocabulary projection, TFLOP/s).
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import CONFIGS, make_tensors, make_workload  # noqa: E402

METRIC = "tree-attn fwd+bwd visible-pair TFLOP/s and tokens/s on 1 GB300; % of bf16 peak"
UNIT = "TFLOP/s"
DEFAULT_CONFIG = "rollout32k"
# kernels of this library per step: plan (tokens with per-tile data, classes, lists and orders),
# RoPE, forward, backward (delta with the loss weights g/K folded in, and dQ-accumulator zeroing;
# dK/dV; dQ finalize)
LAUNCHES_PER_STEP = 3 + 1 + 1 + 3
DKDV_PROFILE = os.path.join(ROOT, "profiles", "k_bwd_dkdv_rollout32k.md")
DKDV_SOURCES = [os.path.join(ROOT, "tree_masked_attention_plan_gb300", "csrc", f) for f in ("attn_bwd.cu", "common.cuh")]


def source_digest(paths):
    import hashlib
    h = hashlib.sha1()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(config):
    """DRAM bytes per k_bwd_dkdv launch from the committed ncu summary, if that summary was taken
    on this workload with the kernel sources as they are now (else None: the counters are stale)."""
    try:
        with open(DKDV_PROFILE) as f:
            kv = dict(line.strip().lstrip("- ").split(": ", 1) for line in f if line.strip().lstrip("- ").startswith(
                ("source_sha1: ", "workload: ", "dram_bytes_per_launch: ")))
    except (OSError, ValueError):
        return None
    if kv.get("workload") != config or kv.get("source_sha1") != source_digest(DKDV_SOURCES):
        return None
    try:
        return int(float(kv["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def reduce_max(vals, device, world):
    """Per-rank timings -> their maximum over the ranks (every rank gets the result)."""
    t = torch.tensor([float(x) for x in vals], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(bf16=float(d["bf16_tflops"]), bf16_sustained=float(d.get("bf16_tflops_sustained", 0)) or None,
                    hbm=float(d["hbm_gbs"]), source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


def host_stats(parent, node_len):
    """N, K, N_pairs and N_flat from parent pointers (plain host loops, no oracle import)."""
    n = len(parent)
    depth_off = np.zeros(n, dtype=np.int64)
    leaves = np.zeros(n, dtype=np.int64)
    has_child = np.zeros(n, dtype=bool)
    for c in range(n):                                  # parents precede children in these trees
        if parent[c] >= 0:
            has_child[parent[c]] = True
    order = sorted(range(n), key=lambda v: _depth(parent, v))
    for v in order:
        if parent[v] >= 0:
            depth_off[v] = depth_off[parent[v]] + node_len[parent[v]]
    for leaf in np.nonzero(~has_child)[0]:
        v = leaf
        while v >= 0:
            leaves[v] += 1
            v = parent[v]
    L = node_len.astype(np.int64)
    n_pairs = int((L * depth_off + L * (L + 1) // 2).sum())
    N = int(L.sum())
    return dict(N=N, K=int((~has_child).sum()), n_pairs=n_pairs, n_flat=int((L * leaves).sum()))


def _depth(parent, v):
    d = 0
    while parent[v] >= 0:
        v = parent[v]
        d += 1
    return d


class ClockSampler:
    """nvidia-smi clock / throttle sampling every 25 ms; the summary keeps the samples whose
    timestamps fall inside the timed region (the region of a short run can be under 0.1 s)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 25

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        # nvidia-smi's start-up (driver queries) must not overlap the timed region: wait for its
        # first sample line (at most 10 s), then a little more
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 10.0:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                pass
            time.sleep(0.05)
        time.sleep(0.3)
        self.t0 = time.time()
        return self

    def __exit__(self, *a):
        self.t1 = time.time()
        time.sleep(2 * self.PERIOD_MS / 1000)     # the sample that covers the region's end
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows, stamps = [], []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    try:
                        stamps.append(datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp())
                    except ValueError:
                        stamps.append(None)
                    rows.append(parts[1:])
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if rows and self.t0 is not None and self.t1 is not None:
            inside = [r for r, t in zip(rows, stamps) if t is not None and self.t0 <= t <= self.t1 + self.PERIOD_MS / 1000]
            if inside:
                rows = inside
            else:                                  # a region shorter than the period: the nearest sample
                mid = 0.5 * (self.t0 + self.t1)
                timed = [(abs(t - mid), i) for i, t in enumerate(stamps) if t is not None]
                rows = [rows[min(timed)[1]]] if timed else rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        under = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": float(np.median(under)) if under else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def run_ours(args, rank, world, dev):
    import tree_masked_attention_plan_gb300 as tam
    torch.cuda.set_device(dev)
    wl = make_workload(args.config)
    st = host_stats(wl.parent, wl.node_len)
    t = make_tensors(wl)
    Hq, Hkv, d, N = wl.Hq, wl.Hkv, wl.d, st["N"]
    if args.shard == "heads":
        # this rank's kv-head group(s) of the one tree: its q / k / v / u heads, the whole plan
        from tree_masked_attention_plan_gb300.shard import kv_head_shard
        sh = kv_head_shard(Hq, Hkv, rank, world)
        t = {"q": t["q"][:, sh.q0:sh.q1].contiguous(), "k": t["k"][:, sh.kv0:sh.kv1].contiguous(),
             "v": t["v"][:, sh.kv0:sh.kv1].contiguous(), "u": t["u"][:, sh.q0:sh.q1].contiguous()}
        Hq, Hkv = sh.Hq, sh.Hkv
    stream = torch.cuda.current_stream()
    q, k, v, u = (t[x].to(dev) for x in ("q", "k", "v", "u"))
    status = tam.new_status(dev)
    plan = tam.tree_plan(wl.parent, wl.node_len, device=dev)
    Np = plan.n_pad
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    o = torch.empty_like(q)
    lse = torch.empty(Hq, Np, dtype=torch.float32, device=dev)
    ws = torch.empty(tam.tree_attn_bwd_workspace(plan, Hq, d), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    # one set of events per timed step: the host enqueues step i+1 (its plan's host pass
    # included) while the GPU runs step i, as a training loop does; the events are read once
    # after the last step
    evs = [{n: [torch.cuda.Event(enable_timing=True) for _ in range(2)] for n in ("step", "fwd", "plan", "rope")}
           for _ in range(max(args.steps, 1))]
    bwd_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(max(args.steps, 1))]
    for b in bwd_evs:                          # creates the CUDA events before the timed region
        tam.tree_set_timing_events(b)
    ev, bwd_ev = evs[0], bwd_evs[0]
    theta = wl.theta

    def step(p):
        ev["rope"][0].record(stream)
        tam.tree_rope_fwd(p, q, k, theta, qr=qr, kr=kr)
        ev["rope"][1].record(stream)
        ev["fwd"][0].record(stream)
        tam.tree_attn_fwd(p, qr, kr, v, o=o, lse=lse, status=status)
        ev["fwd"][1].record(stream)
        # the per-token loss weights g/K are applied inside the backward (no dO pass)
        tam.tree_attn_bwd_weighted(p, qr, kr, v, o, lse, u, rope_theta=theta, workspace=ws, dq=dq, dk=dk, dv=dv,
                                   status=status)

    def full_step():
        ev["step"][0].record(stream)
        ev["plan"][0].record(stream)
        p = tam.tree_plan(wl.parent, wl.node_len, device=dev)
        ev["plan"][1].record(stream)
        step(p)
        ev["step"][1].record(stream)
        return p

    tam.tree_set_timing_events(bwd_ev)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        full_step()
    torch.cuda.synchronize()
    tam.check_status(status, "warmup")
    times = {"step": [], "fwd": [], "bwd": [], "dkdv": [], "plan": [], "rope": []}
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(1.0)
            ev, bwd_ev = evs[i], bwd_evs[i]
            tam.tree_set_timing_events(bwd_ev)
            full_step()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    for e, b in zip(evs[:args.steps], bwd_evs[:args.steps]):
        times["step"].append(e["step"][0].elapsed_time(e["step"][1]))
        times["fwd"].append(e["fwd"][0].elapsed_time(e["fwd"][1]))
        times["plan"].append(e["plan"][0].elapsed_time(e["plan"][1]))
        times["rope"].append(e["rope"][0].elapsed_time(e["rope"][1]))
        times["bwd"].append(b[0].elapsed_time(b[3]))
        times["dkdv"].append(b[1].elapsed_time(b[2]))
    if world > 1:
        torch.distributed.barrier()
    tam.tree_set_timing_events([])
    tam.check_status(status, "timed steps")
    clocks = clk.summary()

    res = dict(st=st, wl=wl, times=times, wall=wall, clocks=clocks, e2e_ms=float("nan"), h2d=0, d2h=0,
               nnz=int(plan.arrays()["counts"][0].item()), Hq_local=Hq, Hkv_local=Hkv, T=plan.n_tiles,
               n_nodes=len(wl.parent))
    if args.no_e2e:
        return res
    # e2e: the same step through the public API from pinned host buffers; every step copies its
    # inputs in and its outputs out.  As a training input pipeline does, step i+1's inputs are
    # copied in and step i's outputs copied out on side streams while the next step computes
    # (two device buffers of each); the timed span runs from the first step's copy-in to the
    # last step's copy-out, divided by the number of steps.  Inputs (671 MB) exceed L2.  Within a
    # step the copies follow the data: K, V, Q come in before U (first read by the loss weights,
    # after the forward), and O goes out as soon as the forward has written it (during the
    # backward), dQ, dK, dV after the backward.
    o_ref, dk_ref, dv_ref = o.clone(), dk.clone(), dv.clone()
    host_in = tuple(t[x].pin_memory() for x in ("q", "k", "v", "u"))
    host_out = tuple(torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (o, dq, dk, dv))
    h2d = sum(x.numel() * x.element_size() for x in host_in) + 8 * len(wl.parent)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    ins = [(q, k, v, u), tuple(torch.empty_like(x) for x in (q, k, v, u))]
    outs = [(o, dq, dk, dv), tuple(torch.empty_like(x) for x in (o, dq, dk, dv))]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    qkv_ready, u_ready, fwd_done, comp_done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(5))

    def copy_in(i):
        b = i % 2
        if i >= 2:
            s_in.wait_event(comp_done[b])          # step i-2 has finished reading these buffers
        with torch.cuda.stream(s_in):
            for j in (1, 2, 0):                    # K, V, Q: what RoPE and the forward read
                ins[b][j].copy_(host_in[j], non_blocking=True)
            qkv_ready[b].record(s_in)
            ins[b][3].copy_(host_in[3], non_blocking=True)
            u_ready[b].record(s_in)

    def compute(i):
        b = i % 2
        qq, kk, vv, uu = ins[b]
        oo, dqq, dkk, dvv = outs[b]
        stream.wait_event(qkv_ready[b])
        if i >= 2:
            stream.wait_event(out_done[b])         # step i-2's outputs have left these buffers
        p = tam.tree_plan(wl.parent, wl.node_len, device=dev)
        tam.tree_rope_fwd(p, qq, kk, theta, qr=qr, kr=kr)
        tam.tree_attn_fwd(p, qr, kr, vv, o=oo, lse=lse, status=status)
        fwd_done[b].record(stream)
        stream.wait_event(u_ready[b])
        tam.tree_attn_bwd_weighted(p, qr, kr, vv, oo, lse, uu, rope_theta=theta, workspace=ws, dq=dqq, dk=dkk, dv=dvv,
                          status=status)
        comp_done[b].record(stream)

    def copy_out(i):
        b = i % 2
        with torch.cuda.stream(s_out):
            s_out.wait_event(fwd_done[b])
            host_out[0].copy_(outs[b][0], non_blocking=True)
            s_out.wait_event(comp_done[b])
            for j in (1, 2, 3):
                host_out[j].copy_(outs[b][j], non_blocking=True)
        out_done[b].record(s_out)

    def pipeline(n, e_start=None, e_end=None):
        if e_start is not None:
            e_start.record(s_in)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)
        if e_end is not None:
            e_end.record(s_out)

    torch.cuda.synchronize()
    pipeline(args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pipeline(args.steps, e0, e1)
    torch.cuda.synchronize()
    e2e_ms = [e0.elapsed_time(e1) / args.steps]
    tam.check_status(status, "e2e steps")
    for name, got, ref in (("o", host_out[0], o_ref), ("dk", host_out[2], dk_ref), ("dv", host_out[3], dv_ref)):
        if not torch.equal(got.to(dev), ref):
            raise RuntimeError(f"e2e pipeline: {name} differs from the device-timed step's")

    res.update(e2e_ms=float(np.mean(e2e_ms)), h2d=h2d, d2h=d2h)
    return res


def run_partitioned(args, dev):
    """The same tree run as partitions (Tree Training explainer, section 8.2): cut below the node
    whose children's subtrees hold the most tokens; parent partition, then each child partition
    with the gateway K/V gathered from the parent's rotated k / v, fp32 gateway gradients summed
    over the children and relayed into the parent's dK, dV.  Timed per step: every partition's
    plan, RoPE, forward and backward, the gateway gathers and the relay.  Each partition's dO
    (whole-tree loss weights) is prepared before the timed region."""
    import tree_masked_attention_plan_gb300 as tam
    from tree_masked_attention_plan_gb300.partition import largest_cut, partition_tree
    torch.cuda.set_device(dev)
    wl = make_workload(args.config)
    st = host_stats(wl.parent, wl.node_len)
    t = make_tensors(wl)
    Hq, Hkv, d, theta = wl.Hq, wl.Hkv, wl.d, wl.theta
    cut = largest_cut(wl.parent, wl.node_len)
    P = partition_tree(wl.parent, wl.node_len, cut)
    status = tam.new_status(dev)
    full_plan = tam.tree_plan(wl.parent, wl.node_len, device=dev)
    dO_full = tam.tree_apply_weights(full_plan, t["u"].to(dev))
    parts = [P["parent"]] + P["children"]
    bufs = []
    for part in parts:
        idx = torch.as_tensor(part.tokens, device=dev)
        q, k, v = (t[x].to(dev)[idx].contiguous() for x in ("q", "k", "v"))
        bufs.append(dict(idx=idx, q=q, k=k, v=v, dO=dO_full[idx].contiguous(), qr=torch.empty_like(q),
                         kr=torch.empty_like(k), o=torch.empty_like(q), dq=torch.empty_like(q),
                         dk=torch.empty_like(k), dv=torch.empty_like(v)))
    A = P["A"]
    rows = torch.as_tensor(P["gw_rows"], dtype=torch.int32, device=dev)
    k_gw = torch.empty(A, Hkv, d, dtype=torch.bfloat16, device=dev)
    v_gw = torch.empty_like(k_gw)
    dk_gw = torch.zeros(A, Hkv, d, dtype=torch.float32, device=dev)
    dv_gw = torch.zeros_like(dk_gw)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        plans = [tam.tree_plan(part.parent, part.node_len, device=dev, pos_offset=part.pos_offset) for part in parts]
        for pl, b in zip(plans, bufs):
            tam.tree_rope_fwd(pl, b["q"], b["k"], theta, qr=b["qr"], kr=b["kr"])
        b0 = bufs[0]
        o0, lse0 = tam.tree_attn_fwd(plans[0], b0["qr"], b0["kr"], b0["v"], o=b0["o"], status=status)
        tam.tree_gather_rows(rows, b0["kr"], out=k_gw)
        tam.tree_gather_rows(rows, b0["v"], out=v_gw)
        tam.tree_attn_bwd(plans[0], b0["qr"], b0["kr"], b0["v"], o0, lse0, b0["dO"], rope_theta=theta,
                          dq=b0["dq"], dk=b0["dk"], dv=b0["dv"], status=status)
        dk_gw.zero_()
        dv_gw.zero_()
        for pl, b in zip(plans[1:], bufs[1:]):
            o, lse = tam.tree_attn_fwd_gateway(pl, k_gw, v_gw, b["qr"], b["kr"], b["v"], o=b["o"], status=status)
            tam.tree_attn_bwd_gateway(pl, k_gw, v_gw, b["qr"], b["kr"], b["v"], o, lse, b["dO"], dk_gw, dv_gw,
                                      rope_theta=theta, dq=b["dq"], dk=b["dk"], dv=b["dv"], status=status)
        tam.tree_relay_add(rows, dk_gw, dv_gw, b0["dk"], b0["dv"])

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    tam.check_status(status, "partitioned warmup")
    # per-step events, read after the last step (the host enqueues ahead of the GPU)
    eps = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for e0, e1 in eps:
            flush.fill_(1.0)
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize()
    ms = [e0.elapsed_time(e1) for e0, e1 in eps]
    tam.check_status(status, "partitioned steps")
    info = dict(cut_node=int(cut), gateway_tokens=A, parent_tokens=int(len(P["parent"].tokens)),
                child_tokens=[int(len(c.tokens)) for c in P["children"]])
    return dict(st=st, wl=wl, ms=float(np.mean(ms)), clocks=clk.summary(), info=info,
                launches=LAUNCHES_PER_STEP * (1 + len(P["children"])) + 3)


CONV_METRIC = "tree causal conv1d fwd+bwd algorithmic GB/s on 1 GB300 (hybrid-layer context, section 9.2)"


def run_conv(args, dev):
    """Hybrid-layer depthwise causal convolution along root paths (Tree Training explainer,
    section 9.2), forward and backward with bias, on the workload's tree: x, dy [N, C] bf16, taps
    [K, C] fp32.  Algorithmic bytes: forward reads x and writes y (4 B per element), backward
    reads x and dy and writes dx (6 B per element); the taps and dw are negligible."""
    import tree_masked_attention_plan_gb300 as tam
    from workloads import make_conv_tensors
    torch.cuda.set_device(dev)
    wl = make_workload(args.config)
    C, K = args.conv_channels, args.conv_k
    plan = tam.tree_plan(wl.parent, wl.node_len, device=dev)
    N = plan.n_tokens
    tree = tam.tree_arrays(wl.parent, wl.node_len, dev)
    t = make_conv_tensors(N, C, K, seed=11)
    x, w, b, dy = t["x"].to(dev), t["w"].to(dev), t["bias"].to(dev), t["u"].to(dev)
    y = torch.empty_like(x)
    ws = torch.empty(tam.tree_conv1d_bwd_workspace(plan, C), dtype=torch.uint8, device=dev)
    dx, dw, db = torch.empty_like(x), torch.empty_like(w), torch.empty_like(b)
    lib = tam._lib()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    status = tam.new_status(dev)
    st = status.data_ptr()

    def step():
        tam._check(lib.tree_conv1d_fwd(plan.ref(), tree[0].data_ptr(), tree[1].data_ptr(), x.data_ptr(), w.data_ptr(),
                                       b.data_ptr(), C, K, y.data_ptr(), st, sp), "conv fwd")
        ev[1].record(stream)
        tam._check(lib.tree_conv1d_bwd(plan.ref(), tree[0].data_ptr(), tree[1].data_ptr(), x.data_ptr(), w.data_ptr(),
                                       dy.data_ptr(), C, K, ws.data_ptr(), dx.data_ptr(), dw.data_ptr(),
                                       db.data_ptr(), st, sp), "conv bwd")

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    fwd, bwd, tot = [], [], []
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for _ in range(args.steps):
            flush.fill_(1.0)
            ev[0].record(stream)
            step()
            ev[2].record(stream)
            torch.cuda.synchronize()
            fwd.append(ev[0].elapsed_time(ev[1]))
            bwd.append(ev[1].elapsed_time(ev[2]))
            tot.append(ev[0].elapsed_time(ev[2]))
    clocks = clk.summary()
    tam.check_status(status, "conv steps")
    # end to end through the public binding: pinned host x, dy in; dx, dw, db out, every step
    hx, hdy = t["x"].pin_memory(), t["u"].pin_memory()
    hdx = torch.empty(N, C, dtype=torch.bfloat16).pin_memory()
    hdw, hdb = torch.empty(K, C).pin_memory(), torch.empty(C).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e = []
    for i in range(args.warmup + args.steps):
        flush.fill_(1.0)
        e0.record(stream)
        x.copy_(hx, non_blocking=True)
        dy.copy_(hdy, non_blocking=True)
        step()
        hdx.copy_(dx, non_blocking=True)
        hdw.copy_(dw, non_blocking=True)
        hdb.copy_(db, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e.append(e0.elapsed_time(e1))
    ms_f, ms_b, ms = (float(np.mean(v)) for v in (fwd, bwd, tot))
    elems = N * C
    algo = 10.0 * elems
    peaks = load_peaks()
    achieved_b = 6.0 * elems / (ms_b * 1e-3) / 1e9
    line = {
        "metric": CONV_METRIC, "value": round(algo / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in/out, fp32 accumulate",
        "data": "synthetic (seeded tree, N(0,1) bf16 x and dy, N(0,1/K) taps)",
        "config": {"workload": f"{wl.name} conv C={C} K={K}", "N": N, "C": C, "K": K, "n_nodes": len(wl.parent),
                   "step": "tree_conv1d_fwd + tree_conv1d_bwd (bias, dw, db)",
                   "l2": "inputs (N C bf16) larger than L2, and flushed between steps"},
        "breakdown_ms": {"fwd": round(ms_f, 4), "bwd": round(ms_b, 4),
                         "fwd_gbs": round(4.0 * elems / (ms_f * 1e-3) / 1e9, 1)},
        "roofline": {"kernel": "tree_conv1d_bwd (zero, k_conv_bwd, finish)", "bound": "hbm",
                     "achieved": round(achieved_b, 1), "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": round(achieved_b / peaks["hbm"], 4), "peak_source": f"{peaks['source']} copy bandwidth",
                     "traffic": None, "algorithmic": "6 B per element (read x, dy; write dx)"},
        "e2e": {"value": round(algo / (float(np.mean(e2e)) * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(float(np.mean(e2e)), 4), "h2d_bytes_per_step": 2 * elems * 2,
                "d2h_bytes_per_step": elems * 2 + (K + 1) * C * 4},
        "gpu_launches": 4 * args.steps, "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = conv_cpu_baseline(wl, t, budget_s=15.0)
    print(json.dumps(line), flush=True)
    return 0


def conv_cpu_baseline(wl, t, budget_s=15.0):
    """The oracle's path-expanded fp64 convolution (forward and gradients) on a channel sample,
    growing the sample until the time budget is spent; credited 10 B per element like the GPU."""
    import oracle
    p = oracle.plan(wl.parent, wl.node_len)
    x, w, b, u = (t[n] for n in ("x", "w", "bias", "u"))
    done, t0, c0 = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < budget_s and c0 < x.shape[1]:
        ch = slice(c0, c0 + 8)
        f64 = [a[..., ch].double().numpy() for a in (x, w, b, u)]
        oracle.conv_paths(wl.parent, wl.node_len, *f64, p=p)
        done += x.shape[0] * 8
        c0 += 8
    el = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dict(value=round(10.0 * done / el / 1e9, 4), unit="GB/s", cores=cores, kind="oracle",
                sample=f"{wl.name}: fp64 path-expanded conv fwd+grads on channels 0-{c0 - 1} of {x.shape[1]}, "
                       f"{el:.1f} s; NumPy default threads")


CE_METRIC = "tree next-token CE fused with the vocabulary projection, fwd+bwd TFLOP/s on 1 GB300 (6 N V D)"


def run_ce(args, dev):
    """The path-averaged next-token cross-entropy fused with the vocabulary projection (Tree
    Training explainer, sections 6.2, 6.3, 12) on the workload's tree: h [N, D] bf16, W [V, D]
    bf16, labels with 10 % ignored.  Algorithmic work 6 N V D (logits, dh, dW); the chunked
    recompute executes 8 N V D on the tensor cores."""
    import tree_masked_attention_plan_gb300 as tam
    torch.cuda.set_device(dev)
    wl = make_workload(args.config)
    D, V, chunk = args.ce_hidden, args.ce_vocab, args.ce_chunk
    plan = tam.tree_plan(wl.parent, wl.node_len, device=dev)
    N = plan.n_tokens
    tree = tam.tree_arrays(wl.parent, wl.node_len, dev)
    gen = torch.Generator().manual_seed(13)
    h_host = torch.randn(N, D, generator=gen).to(torch.bfloat16)
    lab_host = torch.randint(0, V, (N,), generator=gen, dtype=torch.int32)
    lab_host[torch.rand(N, generator=gen) < 0.1] = -100
    gdev = torch.Generator(device=dev).manual_seed(14)
    W = (torch.randn(V, D, generator=gdev, device=dev) / D ** 0.5).to(torch.bfloat16)
    h, labels = h_host.to(dev), lab_host.to(dev)
    ws = torch.empty(tam.tree_ce_workspace(plan, D, V, chunk), dtype=torch.uint8, device=dev)
    out = (torch.empty(1, device=dev), torch.empty(N, device=dev), torch.empty_like(h),
           torch.empty(V, D, dtype=torch.float32, device=dev))
    status = tam.new_status(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def step():
        tam.tree_ce_fwd_bwd(plan, tree, h, W, labels, chunk=chunk, workspace=ws, out=out, status=status)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    tam.check_status(status, "ce warmup")
    ms = []
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for _ in range(args.steps):
            flush.fill_(1.0)
            e0.record(stream)
            step()
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
    clocks = clk.summary()
    tam.check_status(status, "ce steps")
    hp, lp = h_host.pin_memory(), lab_host.pin_memory()
    loss_host = torch.empty(1).pin_memory()
    e2e = []
    for i in range(args.warmup + args.steps):
        flush.fill_(1.0)
        e0.record(stream)
        h.copy_(hp, non_blocking=True)
        labels.copy_(lp, non_blocking=True)
        step()
        loss_host.copy_(out[0], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e.append(e0.elapsed_time(e1))
    t = float(np.mean(ms))
    algo = 6.0 * N * V * D
    executed = 8.0 * N * V * D
    peaks = load_peaks()
    achieved = executed / (t * 1e-3) / 1e12
    line = {
        "metric": CE_METRIC, "value": round(algo / (t * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 operands, fp32 accumulate",
        "data": "synthetic (seeded tree, N(0,1) bf16 hidden states, N(0,1/D) vocabulary matrix, 10 % ignored labels)",
        "config": {"workload": f"{wl.name} CE D={D} V={V} chunk={chunk}", "N": N, "D": D, "V": V, "chunk": chunk,
                   "step": "tree_ce_fwd_bwd (loss, lse, dh, dW)",
                   "l2": "operands larger than L2, and flushed between steps"},
        "roofline": {"kernel": "tree_ce_fwd_bwd (four GEMMs per chunk + small kernels)", "bound": "tensor",
                     "achieved": round(achieved, 1), "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16"], 4), "peak_source": f"{peaks['source']} bf16 burst",
                     "traffic": None, "algorithmic": "8 N V D executed MMA flops per call (6 N V D + recompute)"},
        "e2e": {"value": round(algo / (float(np.mean(e2e)) * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(float(np.mean(e2e)), 4), "h2d_bytes_per_step": N * D * 2 + N * 4,
                "d2h_bytes_per_step": 4},
        # pairs, label logits, loss, loss out + per chunk: 4 GEMMs, LSE merge, label fix-up
        "gpu_launches": (4 + 6 * ((N + chunk - 1) // chunk)) * args.steps, "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = ce_cpu_baseline(wl, h_host, W.cpu(), lab_host, budget_s=15.0)
    print(json.dumps(line), flush=True)
    return 0


def ce_cpu_baseline(wl, h, W, labels, budget_s=15.0):
    """The oracle's row form (fp64 logits, logsumexp and dh rows) on as many rows as fit the
    budget; credited 4 V D flops per row (its logits and dh products)."""
    import oracle
    p = oracle.plan(wl.parent, wl.node_len)
    Wd = W.double().numpy()
    hd = h.double().numpy()
    lab = labels.numpy()
    t0, done = time.perf_counter(), 0
    while time.perf_counter() - t0 < budget_s and done < hd.shape[0]:
        oracle.ce_rows(wl.parent, wl.node_len, hd, Wd, lab, range(done, done + 8), p=p)
        done += 8
    el = time.perf_counter() - t0
    V, D = Wd.shape
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dict(value=round(4.0 * V * D * done / el / 1e12, 6), unit="TFLOP/s", cores=cores, kind="oracle",
                sample=f"{wl.name}: fp64 logits, logsumexp and dh for rows 0-{done - 1} of {hd.shape[0]}, {el:.1f} s "
                       f"(after converting W to fp64); NumPy/BLAS default threads")


def cpu_baseline_sample(config, budget_s=20.0):
    """The oracle as it stands, on the host cores: path-expanded fp64 attention fwd+bwd for q head 0
    over a prefix of the root-to-leaf paths that fits the time budget.  Reported on the GPU line's
    metric: the sample's time is scaled to every path (by the path-expanded causal pairs they
    compute) and every q head, and the whole tree's 14 d Hq N_pairs unique visible-pair flops are
    divided by that time."""
    import oracle
    wl = make_workload(config)
    t = make_tensors(wl)
    p = oracle.plan(wl.parent, wl.node_len)
    path_len = [int(sum(wl.node_len[x] for x in path)) for path in p["paths"]]
    all_path_pairs = sum(L * (L + 1) // 2 for L in path_len)
    done_pairs, t0, n_paths = 0, time.perf_counter(), 0
    sub = dict(p)
    for path, L in zip(p["paths"], path_len):
        sub["paths"] = [path]
        sub["n_paths"] = p["n_paths"]
        oracle.attention_paths(wl.parent, wl.node_len, t["q"][:, :1], t["k"][:, :1], t["v"][:, :1], t["u"][:, :1],
                               heads=[0], p=sub, theta=wl.theta)
        done_pairs += L * (L + 1) // 2
        n_paths += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    whole_tree_s = el * (all_path_pairs / done_pairs) * wl.Hq      # every path, every q head
    n_pairs = host_stats(wl.parent, wl.node_len)["n_pairs"]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dict(value=14 * wl.d * wl.Hq * n_pairs / whole_tree_s / 1e12, unit=UNIT, cores=cores, kind="oracle",
                sample=f"{config}: fp64 path-expanded fwd+bwd, q head 0, first {n_paths} of {p['n_paths']} "
                       f"root-to-leaf paths ({done_pairs} of {all_path_pairs} path-expanded causal pairs) in {el:.1f} s; "
                       f"scaled to all paths and {wl.Hq} q heads ({whole_tree_s:.0f} s) and credited the tree's "
                       f"unique visible-pair flops 14 d Hq N_pairs; NumPy/BLAS default threads",
                seconds=el)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end (host buffers) leg, e.g. under a profiler")
    ap.add_argument("--conv", action="store_true",
                    help="time the hybrid-layer tree convolution (forward + backward) instead of attention")
    ap.add_argument("--ce", action="store_true",
                    help="time the fused vocabulary-projection cross-entropy instead of attention")
    ap.add_argument("--ce-hidden", type=int, default=4096)
    ap.add_argument("--ce-vocab", type=int, default=128256)
    ap.add_argument("--ce-chunk", type=int, default=8192)
    ap.add_argument("--conv-channels", type=int, default=8192)
    ap.add_argument("--conv-k", type=int, default=4)
    ap.add_argument("--shard", default="trees", choices=["trees", "heads"],
                    help="multi-rank split: 'trees' = one tree per rank (weak scaling); 'heads' = one tree "
                         "split by kv-head groups, plan replicated, no exchange (strong scaling)")
    ap.add_argument("--bwd-split", type=int, default=0, choices=[0, 1, 2, 4],
                    help="CTAs per key-tile column in the backward (0: the library's automatic choice)")
    ap.add_argument("--fwd-split", type=int, default=0, choices=[0, 1, 2, 4],
                    help="CTAs per query-tile row in the forward, split-KV (0: automatic)")
    ap.add_argument("--partition", action="store_true",
                    help="run the tree as gateway partitions (parent + children of the largest cut)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args)

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    if args.bwd_split or args.fwd_split:
        import tree_masked_attention_plan_gb300 as tam
        tam.tree_set_bwd_split(args.bwd_split)
        tam.tree_set_fwd_split(args.fwd_split)
    if args.ce:
        if world > 1:
            raise SystemExit("--ce runs on one GPU")
        return run_ce(args, dev)
    if args.conv:
        if world > 1:
            raise SystemExit("--conv runs on one GPU")
        return run_conv(args, dev)
    if args.partition:
        res = run_partitioned(args, dev)
        ms_max, = reduce_max([res["ms"]], dev, world)
        wl, st = res["wl"], res["st"]
        flops = 14.0 * wl.d * wl.Hq * st["n_pairs"]
        peaks = load_peaks()
        value = world * flops / (ms_max * 1e-3) / 1e12
        if rank == 0:
            print(json.dumps({
                "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded tree and N(0,1) bf16 tensors)",
                "config": {"workload": f"{wl.name} as gateway partitions", "N": st["N"], "N_pairs": st["n_pairs"],
                           "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d, "partition": res["info"],
                           "step": "per partition plan+rope+fwd+bwd, gateway gathers, fp32 relay "
                                   "(dO per partition prepared outside the timed region)",
                           "l2": "flushed between steps (256 MiB write, outside the event brackets)",
                           "parallelism": f"one tree per rank x{world}"},
                "tokens_per_s": round(world * st["N"] / (ms_max * 1e-3), 1),
                "pct_bf16_peak": round(100 * value / world / peaks["bf16"], 2),
                "gpu_launches": res["launches"] * args.steps, "clocks": res["clocks"]}), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    res = run_ours(args, rank, world, dev)
    st, wl, times = res["st"], res["wl"], res["times"]
    ms = float(np.mean(times["step"]))
    ms_fwd, ms_bwd, ms_dkdv = (float(np.mean(times[x])) for x in ("fwd", "bwd", "dkdv"))
    ms_max, e2e_max = reduce_max([ms, res["e2e_ms"]], dev, world)
    flops = 14.0 * wl.d * wl.Hq * st["n_pairs"]            # the whole tree, all heads
    peaks = load_peaks()
    heads = args.shard == "heads"
    trees = 1 if heads else world                           # trees the job processes per step
    value = trees * flops / (ms_max * 1e-3) / 1e12
    dkdv_flops = 10.0 * wl.d * res["Hq_local"] * st["n_pairs"]    # this rank's heads
    achieved = dkdv_flops / (ms_dkdv * 1e-3) / 1e12
    ms_plan, ms_rope = (float(np.mean(times[x])) for x in ("plan", "rope"))
    hq_l, hkv_l, T = res["Hq_local"], res["Hkv_local"], res["T"]
    # algorithmic bytes: RoPE reads and writes q, k (bf16) and reads pos; the plan writes 7 int32 /
    # fp32 arrays per padded token, the T x T class table, both CSR index lists and the node block
    rope_bytes = st["N"] * (2 * (hq_l + hkv_l) * wl.d * 2 + 4)
    plan_bytes = 28 * T * 128 + T * T + 8 * res["nnz"] + 32 * res["n_nodes"]
    local_pairs_flops = wl.d * hq_l * st["n_pairs"]
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
            "scaling": "strong" if heads else "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded tree and N(0,1) bf16 tensors)",
            "config": {"workload": wl.name, "N": st["N"], "paths_K": st["K"], "N_pairs": st["n_pairs"],
                       "N_flat": st["n_flat"], "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d, "rope_theta": wl.theta,
                       "nonempty_tiles": res["nnz"], "step": "plan+rope+fwd+bwd (loss weights g/K folded into the backward)",
                       "l2": "flushed between steps (256 MiB write, outside the event brackets)",
                       "parallelism": (f"one tree split by kv-head groups over {world} ranks (plan replicated, "
                                       f"no data-path exchange)") if heads else f"one tree per rank x{world}"},
            "tokens_per_s": round(trees * st["N"] / (ms_max * 1e-3), 1),
            "pct_bf16_peak": round(100 * value / world / peaks["bf16"], 2),
            "breakdown_ms": {"step": round(ms, 4), "plan": round(ms_plan, 4), "rope": round(ms_rope, 4),
                             "fwd": round(ms_fwd, 4), "bwd": round(ms_bwd, 4), "bwd_dkdv": round(ms_dkdv, 4),
                             "attention_fwd_bwd_tflops": round(14 * local_pairs_flops / ((ms_fwd + ms_bwd) * 1e-3)
                                                               / 1e12, 2)},
            "fwd_tflops": round(4 * local_pairs_flops / (ms_fwd * 1e-3) / 1e12, 2),
            "bwd_tflops": round(10 * local_pairs_flops / (ms_bwd * 1e-3) / 1e12, 2),
            "computed_tile_tflops": round(14.0 * wl.d * hq_l * res["nnz"] * 128 * 128 / ((ms_fwd + ms_bwd) * 1e-3)
                                          / 1e12, 2),
            "por": round(1.0 - st["N"] / st["n_flat"], 4),
            "rope_gbs": round(rope_bytes / (ms_rope * 1e-3) / 1e9, 1),
            "plan_gbs": round(plan_bytes / (ms_plan * 1e-3) / 1e9, 1),
            "plan_note": "plan_gbs: algorithmic bytes over the span of tree_plan on the stream (host node pass, one "
                         "node-block copy, three launches)",
            "e2e": None if args.no_e2e else {"value": round(trees * flops / (e2e_max * 1e-3) / 1e12, 2), "unit": UNIT,
                    "ms_per_step": round(e2e_max, 4), "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"],
                    "overlap": "step i+1's copy-in and step i's copy-out on side streams during compute"},
            "roofline": {"kernel": "k_bwd_dkdv", "bound": "tensor", "achieved": round(achieved, 2),
                         "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16"], 4),
                         "peak_source": f"{peaks['source']} bf16 burst", "traffic": profiled_traffic(wl.name),
                         "algorithmic": "10 d Hq N_pairs flops per launch"},
            "gpu_launches": LAUNCHES_PER_STEP * args.steps,
            "clocks": res["clocks"],
            "wall_s_timed_region": round(res["wall"], 3),
        }
        if not args.no_cpu_baseline:
            cb = cpu_baseline_sample(args.config, budget_s=15.0)
            cb.pop("seconds", None)
            line["cpu_baseline"] = cb
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_reference(args):
    """Reference arm: the CPU oracle (the only reference implementation there is), each step a
    bounded sample of the same workload, on the host cores."""
    res = []
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline_sample(args.config, budget_s=4.0)
        if i >= args.warmup:
            res.append(cb)
    value = float(np.mean([r["value"] for r in res]))
    secs = float(np.mean([r["seconds"] for r in res]))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded tree and N(0,1) bf16 tensors)",
            "config": {"workload": args.config, "parallelism": "host cores, rank 0 only"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": res[0]["cores"], "kind": "oracle",
                             "sample": res[0]["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
