#!/usr/bin/env python3
"""Benchmark of the GB300 attention forward (one JSON line on stdout).

Default workload: B=4, H=16, N=2048, d=128, bf16, full (non-causal) attention,
scale 1/sqrt(128) -- the headline configuration of the metric.  A step is one
full forward pass (one launch of the persistent kernel) over that batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I]
                  [--impl ours|reference]

Timing: W >= 3 untimed warm-up steps, then exactly K steps on the launching
stream bracketed by CUDA events, with a barrier + synchronize on both sides;
inputs rotate over enough copies (> 2x the 129 MB L2) that no step reads
another step's inputs from L2.  Under torchrun every rank runs an independent
replica on its own GPU (the forward pass has no cross-GPU exchange); the
reported value is all ranks' FLOPs over the slowest rank's time.

Workload 6 (one causal head of 32768 rows) runs through the split-KV entry
point with the automatic split count (two launches per step: the split
forward and the merge); its line adds the unsplit forward's time on the
same inputs.  Workload 7 (16 causal sequences of 697..3646 rows packed along
the rows) runs through the variable-length entry point, workload 8 (the
headline shape with FP8 E4M3 inputs) through the FP8 entry point, whose
roofline peak is the measured bf16 rate times the nominal fp8/bf16 ratio 2.

``--impl reference`` times the fp64 CPU oracle (the only other place this
script runs it) on rank 0, on bounded row samples of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("attention fwd TFLOP/s (4·B·H·N²·d, ×½ causal) and % of GB300 BF16 "
          "tensor peak")
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}


def _max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks of the default process group (x itself
    without one).  `device` holds the reduction tensor: the rank's GPU under
    NCCL, "cpu" under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _whole_job_tflops(world: int, flops_per_step: float, steps: int, ms: float) -> float:
    """Replicas: every rank runs `steps` steps of the workload; the job's
    rate is all ranks' FLOPs over the slowest rank's time (ms for all
    steps)."""
    return world * flops_per_step * steps / (ms / 1e3) / 1e12


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _kernel_source_hash() -> str:
    """Hash of the sources the forward kernels are compiled from (every file
    under csrc/ but the backward's own, which no forward translation unit
    includes): the key of the recorded ncu counters of forward launches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_10_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))
                    + glob.glob(os.path.join(csrc, "*.h"))):
        if os.path.basename(f).startswith("fa_bwd_"):
            continue
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(wl_name: str):
    """DRAM bytes per launch of the workload's dominant kernel, from the
    machine-readable record (``profiles/*.json``) written beside each ncu
    summary, if it is still current.

    Each record holds the workload name, the kernel-source hash the capture
    was taken at and ``dram_bytes_per_launch``; once the kernel sources
    change the figure no longer applies and None is returned.
    """
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.json"))):
        try:
            with open(path) as f:
                rec = json.load(f)
        except (OSError, ValueError):
            continue
        if rec.get("workload") != wl_name or rec.get("dram_bytes_per_launch") is None:
            continue
        if rec.get("kernel_source_hash") == _kernel_source_hash():
            return float(rec["dram_bytes_per_launch"]), os.path.relpath(path, ROOT)
        return None, os.path.relpath(path, ROOT) + " (stale: kernel sources changed)"
    return None, None


class ClockSampler:
    """nvidia-smi sampled every 200 ms in the background (host timestamps)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        self.error = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if gpu_id is not None:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": f"nvidia-smi unavailable: {self.error}"}
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "sampled during the timed region"
        if not inside:
            inside = [p for (_, p) in self.samples]
            note = "timed region shorter than one sample; all samples of the run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        pw = [num(p[3]) for p in inside if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def _gpu_id_for_smi(torch, dev_index: int):
    try:
        props = torch.cuda.get_device_properties(dev_index)
        dom = getattr(props, "pci_domain_id", None)
        bus = getattr(props, "pci_bus_id", None)
        devn = getattr(props, "pci_device_id", None)
        if bus is not None and devn is not None:
            return f"{dom or 0:08X}:{bus:02X}:{devn:02X}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip()]
    if ids and dev_index < len(ids) and ids[dev_index].strip().isdigit():
        return ids[dev_index].strip()
    return None


def _oracle_rows(wl, q, k, v, rows):
    """The oracle on listed (b, h, i) rows; packed (varlen) workloads are
    evaluated sequence by sequence on [1, H, n, d] views of each sequence.
    Returns the FLOPs of the rows (4*d per admissible key)."""
    import oracle
    lens = wl.seqlens()
    if wl.decode:
        # whole sequences (all heads and query rows) of the sampled rows
        nq, N = wl.n_q, wl.N
        seqs = sorted(set(r[0] for r in rows))
        for b in seqs:
            oracle.attention_varlen_qk(q[b * nq:(b + 1) * nq], k[b * N:(b + 1) * N],
                                       v[b * N:(b + 1) * N], [0, nq], [0, N], wl.scale,
                                       wl.causal)
        return wl.flops / wl.B * len(seqs)
    if wl.dtype == "fp8":
        # Every E4M3 value is a bfloat16 value: widened exactly, the inputs
        # (descales 1) define the same scores, P and O as the FP8 oracle's,
        # which has no row-sampled form.
        import torch
        q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    if not wl.varlen:
        oracle.attention_rows(q, k, v, wl.scale, wl.causal, rows)
    else:
        cu = wl.cu_seqlens()
        for b in sorted(set(r[0] for r in rows)):
            view = lambda t: t[cu[b]:cu[b + 1]].permute(1, 0, 2).unsqueeze(0).contiguous()
            oracle.attention_rows(view(q), view(k), view(v), wl.scale, wl.causal,
                                  [(0, h, i) for (bb, h, i) in rows if bb == b])
    return sum(4.0 * wl.d * ((i + 1) if wl.causal else lens[b]) for (b, _, i) in rows)


def _cpu_baseline(wl, budget_s: float = 12.0):
    """Time the fp64 oracle on whole heads of the workload, about `budget_s`."""
    import oracle
    from workloads import make_qkv
    q, k, v = make_qkv(wl)
    lens = wl.seqlens()
    if wl.decode:
        # whole sequences, as many as the budget allows (at least one)
        t0 = time.perf_counter()
        flops = _oracle_rows(wl, q, k, v, [(0, 0, 0)])
        n = 1
        while time.perf_counter() - t0 < budget_s and n < wl.B:
            flops += _oracle_rows(wl, q, k, v, [(n, 0, 0)])
            n += 1
        dt = time.perf_counter() - t0
        return {"value": flops / dt / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
                "kind": "oracle",
                "sample": f"{n} whole sequences (all heads and query rows) of "
                          f"{wl.describe()}, fp64, {dt:.1f} s"}
    # calibrate on 64 rows of head (0,0), then size the sample to the budget
    probe = [(0, 0, i) for i in range(0, lens[0], max(1, lens[0] // 64))][:64]
    t0 = time.perf_counter()
    probe_flops = _oracle_rows(wl, q, k, v, probe)
    rate = probe_flops / max(time.perf_counter() - t0, 1e-6)
    budget_flops = budget_s * rate
    rows, planned = [], 0.0
    for bh in range(wl.B * wl.H):
        b, h = divmod(bh, wl.H)
        for i in range(lens[b]):
            rows.append((b, h, i))
            planned += 4.0 * wl.d * ((i + 1) if wl.causal else lens[b])
            if planned >= budget_flops:
                break
        if planned >= budget_flops:
            break
    t0 = time.perf_counter()
    flops = _oracle_rows(wl, q, k, v, rows)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{len(rows)} query rows (first rows of heads in order) of "
                      f"{wl.describe()}, fp64, {dt:.1f} s"}


def run_reference(args, wl):
    rank, world, _ = _dist_env()
    if rank != 0:
        return 0
    import oracle
    from workloads import make_qkv
    q, k, v = make_qkv(wl)
    lens = wl.seqlens()
    rows_per_step = 128
    rng = __import__("random").Random(1234)
    step_rows = []
    for s in range(args.warmup + args.steps):
        rows = []
        if wl.decode:
            # decode: one whole sequence per step (all heads and query rows)
            rows.append((rng.randrange(wl.B), 0, 0))
        for _ in range(0 if wl.decode else rows_per_step):
            b = rng.randrange(wl.B)
            rows.append((b, rng.randrange(wl.H), rng.randrange(lens[b])))
        step_rows.append(rows)
    for s in range(args.warmup):
        _oracle_rows(wl, q, k, v, step_rows[s])
    flops = 0.0
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + args.steps):
        flops += _oracle_rows(wl, q, k, v, step_rows[s])
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl, "host cores, fp64 oracle"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": (f"one seeded random sequence per step of {wl.describe()}"
                                    if wl.decode else
                                    f"{rows_per_step} seeded random query rows per step of "
                                    f"{wl.describe()}")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(wl, l2_note):
    return {"workload": f"{wl.name}: {wl.describe()}, scale=1/sqrt(d)", "B": wl.B,
            "H": wl.H, "N": wl.N, "d": wl.d, "causal": wl.causal,
            "input_dtype": wl.dtype, "l2": l2_note, "parallelism": "replicas"}


def _time_dense(fa, torch, wl, dev, sampler, budget_s: float = 0.3, warmup: int = 5):
    """Device time of fa_fwd on a dense workload (inputs resident, rotating
    over enough copies to exceed twice the L2 when one copy does not), for
    the per-workload lines that follow the headline."""
    from workloads import make_qkv
    q, k, v = make_qkv(wl)
    set_bytes = 4 * q.numel() * q.element_size() + wl.B * wl.H * wl.N * 4
    n_sets = max(1, min(8, math.ceil(2.2 * L2_BYTES / set_bytes)))
    sets = []
    for i in range(n_sets):
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        if i > 0:
            qd, kd, vd = qd.clone(), kd.clone(), vd.clone()
        sets.append((qd, kd, vd, torch.empty_like(qd),
                     torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev)))
    stream = torch.cuda.Stream(device=dev)
    dcode = fa.FA_DTYPE_BF16 if wl.dtype == "bf16" else fa.FA_DTYPE_F16

    def step(i):
        qd, kd, vd, od, ld = sets[i % n_sets]
        st_ = fa.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(),
                        ld.data_ptr(), wl.B, wl.H, wl.N, wl.d, wl.scale, int(wl.causal), dcode,
                        stream.cuda_stream)
        if st_ != fa.FA_OK:
            raise RuntimeError(f"forward failed: {fa.fa_status_string(st_)}")

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(warmup):
        step(i)
    e0.record(stream)
    for i in range(3):
        step(i)
    e1.record(stream)
    e1.synchronize()
    per = max(e0.elapsed_time(e1) / 3, 1e-3)
    steps = int(min(20000, max(10, budget_s * 1e3 / per)))
    torch.cuda.synchronize(dev)
    t0 = time.time()
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    st, site = fa.fa_get_device_status(stream.cuda_stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {fa.fa_status_string(st)} (site {site})")
    ms = e0.elapsed_time(e1) / steps
    del sets
    return {"ms_per_step": ms, "steps": steps,
            "tflops": wl.flops / (ms / 1e3) / 1e12,
            "hbm_gbs": wl.hbm_bytes / (ms / 1e3) / 1e9,
            "l2": (f"{n_sets} rotating input sets ({n_sets * set_bytes / 2**20:.0f} MiB)"
                   + (" > L2" if n_sets * set_bytes > L2_BYTES else ", L2-resident")),
            "clocks": sampler.summary(t0, t1) if sampler else None}


def _sweep(fa, torch, dev, indices, peak: float, peak_note: str, gpu_id):
    """The other dense workloads, each timed on its own after the headline
    (same process, same GPU): one entry per workload."""
    from workloads import workload
    sampler = ClockSampler(gpu_id)
    time.sleep(0.25)
    out = []
    try:
        for idx in indices:
            w = workload(idx)
            r = _time_dense(fa, torch, w, dev, sampler)
            r.update({"workload": w.name, "describe": w.describe(),
                      "flops_per_step": w.flops, "hbm_bytes_per_step": w.hbm_bytes,
                      "frac": r["tflops"] / peak, "peak": peak, "peak_source": peak_note})
            traffic, src = _profiled_traffic(w.name)
            r["traffic"] = traffic
            r["traffic_source"] = src
            out.append(r)
    finally:
        sampler.stop()
    return out


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    rank, world, local = _dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}" if world > 1 else "cuda:0")
    torch.cuda.set_device(dev)

    import attention_forward_10_gb300 as fa
    from workloads import make_qkv

    fa.fa_set_max_ctas(0)
    warmup = max(3, args.warmup)
    q, k, v = make_qkv(wl)
    B, H, N, d = wl.B, wl.H, wl.N, wl.d
    # packed (varlen) workloads: [total, H, d] tensors, LSE [H, total];
    # decode workloads: q [B*n_q, H, d], k, v [B*N, H_kv, d], LSE [H, B*n_q]
    total = wl.B * wl.n_q if wl.decode else sum(wl.seqlens())
    lse_shape = (H, total) if (wl.varlen or wl.decode) else (B, H, N)
    cu_dev = torch.tensor(wl.cu_seqlens(), dtype=torch.int32, device=dev) if wl.varlen else None
    max_len = max(wl.seqlens())
    cu_q_dev = cu_k_dev = None
    if wl.decode:
        cu_q_dev = torch.arange(0, B + 1, dtype=torch.int32, device=dev) * wl.n_q
        cu_k_dev = torch.arange(0, B + 1, dtype=torch.int32, device=dev) * N
    set_bytes = (sum(t.numel() * t.element_size() for t in (q, k, v)) +
                 q.numel() * q.element_size() + H * total * 4)
    n_sets = max(1, min(8, math.ceil(2.2 * L2_BYTES / set_bytes)))
    sets = []
    for i in range(n_sets):
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        if i > 0:   # distinct copies (same values) so that no step hits L2
            qd, kd, vd = qd.clone(), kd.clone(), vd.clone()
        sets.append((qd, kd, vd, torch.empty(qd.shape, dtype=torch.bfloat16, device=dev)
                     if wl.dtype == "fp8" else torch.empty_like(qd),
                     torch.empty(lse_shape, dtype=torch.float32, device=dev)))
    stream = torch.cuda.Stream(device=dev)
    handle = stream.cuda_stream
    dcode = fa.FA_DTYPE_BF16 if wl.dtype == "bf16" else fa.FA_DTYPE_F16

    # Split-KV workloads go through fa_fwd_splitkv with the automatic split
    # count; its scratch is allocated once, outside the timed region.
    workspace, ws_bytes, launches_per_call = None, 0, 1

    def ensure_workspace(Bc, Hc):
        nonlocal workspace, ws_bytes, launches_per_call
        st_, need = fa.fa_splitkv_workspace_bytes(Bc, Hc, N, d, int(wl.causal), -1, -1, 0)
        if st_ != fa.FA_OK:
            raise RuntimeError(f"workspace query failed: {fa.fa_status_string(st_)}")
        if need > ws_bytes:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
            ws_bytes = need
        if need > 0:
            launches_per_call = 2
        return need

    def call(qp, kp, vp, op, lp, Bc, Hc, plain=False):
        if wl.dtype == "fp8":
            st_ = fa.fa_fwd_fp8(qp, kp, vp, op, lp, Bc, Hc, Hc, N, d, wl.scale, 1.0, 1.0, 1.0,
                                int(wl.causal), -1, -1, fp8_ws.data_ptr(), fp8_ws.numel(),
                                handle)
        elif wl.varlen:
            st_ = fa.fa_fwd_varlen(qp, kp, vp, op, lp, cu_dev.data_ptr(), B, max_len, total, H,
                                   H, d, wl.scale, int(wl.causal), -1, -1, dcode, handle)
        elif wl.decode:
            st_ = fa.fa_fwd_varlen_qk(qp, kp, vp, op, lp, cu_q_dev.data_ptr(),
                                      cu_k_dev.data_ptr(), None, None, B, wl.n_q, N, total,
                                      B * N, H, wl.kv_heads, d, wl.scale, int(wl.causal), -1,
                                      -1, dcode, handle)
        elif wl.splitkv and not plain:
            st_ = fa.fa_fwd_splitkv(qp, kp, vp, op, lp, Bc, Hc, Hc, N, d, wl.scale,
                                    int(wl.causal), -1, -1, dcode, 0,
                                    workspace.data_ptr() if workspace is not None else None,
                                    ws_bytes, handle)
        else:
            st_ = fa.fa_fwd(qp, kp, vp, op, lp, Bc, Hc, N, d, wl.scale, int(wl.causal),
                            dcode, handle)
        if st_ != fa.FA_OK:
            raise RuntimeError(f"forward failed: {fa.fa_status_string(st_)}")

    fp8_ws = None
    if wl.dtype == "fp8":
        # (two launches per call: the V transpose and the forward)
        st_, need_ = fa.fa_fwd_fp8_workspace_bytes(B, H, N, d)
        fp8_ws = torch.empty(max(need_, 256), dtype=torch.uint8, device=dev)
        launches_per_call = 2

    splits_used = 1
    if wl.splitkv:
        need = ensure_workspace(B, H)
        splits_used = max(1, round(need / (B * H * N * (2 * d + 4)))) if need else 1

    def step(i, plain=False):
        qd, kd, vd, od, ld = sets[i % n_sets]
        call(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), ld.data_ptr(), B, H,
             plain=plain)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    stream.synchronize()
    st, site = fa.fa_get_device_status(handle)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {fa.fa_status_string(st)} (site {site})")
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(5):
        step(i)
    e1.record(stream)
    e1.synchronize()
    per_step_ms = max(e0.elapsed_time(e1) / 5, 1e-3)
    if args.steps is None:
        # about two seconds of timed work, so the clock sampler sees the load
        args.steps = int(min(20000, max(20, 2000.0 / per_step_ms)))
        args.steps = int(_max_over_ranks(args.steps, dev))

    sampler = ClockSampler(_gpu_id_for_smi(torch, dev.index)) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # Soak: at least one second of the same steps, untimed for the metric,
    # right before the timed region, so that the clock record shows the
    # GPU under sustained load (a short timed region sees a cold, boosted
    # GPU); its own rate and clock samples are reported separately.
    soak_steps = int(min(200000, max(args.steps, math.ceil(args.soak_s / max(per_step_ms, 1e-3)
                                                          * 1e3))))
    torch.cuda.synchronize(dev)
    t_soak0 = time.time()
    start.record(stream)
    for i in range(soak_steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_soak1 = time.time()
    soak_ms = start.elapsed_time(end)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    if world > 1:
        dist.barrier()
    ms = start.elapsed_time(end)
    st, site = fa.fa_get_device_status(handle)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {fa.fa_status_string(st)} (site {site})")
    ms = _max_over_ranks(ms, dev)
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    soak = None
    if sampler:
        soak = {"steps": soak_steps, "seconds": soak_ms / 1e3,
                "tflops": wl.flops * soak_steps / (soak_ms / 1e3) / 1e12,
                "ms_per_step": soak_ms / soak_steps,
                "clocks": sampler.summary(t_soak0, t_soak1),
                "note": "untimed for the metric: the same steps for >= "
                        f"{args.soak_s:g} s right before the timed region"}
        sampler.stop()

    ms_per_step = ms / args.steps
    value = _whole_job_tflops(world, wl.flops, args.steps, ms)

    plain_ms = None
    if wl.splitkv:
        # the same steps through the unsplit forward, for comparison
        with torch.cuda.stream(stream):
            for i in range(3):
                step(i, plain=True)
        start.record(stream)
        for i in range(args.steps):
            step(i, plain=True)
        end.record(stream)
        torch.cuda.synchronize(dev)
        plain_ms = start.elapsed_time(end) / args.steps

    def measure_e2e_decode():
        """Decode workload end to end: chunks of whole sequences (about 8);
        each chunk's query rows and cached K/V rows are copied in, computed
        through fa_fwd_varlen_qk on those sequences (offset pointers into
        the device offset arrays, absolute rows), and its O rows copied out;
        the [H][B*n_q] LSE is copied once at the end."""
        nq = wl.n_q
        q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
        o_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        l_h = torch.empty((H, total), dtype=torch.float32).pin_memory()
        dq_, dk_, dv_, do_, dl_ = sets[0]
        per = max(1, B // 8)
        groups = [(b0, min(B, b0 + per)) for b0 in range(0, B, per)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_step():
            root = torch.cuda.current_stream(dev)
            ev0 = torch.cuda.Event()
            ev0.record(root)
            for st_ in (s_in, stream, s_out):
                st_.wait_event(ev0)
            for (g0, g1) in groups:
                with torch.cuda.stream(s_in):
                    dq_[g0 * nq:g1 * nq].copy_(q_h[g0 * nq:g1 * nq], non_blocking=True)
                    dk_[g0 * N:g1 * N].copy_(k_h[g0 * N:g1 * N], non_blocking=True)
                    dv_[g0 * N:g1 * N].copy_(v_h[g0 * N:g1 * N], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                stream.wait_event(ev_in)
                st_ = fa.fa_fwd_varlen_qk(dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                          do_.data_ptr(), dl_.data_ptr(),
                                          cu_q_dev.data_ptr() + 4 * g0,
                                          cu_k_dev.data_ptr() + 4 * g0, None, None, g1 - g0,
                                          nq, N, total, B * N, H, wl.kv_heads, d, wl.scale,
                                          int(wl.causal), -1, -1, dcode, handle)
                if st_ != fa.FA_OK:
                    raise RuntimeError(f"fa_fwd_varlen_qk: {fa.fa_status_string(st_)}")
                ev_c = torch.cuda.Event()
                ev_c.record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_c)
                    o_h[g0 * nq:g1 * nq].copy_(do_[g0 * nq:g1 * nq], non_blocking=True)
            with torch.cuda.stream(s_out):
                s_out.wait_stream(stream)
                l_h.copy_(dl_, non_blocking=True)
            for st_ in (s_in, stream, s_out):
                ev = torch.cuda.Event()
                ev.record(st_)
                root.wait_event(ev)

        e2e_step()
        torch.cuda.synchronize(dev)
        graph = None
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                e2e_step()
            torch.cuda.synchronize(dev)
            graph.replay()
            torch.cuda.synchronize(dev)
        except Exception:  # noqa: BLE001 - any capture failure: run eagerly
            graph = None
            torch.cuda.synchronize(dev)
        steps_ = max(1, min(args.steps, 20))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        root = torch.cuda.current_stream(dev)
        e0.record(root)
        for _ in range(steps_):
            if graph is not None:
                graph.replay()
            else:
                e2e_step()
        e1.record(root)
        torch.cuda.synchronize(dev)
        e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / steps_, dev)
        h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
        d2h = o_h.numel() * o_h.element_size() + l_h.numel() * 4
        return {"value": _whole_job_tflops(world, wl.flops, 1, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "cuda_graph": graph is not None,
                "api": f"{len(groups)} chunks of sequences: cudaMemcpyAsync in/out around "
                       f"fa_fwd_varlen_qk"}

    def measure_e2e():
        if wl.decode:
            return measure_e2e_decode()
        # End to end through the public API with host buffers: each step copies
        # Q, K, V from pinned host memory, runs the forward pass and copies O and
        # LSE back.  Dense bf16/fp16 workloads make one fa_fwd_host call per step
        # (the library chunks the heads and overlaps copies with the kernels).
        # The others (split-KV, packed, FP8) do the same here: the B*H heads are
        # cut into chunks and the copies of one chunk overlap the kernel of the
        # previous one (three streams: H2D, compute, D2H); packed (varlen) batches
        # interleave heads within rows: one chunk.
        host_api = not (wl.splitkv or wl.varlen or wl.dtype == "fp8")
        if wl.varlen:
            rows_e2e, row_shape, l_shape = 1, (total * H * d,), (H * total,)
        else:
            rows_e2e, row_shape, l_shape = B * H, (B * H, N, d), (B * H, N)
        q_h, k_h, v_h = (t.reshape(row_shape).pin_memory() for t in (q, k, v))
        o_h = torch.empty(row_shape, dtype=torch.bfloat16 if wl.dtype == "fp8" else q.dtype)
        o_h = o_h.pin_memory()
        l_h = torch.empty(l_shape, dtype=torch.float32).pin_memory()
        if wl.varlen:
            q_h, k_h, v_h, o_h, l_h = (t.unsqueeze(0) for t in (q_h, k_h, v_h, o_h, l_h))
        n_chunks = max(1, min(8, rows_e2e))
        bounds = [(c * rows_e2e // n_chunks, (c + 1) * rows_e2e // n_chunks)
                  for c in range(n_chunks)]
        dq, dk, dv = (sets[0][t].view(q_h.shape) for t in range(3))
        do_ = sets[0][3].view(o_h.shape)
        dl = sets[0][4].view(l_h.shape)
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        e2e_steps = max(1, min(args.steps, 20))

        def e2e_step():
            """One step: fork the three streams from the current one, copy chunk c
            in, run it, copy it out (chunk c + 1's input copy overlapping chunk
            c's kernel and output copy), join back.  Steps do not overlap."""
            root = torch.cuda.current_stream(dev)
            ev0 = torch.cuda.Event()
            ev0.record(root)
            for st_ in (s_in, stream, s_out):
                st_.wait_event(ev0)
            for (a0, a1) in bounds:
                with torch.cuda.stream(s_in):
                    for dst, src in ((dq, q_h), (dk, k_h), (dv, v_h)):
                        dst[a0:a1].copy_(src[a0:a1], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                stream.wait_event(ev_in)
                call(dq[a0].data_ptr(), dk[a0].data_ptr(), dv[a0].data_ptr(),
                     do_[a0].data_ptr(), dl[a0].data_ptr(), 1, a1 - a0)
                ev_c = torch.cuda.Event()
                ev_c.record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_c)
                    o_h[a0:a1].copy_(do_[a0:a1], non_blocking=True)
                    l_h[a0:a1].copy_(dl[a0:a1], non_blocking=True)
            for st_ in (s_in, stream, s_out):
                ev = torch.cuda.Event()
                ev.record(st_)
                root.wait_event(ev)

        if wl.varlen:
            # Packed batch: chunks of whole sequences (about 8, balanced by
            # rows).  Each chunk's rows are copied into the same rows of the
            # full-size device tensors and fa_fwd_varlen runs on its sequences
            # (cu_seqlens from the chunk's first sequence on, row offsets still
            # global); the [H][total] LSE, strided per chunk, is copied once at
            # the end.
            cu = wl.cu_seqlens()
            target = max(1, total // 8)
            groups, b0 = [], 0
            for b in range(1, B + 1):
                if cu[b] - cu[b0] >= target or b == B:
                    groups.append((b0, b))
                    b0 = b
            lens = wl.seqlens()
            q_v, k_v, v_v = (t.pin_memory() for t in (q, k, v))      # [total, H, d]
            o_v = torch.empty(q.shape, dtype=q.dtype).pin_memory()
            l_v = torch.empty((H, total), dtype=torch.float32).pin_memory()
            dq_v, dk_v, dv_v, do_v, dl_v = sets[0]
            n_chunks = len(groups)

            def e2e_step():
                """One step: fork, per chunk copy in / compute / copy out, join."""
                root = torch.cuda.current_stream(dev)
                ev0 = torch.cuda.Event()
                ev0.record(root)
                for st_ in (s_in, stream, s_out):
                    st_.wait_event(ev0)
                for (g0, g1) in groups:
                    r0, r1 = cu[g0], cu[g1]
                    with torch.cuda.stream(s_in):
                        for dst, src in ((dq_v, q_v), (dk_v, k_v), (dv_v, v_v)):
                            dst[r0:r1].copy_(src[r0:r1], non_blocking=True)
                        ev_in = torch.cuda.Event()
                        ev_in.record(s_in)
                    stream.wait_event(ev_in)
                    st_ = fa.fa_fwd_varlen(dq_v.data_ptr(), dk_v.data_ptr(), dv_v.data_ptr(),
                                           do_v.data_ptr(), dl_v.data_ptr(),
                                           cu_dev.data_ptr() + 4 * g0, g1 - g0,
                                           max(lens[g0:g1]), total, H, H, d, wl.scale,
                                           int(wl.causal), -1, -1, dcode, handle)
                    if st_ != fa.FA_OK:
                        raise RuntimeError(f"fa_fwd_varlen: {fa.fa_status_string(st_)}")
                    ev_c = torch.cuda.Event()
                    ev_c.record(stream)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(ev_c)
                        o_v[r0:r1].copy_(do_v[r0:r1], non_blocking=True)
                with torch.cuda.stream(s_out):
                    s_out.wait_stream(stream)
                    l_v.copy_(dl_v, non_blocking=True)
                for st_ in (s_in, stream, s_out):
                    ev = torch.cuda.Event()
                    ev.record(st_)
                    root.wait_event(ev)

        if host_api:
            H_kv = int(k.shape[1])
            q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
            st_, ws_bytes = fa.fa_fwd_host_workspace_bytes(B, H, H_kv, N, d, 1)
            if st_ != fa.FA_OK:
                raise RuntimeError(f"fa_fwd_host_workspace_bytes: {fa.fa_status_string(st_)}")
            # two requests' outputs and device workspaces: a step may run while
            # the previous one is still in flight on another stream
            outs = [(torch.empty(q.shape, dtype=q.dtype).pin_memory(),
                     torch.empty((B, H, N), dtype=torch.float32).pin_memory(),
                     torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev))
                    for _ in range(2)]
            o_h, l_h = outs[0][0], outs[0][1]
            n_chunks = None

            def e2e_step(slot=0):
                """One step: a single fa_fwd_host call on the current stream."""
                root = torch.cuda.current_stream(dev)
                o_s, l_s, ws_s = outs[slot]
                st_ = fa.fa_fwd_host(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
                                     o_s.data_ptr(), l_s.data_ptr(), B, H, H_kv, N, d, wl.scale,
                                     int(wl.causal), -1, -1, dcode, ws_s.data_ptr(),
                                     ws_s.numel(), root.cuda_stream)
                if st_ != fa.FA_OK:
                    raise RuntimeError(f"fa_fwd_host: {fa.fa_status_string(st_)}")

        if wl.splitkv:
            for (a0, a1) in bounds:
                ensure_workspace(1, a1 - a0)
        e2e_step()
        torch.cuda.synchronize(dev)
        # The step's launches are captured once into a CUDA graph and replayed
        # (host work per step: one graph launch); if capture is refused, the
        # steps are issued eagerly.
        graph = None
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                e2e_step()
            torch.cuda.synchronize(dev)
            graph.replay()
            torch.cuda.synchronize(dev)
        except Exception:  # noqa: BLE001 - any capture failure: run eagerly
            graph = None
            torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        root = torch.cuda.current_stream(dev)
        e0.record(root)
        for _ in range(e2e_steps):
            if graph is not None:
                graph.replay()
            else:
                e2e_step()
        # the last D2H copy (joined into the current stream) closes the timed region
        e1.record(root)
        torch.cuda.synchronize(dev)
        e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
        h2d = q_h.numel() * q_h.element_size() + 2 * k_h.numel() * k_h.element_size()
        d2h = o_h.numel() * o_h.element_size() + H * total * 4
        out = {"value": _whole_job_tflops(world, wl.flops, 1, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "cuda_graph": graph is not None, "in_flight": 1,
               "api": ("fa_fwd_host (C ABI on host buffers)" if host_api else
                       f"{n_chunks} chunks of "
                       f"{'sequences' if wl.varlen else 'heads'}: cudaMemcpyAsync "
                       f"in/out around the C ABI forward")}
        if host_api and graph is not None:
            # Two requests in flight: steps alternate between two streams,
            # each with its own outputs and workspace (one graph per stream),
            # so that a step's input copies overlap the previous step's last
            # kernel and output copies.  Every step still copies its inputs
            # in and its results out inside the timed region.
            streams2 = [torch.cuda.Stream(device=dev) for _ in range(2)]
            graphs2 = []
            for slot in range(2):
                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g2, stream=streams2[slot]):
                    e2e_step(slot)
                graphs2.append(g2)
            torch.cuda.synchronize(dev)
            for slot in range(2):
                with torch.cuda.stream(streams2[slot]):
                    graphs2[slot].replay()
            torch.cuda.synchronize(dev)
            steps2 = 2 * e2e_steps
            e0.record(root)
            for st2 in streams2:
                st2.wait_event(e0)
            for i in range(steps2):
                with torch.cuda.stream(streams2[i % 2]):
                    graphs2[i % 2].replay()
            for st2 in streams2:
                ev = torch.cuda.Event()
                ev.record(st2)
                root.wait_event(ev)
            e1.record(root)
            torch.cuda.synchronize(dev)
            ms2 = _max_over_ranks(e0.elapsed_time(e1) / steps2, dev)
            out.update({"value": _whole_job_tflops(world, wl.flops, 1, ms2),
                        "ms_per_step": ms2, "in_flight": 2,
                        "one_in_flight": {"value": out["value"], "ms_per_step": e2e_ms}})
        return out

    e2e = measure_e2e() if args.e2e else None

    if rank == 0:
        peaks, src = _peaks()
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        peak_note = f"{src} bf16_tflops (burst; kernel timed alone)"
        if wl.dtype == "fp8":
            # FP8 dense tensor rate: the bf16 measurement times the nominal
            # 4.5 / 2.25 PFLOP/s ratio
            peak *= 2.0
            peak_note = f"{src} bf16_tflops x 2 (nominal fp8/bf16 dense ratio)"
        achieved = wl.flops / (ms_per_step / 1e3) / 1e12
        traffic, traffic_src = _profiled_traffic(wl.name)
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_note,
                    "traffic": traffic, "traffic_source": traffic_src,
                    "algorithmic_hbm_bytes": wl.hbm_bytes}
        if wl.flops / wl.hbm_bytes < peak * 1e12 / (float(peaks.get("hbm_gbs", 6800.0)) * 1e9):
            # below the ridge point (the decode workload reads its cache once):
            # bound by HBM bandwidth
            gbs = wl.hbm_bytes / (ms_per_step / 1e3) / 1e9
            hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
            roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                        "frac": gbs / hbm_peak, "peak_source": f"{src} hbm_gbs",
                        "traffic": traffic, "traffic_source": traffic_src,
                        "algorithmic_hbm_bytes": wl.hbm_bytes, "tflops": achieved}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic",
            "config": _config(wl, f"{n_sets} rotating input sets "
                                  f"({n_sets * set_bytes / 2**20:.0f} MiB) > L2"),
            "pct_of_peak": 100.0 * achieved / peak,
            "pct_of_peak_note": "of the tensor peak (the roofline key names the bound)",
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": args.steps * launches_per_call,
            "clocks": clocks,
            "soak": soak,
        }
        if wl.splitkv:
            line["splitkv"] = {"num_splits": splits_used,
                               "unsplit_fa_fwd_ms_per_step": plain_ms,
                               "unsplit_tflops": wl.flops / (plain_ms / 1e3) / 1e12}
        if world == 1 and args.sweep and wl.index == 2:
            # the other dense workloads of the metric, timed after the headline
            line["workloads"] = _sweep(fa, torch, dev, (1, 3, 4, 5), peak, peak_note,
                                       _gpu_id_for_smi(torch, dev.index))
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = _cpu_baseline(wl)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


BWD_METRIC = ("attention bwd TFLOP/s (10·B·H·N²·d = 2.5x the forward's FLOPs, ×½ causal) "
              "and % of GB300 BF16 tensor peak")


def run_backward(args, wl):
    """Time fa_bwd (pre-pass + dK/dV + dQ kernels) on the workload's shapes,
    with Q, K, V, O, LSE and dO resident on the device."""
    import torch
    import torch.distributed as dist
    rank, world, local = _dist_env()
    dev = torch.device(f"cuda:{local}" if world > 1 else "cuda:0")
    torch.cuda.set_device(dev)
    if world > 1:   # replicas: every rank runs the whole workload
        dist.init_process_group("nccl", device_id=dev)
    import attention_forward_10_gb300 as fa
    from workloads import make_qkv
    if wl.splitkv or wl.decode or wl.dtype == "fp8" or wl.d not in (64, 128):
        raise SystemExit("--backward runs the [B,H,N,d] and packed workloads with d = 64 or 128")
    fa.fa_set_max_ctas(0)
    warmup = max(3, args.warmup)
    q, k, v = (t.to(dev) for t in make_qkv(wl))
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(4000 + wl.index))
    dout = dout.to(q.dtype).to(dev)
    if wl.varlen:
        # packed batch ([total, H, d]) through fa_bwd_varlen
        lens = wl.seqlens()
        cu_dev = torch.tensor(wl.cu_seqlens(), dtype=torch.int32, device=dev)
        o, lse = fa.fwd_varlen(q, k, v, cu_dev, max(lens), scale=wl.scale, causal=wl.causal)
        st, need = fa.fa_bwd_workspace_bytes(wl.B, wl.H, max(lens))
    else:
        o, lse = fa.fwd(q, k, v, scale=wl.scale, causal=wl.causal)
        st, need = fa.fa_bwd_workspace_bytes(wl.B, wl.H, wl.N)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.Stream(device=dev)
    dcode = fa.FA_DTYPE_BF16 if wl.dtype == "bf16" else fa.FA_DTYPE_F16

    def step():
        if wl.varlen:
            st_ = fa.fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), cu_dev.data_ptr(), wl.B, max(lens),
                                   int(q.shape[0]), wl.H, wl.H, wl.d, wl.scale, int(wl.causal),
                                   -1, -1, dcode, ws.data_ptr(), ws.numel(), stream.cuda_stream)
        else:
            st_ = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), ws.data_ptr(), ws.numel(), wl.B, wl.H, wl.H, wl.N,
                            wl.d, wl.scale, int(wl.causal), -1, -1, dcode, stream.cuda_stream)
        if st_ != fa.FA_OK:
            raise RuntimeError(f"fa_bwd failed: {fa.fa_status_string(st_)}")

    torch.cuda.synchronize(dev)
    for _ in range(warmup):
        step()
    stream.synchronize()
    if args.steps is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            step()
        e1.record(stream)
        e1.synchronize()
        args.steps = int(min(5000, max(10, 2000.0 / max(e0.elapsed_time(e1) / 3, 1e-3))))
        args.steps = int(_max_over_ranks(args.steps, dev))
    sampler = ClockSampler(_gpu_id_for_smi(torch, dev.index)) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if world > 1:
        dist.barrier()
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    st, site = fa.fa_get_device_status(stream.cuda_stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {fa.fa_status_string(st)} (site {site})")
    ms_all = _max_over_ranks(start.elapsed_time(end), dev)
    ms = ms_all / args.steps
    flops = 2.5 * wl.flops
    peaks, src = _peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms / 1e3) / 1e12  # one replica
    value = _whole_job_tflops(world, flops, args.steps, ms_all)
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {
        "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": _config(wl, "inputs resident; each step reads the same inputs"),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "peak_source": f"{src} bf16_tflops (burst)",
                     "executed_mma_flops_per_algorithmic": 1.4},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about two seconds of work)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=2,
                    help="1..9 (default 2: B=4 H=16 N=2048 d=128 bf16 full; "
                         "6: the split-KV case; 7: a packed variable-length batch; "
                         "8: FP8; 9: decode against a KV cache, GQA 8:1)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="with the default workload, do not time workloads 1, 3, 4 and 5 "
                         "after it")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false",
                    help="skip the end-to-end measurement through host buffers")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="seconds of untimed identical steps right before the timed region")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (fa_bwd) instead of the forward")
    ap.add_argument("--print-kernel-hash", action="store_true",
                    help="print the hash of the kernel sources (the key of the ncu records "
                         "in profiles/) and exit")
    args = ap.parse_args()
    if args.print_kernel_hash:
        print(_kernel_source_hash())
        return 0
    from workloads import workload
    wl = workload(args.workload)
    if args.backward:
        return run_backward(args, wl)
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
