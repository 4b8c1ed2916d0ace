#!/usr/bin/env python
"""Benchmark of the CKDA forward (and decode step) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one ckda_fwd call over the full CKDA-range workload (B=4, H=32,
T=8192, dk=dv=128, bf16 I/O, fp32 state, alpha = tanh(N(0,2)) with exact -1
and 0 entries, beta = 2 sigmoid(N(0,1)), h0 ~ N(0, 0.1)), inputs resident in
HBM.  The inputs (1.07 GB) exceed the 129 MB L2, so no flush is done between
steps.  Prints ONE JSON line on rank 0 with:
  value     whole-job token-heads/s (B*T*H per step, all ranks): two CUDA
            events around the K back-to-back steps
  roofline  the forward's algorithmic bytes / its mean per-call device time
            (the same two events; a call is the status-word clear and the
            kernel) against the measured HBM copy bandwidth
  e2e       the same metric with host (pinned) buffers, H2D and D2H in the
            timed region
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample (rank 0, N=1)
  decode    the decode workload (B=256, H=32, 1000 chained steps): HBM GB/s;
            a summary (GB/s, roofline fraction) is repeated in config.decode
  decode_raw  the same through the step with the input preparation fused in
  prep      the fused input preparation (ckda_prep) on raw inputs of the
            KDA-range shape: HBM GB/s
  bwd       the backward (ckda_bwd) on the KDA-range workload: token-heads/s
  workloads the KDA-range, packed and dk = 64 KDA-range workloads (N=1):
            token-heads/s, roofline
  clocks    SM clocks and throttle reasons sampled during the timed region
--impl reference runs the fp64 oracle as the reference arm on the host cores.
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); timing is max over ranks after a barrier.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CKDA fwd tokens/s (B×T×H) at d=128 bf16 and % of roofline; decode HBM GB/s"
UNIT = "tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_HBM_GBS = 6800.0


def fwd_bytes(B, H, T, dk, dv, nseq, h0, hT, io_bytes=2):
    th = B * H * T
    b = th * ((3 * dk + 2 * dv) * io_bytes + io_bytes)
    st = nseq * H * dk * dv * 4
    return b + (st if h0 else 0) + (st if hT else 0)


def decode_bytes(B, H, dk, dv, io_bytes=2):
    return B * H * (2 * dk * dv * 4 + (3 * dk + 2 * dv) * io_bytes + io_bytes)


def hbm_peak():
    try:
        p = json.load(open(PEAKS_FILE))
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# source files each profiled kernel is built from; a committed DRAM-traffic
# figure only counts while these files are unchanged
KERNEL_SOURCES = {
    "fwd": ["ckda_fwd.cu", "sm103.cuh", "ckda_internal.cuh"],
    "fwd_raw": ["ckda_fwd.cu", "sm103.cuh", "ckda_internal.cuh"],
    "decode128": ["ckda_decode.cu", "ckda_internal.cuh"],
    "decode128_raw": ["ckda_decode.cu", "ckda_internal.cuh"],
    "prep": ["ckda_prep.cu", "ckda_internal.cuh"],
    "prep_bwd": ["ckda_prep.cu", "ckda_internal.cuh"],
    "bwd": ["ckda_bwd.cu", "ckda_internal.cuh"],
}


def kernel_sources_sha(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_ckda_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel]:
        h.update(fn.encode())
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()


def fwd_kernel(dk):
    """The forward kernel a head size runs on (its DRAM-traffic record key)."""
    return "fwd"


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since it was taken; else None."""
    try:
        t = json.load(open(TRAFFIC_FILE))
        e = t["kernels"][kernel]
    except Exception:
        return None
    if e.get("sources_sha256") != kernel_sources_sha(kernel):
        return None
    w = e.get("workloads", {}).get(workload)
    return None if w is None else float(w["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons at 100 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"ckda_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [r for r in rows if r[2] > 250.0] or rows
        sm = sorted(r[0] for r in load)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r[2] for r in rows)}


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- our arm

def time_steps(step_fn, steps, warmup, ws, stream):
    """Runs warmup + timed steps back to back; returns (total seconds, max
    over ranks; the mean per-step device time in ms).  Two CUDA events on the
    launching stream bracket the K steps, with a barrier and a synchronize on
    both sides."""
    import torch
    for _ in range(warmup):
        step_fn()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        step_fn()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    local = t0.elapsed_time(t1) / 1e3
    total = max_over_ranks(local, ws)
    return total, [local / steps * 1e3]


def graph_protocol(step_on, nbytes, kernel, workload, launches=100, warmup=10, trials=3):
    """The scope table's timing protocol, next to the back-to-back timing:
    `warmup` eager steps on a side stream, then `launches` steps captured into
    one CUDA graph, replayed `trials` times, each replay bracketed by CUDA
    events; the median replay over `launches` is the time per step.
    `step_on(stream)` returns a step that launches on that stream."""
    import torch
    s = torch.cuda.Stream()
    step = step_on(s)
    try:
        with torch.cuda.stream(s):
            for _ in range(warmup):
                step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(launches):
                step()
        torch.cuda.synchronize()
        ms = []
        for _ in range(trials):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                g.replay()
                e1.record(s)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1) / launches)
        del g
    except Exception as e:  # a capture the runtime refuses is reported, not fatal
        torch.cuda.synchronize()
        return {"unavailable": f"{type(e).__name__}: {str(e).splitlines()[0][:160]}"}
    med = sorted(ms)[len(ms) // 2]
    return {"protocol": f"CUDA graph of {launches} steps after {warmup} eager warm-ups; median "
                        f"of {trials} replays", "ms_per_step": round(med, 4),
            "trials_ms_per_step": [round(m, 4) for m in ms],
            "roofline": roofline(nbytes, [med], kernel, workload)}


def fwd_case(ck, x, steps, warmup, ws, stream, name):
    import torch
    d = x.to("cuda")
    B, H, T, dk = d.q.shape
    dv = d.v.shape[-1]
    N = d.num_seqs
    o = torch.empty_like(d.v)
    hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device="cuda")
    wsp = ck.new_workspace(N if d.cu_seqlens is not None else 0, H, torch.device("cuda"))

    def step_on(s):
        return lambda: ck.fwd(d.q, d.k, d.v, d.alpha, d.beta, d.h0, d.cu_seqlens, o=o, hT=hT,
                              workspace=wsp, stream=s)

    step = step_on(stream)
    step()
    st = ck.fwd_status(wsp)
    if st != 0:
        raise RuntimeError(f"{name}: device status {ck.STATUS.get(st, st)}")
    total, per = time_steps(step, steps, warmup, ws, stream)
    th = B * H * T
    nbytes = fwd_bytes(B, H, T, dk, dv, N, d.h0 is not None, True)
    launches = 2 if d.cu_seqlens is not None else 1
    return dict(total=total, per=per, th=th, bytes=nbytes, launches=launches, dev=d, o=o, hT=hT,
                wsp=wsp, step_on=step_on)


def dense_case(ck, d, steps, warmup, ws, stream, name, segments):
    """ckda_fwd (segments = 1) or ckda_fwd_split on dense device tensors
    d = (q, k, v, alpha, beta, h0)."""
    import torch
    q, k, v, a, b, h0 = d
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = torch.empty_like(v)
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    wsp = torch.empty(ck.split_workspace_bytes(B, H, T, dk, dv, segments=segments),
                      dtype=torch.uint8, device="cuda")

    def step():
        ck.fwd_split(q, k, v, a, b, h0, segments=segments, o=o, hT=hT, workspace=wsp,
                     stream=stream)

    step()
    st = ck.fwd_status(wsp)
    if st != 0:
        raise RuntimeError(f"{name}: device status {ck.STATUS.get(st, st)}")
    total, per = time_steps(step, steps, warmup, ws, stream)
    th = B * H * T
    nbytes = fwd_bytes(B, H, T, dk, dv, B, h0 is not None, True)
    launches = 3 if segments >= 3 else (2 if segments == 2 else 1)
    return {"value": round(th * steps / total, 1), "unit": UNIT,
            "ms_per_step": round(total / steps * 1e3, 4), "steps": steps, "token_heads": th,
            "segments": segments, "launches_per_step": launches,
            "roofline": roofline(nbytes, per, "fwd", name)}


def fig5_sweep(ck, steps, ws, stream):
    """The paper's Fig. 5 shapes (16 heads, d = 128, 32k tokens per step, B x T from 16 x 2k
    down) plus 1 x 32k, each through one pass (ckda_fwd) and the sequence split at its
    automatic segment count.  Every point views the one `long_seq` draw as
    [B, 16, 32768 / B, 128], with its h0 repeated over B."""
    import synth
    x = synth.make_workload("long_seq").to("cuda")
    H, Ttot, dk = x.q.shape[1], x.q.shape[2], x.q.shape[3]
    out = {}
    for B in (16, 8, 4, 2, 1):
        T = Ttot // B
        v4 = lambda t: t.view(B, H, T, t.shape[-1])
        d = (v4(x.q), v4(x.k), v4(x.v), v4(x.alpha), x.beta.view(B, H, T),
             x.h0.expand(B, H, dk, dk).contiguous())
        S = ck.split_segments(B, H, T, dk, 128)
        name = "long_seq" if B == 1 else f"fig5_{B}x{T // 1024}k"
        pt = {"B": B, "T": T, "plain": dense_case(ck, d, steps, 3, ws, stream, name, 1)}
        if S > 1:
            pt["split"] = dense_case(ck, d, 2 * steps, 3, ws, stream, name, S)
            pt["split"]["roofline"]["traffic"] = None
        out[f"{B}x{T // 1024}k"] = pt
    return out


def varlen_split_case(ck, steps, ws, stream):
    """One 32k-token sequence packed with 63 of 1k tokens (16 heads, d = 128,
    KDA gates, h0): ckda_fwd on the packed input, where the long sequence's
    16 heads run 512 chunks each while the short ones finish early, against
    ckda_fwd_split_varlen at its automatic segment length."""
    import torch
    import synth
    lengths = [1024] * 31 + [32768] + [1024] * 32
    x = synth.make_varlen(lengths, 16, 128, dist="kda", dtype="bf16", h0=True, seed=54)
    name = "varlen_long_tail"
    plain = fwd_case(ck, x, steps, 3, ws, stream, name)
    d = plain["dev"]
    B, H, T, dk = d.q.shape
    N = d.num_seqs
    sl = ck.split_varlen_seg_len(N, H, T, dk, 128)
    wsp = torch.empty(ck.split_varlen_workspace_bytes(N, H, T, dk, sl), dtype=torch.uint8,
                      device="cuda")
    o, hT = plain["o"], plain["hT"]

    def step():
        ck.fwd_split_varlen(d.q, d.k, d.v, d.alpha, d.beta, d.cu_seqlens, h0=d.h0, seg_len=sl,
                            o=o, hT=hT, workspace=wsp, stream=stream)

    step()
    st = ck.fwd_status(wsp)
    if st != 0:
        raise RuntimeError(f"{name} split: device status {ck.STATUS.get(st, st)}")
    total, per = time_steps(step, steps, 3, ws, stream)
    out = {"config": {"lengths": "31 x 1024, 32768, 32 x 1024", "H": H, "d": dk, "h0": True,
                      "dist": "kda", "T": T}}
    for key, tot, pr, launches in (("plain", plain["total"], plain["per"], plain["launches"]),
                                   ("split", total, per, 5)):
        r = roofline(plain["bytes"], pr, "fwd", name)
        r["traffic"] = None
        out[key] = {"value": round(plain["th"] * steps / tot, 1), "unit": UNIT,
                    "ms_per_step": round(tot / steps * 1e3, 4), "launches_per_step": launches,
                    "roofline": r}
    out["split"]["seg_len"] = sl
    return out


def roofline(nbytes, per_ms, kernel, workload):
    peak, src = hbm_peak()
    mean_s = sum(per_ms) / len(per_ms) / 1e3
    ach = nbytes / mean_s / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
            "frac": round(ach / peak, 4), "traffic": traffic_for(kernel, workload),
            "algorithmic_bytes": nbytes, "mean_launch_ms": round(mean_s * 1e3, 4),
            "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
            else "fallback 6.8 TB/s"}


def e2e_packed(ck, x, steps, ws, stream):
    """Packed input (ckda_fwd_host takes dense input only): pinned host inputs
    copied to the device, ckda_fwd on them, o and hT copied back, all on the
    stream and inside the timed region."""
    import torch
    B, H, T, dk = x.q.shape
    dv = x.v.shape[-1]
    N = x.cu_seqlens.numel() - 1
    host = [t.pin_memory() for t in (x.q, x.k, x.v, x.alpha, x.beta, x.cu_seqlens)]
    hh0 = None if x.h0 is None else x.h0.pin_memory()
    dev = [torch.empty_like(t, device="cuda") for t in host]
    dh0 = None if hh0 is None else torch.empty_like(hh0, device="cuda")
    o = torch.empty((B, H, T, dv), dtype=x.q.dtype, device="cuda")
    hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device="cuda")
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hh = torch.empty(hT.shape, dtype=torch.float32).pin_memory()
    wsp = ck.new_workspace(N, H, torch.device("cuda"))

    def step():
        with torch.cuda.stream(stream):
            for d, h in zip(dev, host):
                d.copy_(h, non_blocking=True)
            if dh0 is not None:
                dh0.copy_(hh0, non_blocking=True)
            q, k, v, a, b, cu = dev
            ck.fwd(q, k, v, a, b, dh0, cu, o=o, hT=hT, workspace=wsp, stream=stream)
            ho.copy_(o, non_blocking=True)
            hh.copy_(hT, non_blocking=True)

    total, _ = time_steps(step, steps, 3, ws, stream)
    h2d = sum(t.numel() * t.element_size() for t in host) + \
        (0 if hh0 is None else hh0.numel() * 4)
    d2h = ho.numel() * ho.element_size() + hh.numel() * 4
    return {"value": round(ws * B * H * T * steps / total, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "path": "copies in, ckda_fwd (packed), copies out; not overlapped"}


def e2e_fwd(ck, x, steps, ws, stream):
    """Host (pinned) inputs -> ckda_fwd_host -> host outputs, the whole call
    timed: it copies each slice of tokens in, computes it and copies its o
    out, the copies of one slice overlapping the computation of another."""
    import torch
    if x.cu_seqlens is not None:
        return e2e_packed(ck, x, steps, ws, stream)
    B, H, T, dk = x.q.shape
    dv = x.v.shape[-1]
    hq, hk, hv, ha, hb = (t.pin_memory() for t in (x.q, x.k, x.v, x.alpha, x.beta))
    hh0 = None if x.h0 is None else x.h0.pin_memory()
    ho = torch.empty((B, H, T, dv), dtype=x.q.dtype).pin_memory()
    hh = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()
    scratch = torch.empty(ck.host_scratch_bytes(B, H, T, dk, dv, x.q.dtype), dtype=torch.uint8,
                          device="cuda")

    def step():
        ck.fwd_host(hq, hk, hv, ha, hb, hh0, o=ho, hT=hh, scratch=scratch, stream=stream)

    total, _ = time_steps(step, steps, 3, ws, stream)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ha, hb)) + \
        (0 if hh0 is None else hh0.numel() * 4)
    d2h = ho.numel() * ho.element_size() + hh.numel() * 4
    return {"value": round(ws * B * H * T * steps / total, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps}


def decode_case(ck, steps, warmup, ws, stream, pool=32, raw=False):
    """The decode workload; with raw=True through ckda_decode_step_raw (the
    same seeded tensors read as raw q, k and gate logits: the same bytes)."""
    import torch
    import synth
    w = synth.WORKLOADS["ckda_decode"]
    B, H, d = w["B"], w["H"], w["d"]
    S = synth.make_decode_state(B, H, d, seed=w["seed"]).cuda()
    ins = [tuple(t.cuda() for t in synth.make_decode_step(B, H, d, seed=w["seed"], step=i))
           for i in range(pool)]
    o = torch.empty((B, H, d), dtype=torch.bfloat16, device="cuda")
    it = [0]

    def step_on(s):
        def step():
            q, k, v, a, b = ins[it[0] % pool]
            it[0] += 1
            if raw:
                ck.decode_step_raw(q, k, v, a, b, S, o=o, stream=s)
            else:
                ck.decode_step(q, k, v, a, b, S, o=o, stream=s)
        return step

    total, per = time_steps(step_on(stream), steps, warmup, ws, stream)
    nbytes = decode_bytes(B, H, d, d)
    kern = "decode128_raw" if raw else "decode128"
    rl = roofline(nbytes, per, kern, "ckda_decode")
    gp = graph_protocol(step_on, nbytes, kern, "ckda_decode")
    return {"value": round(ws * nbytes * steps / total / 1e9, 1), "unit": "GB/s",
            "steps": steps, "ms_per_step": round(total / steps * 1e3, 4),
            "config": {"workload": "ckda_decode", "B": B, "H": H, "d": d,
                       "inputs": f"pool of {pool} seeded steps cycled"},
            "roofline": rl, "graph_protocol": gp, "gpu_launches": steps}


def prep_bytes(rows, dk, io_bytes=2, with_q=True):
    nt = 3 if with_q else 2
    return rows * 2 * (nt * dk * io_bytes + io_bytes)


def prep_case(ck, x, steps, warmup, ws, stream, name):
    """ckda_prep on raw inputs of the workload's shape: q and k unnormalised,
    gate logits a ~ N(0, 2), b ~ N(0, 1); HBM bytes read and written once."""
    import torch
    B, H, T, dk = x.q.shape
    g = torch.Generator().manual_seed(21)
    raw = [torch.randn(sh, generator=g).to(torch.bfloat16).cuda()
           for sh in ((B, H, T, dk), (B, H, T, dk), (B, H, T, dk), (B, H, T))]
    qr, kr, ar, br = raw
    qr.mul_(3)
    ar.mul_(2)
    out = (torch.empty_like(qr), torch.empty_like(kr), torch.empty_like(ar), torch.empty_like(br))

    def step():
        ck.prep(kr, ar, br, q_raw=qr, out=out, stream=stream)

    total, per = time_steps(step, steps, warmup, ws, stream)
    rows = B * H * T
    nbytes = prep_bytes(rows, dk)
    peak, src = hbm_peak()
    ms = sum(per) / len(per)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del raw, out
    return {"value": round(nbytes * steps / total / 1e9, 1), "unit": "GB/s", "steps": steps,
            "ms_per_step": round(total / steps * 1e3, 4),
            "config": {"workload": f"raw inputs of the {name} shape", "rows": rows, "dk": dk,
                       "io": "bf16", "normalize_q": True},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": traffic_for("prep", name),
                         "algorithmic_bytes": nbytes, "mean_launch_ms": round(ms, 4),
                         "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"
                         if src == "measured" else src},
            "gpu_launches": steps}


def prep_bwd_bytes(rows, dk, io_bytes=2):
    """Algorithmic bytes of ckda_prep_bwd with q: q_raw, k_raw, a_raw and the
    gradients of q, k, alpha in, those of the raw three out (dk each), plus
    b_raw and d_beta in and d_b_raw out."""
    return rows * (9 * dk + 3) * io_bytes


def prep_bwd_case(ck, x, steps, warmup, ws, stream, name):
    """ckda_prep_bwd on raw inputs of the workload's shape (as prep_case) and
    unit-normal upstream gradients; HBM bytes read and written once."""
    import torch
    B, H, T, dk = x.q.shape
    g = torch.Generator().manual_seed(22)
    shapes = ((B, H, T, dk),) * 3 + ((B, H, T),) + ((B, H, T, dk),) * 3 + ((B, H, T),)
    t = [torch.randn(sh, generator=g).to(torch.bfloat16).cuda() for sh in shapes]
    qr, kr, ar, br, dq, dk_, da, db = t
    qr.mul_(3)
    ar.mul_(2)
    out = (torch.empty_like(qr), torch.empty_like(kr), torch.empty_like(ar), torch.empty_like(br))

    def step():
        ck.prep_bwd(kr, ar, br, dk_, da, db, q_raw=qr, d_q=dq, out=out, stream=stream)

    total, per = time_steps(step, steps, warmup, ws, stream)
    rows = B * H * T
    nbytes = prep_bwd_bytes(rows, dk)
    peak, src = hbm_peak()
    ms = sum(per) / len(per)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del t, out
    return {"value": round(nbytes * steps / total / 1e9, 1), "unit": "GB/s", "steps": steps,
            "ms_per_step": round(total / steps * 1e3, 4),
            "config": {"workload": f"raw inputs and upstream gradients of the {name} shape",
                       "rows": rows, "dk": dk, "io": "bf16", "normalize_q": True},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": traffic_for("prep_bwd", name),
                         "algorithmic_bytes": nbytes, "mean_launch_ms": round(ms, 4),
                         "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"
                         if src == "measured" else src},
            "gpu_launches": steps}


def fwd_raw_case(ck, x, steps, warmup, ws, stream, name):
    """The forward on raw inputs of the workload's shape: ckda_fwd_raw (the
    preparation inside the forward kernel) against ckda_prep followed by
    ckda_fwd.  Both read raw q, k, a, b and v and write o and hT; the
    algorithmic bytes are the forward's (the prepared tensors need not touch
    HBM)."""
    import torch
    B, H, T, dk = x.q.shape
    g = torch.Generator().manual_seed(23)
    qr, kr, ar = (torch.randn((B, H, T, dk), generator=g).to(torch.bfloat16).cuda()
                  for _ in range(3))
    br = torch.randn((B, H, T), generator=g).to(torch.bfloat16).cuda()
    v = x.v.cuda()
    h0 = None if x.h0 is None else x.h0.cuda()
    o = torch.empty_like(v)
    hT = torch.empty((B, H, dk, v.shape[-1]), dtype=torch.float32, device="cuda")
    wsp = ck.new_workspace(0, H, torch.device("cuda"))
    prepped = (torch.empty_like(qr), torch.empty_like(kr), torch.empty_like(ar),
               torch.empty_like(br))

    def fused():
        ck.fwd_raw(qr, kr, v, ar, br, h0, o=o, hT=hT, workspace=wsp, stream=stream)

    def two_pass():
        q, k, a, b = ck.prep(kr, ar, br, q_raw=qr, out=prepped, stream=stream)
        ck.fwd(q, k, v, a, b, h0, o=o, hT=hT, workspace=wsp, stream=stream)

    fused()
    st = ck.fwd_status(wsp)
    if st != 0:
        raise RuntimeError(f"{name} raw: device status {ck.STATUS.get(st, st)}")
    th = B * H * T
    nbytes = fwd_bytes(B, H, T, dk, v.shape[-1], B, h0 is not None, True)
    out = {}
    for key, fn, launches in (("fused", fused, 1), ("prep_then_fwd", two_pass, 2)):
        total, per = time_steps(fn, steps, warmup, ws, stream)
        r = roofline(nbytes, per, "fwd_raw", name)
        if key != "fused":
            r["traffic"] = None  # two kernels
        out[key] = {"value": round(th * steps / total, 1), "unit": UNIT,
                    "ms_per_step": round(total / steps * 1e3, 4), "launches_per_step": launches,
                    "roofline": r}
    del qr, kr, ar, br, prepped
    return out


def bwd_bytes(B, H, T, dk, dv, io_bytes=2):
    """Algorithmic bytes of ckda_bwd: q, k, alpha, v, do, beta in; dq, dk,
    dalpha, dv, dbeta out (the states it stores and reads back are not)."""
    return B * H * T * (6 * dk + 3 * dv + 2) * io_bytes


def bwd_case(ck, x, steps, warmup, ws, stream, units=0, name="ckda_full"):
    """ckda_bwd on the workload (or, with units > 0, on its first `units`
    (batch, head) pairs: a smaller workspace, the same per-unit work)."""
    import torch
    import synth
    if units > 0:
        B0, H0 = x.q.shape[:2]
        nb, nh = max(1, units // H0), min(units, H0)
        sl = lambda t: None if t is None else t[:nb, :nh].contiguous()
        x = synth.FwdInputs(sl(x.q), sl(x.k), sl(x.v), sl(x.alpha), sl(x.beta), sl(x.h0), None)
    d = x.to("cuda")
    B, H, T, dk = d.q.shape
    dv = d.v.shape[-1]
    g = torch.Generator().manual_seed(31)
    do = torch.randn(tuple(d.v.shape), generator=g).to(d.v.dtype).cuda()
    need = ck.bwd_workspace_bytes(B, H, T, dk, dv)
    wsp = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")

    def step():
        ck.bwd(d.q, d.k, d.v, d.alpha, d.beta, do, h0=d.h0, workspace=wsp, stream=stream)

    total, per = time_steps(step, steps, warmup, ws, stream)
    th = B * H * T
    nbytes = bwd_bytes(B, H, T, dk, dv)
    peak, src = hbm_peak()
    ms = sum(per) / len(per)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del wsp, do, d
    return {"value": round(th * steps / total, 1), "unit": UNIT, "steps": steps,
            "ms_per_step": round(total / steps * 1e3, 4), "token_heads": th,
            "config": {"workload": name if units <= 0 else f"{name}, {B * H} units",
                       "kernel": "token-serial, CUDA cores, fp32", "workspace_bytes": need},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4),
                         "traffic": traffic_for("bwd", name) if units <= 0 else None,
                         "algorithmic_bytes": nbytes, "mean_launch_ms": round(ms, 4),
                         "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"
                         if src == "measured" else src},
            "gpu_launches": steps}


def cpu_baseline(x, target_s=12.0):
    """The oracle, as it stands, on a bounded sample of the workload's units."""
    import oracle
    B, H, T, _ = x.q.shape
    units = [(b, h) for b in range(B) for h in range(H)]
    n = min(len(units), max(1, oracle.max_threads()))
    t_used, th_done, reps = 0.0, 0, 0
    while True:
        sel = units[(reps * n) % len(units):][:n]
        bs = sorted({b for b, _ in sel})
        hs = sorted({h for _, h in sel})
        sub = lambda t: t[bs][:, hs]
        t0 = time.perf_counter()
        oracle.fwd(sub(x.q), sub(x.k), sub(x.v), sub(x.alpha), sub(x.beta),
                   None if x.h0 is None else sub(x.h0))
        dt = time.perf_counter() - t0
        t_used += dt
        th_done += len(bs) * len(hs) * T
        reps += 1
        if t_used >= target_s or reps >= 50:
            break
        if dt < target_s / 8 and n < len(units):
            n = min(len(units), n * 2)
    return {"value": round(th_done / t_used, 1), "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{reps} runs over {th_done} token-heads (whole (batch, head) sequences of "
                      f"T={T}) of the same workload, {t_used:.1f} s, fp64 C + OpenMP"}


def run_ours(args):
    import torch
    import gated_delta_rule_ckda_gb300 as ck
    import synth
    ws, rank, local = dist_setup()
    ck.lib()
    stream = torch.cuda.current_stream()
    name = args.workload
    x = synth.make_workload(name)
    clocks = ClockSampler(local)
    clocks.start()
    r = fwd_case(ck, x, args.steps, args.warmup, ws, stream, name)
    clk = clocks.stop()
    B, H, T, dk = x.q.shape
    value = ws * r["th"] * args.steps / r["total"]
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(r["total"] / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "H": H, "T": T, "dk": dk, "dv": x.v.shape[-1],
                   "io": "bf16", "state": "fp32", "chunk": 64,
                   "precision": "bf16 I/O; fp16/bf16 tensor-core operands; fp32 accumulation, "
                                "gate products, T and state",
                   "l2": "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": roofline(r["bytes"], r["per"], fwd_kernel(dk), name),
        "gpu_launches": r["launches"] * args.steps,
        "clocks": clk,
    }
    if ws == 1:
        out["graph_protocol"] = graph_protocol(r["step_on"], r["bytes"], fwd_kernel(dk), name)
    out["e2e"] = e2e_fwd(ck, x, max(3, min(args.steps, args.e2e_steps)), ws, stream)
    extras = [] if args.no_extras else [e for e in args.extras.split(",") if e and e != "none"]
    if ws == 1 and "decode" in extras:
        out["decode"] = decode_case(ck, args.decode_steps, 10, ws, stream)
        dr = out["decode"]["roofline"]
        # the metric's second half, kept where the one-line record is read
        out["config"]["decode"] = {"workload": "ckda_decode (B=256, H=32, d=128, 1000 chained "
                                               "steps)", "GB/s": out["decode"]["value"],
                                   "roofline_frac": dr["frac"], "ms_per_step":
                                   out["decode"]["ms_per_step"]}
    if ws == 1 and "decode_raw" in extras:
        out["decode_raw"] = decode_case(ck, args.decode_steps, 10, ws, stream, raw=True)
    if ws == 1 and "prep" in extras:
        out["prep"] = prep_case(ck, x, 200, 10, ws, stream, args.workload)
    if ws == 1 and "fwd_raw" in extras:
        out["fwd_raw"] = fwd_raw_case(ck, x, 100, 5, ws, stream, args.workload)
    if ws == 1 and "prep_bwd" in extras:
        out["prep_bwd"] = prep_bwd_case(ck, x, 200, 10, ws, stream, args.workload)
    if ws == 1 and "bwd" in extras:
        out["bwd"] = bwd_case(ck, x, 10, 3, ws, stream, units=args.bwd_units, name=args.workload)
    if ws == 1 and any(e in extras for e in ("kda_range", "ckda_full", "ckda_varlen",
                                             "kda_range_dk64")):
        wl = {}
        for nm, steps in (("kda_range", 200), ("ckda_full", 20), ("ckda_varlen", 10),
                          ("kda_range_dk64", 200)):
            if nm not in extras or nm == name:
                continue
            xx = synth.make_workload(nm)
            rr = fwd_case(ck, xx, steps, 3, ws, stream, nm)
            wl[nm] = {"value": round(rr["th"] * steps / rr["total"], 1), "unit": UNIT,
                      "ms_per_step": round(rr["total"] / steps * 1e3, 4), "steps": steps,
                      "token_heads": rr["th"],
                      "roofline": roofline(rr["bytes"], rr["per"], fwd_kernel(xx.q.shape[-1]), nm),
                      "graph_protocol": graph_protocol(
                          rr["step_on"], rr["bytes"], fwd_kernel(xx.q.shape[-1]), nm,
                          launches=10 if nm == "ckda_varlen" else 100)}
            del xx, rr
        out["workloads"] = wl
    if ws == 1 and "varlen_split" in extras:
        out["varlen_split"] = varlen_split_case(ck, 20, ws, stream)
    if ws == 1 and "fig5_sweep" in extras:
        # 32k tokens per step of 16 heads at B x T = 16 x 2k .. 1 x 32k: one pass fills
        # B x 16 SMs; the split runs the long sequences as segments
        out["fig5_sweep"] = fig5_sweep(ck, 5, ws, stream)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(x, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out))


# ----------------------------------------------------------- reference arm

def run_reference(args):
    """The fp64 oracle on the host cores, as the reference arm."""
    import numpy as np  # noqa: F401
    import oracle
    import synth
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    name = args.workload
    x = synth.make_workload(name)
    B, H, T, dk = x.q.shape
    budget = 150.0 / (args.steps + args.warmup)  # seconds per step
    # one step: whole (batch, head) units, as many as fit the per-step budget
    probe_t0 = time.perf_counter()
    sub = lambda t, n: t[:1, :n]
    oracle.fwd(sub(x.q, 1), sub(x.k, 1), sub(x.v, 1), sub(x.alpha, 1), sub(x.beta, 1))
    per_unit = time.perf_counter() - probe_t0
    cores = oracle.max_threads()
    n_units = int(max(1, min(H, cores * max(1.0, budget / max(per_unit, 1e-6)))))
    n_units = min(n_units, H)
    Tm = T
    if per_unit > budget:  # even one unit is too slow: shorten the sample
        Tm = max(64, int(T * budget / per_unit))
    args_ = [t[:1, :n_units, :Tm] for t in (x.q, x.k, x.v, x.alpha, x.beta)]
    for _ in range(args.warmup):
        oracle.fwd(*args_)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.fwd(*args_)
    total = time.perf_counter() - t0
    th = n_units * Tm * args.steps
    value = th / total
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": name, "B": B, "H": H, "T": T, "dk": dk, "dv": x.v.shape[-1],
                   "io": "bf16 inputs widened to fp64", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step: {n_units} (batch, head) units x {Tm} tokens of "
                                   f"the {name} workload"},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ckda_full",
                    choices=["kda_range", "ckda_full", "ckda_varlen"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--extras",
                    default="decode,decode_raw,prep,prep_bwd,fwd_raw,bwd,kda_range,ckda_varlen,"
                            "kda_range_dk64,fig5_sweep,varlen_split",
                    help="comma list of extra measurements: decode, decode_raw, prep, prep_bwd, fwd_raw, bwd, "
                         "varlen_split, "
                         "kda_range, ckda_full, ckda_varlen, kda_range_dk64, fig5_sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd-units", type=int, default=0,
                    help="run the bwd extra on the first N (batch, head) units only")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
