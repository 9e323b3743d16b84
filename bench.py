#!/usr/bin/env python
"""Prefill throughput of the gated delta rule forward pass (chunk-parallel WY
form) on GB300, with its roofline and the fp64 oracle timed on the host cores.

One step = one pass of the whole hot path (chunk-prep kernel + scan kernel)
over one batch of synthetic input.  Default workload: the 32k-token spot of
stratat pull #1296 ("Measured verdict on gfx1100": 32k tokens, HV = 48 value
heads, state 128) as bf16 GDN with 16 q/k heads and chunk 64.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  Multi-GPU (torchrun, one rank per GPU): every
rank runs its own copy of the workload (independent sequences, no collective
on the data path) -> weak scaling; the value is all ranks' tokens over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s (gated delta-rule fwd, 1 GB300) and % of HBM/tensor roofline"
METRIC_DECODE = "decode tokens/s (gated delta-rule step, T = 1, 1 GB300) and % of HBM roofline"
METRIC_PREPOST = ("pre/post ops tokens/s (causal conv + q/k L2 norm + gated RMS norm, 1 GB300) "
                  "and % of HBM roofline")


def metric_of(c) -> str:
    """The metric a workload's line reports (the same for both arms)."""
    if c.name.startswith("prepost"):
        return METRIC_PREPOST
    if c.T == 1 and "decode" in c.name:
        return METRIC_DECODE
    return METRIC
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "gdn_bf16_t32768"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-lockstep", action="store_true",
                    help="skip the lockstep launch's timing pass")
    ap.add_argument("--in-flight", type=int, default=3,
                    help="independent batches in flight in the throughput pass (3 measured "
                         "best at 32k tokens: 2 / 3 / 4 give 39.6 / 41.8 / 41.1 M tokens/s)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# workload arithmetic (per-token bytes and FLOPs of the roofline)
# ---------------------------------------------------------------------------
def algorithmic_bytes(c, which="path"):
    """HBM bytes each kernel must move at least once: q, k, v, g, beta read,
    o written (states excluded, <= ~1% here)."""
    es = 2 if c.dtype_name == "bf16" else 4
    n = c.tokens
    qk = 2 * n * c.H * c.dk * es
    vo = 2 * n * c.HV * c.dv * es
    gb = n * c.HV * (1 if c.gate_mode == 0 else c.dk) * 4
    bb = n * c.HV * 4
    if which == "prep":  # reads q, k, g, beta
        return qk + gb + bb
    return qk + vo + gb + bb  # scan and whole path: everything once


# what each kernel of the split design reads and writes at least once, per
# chunk slot: the scalar-gate bf16 path's prep writes one 32 KB operand image
# per value head and one 32 KB [K_next; Q] image per q/k head, the per-key-gate
# path's prep an operand image and a gated [Kg; Qg] image per value head, and
# the scan reads them back
KERNEL_BYTES_NOTE = {
    ("scan", "bf16", 0): "v, o, g, beta plus the prep's operand images read back "
                         "(HV x 32 KB and H x 32 KB per chunk)",
    ("prep", "bf16", 0): "q, k, g, beta plus the operand images written "
                         "(HV x 32 KB and H x 32 KB per chunk)",
    ("scan", "bf16", 1): "v, o, beta plus the prep's images read back (per chunk and value "
                         "head: [P1; AqkT] and the gated [Kg; Qg], 10 + 16 KB at chunk 32, "
                         "24 + 32 KB at chunk 64, and dk decays)",
    ("prep", "bf16", 1): "q, k, the per-channel g, beta plus the images written (per chunk "
                         "and value head: 10 + 16 KB at chunk 32, 24 + 32 KB at chunk 64, and "
                         "dk decays)",
}


def kernel_design_bytes(c, which, case, cu_seqlens=None):
    """Bytes one kernel of the bf16 split design must move; None for the fp32
    path.  ``cu_seqlens``: the packed cuts of a varlen workload."""
    if (which, c.dtype_name, c.gate_mode) not in KERNEL_BYTES_NOTE:
        return None
    n = c.tokens
    slots = n // c.chunk + case.num_states  # chunk slots the workspace holds (upper bound)
    chunks = sum(-(-L // c.chunk) for L in seq_lengths(case, cu_seqlens))
    assert chunks <= slots
    if c.gate_mode == 1:  # per-key gate: per (chunk, value head) images and decays
        per = (10240 + (c.dk // 64) * 8192) if c.chunk == 32 else (24576 + (c.dk // 64) * 16384)
        images = chunks * c.HV * (per + c.dk * 4)
        if which == "scan":
            return 2 * n * c.HV * c.dv * 2 + n * c.HV * 4 + images
        return 2 * n * c.H * c.dk * 2 + n * c.HV * c.dk * 4 + n * c.HV * 4 + images
    images = chunks * (c.HV * 32768 + c.H * (c.dk // 64) * 16384)
    if which == "scan":
        return 2 * n * c.HV * c.dv * 2 + 2 * n * c.HV * 4 + images
    return 2 * n * c.H * c.dk * 2 + 2 * n * c.HV * 4 + images


def seq_lengths(case, cu_seqlens=None):
    """Lengths of the sequences of a workload."""
    if case.n_seqs > 0:
        cu = [int(v) for v in cu_seqlens]
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    return [case.T] * case.B


def algorithmic_flops(c):
    """Chunk-GEMM FLOPs, dense count: per token and value head
    2 (3 C dk + 2 C dv + 3 dk dv): Gram, W, Aqk; U, O_intra; W S, Qg S, Kt^T Vn."""
    C, dk, dv = c.chunk, c.dk, c.dv
    return c.tokens * c.HV * 2 * (3 * C * dk + 2 * C * dv + 3 * dk * dv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


def kernel_source_sha(source):
    """Hash of one kernel's translation unit and every header of csrc/ (the
    structs and device helpers it compiles with)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunkwise_gated_delta_gdn_gb300", "csrc")
    names = [source] + sorted(n for n in os.listdir(csrc) if n.endswith((".h", ".cuh")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, kernel, units):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; scaled by units processed when the capture
    ran a smaller case."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None, None
    for e in rec.get("entries", []):
        src = e.get("source")
        if (e.get("kernel") == kernel and e.get("workload") == workload and src
                and e.get("source_sha") == kernel_source_sha(src)):
            per_unit = float(e["dram_bytes"]) / float(e["tokens"])
            return per_unit * units, e.get("note")
    return None, None


# ---------------------------------------------------------------------------
# ranks: one process per GPU, independent replicas, timed by the slowest
# ---------------------------------------------------------------------------
def rank_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(x: float, dev) -> float:
    """The largest x over all ranks (every rank gets the slowest rank's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ms_step: float, world: int) -> float:
    """Units all ranks processed per second at the slowest rank's step time."""
    return world * units_per_rank / (ms_step / 1e3)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU side: the oracle
# ---------------------------------------------------------------------------
def oracle_sample(c, x, n_tokens):
    """Run the token-serial oracle on the first n_tokens of every sequence
    row (all value heads); returns (seconds, tokens processed)."""
    import numpy as np
    import oracle

    Bq = x["q"].shape[0]
    n_tokens = max(1, min(n_tokens, x["q"].shape[1]))
    if x["cu_seqlens"] is not None:  # packed: the first sequence's prefix
        first = int(x["cu_seqlens"][1])
        n_tokens = min(n_tokens, first)
        Bq = 1
    q = x["q"][:Bq, :n_tokens].reshape(-1, c.H, c.dk)
    k = x["k"][:Bq, :n_tokens].reshape(-1, c.H, c.dk)
    v = x["v"][:Bq, :n_tokens].reshape(-1, c.HV, c.dv)
    g = x["g"][:Bq, :n_tokens].reshape((-1,) + tuple(x["g"].shape[2:]))
    beta = x["beta"][:Bq, :n_tokens].reshape(-1, c.HV)
    h0 = x["h0"][:Bq] if x["h0"] is not None else None
    cu = np.arange(Bq + 1, dtype=np.int64) * n_tokens
    t = time.perf_counter()
    oracle.token_serial(q, k, v, g, beta, h0, cu, c.scale, c.gate_mode)
    return time.perf_counter() - t, Bq * n_tokens


def oracle_sample_text(c0, x, n):
    """What oracle_sample processed, from the tokens it reports."""
    if x["cu_seqlens"] is not None:
        where = f"the first {n} tokens of the first packed sequence"
    elif x["q"].shape[0] == 1:
        where = f"the first {n} tokens"
    else:
        rows = x["q"].shape[0]
        where = f"the first {n // rows} tokens of each of the {rows} batch rows ({n} tokens)"
    return f"fp64 token-serial oracle on {where} (all {c0.HV} value heads) of {c0.name}"


def calibrate_oracle(c, x, target_s):
    sec, n = oracle_sample(c, x, 64)
    per_token = sec / n
    return max(16, int(target_s / max(per_token, 1e-9)))


# ---------------------------------------------------------------------------
def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.gpus > 1 and world == 1:
        raise SystemExit("--gpus N > 1 must be launched with torchrun (one rank per GPU)")

    from chunkwise_gated_delta_gdn_gb300 import synth

    c0 = synth.case(args.workload)

    class W:  # workload view with the fields the arithmetic needs
        pass

    wl = W()
    for f in ("H", "HV", "dk", "dv", "chunk", "gate_mode", "scale"):
        setattr(wl, f, getattr(c0, f))
    wl.tokens = c0.tokens
    wl.dtype_name = "bf16" if str(c0.dtype).endswith("bfloat16") else "f32"
    config = {"workload": c0.name, "B": c0.B, "T": c0.T, "H": c0.H, "HV": c0.HV,
              "dk": c0.dk, "dv": c0.dv, "chunk": c0.chunk,
              "gate": "scalar (GDN)" if c0.gate_mode == 0 else "per-key (KDA)",
              "n_seqs": c0.num_states, "h0": c0.h0_std is not None}

    if args.impl == "reference":
        run_reference(args, rank, world, c0, wl, config)
        return
    if c0.T == 1 and "decode" in c0.name:
        bench_decode(args, rank, world, local_rank, c0, wl, config)
        return
    if c0.name.startswith("prepost"):
        bench_prepost(args, rank, world, local_rank, c0, wl, config)
        return

    import torch
    import torch.distributed as dist

    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    from chunkwise_gated_delta_gdn_gb300 import build as cuda_build
    from chunkwise_gated_delta_gdn_gb300 import gdn

    gdn.load(cuda_build.build())
    x = synth.make_inputs(c0)
    names = ("q", "k", "v", "g", "beta", "h0", "cu_seqlens")
    d = {n: (x[n].to(dev) if x[n] is not None else None) for n in names}
    B, T = x["q"].shape[0], x["q"].shape[1]
    n_states = c0.num_states
    o = torch.empty((B, T, c0.HV, c0.dv), dtype=c0.dtype, device=dev)
    hT = torch.empty((n_states, c0.HV, c0.dk, c0.dv), dtype=torch.float32, device=dev)
    dt = gdn.GDN_BF16 if c0.dtype == torch.bfloat16 else gdn.GDN_F32
    ws_bytes = gdn.gdn_chunk_fwd_workspace_bytes(B, T, c0.H, c0.HV, c0.dk, c0.dv, c0.chunk,
                                                 c0.gate_mode, n_states, dt)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    kw = dict(workspace=ws, o=o, hT=hT, scale=c0.scale, chunk=c0.chunk,
              cu_seqlens=d["cu_seqlens"])
    args_in = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])

    def step():
        gdn.gdn_chunk_fwd_prep(*args_in, **kw)
        gdn.gdn_chunk_fwd_scan(*args_in, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags = gdn.gdn_read_device_flags(ws)

    K = args.steps
    # (1) kernel pass: steps one after another on one stream, CUDA events
    # around each launch -> per-kernel times for the kernel roofline
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        ev[i][0].record()
        gdn.gdn_chunk_fwd_prep(*args_in, **kw)
        ev[i][1].record()
        gdn.gdn_chunk_fwd_scan(*args_in, **kw)
        ev[i][2].record()
    torch.cuda.synchronize()
    prep_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    scan_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K

    # (1b) single calls: whole gdn_chunk_fwd passes one after another on one
    # stream, each finishing before the next starts (what a prefill layer that
    # must complete before the next layer gets)
    ev_a = torch.cuda.Event(enable_timing=True)
    ev_b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev_a.record()
    for _ in range(K):
        gdn.gdn_chunk_fwd(*args_in, **kw)
    ev_b.record()
    torch.cuda.synchronize()
    single_ms = max_over_ranks(ev_a.elapsed_time(ev_b) / K, dev)

    # (1c) the lockstep launch (prep and scan in one cooperative grid), where
    # the path has one: single calls one after another, as (1b)
    lock_ms, lock_refused = None, None
    if wl.dtype_name == "bf16" and c0.gate_mode == 0 and not args.no_lockstep:
        try:
            gdn.gdn_chunk_fwd_lockstep(*args_in, **kw)
        except gdn.GdnError as e:  # e.g. more scan blocks than SMs: refused on the host
            lock_refused = str(e)
        if lock_refused is None:
            gdn.gdn_chunk_fwd_lockstep(*args_in, **kw)
            torch.cuda.synchronize()
            ev_a.record()
            for _ in range(K):
                gdn.gdn_chunk_fwd_lockstep(*args_in, **kw)
            ev_b.record()
            torch.cuda.synchronize()
            lock_ms = max_over_ranks(ev_a.elapsed_time(ev_b) / K, dev)

    # (2) throughput pass (the reported value): independent batches in flight
    # on their own streams, each with its own workspace and outputs, so one
    # batch's prep fills the SMs another's scan leaves idle.  Every step is
    # still one whole forward pass over one batch.
    nf = max(1, args.in_flight)
    ws2 = [ws] + [torch.empty_like(ws) for _ in range(nf - 1)]
    outs2 = [(o, hT)] + [(torch.empty_like(o), torch.empty_like(hT)) for _ in range(nf - 1)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(nf)]
    main = torch.cuda.current_stream(dev)

    def step2(i):
        b = i % nf
        with torch.cuda.stream(streams[b]):
            gdn.gdn_chunk_fwd(*args_in, o=outs2[b][0], hT=outs2[b][1], workspace=ws2[b],
                              scale=c0.scale, chunk=c0.chunk, cu_seqlens=d["cu_seqlens"],
                              stream=streams[b])

    for i in range(max(args.warmup, nf)):
        step2(i)
    torch.cuda.synchronize()
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.25)  # let the sampler come up before the timed region
    ev_start.record(main)
    for s_ in streams:
        s_.wait_event(ev_start)
    for i in range(K):
        step2(i)
    for s_ in streams:
        main.wait_stream(s_)
    ev_end.record(main)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = ev_start.elapsed_time(ev_end)
    ms_step = max_over_ranks(ms_total / K, dev)
    tokens_per_rank = c0.tokens
    value = whole_job_rate(tokens_per_rank, ms_step, world)

    # ---- end to end through the public binding, host buffers ----
    # Every step copies its inputs in from pinned host memory and its results
    # (o and hT) back out.  Steps are pipelined the way a serving loop would
    # run them: double-buffered device inputs and outputs, host-to-device
    # copies on one stream, the forward pass on a second, device-to-host
    # copies on a third, ordered by events; the timed region runs from the
    # first copy in to the last copy out.
    e2e = None
    if not args.no_e2e:
        host = {n: (x[n].pin_memory() if x[n] is not None else None) for n in names}
        o_hosts = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
        h_hosts = [torch.empty(hT.shape, dtype=hT.dtype).pin_memory() for _ in range(2)]
        h2d = sum(host[n].numel() * host[n].element_size() for n in names if host[n] is not None)
        d2h = o.numel() * o.element_size() + hT.numel() * hT.element_size()
        dbuf = [d] + [{n: (torch.empty_like(d[n]) if d[n] is not None else None) for n in names}]
        obuf = [(o, hT), (torch.empty_like(o), torch.empty_like(hT))]
        s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_run = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        started = [False, False]

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if started[b]:
                    s_in.wait_event(ev_run[b])  # step i-2 is done reading buffer b
                for n in names:
                    if host[n] is not None:
                        dbuf[b][n].copy_(host[n], non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev_in[b])
                if started[b]:
                    s_run.wait_event(ev_out[b])  # step i-2's results have left buffer b
                db, (ob, hb) = dbuf[b], obuf[b]
                gdn.gdn_chunk_fwd(db["q"], db["k"], db["v"], db["g"], db["beta"], db["h0"], o=ob,
                                  hT=hb, workspace=ws, scale=c0.scale, chunk=c0.chunk,
                                  cu_seqlens=db["cu_seqlens"], stream=s_run)
                ev_run[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[b])
                o_hosts[b].copy_(obuf[b][0], non_blocking=True)
                h_hosts[b].copy_(obuf[b][1], non_blocking=True)
                ev_out[b].record(s_out)
            started[b] = True

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        for i in range(args.e2e_steps):
            e2e_step(i)
        b_ev.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b_ev) / args.e2e_steps, dev)
        e2e = {"value": whole_job_rate(tokens_per_rank, e2e_ms, world), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "pipeline": "double-buffered; copies in, forward pass and copies out on "
                           "three streams"}

    # ---- roofline ----
    peaks, peak_src = load_peaks()
    dominant = "scan" if scan_ms >= prep_ms else "prep"
    kern_ms = scan_ms if dominant == "scan" else prep_ms
    kbytes = algorithmic_bytes(wl, dominant)
    achieved = kbytes / (kern_ms / 1e3) / 1e9
    traffic, traffic_note = measured_traffic(c0.name, dominant, c0.tokens)
    kernel_names = {  # kernels gdn_chunk_fwd launches for this workload
        ("prep", "bf16", 0): "gdn_prep_tmem_kernel", ("scan", "bf16", 0): "gdn_scan_la_kernel",
        ("prep", "bf16", 1): "gdn_prep_tc_kernel", ("scan", "bf16", 1): "gdn_scan_tc_kernel",
        ("prep", "f32", 0): "gdn_prep_kernel", ("scan", "f32", 0): "gdn_scan_kernel",
        ("prep", "f32", 1): "gdn_prep_kernel", ("scan", "f32", 1): "gdn_scan_kernel"}
    kname = kernel_names[(dominant, wl.dtype_name, c0.gate_mode)]
    if kname == "gdn_prep_tc_kernel" and c0.chunk == 32:
        kname = "gdn_prep_kda_kernel"  # the per-key-gate prep at chunk 32
    roofline = {"bound": "hbm", "kernel": kname,
                "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": traffic, "algorithmic_bytes": kbytes, "kernel_ms": kern_ms,
                "peak_source": f"hbm_gbs of {peak_src}"}
    if traffic_note:
        roofline["traffic_note"] = traffic_note
    roofline["frac_note"] = ("achieved charges the whole path's algorithmic bytes (q, k, v, o, "
                             "g, beta read or written once) to this one kernel's launch time")
    own = kernel_design_bytes(wl, dominant, c0, x["cu_seqlens"])
    if own is not None:
        roofline["kernel_own"] = {
            "bytes": own, "achieved": own / (kern_ms / 1e3) / 1e9,
            "frac": own / (kern_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "note": "bytes this kernel must move in the split design: " + KERNEL_BYTES_NOTE[
                (dominant, wl.dtype_name, c0.gate_mode)]}
    path_bytes = algorithmic_bytes(wl, "path")
    path_flops = algorithmic_flops(wl)
    t_hbm = path_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = path_flops / (peaks["bf16_tflops_sustained"] * 1e12)
    t_tc_burst = path_flops / (peaks["bf16_tflops"] * 1e12)
    path = {"bytes": path_bytes, "flops": path_flops, "t_hbm_us": t_hbm * 1e6,
            "t_tensor_us": t_tc * 1e6, "t_tensor_burst_us": t_tc_burst * 1e6,
            "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "frac": max(t_hbm, t_tc) / (ms_step / 1e3 / world) if ms_step > 0 else None,
            "frac_burst": max(t_hbm, t_tc_burst) / (ms_step / 1e3 / world) if ms_step > 0 else None,
            "frac_single_call": max(t_hbm, t_tc) / (single_ms / 1e3) if single_ms > 0 else None,
            "note": f"whole path vs max(HBM, tensor) roofline of {peak_src} peaks; frac uses the "
                    "sustained bf16 peak (a kernel timed inside a long loop), frac_burst the "
                    "burst peak"}

    # ---- CPU baseline (oracle) on rank 0 at N = 1 ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n_tok = calibrate_oracle(wl, x, args.cpu_seconds)
        sec, n = oracle_sample(wl, x, n_tok)
        cpu = {"value": n / sec, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{oracle_sample_text(c0, x, n)}, {sec:.1f} s"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype_name,
            "data": "synthetic (seeded; no dataset)",
            "config": dict(config, l2="inputs 1 GB+ and workspace exceed the 129 MB L2; no flush",
                           parallelism=f"replicas x{world}",
                           in_flight=f"{nf} independent batches on {nf} streams (own workspace "
                                     "and outputs each); every step is one whole forward pass",
                           kernels_ms="from a separate pass, one step after another"),
            "roofline": roofline, "path_roofline": path, "cpu_baseline": cpu, "e2e": e2e,
            "lockstep": ({"unavailable": lock_refused} if lock_refused else None) if lock_ms is None else {
                "value": whole_job_rate(tokens_per_rank, lock_ms, world), "unit": UNIT,
                "ms_per_step": lock_ms,
                "note": "gdn_chunk_fwd_lockstep (a prep launch over the first chunks as a head "
                        "start, then prep and scan in one cooperative launch), one call after "
                        "another"},
            "single_call": {"value": whole_job_rate(tokens_per_rank, single_ms, world),
                            "unit": UNIT, "ms_per_step": single_ms,
                            "note": "one gdn_chunk_fwd after another on one stream, no batches "
                                    "in flight"},
            "clocks": clocks, "gpu_launches": 2 * K,
            "kernels_ms": {"prep": prep_ms, "scan": scan_ms}, "device_flags": flags}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def decode_bytes(c):
    """HBM bytes one decode step must move: every state read and written once,
    plus q, k, v, g, beta read and o written."""
    es = 2 if str(c.dtype).endswith("bfloat16") else 4
    n = c.B
    state = n * c.HV * c.dk * c.dv * 4
    qk = 2 * n * c.H * c.dk * es
    vo = 2 * n * c.HV * c.dv * es
    gb = n * c.HV * ((1 if c.gate_mode == 0 else c.dk) + 1) * 4
    return 2 * state + qk + vo + gb


def bench_decode(args, rank, world, local_rank, c0, wl, config):
    """One decode step (T = 1) of a batch of sequences through the token-serial
    kernel, the states updated in place on the device as a serving loop keeps
    them.  Tokens/s = sequences per step / step time."""
    import torch
    import torch.distributed as dist

    from chunkwise_gated_delta_gdn_gb300 import build as cuda_build
    from chunkwise_gated_delta_gdn_gb300 import gdn, synth

    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    gdn.load(cuda_build.build())
    x = synth.make_inputs(c0)
    names = ("q", "k", "v", "g", "beta")
    d = {n: x[n].to(dev) for n in names}
    state = x["h0"].to(dev)
    o = torch.empty((c0.B, 1, c0.HV, c0.dv), dtype=c0.dtype, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(dd, ob):
        gdn.gdn_recurrent_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], state, hT=state,
                              o=ob, scale=c0.scale)

    gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], state, hT=state, o=o,
                          scale=c0.scale, flags=flags)
    dev_flags = gdn.gdn_read_device_flags(flags)
    for _ in range(args.warmup):
        step(d, o)
    torch.cuda.synchronize()
    K = args.steps
    main = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.25)
    a.record(main)
    for _ in range(K):
        step(d, o)
    b.record(main)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_step = max_over_ranks(a.elapsed_time(b) / K, dev)
    value = whole_job_rate(c0.B, ms_step, world)

    # end to end: each step's token inputs copied in from pinned host memory
    # and its outputs o copied back; the states stay resident on the device.
    # Steps are pipelined like a serving loop: double-buffered token inputs and
    # outputs, copies in on one stream, the step on a second, copies out on a
    # third, ordered by events (the steps themselves stay in order: each
    # updates the states the next one reads).
    e2e = None
    if not args.no_e2e:
        host = {n: x[n].pin_memory() for n in names}
        o_hosts = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = o.numel() * o.element_size()
        dbuf = [d, {n: torch.empty_like(d[n]) for n in names}]
        obuf = [o, torch.empty_like(o)]
        s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_run = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        started = [False, False]

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if started[b]:
                    s_in.wait_event(ev_run[b])  # step i-2 is done reading buffer b
                for n in names:
                    dbuf[b][n].copy_(host[n], non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev_in[b])
                if started[b]:
                    s_run.wait_event(ev_out[b])  # step i-2's o has left buffer b
                db = dbuf[b]
                gdn.gdn_recurrent_fwd(db["q"], db["k"], db["v"], db["g"], db["beta"], state,
                                      hT=state, o=obuf[b], scale=c0.scale, stream=s_run)
                ev_run[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[b])
                o_hosts[b].copy_(obuf[b], non_blocking=True)
                ev_out[b].record(s_out)
            started[b] = True

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        rank_barrier()
        a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a2.record(s_in)
        for i in range(args.e2e_steps):
            e2e_step(i)
        b2.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a2.elapsed_time(b2) / args.e2e_steps, dev)
        e2e = {"value": whole_job_rate(c0.B, e2e_ms, world), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "note": "token inputs in and o out every step, double-buffered on their own "
                       "streams; the states stay resident on the device"}

    peaks, peak_src = load_peaks()
    kbytes = decode_bytes(c0)
    achieved = kbytes / (ms_step / 1e3) / 1e9
    traffic, traffic_note = measured_traffic(c0.name, "recurrent", c0.B)
    roofline = {"bound": "hbm", "kernel": "gdn_recurrent_kernel", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": traffic, "algorithmic_bytes": kbytes, "kernel_ms": ms_step,
                "peak_source": f"hbm_gbs of {peak_src}"}
    if traffic_note:
        roofline["traffic_note"] = traffic_note

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t0, n_done = time.perf_counter(), 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 10.0) or n_done == 0:
            _, n = oracle_sample(wl, x, 1)
            n_done += n
        sec = time.perf_counter() - t0
        cpu = {"value": n_done / sec, "unit": UNIT, "cores": oracle.num_threads(),
               "kind": "oracle",
               "sample": f"fp64 token-serial oracle, {n_done // c0.B} whole decode steps of "
                         f"{c0.name} ({c0.B} sequences x {c0.HV} value heads), {sec:.1f} s"}

    line = {"metric": METRIC_DECODE,
            "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype_name, "data": "synthetic (seeded; no dataset)",
            "config": dict(config, l2="states exceed the 129 MB L2; no flush",
                           parallelism=f"replicas x{world}",
                           state="updated in place (hT = h0), resident on the device"),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": K, "device_flags": dev_flags}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_prepost(args, rank, world, local_rank, c0, wl, config):
    """One pass of the operations either side of the recurrence over the
    workload's tokens: causal convolution (width 4, SiLU, with history) of the
    q, k and v channels, L2 norm of q and k, gated RMS norm of o.  Each is
    memory-bound; the roofline is HBM for every kernel."""
    import torch
    import torch.distributed as dist

    from chunkwise_gated_delta_gdn_gb300 import build as cuda_build
    from chunkwise_gated_delta_gdn_gb300 import gdn, synth

    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    gdn.load(cuda_build.build())
    xin = synth.make_prepost_inputs(c0)
    d = {k: v.to(dev) for k, v in xin.items()}
    B, T, D = d["x"].shape
    W = d["w"].shape[1]
    y = torch.empty_like(d["x"])
    hT = torch.empty_like(d["h0"])
    qdim = c0.H * c0.dk
    on = torch.empty_like(d["o"])
    es = 2
    n_tok = B * T
    kbytes = {"conv": 2 * n_tok * D * es, "l2norm_qk": 2 * 2 * n_tok * qdim * es,
              "rmsnorm_gated": 3 * n_tok * c0.HV * c0.dv * es}

    def conv():
        gdn.gdn_causal_conv1d_fwd(d["x"], d["w"], d["bias"], d["h0"], y=y, hT=hT,
                                  activation=gdn.GDN_ACT_SILU)

    # q and k rows (as the recurrence takes them: contiguous [B, T, H, dk] each),
    # normalised in place
    qk = torch.empty((2, B, T, c0.H, c0.dk), dtype=c0.dtype, device=dev)
    qk.copy_(d["x"][..., :2 * qdim].reshape(B, T, 2, c0.H, c0.dk).permute(2, 0, 1, 3, 4))

    def l2_packed():
        gdn.gdn_l2norm_fwd(qk, eps=1e-6, y=qk)

    def norm():
        gdn.gdn_rmsnorm_gated_fwd(d["o"], d["norm_weight"], d["z"], eps=1e-6, y=on)

    kern = {"conv": conv, "l2norm_qk": l2_packed, "rmsnorm_gated": norm}
    for _ in range(args.warmup):
        for f in kern.values():
            f()
    torch.cuda.synchronize()
    rank_barrier()
    K = args.steps
    ev = {n: [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)] for n in kern}
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.25)
    main = torch.cuda.current_stream(dev)
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(main)
    for i in range(K):
        for n, f in kern.items():
            ev[n][2 * i].record(main)
            f()
            ev[n][2 * i + 1].record(main)
    b_ev.record(main)
    torch.cuda.synchronize()
    rank_barrier()
    clocks = sampler.stop()
    ms_step = max_over_ranks(a_ev.elapsed_time(b_ev) / K, dev)
    kms = {n: sum(ev[n][2 * i].elapsed_time(ev[n][2 * i + 1]) for i in range(K)) / K for n in kern}
    peaks, peak_src = load_peaks()
    per_kernel = {n: {"ms": kms[n], "algorithmic_bytes": kbytes[n],
                      "achieved_gbs": kbytes[n] / (kms[n] / 1e3) / 1e9,
                      "frac": kbytes[n] / (kms[n] / 1e3) / 1e9 / peaks["hbm_gbs"]} for n in kern}
    dom = max(kms, key=kms.get)
    roofline = {"bound": "hbm", "kernel": {"conv": "gdn_conv1d_kernel",
                                           "l2norm_qk": "gdn_rownorm_kernel (L2)",
                                           "rmsnorm_gated": "gdn_rownorm_kernel (gated RMS)"}[dom],
                "achieved": per_kernel[dom]["achieved_gbs"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": per_kernel[dom]["frac"],
                "traffic": measured_traffic(c0.name, dom, n_tok)[0],
                "algorithmic_bytes": kbytes[dom], "kernel_ms": kms[dom],
                "peak_source": f"hbm_gbs of {peak_src}"}
    value = whole_job_rate(n_tok, ms_step, world)

    # end to end: each step copies x, o and z in from pinned host memory and the
    # convolution output and the normed o back out.  Steps are pipelined like
    # a serving loop: double-buffered device inputs and outputs, copies in on
    # one stream, the three operations on a second, copies out on a third,
    # ordered by events.
    e2e = None
    if not args.no_e2e:
        hx, ho, hz = (xin[n].pin_memory() for n in ("x", "o", "z"))
        hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
        hon = [torch.empty(on.shape, dtype=on.dtype).pin_memory() for _ in range(2)]
        dx, dob, dz = [d["x"], torch.empty_like(d["x"])], [d["o"], torch.empty_like(d["o"])], \
            [d["z"], torch.empty_like(d["z"])]
        dy, dh, don = [y, torch.empty_like(y)], [hT, torch.empty_like(hT)], [on, torch.empty_like(on)]
        s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        ev_in, ev_run, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
        started = [False, False]

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if started[b]:
                    s_in.wait_event(ev_run[b])  # step i-2 is done reading buffer b
                dx[b].copy_(hx, non_blocking=True)
                dob[b].copy_(ho, non_blocking=True)
                dz[b].copy_(hz, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev_in[b])
                if started[b]:
                    s_run.wait_event(ev_out[b])  # step i-2's results have left buffer b
                gdn.gdn_causal_conv1d_fwd(dx[b], d["w"], d["bias"], d["h0"], y=dy[b], hT=dh[b],
                                          activation=gdn.GDN_ACT_SILU, stream=s_run)
                gdn.gdn_l2norm_fwd(qk, eps=1e-6, y=qk, stream=s_run)
                gdn.gdn_rmsnorm_gated_fwd(dob[b], d["norm_weight"], dz[b], eps=1e-6, y=don[b],
                                          stream=s_run)
                ev_run[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[b])
                hy[b].copy_(dy[b], non_blocking=True)
                hon[b].copy_(don[b], non_blocking=True)
                ev_out[b].record(s_out)
            started[b] = True

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        rank_barrier()
        a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e = max(4, min(args.e2e_steps, 10))
        a2.record(s_in)
        for i in range(n_e):
            e2e_step(i)
        b2.record(s_out)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a2.elapsed_time(b2) / n_e, dev)
        h2d = sum(t.numel() * t.element_size() for t in (hx, ho, hz))
        d2h = sum(t.numel() * t.element_size() for t in (hy[0], hon[0]))
        e2e = {"value": whole_job_rate(n_tok, e_ms, world), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms, "steps": n_e,
               "note": "x, o and z copied in, the convolution output and the normed o copied "
                       "out, every step; double-buffered, copies in, the operations and copies "
                       "out on three streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # noqa: F401  (the package; the pre/post oracle is numpy)
        from oracle import prepost
        n_s = 512
        t0 = time.perf_counter()
        prepost.causal_conv1d(xin["x"][0, :n_s], xin["w"], xin["bias"], xin["h0"][:1], [0, n_s], 1)
        prepost.l2norm(xin["x"][0, :n_s, :2 * qdim].reshape(n_s, 2 * c0.H, c0.dk), 1e-6)
        prepost.rmsnorm_gated(xin["o"][0, :n_s], xin["norm_weight"], xin["z"][0, :n_s], 1e-6)
        sec = time.perf_counter() - t0
        cpu = {"value": n_s / sec, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"fp64 numpy oracle of the three operations on the first {n_s} tokens "
                         f"of {c0.name}, {sec:.2f} s"}

    line = {"metric": METRIC_PREPOST,
            "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; no dataset)",
            "config": dict(config, conv_channels=D, conv_width=W, activation="silu",
                           l2="inputs exceed the 129 MB L2; no flush",
                           parallelism=f"replicas x{world}"),
            "roofline": roofline, "kernels": per_kernel, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "gpu_launches": K * 4}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args, rank, world, c0, wl, config):
    """The oracle as it stands, timed on the host cores (the reference arm)."""
    if rank != 0:
        return
    import oracle
    from chunkwise_gated_delta_gdn_gb300 import synth

    total = args.steps + args.warmup
    per_step_s = min(10.0, 150.0 / max(total, 1))
    if c0.name.startswith("prepost"):
        # the pre/post operations' numpy oracle on a prefix of the tokens
        from oracle import prepost
        xin = synth.make_prepost_inputs(c0)
        qdim = c0.H * c0.dk

        def sample(n_s):
            t0 = time.perf_counter()
            prepost.causal_conv1d(xin["x"][0, :n_s], xin["w"], xin["bias"], xin["h0"][:1],
                                  [0, n_s], prepost.ACT_SILU)
            prepost.l2norm(xin["x"][0, :n_s, :2 * qdim].reshape(n_s, 2 * c0.H, c0.dk), 1e-6)
            prepost.rmsnorm_gated(xin["o"][0, :n_s], xin["norm_weight"], xin["z"][0, :n_s], 1e-6)
            return time.perf_counter() - t0, n_s

        sec, n_s = sample(64)
        n_tok = int(min(c0.T, max(64, per_step_s / max(sec / n_s, 1e-9))))
        describe = lambda n: (f"the numpy fp64 oracle of the three operations on the first "
                              f"{n} tokens of {c0.name}")
        cores = 1
    else:
        x = synth.make_inputs(c0)
        n_tok = calibrate_oracle(wl, x, per_step_s)

        def sample(n_s):
            return oracle_sample(wl, x, n_s)

        describe = lambda n: oracle_sample_text(c0, x, n)
        cores = oracle.num_threads()
    for _ in range(args.warmup):
        sample(n_tok)
    times, n = [], 0
    for _ in range(args.steps):
        sec, n = sample(n_tok)
        times.append(sec)
    ms_step = 1e3 * sum(times) / len(times)
    value = n / (ms_step / 1e3)
    line = {"impl": "reference", "metric": metric_of(c0), "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; no dataset)",
            "config": config,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: {describe(n)}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
