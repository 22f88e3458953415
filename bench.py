"""Benchmark: attention TFLOP/s (forward + backward) on one GB300.

One step = the whole hot path over one batch: fa_forward (tile schedule,
TMA loads, S = QK^T, mask, online softmax, O += PV, epilogue) then the
backward (preprocess, recompute kernel, dQ conversion), all through the C
ABI.  Default workload: the largest single-GPU shape of the long-sequence
sweep, B=1 H=16 N=16384 d=128, non-causal (the long-range workload's shape
without its causal mask), bf16 inputs drawn N(0,1) from a seeded generator
with 1% of the keys scaled by 8.  --workload bert_large times the
BERT-large-shaped step (B=8 H=16 N=512 d=64).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed

L2 is flushed (a 256 MiB device write) before every timed step, outside the
per-step CUDA events; the default workload's inputs (268 MB) are also larger
than L2, the BERT-shaped ones (34 MB) are not.  Under torchrun every rank runs its own replica (weak
scaling); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "longseq_dense_n16384_d128"
METRIC = "attention TFLOP/s fwd and fwd+bwd (bf16, 1×GB300) and % of dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def kernel_source_hash(files):
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, "io_aware_exact_15_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def workload_of(args):
    """The named workload; --sparse-density replaces the random-tile density
    of a block-sparse one (the sparsity-scaling runs)."""
    import dataclasses

    import fa_workloads as W
    w = W.WORKLOADS[args.workload]
    dens = getattr(args, "sparse_density", None)
    if dens is not None:
        if w.sparse_density is None:
            raise SystemExit("--sparse-density applies to block-sparse workloads")
        w = dataclasses.replace(w, sparse_density=float(dens),
                                note=f"{w.note}; random-tile density {dens}")
    return w


def bwd_compulsory_bytes(rows_q, rows_kv, d, deterministic=False):
    """Bytes the backward main kernel must move at least once: Q, dO (bf16)
    and lse, D (fp32) per query row; K, V read and dK, dV written (bf16) per
    key/value row; the fp32 dQ accumulator read and written once per query
    row (the deterministic pass writes bf16 dQ instead)."""
    per_q = 2 * d * 2 + 2 * 4 + (2 * d if deterministic else 2 * 4 * d)
    per_kv = 2 * d * 2 + 2 * d * 2
    return int(rows_q * per_q + rows_kv * per_kv)


def max_over_ranks(x, dist, device):
    """The largest x over all ranks (x itself on one rank): the job's time is
    that of its slowest rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_rank_step, ms_per_step):
    """Whole-job throughput: every rank runs its own replica of the step
    (weak scaling), all of them within the slowest rank's step time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def ncu_traffic(kernel_key, src_hash):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != src_hash:
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loop runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=100):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world, dist):
    import numpy as np
    import torch

    import fa_workloads as W
    import io_aware_exact_15_gb300 as fa

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    w = workload_of(args)
    B, H, N, d = w.B, w.H, w.N, w.d
    Hkv = w.kv_heads
    varlen = w.varlen
    gqa = Hkv != H
    drop = (w.dropout, W.DROPOUT_SEED, 0)
    det = bool(getattr(args, "deterministic", False))
    if det and (varlen or gqa or w.dropout > 0 or w.sparse_density is not None):
        raise SystemExit("--deterministic applies to dense or causal equal-length workloads")
    combined = varlen or gqa or w.dropout > 0 or det  # no split backward entry point
    if varlen:
        q, k, v, do, cu = W.make_varlen_inputs(w, with_do=True)
        mask = None
        T = int(cu[-1])
        max_seqlen = int(np.max(np.diff(cu)))
        lse_shape = (H, T)
        rows_b, rows_n = 1, T  # the packed batch as one (1, H, T) row problem
    else:
        q, k, v, do, mask = W.make_inputs(w, with_do=True)
        cu = None
        lse_shape = (B, H, N)
        rows_b, rows_n = B, N
    stream = torch.cuda.Stream(device=dev)
    K = args.steps
    s_ptr = stream.cuda_stream
    sparse = mask is not None
    mh = mask.shape[0] if sparse else 1
    with torch.cuda.stream(stream):
        qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
        md = torch.from_numpy(np.ascontiguousarray(mask)).to(dev) if sparse else None
        cud = torch.from_numpy(cu).to(dev) if varlen else None
        o = torch.empty_like(qd)
        lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
        dq = torch.empty_like(qd)
        dk, dv = torch.empty_like(kd), torch.empty_like(vd)
        nbytes = (fa.fa_blocksparse_workspace_size(B, H, N, d, mh) if sparse
                  else fa.fa_backward_workspace_size(rows_b, H, rows_n, d))
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    lists_bytes = nbytes - fa.fa_backward_workspace_size(B, H, N, d) if sparse else 0

    def check(st, what):
        if st != fa.FA_OK:
            raise RuntimeError(f"{what}: {fa.fa_status_string(st)}")

    bws = ws[lists_bytes:] if sparse else ws
    bwb = nbytes - lists_bytes

    # device buffers of one step (the double-buffered e2e loop uses two sets)
    # One allocation per direction: a step's inputs (q, k, v, dO and the mask
    # or sequence offsets) and its outputs (o, lse, dq, dk, dv) are views into
    # a single buffer, 256-byte aligned, so each moves in one copy.
    in_specs = [(tuple(t.shape), t.dtype) for t in (qd, kd, vd, dod)]
    if md is not None:
        in_specs.append((tuple(md.shape), md.dtype))
    if cud is not None:
        in_specs.append((tuple(cud.shape), cud.dtype))
    out_specs = [(tuple(t.shape), t.dtype) for t in (o, lse, dq, dk, dv)]

    def packed(specs, device=None, pin=False):
        sizes = [int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
                 for shape, dt in specs]
        offs, total = [], 0
        for n in sizes:
            offs.append(total)
            total += (n + 255) // 256 * 256
        buf = torch.empty(total, dtype=torch.uint8, device=device)
        if pin:
            buf = buf.pin_memory()
        views = [buf[a:a + n].view(dt).view(shape)
                 for (shape, dt), a, n in zip(specs, offs, sizes)]
        return buf, views

    def buffer_set():
        with torch.cuda.stream(stream):
            din, iv = packed(in_specs, device=dev)
            dout, ov = packed(out_specs, device=dev)
        bs = types.SimpleNamespace(din=din, dout=dout, qd=iv[0], kd=iv[1], vd=iv[2], dod=iv[3],
                                   md=None, cud=None, o=ov[0], lse=ov[1], dq=ov[2], dk=ov[3],
                                   dv=ov[4])
        rest = iv[4:]
        if md is not None:
            bs.md = rest.pop(0)
        if cud is not None:
            bs.cud = rest.pop(0)
        return bs

    b0 = types.SimpleNamespace(qd=qd, kd=kd, vd=vd, dod=dod, md=md, cud=cud, o=o, lse=lse,
                               dq=dq, dk=dk, dv=dv)

    def forward(bs):
        if varlen:
            check(fa.fa_forward_varlen(bs.qd, bs.kd, bs.vd, bs.o, bs.lse, bs.cud, B, max_seqlen, T, H, Hkv, d,
                                       w.scale, w.causal, *drop, s_ptr), "forward")
        elif w.dropout > 0:
            check(fa.fa_forward_dropout(bs.qd, bs.kd, bs.vd, bs.o, bs.lse, B, H, N, d, w.scale, w.causal, *drop,
                                        s_ptr), "forward")
        elif gqa:
            check(fa.fa_forward_gqa(bs.qd, bs.kd, bs.vd, bs.o, bs.lse, B, H, Hkv, N, d, w.scale, w.causal,
                                    s_ptr), "forward")
        else:
            check(fa.fa_forward(bs.qd, bs.kd, bs.vd, bs.o, bs.lse, B, H, N, d, w.scale, w.causal, s_ptr),
                  "forward")

    def backward_whole(bs):
        if det:
            check(fa.fa_backward_deterministic(bs.qd, bs.kd, bs.vd, bs.o, bs.dod, bs.lse, bs.dq, bs.dk, bs.dv, B, H, N, d,
                                               w.scale, w.causal, ws, nbytes, s_ptr), "backward")
        elif varlen:
            check(fa.fa_backward_varlen(bs.qd, bs.kd, bs.vd, bs.o, bs.dod, bs.lse, bs.dq, bs.dk, bs.dv, bs.cud, B, max_seqlen,
                                        T, H, Hkv, d, w.scale, w.causal, *drop, ws, nbytes,
                                        s_ptr), "backward")
        elif w.dropout > 0:
            check(fa.fa_backward_dropout(bs.qd, bs.kd, bs.vd, bs.o, bs.dod, bs.lse, bs.dq, bs.dk, bs.dv, B, H, N, d, w.scale,
                                         w.causal, *drop, ws, nbytes, s_ptr), "backward")
        else:
            check(fa.fa_backward_gqa(bs.qd, bs.kd, bs.vd, bs.o, bs.dod, bs.lse, bs.dq, bs.dk, bs.dv, B, H, Hkv, N, d,
                                     w.scale, w.causal, ws, nbytes, s_ptr), "backward")

    # One step; `ev` (5 events) splits it into its kernels.  Grouped-head and
    # variable-length batches have no split backward entry point: the split
    # step then brackets their whole backward and times the row-wise
    # preprocess and dQ conversion beside it (the main kernel's time is the
    # difference); the unsplit step is exactly forward + backward.
    def step(ev=None, bs=None):
        bs = bs or b0
        rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        if sparse:
            check(fa.fa_blocksparse_forward(bs.qd, bs.kd, bs.vd, bs.o, bs.lse, B, H, N, d, w.scale, w.causal, bs.md,
                                            mh, ws, nbytes, s_ptr), "forward")
            rec(1)
            rec(2)
            check(fa.fa_blocksparse_backward(bs.qd, bs.kd, bs.vd, bs.o, bs.dod, bs.lse, bs.dq, bs.dk, bs.dv, B, H, N, d,
                                             w.scale, w.causal, bs.md, mh, ws, nbytes, s_ptr),
                  "backward")
            rec(3)
            rec(4)
            return
        forward(bs)
        rec(1)
        if combined:
            if ev:
                check(fa.fa_backward_preprocess(bs.o, bs.dod, rows_b, H, rows_n, d, bws, bwb, s_ptr),
                      "preprocess")
            rec(2)
            backward_whole(bs)
            rec(3)
            if ev and not det:  # the deterministic backward has no conversion pass
                check(fa.fa_backward_dq_convert(bs.dq, rows_b, H, rows_n, d, w.scale, bws, bwb,
                                                s_ptr), "convert")
            rec(4)
            return
        check(fa.fa_backward_preprocess(bs.o, bs.dod, B, H, N, d, bws, bwb, s_ptr), "preprocess")
        rec(2)
        check(fa.fa_backward_main(bs.qd, bs.kd, bs.vd, bs.dod, bs.lse, bs.dk, bs.dv, B, H, N, d, w.scale, w.causal,
                                  bws, bwb, s_ptr), "backward")
        rec(3)
        check(fa.fa_backward_dq_convert(bs.dq, B, H, N, d, w.scale, bws, bwb, s_ptr), "convert")
        rec(4)

    launches_per_step = (2 + 4) if sparse else 4
    ff = W.fwd_flops(w, mask)
    fb = W.fwd_bwd_flops(w, mask)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = fa.fa_get_device_status(s_ptr)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after warm-up: {fa.fa_status_string(st)}")

    def timed_loop(K, split):
        """K steps, each after an L2 flush; returns per-step event lists."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5 if split else 2)]
               for _ in range(K)]
        with torch.cuda.stream(stream):
            torch.cuda._sleep(40_000_000)  # head start so launches queue ahead of the GPU
        for i in range(K):
            with torch.cuda.stream(stream):
                flush.fill_(i & 0xFF)
            if split:
                step(evs[i])
            else:
                evs[i][0].record(stream)
                step()
                evs[i][1].record(stream)
        return evs

    K = args.steps
    clocks = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    evs = timed_loop(K, split=False)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms = statistics.fmean(step_ms)
    # per-kernel split on a shorter loop of the same steps
    Ks = max(10, min(K, 300))
    sev = timed_loop(Ks, split=True)
    torch.cuda.synchronize(dev)
    st = fa.fa_get_device_status(s_ptr)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after timing: {fa.fa_status_string(st)}")
    per = [[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in sev]
    fwd_ms = statistics.fmean(p[0] for p in per)
    pre_ms = statistics.fmean(p[1] for p in per)
    main_ms = statistics.fmean(p[2] for p in per)
    conv_ms = statistics.fmean(p[3] for p in per)
    if combined:  # p[2] bracketed preprocess + main (+ dQ pass or convert)
        main_ms = main_ms - pre_ms - (0.0 if det else conv_ms)
    ms_max = max_over_ranks(ms, dist, dev)
    value = whole_job_tflops(world, fb, ms_max)

    # end to end through the public API with host buffers (pinned)
    hin, hiv = packed(in_specs, pin=True)
    hout, _ = packed(out_specs, pin=True)
    host_inputs = [q, k, v, do]
    if sparse:
        host_inputs.append(torch.from_numpy(np.ascontiguousarray(mask)))
    if varlen:
        host_inputs.append(torch.from_numpy(cu))
    for dst, src in zip(hiv, host_inputs):
        dst.copy_(src)
    h2d = hin.numel()   # bytes copied per step (payload plus <= 255 B alignment per tensor)
    d2h = hout.numel()

    # Streamed batches: step i's inputs go up on `cin`, its forward + backward
    # run on the compute stream, its outputs come down on `cout`; two buffer
    # sets let the copies of steps i+1 and i-1 overlap the compute of step i.
    # Every step's host -> device and device -> host copies are inside the
    # timed region.
    sets = [buffer_set(), buffer_set()]
    cin = torch.cuda.Stream(device=dev)
    cout = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of set s loaded
    ev_done = [torch.cuda.Event() for _ in range(2)]    # compute on set s finished
    ev_out = [torch.cuda.Event() for _ in range(2)]     # outputs of set s copied out
    used = [False, False]

    def e2e_step(i):
        sidx = i & 1
        bs = sets[sidx]
        with torch.cuda.stream(cin):
            if used[sidx]:
                cin.wait_event(ev_done[sidx])  # the set's previous inputs are consumed
            bs.din.copy_(hin, non_blocking=True)
            ev_in[sidx].record(cin)
        stream.wait_event(ev_in[sidx])
        if used[sidx]:
            stream.wait_event(ev_out[sidx])  # the set's previous outputs are copied out
        step(bs=bs)
        ev_done[sidx].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_done[sidx])
            hout.copy_(bs.dout, non_blocking=True)
            ev_out[sidx].record(cout)
        used[sidx] = True

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    Ke = max(3, min(K, 200))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cin)
    for i in range(Ke):
        e2e_step(i)
    b.record(cout)
    torch.cuda.synchronize(dev)
    ems = a.elapsed_time(b) / Ke
    # the same steps one after another on one stream, for comparison
    def serial_step():
        bs = sets[0]
        with torch.cuda.stream(stream):
            bs.din.copy_(hin, non_blocking=True)
        step(bs=bs)
        with torch.cuda.stream(stream):
            hout.copy_(bs.dout, non_blocking=True)
    serial_step()
    torch.cuda.synchronize(dev)
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a2.record(stream)
    for _ in range(Ke):
        serial_step()
    b2.record(stream)
    torch.cuda.synchronize(dev)
    ems_serial = a2.elapsed_time(b2) / Ke
    ems = max_over_ranks(ems, dist, dev)
    e2e = {"value": round(whole_job_tflops(world, fb, ems), 3), "unit": "TFLOP/s",
           "ms_per_step": round(ems, 4), "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h),
           "path": "per step: one pinned host -> device copy of the packed inputs (q, k, v, dO), "
                   "forward + backward via the C ABI, one device -> host copy of the packed "
                   "outputs (o, lse, dq, dk, dv); streamed with two device buffer sets so the "
                   "copies of neighbouring steps overlap compute",
           "serial_ms_per_step": round(ems_serial, 4)}

    src_hash = kernel_source_hash(["fa_bwd.cu", "fa_ptx.cuh", "fa_sched.cuh"])
    main_flops = 2.5 * ff
    achieved = main_flops / (main_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    traffic = ncu_traffic(f"fa_bwd_kernel:{args.workload}", src_hash)
    rows_q = H * T if varlen else B * H * N
    rows_kv = Hkv * T if varlen else B * Hkv * N
    comp = bwd_compulsory_bytes(rows_q, rows_kv, d, det)
    kname = ("fa_bwd_kernel without dQ + fa_bwd_dq_kernel (deterministic backward; algorithmic "
             "FLOPs count the five products once)" if det else
             "fa_bwd_kernel (recompute: S, dP, dV, dK, dQ MMAs)")
    roofline = {"kernel": kname, "bound": "tensor",
                "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "peak_source": f"{peaks['source']} bf16 burst",
                "traffic": traffic,
                "hbm": {"compulsory_bytes": comp,
                        "compulsory_gbs": round(comp / (main_ms * 1e-3) / 1e9, 1),
                        "traffic_gbs": (round(traffic / (main_ms * 1e-3) / 1e9, 1)
                                        if traffic else None),
                        "peak_gbs": peaks["hbm_gbs"],
                        "what": "inputs read once and outputs written once (Q, K, V, dO, lse, "
                                "D, dK, dV; the fp32 dQ accumulator read and written once), "
                                "and the ncu DRAM bytes, per launch over avg_launch_ms"},
                "main_time": ("deterministic backward minus the separately timed preprocess: "
                              "key-tile pass + query-tile dQ pass together" if det else
                              "combined backward minus separately timed preprocess and convert"
                              if combined else "CUDA events around the kernel's launch"),
                "algorithmic_flops_per_launch": main_flops,
                "avg_launch_ms": round(main_ms, 5),
                "timing_note": "per-kernel events sit between launches and stop programmatic "
                               "dependent launch from overlapping a kernel with its neighbours: "
                               "avg_launch_ms is an upper bound on the kernel's time inside "
                               "the unsplit step, so frac is a lower bound"}
    fwd_tf = ff / (fwd_ms * 1e-3) / 1e12
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": f"{w.name}: {w.note}", "B": B, "H": H, "N": N, "d": d,
                   "causal": w.causal, "sparse": sparse, "Hkv": Hkv, "dropout": w.dropout,
                   "deterministic_backward": det,
                   **({"total_tokens": T, "max_seqlen": max_seqlen,
                       "seq_lens": [int(x) for x in np.diff(cu)]} if varlen else {}),
                   **({"sparse_density": w.sparse_density,
                       "kept_tiles": int(np.count_nonzero(mask)),
                       "tiles": int(mask.size)} if sparse else {}),
                   "l2": "flushed before every timed step (256 MiB device write, outside events)",
                   "parallelism": f"replicas x{world} (independent heads per GPU)"},
        "fwd": {"ms": round(fwd_ms, 5), "tflops": round(fwd_tf, 2),
                "frac_of_peak": round(fwd_tf / peak, 4)},
        "fwd_bwd": {"ms": round(ms, 5), "tflops": round(fb / (ms * 1e-3) / 1e12, 2),
                    "frac_of_peak": round(fb / (ms * 1e-3) / 1e12 / peak, 4)},
        "kernels_ms": {"fa_fwd_kernel": round(fwd_ms, 5), "fa_bwd_pre_kernel": round(pre_ms, 5),
                       "fa_bwd_kernel": round(main_ms, 5),
                       "fa_dq_convert_kernel": round(conv_ms, 5)},
        "roofline": roofline, "e2e": e2e, "gpu_launches": launches_per_step * K,
        "split_steps": Ks,
        "clocks": clk, "wall_s_timed": round(wall, 3),
        "peaks": {k_: peaks[k_] for k_ in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")},
    }
    return result


# ---------------------------------------------------------------------------- CPU oracle
def oracle_job(w):
    """(sample(n), units, flops_per_unit): sample(n) runs the fp64 oracle
    forward + backward on the first n units of the workload: (batch, head)
    slices, or heads of a packed variable-length batch.  Grouped heads are
    sampled per query head with its key/value head."""
    import numpy as np

    import fa_workloads as W
    import oracle
    f = lambda t: t.float().double().numpy()
    drop = (w.dropout, W.DROPOUT_SEED, 0) if w.dropout > 0 else None
    if w.varlen:
        q, k, v, do, cu = W.make_varlen_inputs(w, with_do=True)
        G = w.H // w.kv_heads

        def sample(n, nthreads):
            kv = np.arange(n) // G
            oracle.forward_varlen(f(q[:n]), f(k[kv]), f(v[kv]), cu, w.scale, causal=w.causal,
                                  nthreads=nthreads, dropout=drop)
            oracle.backward_varlen(f(q[:n]), f(k[kv]), f(v[kv]), f(do[:n]), cu, w.scale,
                                   causal=w.causal, nthreads=nthreads, dropout=drop)
        return sample, w.H, W.fwd_bwd_flops(w) / w.H
    q, k, v, do, mask = W.make_inputs(w, with_do=True)
    B, H, N, d = q.shape
    G = H // k.shape[1]
    if G > 1:
        k, v = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    r = lambda t, n: f(t.reshape(1, B * H, N, d)[:, :n])

    def sample(n, nthreads):
        oracle.forward(r(q, n), r(k, n), r(v, n), w.scale, causal=w.causal, block_mask=mask,
                       nthreads=nthreads, dropout=drop)
        oracle.backward(r(q, n), r(k, n), r(v, n), r(do, n), w.scale, causal=w.causal,
                        block_mask=mask, nthreads=nthreads, dropout=drop)
    return sample, B * H, W.fwd_bwd_flops(w, mask) / (B * H)


def calibrate_units(sample, total, nthreads, budget_s):
    """Units whose oracle forward + backward take about budget_s seconds, and
    the last calibration run (units, seconds)."""
    n = 1
    while True:
        t0 = time.perf_counter()
        sample(n, nthreads)
        dt = time.perf_counter() - t0
        if n >= total or dt >= 0.2 * budget_s:
            break
        n = min(total, n * 4)
    return max(1, min(total, int(n * budget_s / max(dt, 1e-3)))), (n, dt)


def cpu_baseline(w, budget_s=12.0, single_thread_s=4.0):
    """The oracle on all host threads over a sample of the workload, and on
    one thread over a sample of the BERT-large-shaped workload."""
    import fa_workloads as W
    sample, total, per_unit = oracle_job(w)
    nthreads = os.cpu_count() or 1
    n, (n_cal, dt_cal) = calibrate_units(sample, total, nthreads, budget_s)
    passes = 1
    if n == n_cal and dt_cal >= 0.5 * budget_s:
        dt = dt_cal  # one unit already takes the budget: keep that run
    else:
        if n >= total:  # the whole workload takes less than the budget: repeat it
            t0 = time.perf_counter()
            sample(n, nthreads)
            passes = max(1, int(budget_s / max(time.perf_counter() - t0, 1e-3)))
        t0 = time.perf_counter()
        for _ in range(passes):
            sample(n, nthreads)
        dt = time.perf_counter() - t0
    unit = "heads of the packed batch" if w.varlen else "(batch, head) slices"
    out = {"value": round(per_unit * n * passes / dt / 1e12, 9), "unit": "TFLOP/s",
           "cores": nthreads, "kind": "oracle",
           "sample": f"fp64 C oracle forward+backward on {n} of {total} {unit} "
                     f"of {w.name}, {passes} pass(es), {dt:.2f} s wall"}
    wb = W.WORKLOADS["bert_large"]
    s1, total1, per1 = oracle_job(wb)
    n1, (nc1, dc1) = calibrate_units(s1, total1, 1, single_thread_s)
    t0 = time.perf_counter()
    s1(n1, 1)
    d1 = time.perf_counter() - t0
    out["single_thread"] = {
        "value": round(per1 * n1 / d1 / 1e12, 9), "unit": "TFLOP/s", "cores": 1,
        "workload": wb.name,
        "sample": f"fp64 C oracle forward+backward on {n1} of {total1} (batch, head) slices "
                  f"of {wb.name} on one thread, {d1:.2f} s wall"}
    return out


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle timed on the host cores, on a
    bounded sample of the same workload each step (rank 0 only)."""
    import fa_workloads as W
    if rank != 0:
        return None
    w = workload_of(args)
    sample, total, per_unit = oracle_job(w)
    nthreads = os.cpu_count() or 1
    per_step_budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    n, (n_cal, dt_cal) = calibrate_units(sample, total, nthreads, per_step_budget)
    # a calibration run of exactly one step's sample is that step's warm-up
    done = 1 if n == n_cal else 0
    for _ in range(max(0, args.warmup - done)):
        sample(n, nthreads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        sample(n, nthreads)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.fmean(times)
    value = per_unit * n / (ms * 1e-3) / 1e12
    sample_txt = f"fp64 C oracle forward+backward on {n} of {total} units per step ({w.name})"
    return {"metric": METRIC, "value": round(value, 9), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, upcast to fp64)",
            "config": {"workload": f"{w.name}: {w.note}", "B": w.B, "H": w.H, "N": w.N,
                       "d": w.d, "causal": w.causal},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "cores": nthreads,
                             "kind": "oracle", "sample": sample_txt},
            "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def tile_model_kv_bytes(B, H, N, d, rows, causal):
    """K and V bytes the forward's CTAs stream with no reuse between CTAs
    (the K/V term of the tile IO model): every CTA of `rows` query rows reads
    every 128-key tile it needs, all of them (dense) or those up to its last
    row (causal).  The row block, not the key tile, sets this."""
    nT = (N + 127) // 128
    per = rows // 128
    ctas = (nT + per - 1) // per
    if causal:
        tiles = sum(min(nT, per * (c + 1)) for c in range(ctas))
    else:
        tiles = ctas * nT
    return int(B * H * tiles * 2 * 128 * d * 2)


SWEEP_STAGES = {(128, 128): (2, 3, 4, 5), (128, 64): (4, 8), (128, 256): (2,),
                (64, 128): (2, 4, 8), (64, 64): (8, 16), (64, 256): (2, 4)}


def sweep_configs(d):
    """(rows per CTA, key tile, K/V stages) the library builds for head dim d;
    a 256-key tile takes one query tile per CTA."""
    return [(rows, bc, st) for (dd, bc), sts in SWEEP_STAGES.items() if dd == d for st in sts
            for rows in ((128,) if bc == 256 else (128, 256))]


def run_tile_sweep(args):
    """Block-size experiment: forward time per (rows per CTA, key tile,
    K/V stages), one JSON line each.  DRAM bytes per configuration come from
    running this mode under ncu (dram__bytes_read.sum +
    dram__bytes_write.sum)."""
    import torch

    import fa_workloads as W
    import io_aware_exact_15_gb300 as fa

    dev = torch.device("cuda", 0)
    w = workload_of(args)
    B, H, N, d = w.B, w.H, w.N, w.d
    q, k, v, _, _ = W.make_inputs(w, with_do=False)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ff = W.fwd_flops(w)
    peak = load_peaks()["bf16_tflops"]
    for rows, bc, st in sweep_configs(d) + [("default", 128, None)]:
        def call():
            if st is None:
                r = fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, w.scale, w.causal)
            else:
                r = fa.fa_debug_forward_config(qd, kd, vd, o, lse, B, H, N, d, w.scale, w.causal,
                                               rows, bc, st)
            if r != fa.FA_OK:
                raise RuntimeError(fa.fa_status_string(r))
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            call()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        br = 256 if rows == "default" else rows
        print(json.dumps({"sweep": "forward tile configuration", "workload": w.name,
                          "rows_per_cta": br, "key_tile": bc,
                          "kv_stages": st if st else "fa_forward",
                          "ms": round(ms, 4), "tflops": round(ff / (ms * 1e-3) / 1e12, 1),
                          "frac_of_peak": round(ff / (ms * 1e-3) / 1e12 / peak, 4),
                          "tile_model_kv_bytes": tile_model_kv_bytes(B, H, N, d, br,
                                                                     w.causal)}), flush=True)
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status after the sweep")


def run_host_overhead(args, calls=200, batches=10):
    """Host time of one C-ABI call (argument checks, cached tensor maps,
    launches), measured around the raw ctypes calls on a problem small
    enough that the GPU keeps up; a host-only library call gives the floor
    of the ctypes call itself."""
    import torch

    import io_aware_exact_15_gb300 as fa

    lib = fa.load()
    dev = torch.device("cuda", 0)
    out = {}
    for (B, H, N, d) in ((1, 1, 128, 64), (8, 16, 512, 64)):
        q, k, v, o, do, dq, dk, dv = (torch.zeros((B, H, N, d), dtype=torch.bfloat16, device=dev)
                                      for _ in range(8))
        lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
        nb = fa.fa_backward_workspace_size(B, H, N, d)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        s_ = torch.cuda.current_stream().cuda_stream
        p = lambda t: t.data_ptr()
        fargs = (p(q), p(k), p(v), p(o), p(lse), B, H, N, d, 0.125, 0, s_)
        bargs = (p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv), B, H, N, d, 0.125, 0,
                 p(ws), nb, s_)
        cases = {"fa_forward": (lib.fa_forward, fargs), "fa_backward": (lib.fa_backward, bargs),
                 "ctypes_floor": (lib.fa_backward_workspace_size, (B, H, N, d))}
        res = {}
        for name, (fn, a) in cases.items():
            for _ in range(20):
                fn(*a)
            torch.cuda.synchronize()
            tot = 0.0
            for _ in range(batches):
                t0 = time.perf_counter()
                for _ in range(calls):
                    fn(*a)
                tot += time.perf_counter() - t0
                torch.cuda.synchronize()
            res[name] = round(1e6 * tot / (calls * batches), 2)
        out[f"B{B} H{H} N{N} d{d}"] = res
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status after the host-overhead loop")
    print(json.dumps({"host_us_per_call": out}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="time fa_backward_deterministic instead of fa_backward")
    ap.add_argument("--tile-sweep", action="store_true",
                    help="time the forward per tile configuration (block-size experiment)")
    ap.add_argument("--sparse-density", type=float, default=None,
                    help="random-tile density of a block-sparse workload (default: its own)")
    ap.add_argument("--host-overhead", action="store_true",
                    help="time the host side of one fa_forward / fa_backward call")
    args = ap.parse_args()
    if args.tile_sweep:
        run_tile_sweep(args)
        return
    if args.host_overhead:
        run_host_overhead(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    # the oracle pool starts before the first GPU call (threads, no fork)
    res = run_gpu(args, rank, world, dist)
    if rank == 0:
        import fa_workloads as W
        if not args.no_cpu_baseline and world >= 1:
            res["cpu_baseline"] = cpu_baseline(workload_of(args))
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
