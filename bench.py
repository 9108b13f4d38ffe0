#!/usr/bin/env python
"""Ring-chunked exact attention, forward + backward, on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
the ring-chunked forward (online LSE merge) and the ring-chunked backward
(row statistics, the recomputing backward kernel, dQ conversion) of the
long-context video workload B=1, S=32760, H=24, D=128, P=8 ring chunks.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  The throughput unit is TFLOP/s with the
algorithmic flop count 14 * B * Hq * S^2 * D per step (4 forward, 10 for the
backward that recomputes the probabilities).  N > 1 runs N independent
replicas of the workload (the ring is emulated on one GPU; there is no
data-path collective), launched by torchrun.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from seeded_inputs import (GQA_D256_S1024, HYBRID_RING, HYBRID_S65536, HYBRID_ULYSSES,  # noqa: E402
                           VIDEO_S32760_P8, AttnShape, attn_inputs, exchange_input)

METRIC = "fwd+bwd attention TFLOP/s at 1 GB300 (ring P chunks), % of dense bf16 peak"
UNIT = "TFLOP/s"
WORKLOAD = VIDEO_S32760_P8
WORKLOAD_NAME = "video-DiT long context MHA fwd+bwd, B=1 S=32760 H=24 D=128, P=8 ring chunks (8 x 4095)"
L2_NOTE = "inputs larger than L2 (q/k/v/dout 805 MB vs 126.5 MB L2); no flush"

# dram traffic per launch of the backward kernel from one ncu capture (see
# profiles/); valid only while the kernel source is the one it was taken on.
NCU_BWD = {"bytes_per_launch": 1320996352 + 850899712,  # dram read + write, S=32760 H=24 D=128 P=8
           "source_sha256": "2bcf66524566ddefaea9a26f4a35ec781a902d54c39579cef1259735577b8322"}


# Dense bf16 tensor-core rate of one SM per clock: one M=128, N=128, K=16
# tcgen05 product (2 flop per multiply-add) every 64 clocks.
TC_FLOP_PER_CLK_SM = 128 * 128 * 16 * 2 // 64


def flops_fwd(sh: AttnShape) -> float:
    return 4.0 * sh.B * sh.Hq * sh.S * sh.S * sh.D


def flops_bwd(sh: AttnShape) -> float:
    return 10.0 * sh.B * sh.Hq * sh.S * sh.S * sh.D


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"bf16": pk["bf16_tflops"], "bf16_sustained": pk["bf16_tflops_sustained"],
                "hbm": pk["hbm_gbs"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def tensor_peaks(peaks, clocks, n_sm):
    """The denominators of the tensor-core roofline for a kernel timed under
    `clocks` (the nvidia-smi samples of the timed region):
      measured -- the cuBLAS bf16 GEMM of MEASURED_PEAKS.json: the burst figure
                  when the SM clock's median sat at its maximum (no power or
                  thermal cap held it down), else the sustained one;
      clock    -- the tensor cores' own rate at the sampled median SM clock:
                  SMs x MHz x TC_FLOP_PER_CLK_SM."""
    mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    at_max = bool(mhz and mx and mhz >= 0.97 * mx)
    measured = peaks["bf16"] if at_max else peaks["bf16_sustained"]
    kind = (f"bf16 dense, {'burst' if at_max else 'sustained'} ({peaks['source']}): "
            f"SM clock median {mhz} of {mx} MHz in the timed region")
    clock = n_sm * mhz * 1e6 * TC_FLOP_PER_CLK_SM / 1e12 if mhz else None
    return measured, kind, clock


def roofline_entry(kernel, achieved, peaks, clocks, n_sm, **extra):
    measured, kind, clock = tensor_peaks(peaks, clocks, n_sm)
    d = {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": measured, "unit": "TFLOP/s",
         "frac": achieved / measured, "peak_kind": kind,
         "frac_burst": achieved / peaks["bf16"], "frac_sustained": achieved / peaks["bf16_sustained"],
         "clock_peak": clock, "frac_clock_peak": achieved / clock if clock else None,
         "sm_mhz": clocks.get("sm_mhz")}
    d.update(extra)
    return d


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest x over the ranks of the default process group (the
    slowest replica's time); x itself without one."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def replica_throughput(flops_per_step: float, steps: int, ms: float, world: int) -> float:
    """Whole-job TFLOP/s of `world` independent replicas, each doing `steps`
    steps, timed by the slowest replica (ms)."""
    return world * flops_per_step * steps / (ms / 1e3) / 1e12


def cpu_sample(S_sample: int):
    """Times the fp64 oracle (forward + analytic backward) on head 0 of the
    workload truncated to its first S_sample rows; returns (TFLOP/s, seconds)."""
    import oracle

    sh = AttnShape(B=1, S=S_sample, Hq=1, Hkv=1, D=WORKLOAD.D, P=1)
    q, k, v, do = attn_inputs(sh, seed=777)
    oracle.build()
    # every host core (torchrun pins OMP_NUM_THREADS to 1 per rank, and only
    # rank 0 runs the oracle)
    oracle.set_threads(os.cpu_count())
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v)
    oracle.attn_bwd(q, k, v, do)
    dt = time.perf_counter() - t0
    return 14.0 * S_sample * S_sample * sh.D / dt / 1e12, dt


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    S_step = 4095  # one ring chunk of head 0 per step
    for _ in range(args.warmup):
        cpu_sample(S_step)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_sample(S_step)
    dt = time.perf_counter() - t0
    val = args.steps * 14.0 * S_step * S_step * WORKLOAD.D / dt / 1e12
    cores = os.cpu_count()
    sample = (f"fp64 oracle forward + analytic backward of head 0 of the workload truncated to "
              f"its first ring chunk (S={S_step}, D={WORKLOAD.D}) per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def config_dict():
    sh = WORKLOAD
    return {"workload": WORKLOAD_NAME, "B": sh.B, "S": sh.S, "Hq": sh.Hq, "Hkv": sh.Hkv, "D": sh.D,
            "P": sh.P, "layout": sh.layout, "causal": False, "l2": L2_NOTE}


def measure_exchange(ctx, dev, stream, barrier, peaks):
    """Ulysses exchange of the hybrid workload's q, [1,65536,32,128] bf16,
    ring 4 x ulysses 2: forward and inverse, bytes read + written."""
    xq = exchange_input(1, 65536, 32, 128, seed=5).to(dev)
    y = ctx.seq_head_exchange(xq, 4, 2, 0, "bshd")
    back = ctx.seq_head_exchange(y, 4, 2, 1, "bshd", S=65536, B=1, H=32)
    barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    x0.record(stream)
    for _ in range(reps):
        ctx.seq_head_exchange(xq, 4, 2, 0, "bshd", y=y)
        ctx.seq_head_exchange(y, 4, 2, 1, "bshd", y=back, S=65536, B=1, H=32)
    x1.record(stream)
    barrier()
    xms = x0.elapsed_time(x1) / (2 * reps)
    xbytes = 2 * xq.numel() * xq.element_size()
    gbs = xbytes / (xms / 1e3) / 1e9
    return {"shape": [1, 65536, 32, 128], "ring": 4, "ulysses": 2, "bound": "hbm", "achieved": gbs,
            "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"], "ms": xms,
            "bytes": xbytes}


def measure_d256(ctx, dev, stream, barrier, peaks):
    """Head dimension 256: the 24/4-head causal language model (1024 tokens,
    P=2; inputs 14 MB, resident in L2) and a long-context case of the same
    heads (16384 tokens, P=8)."""
    return measure_causal(ctx, dev, stream, barrier, peaks,
                          (("24/4-head D=256 causal LM, S=1024, P=2", GQA_D256_S1024, 50),
                           ("same heads, long context S=16384, P=8",
                            AttnShape(B=1, S=16384, Hq=24, Hkv=4, D=256, P=8), 5)))


def measure_causal(ctx, dev, stream, barrier, peaks, cases):
    """Causal fwd + bwd steps, eager and replayed from a CUDA graph, with the
    kernels' own event times.  Causal flop count: the S (S + 1) / 2 visible
    pairs, 4 D flop each forward and 10 D backward, per query head."""
    res = []
    for name, sh, reps in cases:
        q, k, v, do = (t.to(dev) for t in attn_inputs(sh))
        out, lse = ctx.attn_fwd(q, k, v, sh.P, causal=True)
        ws = torch.empty(ctx.workspace_size(sh.B, sh.S, sh.Hq, sh.Hkv, sh.D, sh.P), dtype=torch.uint8,
                         device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def step():
            ctx.attn_fwd(q, k, v, sh.P, causal=True, out=out, lse=lse)
            ctx.attn_bwd(q, k, v, out, lse, do, sh.P, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)

        for _ in range(3):
            step()
        barrier()
        ctx.profile_enable(True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            step()
        e1.record(stream)
        barrier()
        ctx.profile_enable(False)
        if ctx.device_status() != 0:
            raise RuntimeError(f"device-side wait timed out ({name})")
        ms = e0.elapsed_time(e1) / reps
        # the same step captured once in a CUDA graph and replayed (no
        # per-launch host overhead: matters at 1024 tokens)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        barrier()
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
        barrier()
        if ctx.device_status() != 0:
            raise RuntimeError(f"device-side wait timed out ({name}, graph)")
        ms_graph = e0.elapsed_time(e1) / reps
        pairs = sh.B * sh.Hq * sh.S * (sh.S + 1) / 2.0
        fl_f, fl_b = 4.0 * pairs * sh.D, 10.0 * pairs * sh.D
        f_ms, f_n = ctx.profile_read("fwd")
        b_ms, b_n = ctx.profile_read("bwd")
        f_avg, b_avg = f_ms / max(f_n, 1), b_ms / max(b_n, 1)
        fname, bname = (("attn_fwd256_kernel", "attn_bwd256_kernel") if sh.D == 256
                        else (f"attn_fwd_kernel<{sh.D}>", f"attn_bwd_kernel<{sh.D}>"))
        res.append({"workload": name, "B": sh.B, "S": sh.S, "Hq": sh.Hq, "Hkv": sh.Hkv, "D": sh.D,
                    "P": sh.P, "causal": True, "ms_per_step": ms,
                    "value": (fl_f + fl_b) / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
                    "graph": {"ms_per_step": ms_graph, "value": (fl_f + fl_b) / (ms_graph / 1e3) / 1e12},
                    "fwd_kernel": {"kernel": fname, "avg_ms": f_avg,
                                   "achieved": fl_f / (f_avg / 1e3) / 1e12,
                                   "frac": fl_f / (f_avg / 1e3) / 1e12 / peaks["bf16"]},
                    "bwd_kernel": {"kernel": bname, "avg_ms": b_avg,
                                   "achieved": fl_b / (b_avg / 1e3) / 1e12,
                                   "frac": fl_b / (b_avg / 1e3) / 1e12 / peaks["bf16"]},
                    "peak": peaks["bf16"], "peak_kind": f"bf16 dense, burst ({peaks['source']})"})
        del q, k, v, do, out, lse, ws, dq, dk, dv, graph
    return res


def measure_hybrid(ctx, dev, stream, barrier, steps=2):
    """The ring 4 x ulysses 2 hybrid at full size, one step = the exchange of
    q, k, v ([1,65536,32,128], k and v with 8 heads), GQA 32/8 ring attention
    over 4 chunks on the exchanged tensors (forward and backward, both head
    groups in one call each), the exchange of dout and the inverse exchange
    of out, dq, dk, dv.  TFLOP/s over the attention's algorithmic flops."""
    sh, R, U = HYBRID_S65536, HYBRID_RING, HYBRID_ULYSSES
    q, k, v, do = (t.to(dev) for t in attn_inputs(sh))
    W = R * U
    Ssh = -(-sh.S // W)
    offs = [min(r * U * Ssh, sh.S) for r in range(R)] + [sh.S]  # rank (r, u) holds these rows
    ex = [torch.empty(ctx.exchanged_shape(sh.B, sh.S, t.shape[2], sh.D, R, U, "bshd"), dtype=t.dtype, device=dev)
          for t in (q, k, v, do)]
    views = [ctx.exchanged_view(t, sh.S, "bshd") for t in ex]
    vq, vk, vv, vdo = views
    out, lse = ctx.attn_fwd(vq, vk, vv, R, chunk_offsets=offs)
    dq, dk, dv = ctx.attn_bwd(vq, vk, vv, out, lse, vdo, R, chunk_offsets=offs)
    ws = torch.empty(ctx.workspace_size(U * sh.B, sh.S, sh.Hq // U, sh.Hkv // U, sh.D, R), dtype=torch.uint8,
                     device=dev)
    back = [torch.empty_like(t) for t in (q, q, k, v)]
    assert sh.S % W == 0  # no padding rows: the attention's outputs are the dense exchanged layout
    grp = lambda t: t.view(U, sh.B, sh.S, t.shape[2], sh.D)

    def step():
        for x, y in zip((q, k, v), ex[:3]):
            ctx.seq_head_exchange(x, R, U, 0, "bshd", y=y)
        ctx.attn_fwd(vq, vk, vv, R, chunk_offsets=offs, out=out, lse=lse)
        ctx.seq_head_exchange(grp(out), R, U, 1, "bshd", y=back[0], S=sh.S, B=sh.B, H=sh.Hq)
        ctx.seq_head_exchange(do, R, U, 0, "bshd", y=ex[3])
        ctx.attn_bwd(vq, vk, vv, out, lse, vdo, R, chunk_offsets=offs, dq=dq, dk=dk, dv=dv, workspace=ws)
        for g_, y, H in ((dq, back[1], sh.Hq), (dk, back[2], sh.Hkv), (dv, back[3], sh.Hkv)):
            ctx.seq_head_exchange(grp(g_), R, U, 1, "bshd", y=y, S=sh.S, B=sh.B, H=H)

    step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    barrier()
    if ctx.device_status() != 0:
        raise RuntimeError("device-side wait timed out (hybrid)")
    ms = e0.elapsed_time(e1) / steps
    # fused exchange + attention: the attention reads the un-exchanged
    # tensors through a strided view that makes the head group the batch
    # index ([U, S, H/U, D], B = 1) and writes out, dq, dk, dv straight into
    # the un-exchanged layout: no exchange copies at all
    Hu, Hku = sh.Hq // U, sh.Hkv // U
    gview = lambda t, Hg: t[0].view(sh.S, U, Hg, sh.D).permute(1, 0, 2, 3)
    out_f, dq_f = torch.empty_like(q), torch.empty_like(q)
    dk_f, dv_f = torch.empty_like(k), torch.empty_like(v)
    lse_f = torch.empty(U, Hu, sh.S, dtype=torch.float32, device=dev)
    fq, fk, fv, fdo = gview(q, Hu), gview(k, Hku), gview(v, Hku), gview(do, Hu)
    fout, fdq, fdk, fdv = gview(out_f, Hu), gview(dq_f, Hu), gview(dk_f, Hku), gview(dv_f, Hku)
    ws_f = torch.empty(ctx.workspace_size(U, sh.S, Hu, Hku, sh.D, R), dtype=torch.uint8, device=dev)

    def fused_step():
        ctx.attn_fwd(fq, fk, fv, R, chunk_offsets=offs, out=fout, lse=lse_f)
        ctx.attn_bwd(fq, fk, fv, fout, lse_f, fdo, R, chunk_offsets=offs, dq=fdq, dk=fdk, dv=fdv, workspace=ws_f)

    fused_step()
    barrier()
    e0.record(stream)
    for _ in range(steps):
        fused_step()
    e1.record(stream)
    barrier()
    if ctx.device_status() != 0:
        raise RuntimeError("device-side wait timed out (hybrid, fused)")
    ms_fused = e0.elapsed_time(e1) / steps
    flops = flops_fwd(sh) + flops_bwd(sh)
    res = {"workload": "ring 4 x ulysses 2 hybrid, [1,65536,32,128] (k, v 8 heads), GQA 32/8, P=4",
           "ms_per_step": ms, "value": flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "steps": steps,
           "exchanges_per_step": 8,
           "fused": {"ms_per_step": ms_fused, "value": flops / (ms_fused / 1e3) / 1e12,
                     "note": "one call over strided head-group views of the un-exchanged tensors; "
                             "outputs written in place, no exchange"}}
    del q, k, v, do, ex, views, out, lse, dq, dk, dv, ws, back, out_f, dq_f, dk_f, dv_f, lse_f, ws_f
    return res


def measure_e2e(ctx, dev, sh, host_inputs, ws, steps, barrier, world):
    """End to end through the public API: every step copies that step's
    inputs (q, k, v, dout) from pinned host memory to the GPU, runs the
    forward and backward, and copies the results (out, lse, dq, dk, dv) back
    to pinned host memory.  Input and output buffers are double-buffered and
    the copies run on their own streams, so step k's copies overlap the
    compute of its neighbours, as a pipeline fed with a stream of batches
    would run.  Within a step the forward starts once q, k, v are in and
    out, lse are copied back while the backward runs.  The timed region
    spans the first input copy to the last result copy.  Returns the e2e
    dict of the JSON line."""
    pin = lambda t: t.contiguous().pin_memory()
    h_in = [pin(t) for t in host_inputs]
    nbuf = 2
    d_in = [[torch.empty(t.shape, dtype=t.dtype, device=dev) for t in h_in] for _ in range(nbuf)]
    oshape = [(sh.B, sh.S, sh.Hq, sh.D), (sh.B, sh.Hq, sh.S), (sh.B, sh.S, sh.Hq, sh.D),
              (sh.B, sh.S, sh.Hkv, sh.D), (sh.B, sh.S, sh.Hkv, sh.D)]
    odt = [torch.bfloat16, torch.float32, torch.bfloat16, torch.bfloat16, torch.bfloat16]
    d_out = [[torch.empty(s_, dtype=t_, device=dev) for s_, t_ in zip(oshape, odt)] for _ in range(nbuf)]
    h_out = [[torch.empty(s_, dtype=t_, pin_memory=True) for s_, t_ in zip(oshape, odt)] for _ in range(nbuf)]
    compute = torch.cuda.current_stream(dev)
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev() for _ in range(nbuf)], [ev() for _ in range(nbuf)]
    out_ready, out_free = [ev() for _ in range(nbuf)], [ev() for _ in range(nbuf)]
    fwd_in, fwd_done = [ev() for _ in range(nbuf)], [ev() for _ in range(nbuf)]

    def run(k):
        b = k % nbuf
        h2d_s.wait_event(in_free[b])  # the compute of step k - 2 has read these inputs
        with torch.cuda.stream(h2d_s):
            for j, (d, h) in enumerate(zip(d_in[b], h_in)):
                d.copy_(h, non_blocking=True)
                if j == 2:
                    fwd_in[b].record(h2d_s)  # q, k, v: the forward can start
        in_ready[b].record(h2d_s)
        compute.wait_event(fwd_in[b])
        compute.wait_event(out_free[b])  # the results of step k - 2 have been copied out
        q, k_, v, do = d_in[b]
        out, lse, dq, dk, dv = d_out[b]
        ctx.attn_fwd(q, k_, v, sh.P, out=out, lse=lse)
        fwd_done[b].record(compute)
        compute.wait_event(in_ready[b])  # dout
        ctx.attn_bwd(q, k_, v, out, lse, do, sh.P, dq=dq, dk=dk, dv=dv, workspace=ws)
        in_free[b].record(compute)
        out_ready[b].record(compute)
        d2h_s.wait_event(fwd_done[b])  # out and lse leave while the backward runs
        with torch.cuda.stream(d2h_s):
            for j, (h, d) in enumerate(zip(h_out[b], d_out[b])):
                if j == 2:
                    d2h_s.wait_event(out_ready[b])
                h.copy_(d, non_blocking=True)
        out_free[b].record(d2h_s)

    for k in range(2):
        run(k)
    barrier()
    # the copies alone, outside the timed region: the link's bandwidth on this machine
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(h2d_s):
        c0.record(h2d_s)
        for d, h in zip(d_in[0], h_in):
            d.copy_(h, non_blocking=True)
        c1.record(h2d_s)
    barrier()
    h2d_ms = c0.elapsed_time(c1)
    with torch.cuda.stream(d2h_s):
        c0.record(d2h_s)
        for h, d in zip(h_out[0], d_out[0]):
            h.copy_(d, non_blocking=True)
        c1.record(d2h_s)
    barrier()
    d2h_ms = c0.elapsed_time(c1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    h2d_s.wait_event(e0)
    for k in range(steps):
        run(k)
    compute.wait_event(out_free[(steps - 1) % nbuf])
    e1.record(compute)
    barrier()
    ems = max_over_ranks(e0.elapsed_time(e1), dev)
    flops_step = flops_fwd(sh) + flops_bwd(sh)
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    return {"value": replica_throughput(flops_step, steps, ems, world), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems / steps,
            "copies_alone": {"h2d_ms": h2d_ms, "h2d_gbs": h2d / (h2d_ms / 1e3) / 1e9,
                             "d2h_ms": d2h_ms, "d2h_gbs": d2h / (d2h_ms / 1e3) / 1e9},
            "overlap": "copies on their own streams, inputs/outputs double-buffered; the forward starts "
                       "once q, k, v are in, out and lse are copied back during the backward",
            "gpu_launches": 4 * steps}


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-exchange", action="store_true")
    ap.add_argument("--no-d256", action="store_true")
    ap.add_argument("--no-hybrid", action="store_true")
    ap.add_argument("--no-causal", action="store_true")
    ap.add_argument("--shape", default=None,
                    help="S,Hq,Hkv,D,P: a smaller case of the same kernels (profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    global WORKLOAD, WORKLOAD_NAME, L2_NOTE
    if args.shape:
        S, Hq, Hkv, D, P = (int(x) for x in args.shape.split(","))
        WORKLOAD = AttnShape(B=1, S=S, Hq=Hq, Hkv=Hkv, D=D, P=P)
        WORKLOAD_NAME = f"profiling case B=1 S={S} Hq={Hq} Hkv={Hkv} D={D} P={P}"
        L2_NOTE = f"q/k/v/dout {4 * S * Hq * D * 2 / 1e6:.0f} MB; no flush"

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import context_attention_fwd_gb300 as ctx

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ctx.load_library(build_if_missing=True)
    sh = WORKLOAD
    peaks = load_peaks()

    q_h, k_h, v_h, do_h = attn_inputs(sh)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    out = torch.empty_like(q)
    lse = torch.empty(sh.B, sh.Hq, sh.S, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ctx.workspace_size(sh.B, sh.S, sh.Hq, sh.Hkv, sh.D, sh.P), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ctx.attn_fwd(q, k, v, sh.P, out=out, lse=lse)
        ctx.attn_bwd(q, k, v, out, lse, do, sh.P, dq=dq, dk=dk, dv=dv, workspace=ws)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    if ctx.device_status() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    # ------------------------------------------------ device-resident timing
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx.profile_enable(True)
    with ClockSampler(local) as clk:
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
    ctx.profile_enable(False)
    ms = max_over_ranks(ev0.elapsed_time(ev1), dev)
    if ctx.device_status() != 0:
        raise RuntimeError("device-side wait timed out during the timed region")
    flops_step = flops_fwd(sh) + flops_bwd(sh)
    value = replica_throughput(flops_step, args.steps, ms, world)
    bwd_ms, bwd_n = ctx.profile_read("bwd")
    fwd_ms, fwd_n = ctx.profile_read("fwd")
    bwd_avg, fwd_avg = bwd_ms / max(bwd_n, 1), fwd_ms / max(fwd_n, 1)
    bwd_tf = flops_bwd(sh) / (bwd_avg / 1e3) / 1e12
    fwd_tf = flops_fwd(sh) / (fwd_avg / 1e3) / 1e12
    bwd_src = os.path.join(ROOT, "context_attention_fwd_gb300", "csrc", "attn_bwd.cu")
    # the ncu bytes were taken on the default workload, with this source
    traffic = (NCU_BWD["bytes_per_launch"]
               if not args.shape and NCU_BWD["source_sha256"] == source_sha(bwd_src) else None)
    kname = "attn_fwd256_kernel" if sh.D == 256 else f"attn_fwd_kernel<{sh.D}>"
    bname = "attn_bwd256_kernel" if sh.D == 256 else f"attn_bwd_kernel<{sh.D}>"
    clocks = clk.summary()
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    _, _, clock_peak = tensor_peaks(peaks, clocks, n_sm)

    # ------------------------------------------------ end to end, host buffers
    e2e = None
    if not args.no_e2e:
        del out, lse, dq, dk, dv
        e2e = measure_e2e(ctx, dev, sh, (q_h, k_h, v_h, do_h), ws, args.steps, barrier, world)

    # ------------------------------------------------ the exchange (HBM bound)
    exchange = None
    if not args.no_exchange:
        exchange = measure_exchange(ctx, dev, stream, barrier, peaks)

    # ------------------------------------------------ the ring x ulysses hybrid at full size
    hybrid = None
    if not args.no_hybrid and not args.shape:
        hybrid = measure_hybrid(ctx, dev, stream, barrier)

    # ------------------------------------------------ head dimension 256 (GQA 24/4, causal)
    d256 = None
    if not args.no_d256:
        d256 = measure_d256(ctx, dev, stream, barrier, peaks)

    # ------------------------------------------------ the long-context workload with causal masking
    causal = None
    if not args.no_causal and not args.shape:
        causal = measure_causal(ctx, dev, stream, barrier, peaks,
                                (("video-DiT shape with causal masking, B=1 S=32760 H=24 D=128, P=8",
                                  AttnShape(B=1, S=32760, Hq=24, Hkv=24, D=128, P=8), 3),))

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(),
        "pct_of_peak": {"burst": 100.0 * value / world / peaks["bf16"],
                        "sustained": 100.0 * value / world / peaks["bf16_sustained"],
                        "clock_derived": (100.0 * value / world / clock_peak) if clock_peak else None,
                        "clock_derived_tflops": clock_peak,
                        "peaks_source": peaks["source"],
                        "note": "burst / sustained: the measured cuBLAS bf16 GEMM; clock_derived: "
                                f"{n_sm} SMs x median SM MHz x {TC_FLOP_PER_CLK_SM} flop/clk/SM"},
        "clocks": clocks,
        "gpu_launches": 4 * args.steps,
        "roofline": roofline_entry(bname, bwd_tf, peaks, clocks, n_sm, traffic=traffic,
                                   launches=bwd_n, avg_ms=bwd_avg),
        "roofline_fwd": roofline_entry(kname, fwd_tf, peaks, clocks, n_sm, launches=fwd_n, avg_ms=fwd_avg),
        "exchange": exchange,
        "d256": d256,
        "causal": causal,
        "hybrid": hybrid,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, secs = cpu_sample(16380)
        line["cpu_baseline"] = {
            "value": val, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": ("fp64 oracle forward + analytic backward of head 0 of the workload truncated "
                       f"to its first four ring chunks (S=16380, D=128), {secs:.1f} s")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
