"""Throughput of the Ulysses attention step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is the whole hot path over one batch of synthetic input, already
resident in HBM:
    seq->head relayout of Q/K/V, attention forward, head->seq relayout of O,
    seq->head relayout of dO, attention backward (row statistics, main kernel,
    dQ convert), head->seq relayout of dQ/dK/dV.
The metric is causal attention fwd+bwd TFLOP/s (fwd = 4*b*h*s^2*d/2 flops for a
causal square, backward 2.5x the forward), with the bf16 tensor-core fraction
and the relayout GB/s against the measured HBM copy bandwidth beside it.

N > 1 (one process per GPU under torch.distributed.run): every rank runs the
same step on its own GPU with no collective on the data path (weak scaling);
the timed region is bracketed by barriers and the slowest rank's time is used.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import contextlib
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sequence_head_attention_seq_b300 import workloads  # noqa: E402

METRIC = "causal MHA fwd+bwd TFLOP/s and % bf16 tensor peak; relayout GB/s vs HBM"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "llama70b"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ---------------------------------------------------------------- accounting

def attn_fwd_flops(w) -> float:
    """4*b*h*sq*sk*d for the two GEMMs of the forward, halved for a causal square."""
    f = 4.0 * w.b * w.h * w.s * w.s * w.d
    return f / 2 if w.causal else f


def valid_pairs(w, key_len=None) -> int:
    """Exact (query row, key) pairs that take part, summed over batch rows and heads: the
    causal square counts sum_i (i + 1); padded keys drop out (key j < key_len[b])."""
    lens = [w.s] * w.b if key_len is None else [int(x) for x in key_len.tolist()]
    total = 0
    for n in lens:
        n = max(0, min(n, w.s))
        if w.causal:
            # row i sees keys 0..min(i, n-1)
            full = min(n, w.s)
            total += full * (full + 1) // 2 + (w.s - full) * n
        else:
            total += w.s * n
    return total * w.h


MUFU_EX2_PER_CLK_SM = 32    # ex2.approx.f32 lanes per clock per SM, measured on B300


def step_flops(w) -> float:
    return 3.5 * attn_fwd_flops(w)          # forward + backward (2.5x forward)


def proj_flops(w) -> float:
    """Projections of the attention layer (hidden = h*d): forward 2*M*dim*3hd (q, k, v) +
    2*M*hd*dim (output), backward twice that (input and weight gradients)."""
    M, dim, hd = w.b * w.s, w.h * w.d, w.h * w.d
    return 3 * (2.0 * M * dim * 3 * hd + 2.0 * M * hd * dim)


def tensor_bytes(w) -> int:
    return w.b * w.s * w.h * w.d * 2


def relayout_bytes_per_step(w) -> int:
    """Each relayout reads and writes every tensor once: Q, K, V, O, dO, dQ, dK, dV."""
    return 0 if w.N == 1 else 8 * 2 * tensor_bytes(w)


def launches_per_step(w, ring_chunks: int = 0, fused: bool = False) -> int:
    relayouts = 0 if (w.N == 1 or fused) else 4
    if ring_chunks > 1:                   # per chunk: fwd + merge, main + dQ convert;
        return relayouts + ring_chunks * 4 + 1   # statistics once (later chunks reuse them)
    return relayouts + 1 + 3              # fwd; bwd = statistics + main + dQ convert


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest(names) -> str:
    """sha256 (16 hex digits) of the kernel sources' code: comments and white space are
    removed first, so a change of wording leaves it alone and a change of code does not."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sequence_head_attention_seq_b300", "csrc", n)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()[:16]


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per sp_attn_bwd call of the
# LLaMA-70B-shaped workload, keyed by the digest of the kernel code they were measured on:
# a changed kernel has no recorded traffic until it is captured again.  Captured on the
# same sequence with 8 heads (one call: statistics, main and dQ-convert kernels, 1.019 GB)
# and scaled by the 8x heads of the full workload, whose CTAs run one head at a time.
RECORDED_BWD_TRAFFIC = {
    "workload": "llama70b",
    "sources": ["attn_bwd.cu", "ptx.cuh"],
    "by_digest": {"a9dc8b946333eecf": 8151209984},
}


def recorded_traffic(workload_name: str) -> int | None:
    """DRAM bytes per sp_attn_bwd call for this workload if its kernel code is unchanged
    since the capture, else None."""
    rec = RECORDED_BWD_TRAFFIC
    if workload_name != rec["workload"]:
        return None
    return rec["by_digest"].get(source_digest(rec["sources"]))


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, device) -> float:
    if dist.is_available() and dist.is_initialized():
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return x


def barrier():
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(REASON_NAMES, parts[3:]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_index_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------- CPU oracle sample

def oracle_sample(w, heads: int, prefix: int):
    """Causal fwd+bwd of `heads` heads over the first `prefix` positions of workload w,
    drawn with the workload's seeds and scale (a bounded sample of the same problem)."""
    import oracle
    orc = oracle.default()
    heads, prefix = min(heads, w.h), min(prefix, w.s)
    shape = (1, prefix, heads, w.d)
    q = workloads.randn_bf16(shape, w.seed("q"), w.scale).double().numpy()
    k = workloads.randn_bf16(shape, w.seed("k"), w.scale).double().numpy()
    v = workloads.randn_bf16(shape, w.seed("v"), w.scale).double().numpy()
    do = workloads.randn_bf16(shape, w.seed("dout"), 1.0).double().numpy()
    t0 = time.perf_counter()
    orc.attn_fwd(q, k, v, w.causal)
    orc.attn_bwd(q, k, v, do, w.causal)
    dt = time.perf_counter() - t0
    flops = 3.5 * 4.0 * heads * prefix * prefix * w.d / (2 if w.causal else 1)
    return flops, dt, orc.threads(), heads, prefix


def head_of(t: torch.Tensor, w, j: int):
    """Head j of a shard-layout tensor [N][b][s/N][h][d] over the whole sequence of batch
    row 0, as the oracle's [1][s][1][d] fp64 array (the shards in order are the sequence)."""
    return t[:, 0, :, j, :].reshape(1, w.s, 1, w.d).double().cpu().numpy()


def cpu_baseline(w, ins, head=0):
    """The oracle on the host cores over one whole head of the timed workload (every query
    row and every key; inputs copied from the device), extrapolated linearly in heads to
    the full workload, plus the same oracle on one core over a shorter sequence."""
    import oracle
    orc = oracle.default()
    q, k, v, do = (head_of(ins[n], w, head) for n in ("q", "k", "v", "dout"))
    kl = None if ins["key_len"] is None else ins["key_len"][:1].tolist()
    t0 = time.perf_counter()
    orc.attn_fwd(q, k, v, w.causal, 0, kl)
    orc.attn_bwd(q, k, v, do, w.causal, 0, kl)
    dt = time.perf_counter() - t0
    flops = step_flops(w) / (w.b * w.h)            # one head of one batch row
    full_s = dt * w.b * w.h
    line = {"value": flops / dt / 1e12, "unit": UNIT, "cores": orc.threads(), "kind": "oracle",
            "sample": f"fp64 C oracle, fwd+bwd of head {head} of batch row 0 over all {w.s} "
                      f"positions of {w.name} (d={w.d}), inputs copied from the device: "
                      f"{flops / 1e9:.1f} GFLOP in {dt:.1f} s",
            "full_workload_s": full_s,
            "full_workload_s_kind": f"extrapolated linearly in heads ({w.b * w.h} heads), "
                                    "not measured"}
    # the same oracle on one core, on a shorter sequence of the same problem
    threads = orc.threads()
    orc.set_threads(1)
    try:
        f1, dt1, _, h1, p1 = oracle_sample(w, 1, 2048)
    finally:
        orc.set_threads(threads)
    line["single_core"] = {"value": f1 / dt1 / 1e12, "unit": UNIT, "cores": 1,
                           "sample": f"1 head over the first {p1} positions; "
                                     f"{f1 / 1e9:.1f} GFLOP in {dt1:.1f} s"}
    line["relayout"] = cpu_relayout(w, ins)
    return line


def cpu_relayout(w, ins):
    """The regrouping on the host: the oracle's scalar copy loop (one thread) over one
    whole tensor of the workload (Q, sequence shards -> head groups), in GB/s of bytes
    read + written; None when the workload has a single shard (nothing to regroup)."""
    if w.N == 1:
        return None
    import oracle
    bits = ins["q"].contiguous().cpu().view(torch.int16).numpy().view("uint16")
    t0 = time.perf_counter()
    oracle.default().seq2head(bits, w.N, w.b, w.s, w.h, w.d)
    dt = time.perf_counter() - t0
    return {"value": 2 * bits.nbytes / dt / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"seq2head of one {bits.nbytes / 2**20:.0f} MiB tensor (Q) of {w.name}, "
                      f"N={w.N}: {dt:.2f} s"}


# ---------------------------------------------------------------- arms

def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    heads, prefix = 1, 8192
    for _ in range(args.warmup):
        oracle_sample(w, heads, prefix)
    total_flops, total_t, cores = 0.0, 0.0, 1
    for _ in range(args.steps):
        f, dt, cores, heads, prefix = oracle_sample(w, heads, prefix)
        total_flops += f
        total_t += dt
    value = total_flops / total_t / 1e12
    sample = (f"fp64 C oracle, causal fwd+bwd of {heads} head over the first {prefix} positions "
              f"of {w.name} per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_note(w) -> str:
    """Whether a step's data outruns L2 between timed steps: a step reads and writes the
    eight shard tensors and their eight head-group copies."""
    ws = 16 * tensor_bytes(w)
    per = f"{tensor_bytes(w) / 2**20:.0f} MiB per tensor, {ws / 2**20:.0f} MiB touched per step"
    if ws > 126e6:
        return f"inputs larger than L2 ({per}, 126 MB L2)"
    return f"working set within the 126 MB L2 ({per}); not flushed between steps"


def config_of(w, ring_chunks: int = 0):
    extra = {"ring_chunks": ring_chunks} if ring_chunks > 1 else {}
    return {**extra, "workload": w.name, "b": w.b, "heads": w.h, "head_dim": w.d, "seq_len": w.s,
            "sp_degree": w.N, "heads_per_group": w.h_local, "causal": w.causal,
            "input_scale": w.scale,
            "l2": l2_note(w),
            "flops_convention": "fwd 4*b*h*s^2*d/2 (causal), bwd 2.5x fwd"}


class EventTimer:
    """CUDA events around each library call, recorded on the current (launching) stream."""

    def __init__(self):
        self.enabled = False
        self.pairs = {}

    @contextlib.contextmanager
    def __call__(self, name):
        if not self.enabled:
            yield
            return
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        yield
        b.record()
        self.pairs.setdefault(name, []).append((a, b))

    def mean_ms(self):
        return {n: sum(a.elapsed_time(b) for a, b in ps) / len(ps) for n, ps in self.pairs.items()}

    def per_step_ms(self, steps):
        return {n: sum(a.elapsed_time(b) for a, b in ps) / steps for n, ps in self.pairs.items()}


def merge_bytes_per_step(w, chunks: int) -> int:
    """sp_attn_merge over `chunks` key chunks: every call reads the bf16 partial (2 B per
    element) and writes the fp32 accumulator (4 B); all but the first also read it (4 B);
    the last also writes the bf16 output (2 B); plus 4-byte lse values per row (read the
    partial's, read and write the accumulator's)."""
    elems = w.b * w.s * w.h * w.d
    rows = w.b * w.s * w.h
    per_elem = 6 + 10 * (chunks - 2) + 12 if chunks > 1 else 8
    per_row = 8 + 12 * (chunks - 1)
    return elems * per_elem + rows * per_row


# Workloads measured after the headline in the default run (name, timed steps, graph
# replay too): the other configurations, so that each reports its step rate, roofline
# fraction and relayout rate.  The short ones (sub-millisecond steps of eight launches)
# are also timed replayed from a CUDA graph, where the host's per-call cost shows.
OTHER_WORKLOADS = [("ulysses131k", 3, False), ("llama7b", 20, True), ("padded", 20, True)]


def host_link(host_in, host_out, device, reps: int = 2):
    """Copy rates between the step's page-locked host buffers and the device: each
    direction alone and both at once (the end-to-end step moves both directions while
    its kernels run), timed with CUDA events around plain whole-tensor copies."""
    dev_in = [torch.empty(t.shape, dtype=t.dtype, device=device) for t in host_in]
    dev_out = [torch.empty(t.shape, dtype=t.dtype, device=device) for t in host_out]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    legs = {"h2d": (s_in, list(zip(dev_in, host_in))), "d2h": (s_out, list(zip(host_out, dev_out)))}

    def run(which):
        cur = torch.cuda.current_stream(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        ends = []
        for name in which:
            st, pairs = legs[name]
            st.wait_event(e0)
            with torch.cuda.stream(st):
                for _ in range(reps):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(st)
            ends.append(ev)
        for ev in ends:
            cur.wait_event(ev)
        e1.record(cur)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps

    run(("h2d", "d2h"))   # warm-up
    nbytes = sum(t.numel() * t.element_size() for t in host_in)
    ms = {k: run(v) for k, v in (("h2d", ("h2d",)), ("d2h", ("d2h",)),
                                 ("both", ("h2d", "d2h")))}
    return {"h2d_gbs": nbytes / (ms["h2d"] * 1e-3) / 1e9,
            "d2h_gbs": nbytes / (ms["d2h"] * 1e-3) / 1e9,
            "both_gbs_each_way": nbytes / (ms["both"] * 1e-3) / 1e9,
            "both_ms": ms["both"], "bytes_each_way": nbytes}


def graph_replay_ms(one_step, steps, warmup, device) -> float:
    """The step captured once in a CUDA graph and replayed `steps` times after `warmup`
    replays: CUDA-event milliseconds per step (this rank).  The same launches with the
    same arguments as the eager step, without the host's per-call launch cost."""
    from sequence_head_attention_seq_b300 import sp_get_device_status
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        one_step()                       # settles any first-call setup off the capture
        side.synchronize()
        with torch.cuda.graph(cg, stream=side):
            one_step()
    torch.cuda.current_stream(device).wait_stream(side)
    for _ in range(warmup):
        cg.replay()
    torch.cuda.synchronize()
    barrier()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(steps):
        cg.replay()
    g1.record()
    torch.cuda.synchronize()
    barrier()
    if sp_get_device_status() != 0:
        raise RuntimeError("device status reported an error during graph replay")
    ms = g0.elapsed_time(g1) / steps
    del cg
    return ms


def measure_workload(w, steps, warmup, device, peaks, graph: bool = False):
    """Time `steps` device-resident steps of workload w (after `warmup` untimed ones) with
    CUDA events on the launching stream, and each library call inside them; with
    `graph`, also the same step replayed from a CUDA graph."""
    from sequence_head_attention_seq_b300 import UlyssesAttention, sp_get_device_status
    ins = workloads.make_inputs(w, device=device)
    timer = EventTimer()
    step = UlyssesAttention(w.N, w.b, w.s, w.h, w.d, w.causal, key_len=ins["key_len"],
                            device=device, timer=timer)
    for _ in range(warmup):
        step.forward(ins["q"], ins["k"], ins["v"])
        step.backward(ins["dout"])
    torch.cuda.synchronize()
    # the step rate from a loop without per-call events (on sub-millisecond steps the
    # twelve event records per step would show), then the per-call times from a second,
    # instrumented loop of the same steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step.forward(ins["q"], ins["k"], ins["v"])
        step.backward(ins["dout"])
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    timer.enabled = True
    for _ in range(steps):
        step.forward(ins["q"], ins["k"], ins["v"])
        step.backward(ins["dout"])
    torch.cuda.synchronize()
    timer.enabled = False
    if sp_get_device_status() != 0:
        raise RuntimeError(f"device status reported an error in workload {w.name}")
    per_step = timer.per_step_ms(steps)
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    fwd_f = attn_fwd_flops(w)
    tf = step_flops(w) / (ms * 1e-3) / 1e12
    out = {"steps": steps, "warmup": warmup, "ms_per_step": ms, "tflops": tf,
           "frac_of_burst": tf / burst,
           "attn_fwd_tflops": fwd_f / (per_step["attn_fwd"] * 1e-3) / 1e12,
           "attn_bwd_tflops": 2.5 * fwd_f / (per_step["attn_bwd"] * 1e-3) / 1e12,
           "valid_tflops": 14.0 * w.d * valid_pairs(w, ins["key_len"]) / (ms * 1e-3) / 1e12,
           "config": config_of(w)}
    relayout_ms = sum(per_step.get(n, 0.0) for n in ("seq2head_qkv", "head2seq_o", "seq2head_do",
                                                       "head2seq_grads"))
    if relayout_ms > 0:
        gbs = relayout_bytes_per_step(w) / (relayout_ms * 1e-3) / 1e9
        out["relayout"] = {"gbs": gbs, "frac": gbs / hbm, "ms_per_step": relayout_ms}
    if graph:
        def one_step():
            step.forward(ins["q"], ins["k"], ins["v"])
            step.backward(ins["dout"])
        gms = graph_replay_ms(one_step, steps, warmup, device)
        gtf = step_flops(w) / (gms * 1e-3) / 1e12
        out["graph"] = {"ms_per_step": gms, "tflops": gtf, "frac_of_burst": gtf / burst,
                        "what": "the same step captured once in a CUDA graph and replayed"}
    return out


# a workload whose whole fwd+bwd the oracle finishes in about half a minute or less on the
# host cores (about 0.04 TFLOP/s on 16) is timed in full beside its GPU line
ORACLE_WHOLE_MAX_FLOPS = 1.0e12


def oracle_whole(w, ins):
    """The oracle on the host cores over the whole workload: every head, query row and key
    of forward and backward (the regroupings are not part of it)."""
    import oracle
    orc = oracle.default()

    def plain(t):   # shards [N][b][s/N][h][d] -> [b][s][h][d] (the shards in order)
        return t.permute(1, 0, 2, 3, 4).reshape(w.b, w.s, w.h, w.d).double().cpu().numpy()

    q, k, v, do = (plain(ins[n]) for n in ("q", "k", "v", "dout"))
    kl = None if ins["key_len"] is None else ins["key_len"].tolist()
    t0 = time.perf_counter()
    orc.attn_fwd(q, k, v, w.causal, 0, kl)
    orc.attn_bwd(q, k, v, do, w.causal, 0, kl)
    dt = time.perf_counter() - t0
    return {"value": step_flops(w) / dt / 1e12, "unit": UNIT, "cores": orc.threads(),
            "kind": "oracle",
            "sample": f"fp64 C oracle, fwd+bwd of the whole {w.name} workload (all {w.b * w.h} "
                      f"heads, every row and key; inputs of the same shapes and distributions "
                      f"generated on the host): {step_flops(w) / 1e9:.1f} GFLOP in {dt:.1f} s"}


def measure_other_workloads(warmup, device, peaks, local):
    clocks = ClockSampler(gpu_index_for(local))
    clocks.start()
    res = {}
    try:
        for name, steps, graph in OTHER_WORKLOADS:
            res[name] = measure_workload(workloads.WORKLOADS[name], steps, warmup, device, peaks,
                                         graph)
            torch.cuda.empty_cache()
    finally:
        clocks.stop()
    res["clocks"] = clocks.summary()
    # the oracle after the GPU timing, so that the clock record covers the kernels only
    for name, _, _ in OTHER_WORKLOADS:
        w = workloads.WORKLOADS[name]
        if step_flops(w) <= ORACLE_WHOLE_MAX_FLOPS:
            res[name]["cpu_baseline"] = oracle_whole(w, workloads.make_inputs(w, device="cpu"))
    res["peaks"] = "burst bf16 and HBM copy from " + ("MEASURED_PEAKS.json" if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else "the fallback figures")
    return res


def run_ours(args, w):
    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from sequence_head_attention_seq_b300 import UlyssesAttention, sp_get_device_status

    peaks, peak_kind = load_peaks()
    ins = workloads.make_inputs(w, device=device)
    timer = EventTimer()
    key_len, key_mask = ins["key_len"], None
    if args.key_mask:
        if key_len is None:
            raise SystemExit("--key-mask needs a workload with padded keys")
        # the same right padding, expressed as a general per-key mask
        key_mask = torch.arange(w.s)[None, :] < key_len[:, None]
        key_len = None
    if args.layer:
        # the whole attention layer with synthetic weights (hidden = h * d)
        from sequence_head_attention_seq_b300 import AttentionLayer
        dim = w.h * w.d
        lshape = (w.N, w.b, w.s_local, dim)
        x = workloads.randn_bf16(lshape, w.seed("q"), w.scale, device)
        wqkv = workloads.randn_bf16((3 * w.h * w.d, dim), 1000 * w.index + 5, dim ** -0.5, device)
        wo = workloads.randn_bf16((dim, w.h * w.d), 1000 * w.index + 6, (w.h * w.d) ** -0.5,
                                  device)
        ldout = workloads.randn_bf16(lshape, w.seed("dout"), 1.0, device)
        step = AttentionLayer(w.N, w.b, w.s, w.h, w.d, dim, w.causal, device=device, timer=timer)

        def one_step():
            step.forward(x, wqkv, wo)
            step.backward(ldout)
    else:
        step = UlyssesAttention(w.N, w.b, w.s, w.h, w.d, w.causal, key_len=key_len,
                                device=device, timer=timer, ring_chunks=args.ring,
                                key_mask=key_mask, fused=args.fused)

        def one_step():
            step.forward(ins["q"], ins["k"], ins["v"])
            step.backward(ins["dout"])

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if sp_get_device_status() != 0:
        raise RuntimeError("device status reported an error during warm-up")

    clocks = ClockSampler(gpu_index_for(local))
    clocks.start()
    timer.enabled = True
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.steps):
        one_step()
    end.record()
    torch.cuda.synchronize()
    barrier()
    timer.enabled = False
    clocks.stop()
    local_ms = start.elapsed_time(end)
    calls = timer.mean_ms()
    status = sp_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    total_ms = reduce_max(local_ms, device)
    ms_per_step = total_ms / args.steps
    flops = step_flops(w) + (proj_flops(w) if args.layer else 0.0)
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12

    # the same step captured once in a CUDA graph and replayed (no per-call host launch
    # cost); reported beside the eager number, which stays the headline
    graph = None
    if args.graph:
        gms = reduce_max(graph_replay_ms(one_step, args.steps, args.warmup, device), device)
        graph = {"value": world * flops / (gms * 1e-3) / 1e12, "unit": UNIT,
                 "ms_per_step": gms}

    # end to end through the public API: pinned host buffers in, results back out
    e2e = None
    if not args.no_e2e and not args.layer:
        host_in = {n: ins[n].cpu().pin_memory() for n in ("q", "k", "v", "dout")}
        host_out = [torch.empty(ins["q"].shape, dtype=torch.bfloat16).pin_memory()
                    for _ in range(4)]
        if not args.ring and not args.key_mask:
            # the host-buffer entry point: transfers overlapped with the kernels
            from sequence_head_attention_seq_b300 import UlyssesHostStep
            del step
            torch.cuda.empty_cache()
            host_step = UlyssesHostStep(w.N, w.b, w.s, w.h, w.d, w.causal, key_len=key_len,
                                        device=device)
            e2e_api = "UlyssesHostStep.step (sp_ulysses_step_host)"

            def e2e_step():
                host_step.step(host_in["q"], host_in["k"], host_in["v"], host_in["dout"],
                               *host_out)
        else:
            dev_in = {n: torch.empty_like(ins[n]) for n in host_in}
            e2e_api = "copies + UlyssesAttention.forward/backward"

            def e2e_step():
                for n in host_in:
                    dev_in[n].copy_(host_in[n], non_blocking=True)
                step.forward(dev_in["q"], dev_in["k"], dev_in["v"])
                step.backward(dev_in["dout"])
                for dst, src in zip(host_out, (step.o, step.dq, step.dk, step.dv)):
                    dst.copy_(src, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        e2e_steps = max(1, min(args.steps, 5))
        for _ in range(e2e_steps):
            e2e_step()
        e1.record()
        torch.cuda.synchronize()
        barrier()
        e2e_ms = reduce_max(e0.elapsed_time(e1), device) / e2e_steps
        e2e = {"value": world * step_flops(w) / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": 4 * tensor_bytes(w), "d2h_bytes_per_step": 4 * tensor_bytes(w),
               "ms_per_step": e2e_ms, "api": e2e_api}
        # the end-to-end step can take no less than the longer of the device step and
        # the time the host link needs to move its inputs in and its results out at once
        link = host_link(list(host_in.values()), host_out, device)
        bound = max(link["both_ms"], ms_per_step)
        e2e["link"] = {**link, "bound_ms": bound, "frac_of_bound": bound / e2e_ms,
                       "bound_basis": "max(device step, both directions' copies measured at "
                                      "once on these buffers)"}

    clock_summary = clocks.summary()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    per_step = timer.per_step_ms(args.steps)
    ring = args.ring > 1
    fwd_ms = per_step.get("ring_chunk_fwd" if ring else "attn_fwd")
    bwd_ms = per_step.get("ring_chunk_bwd" if ring else "attn_bwd")
    fwd_f = attn_fwd_flops(w)
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    bwd_tf = 2.5 * fwd_f / (bwd_ms * 1e-3) / 1e12
    plain = not (ring or args.heads is not None or args.key_mask or args.fused or args.layer)
    traffic = recorded_traffic(w.name) if plain else None
    relayout_ms = sum(calls.get(n, 0.0) for n in ("seq2head_qkv", "head2seq_o", "seq2head_do",
                                                    "head2seq_grads"))
    relayout = None
    if relayout_ms > 0:
        gbs = relayout_bytes_per_step(w) / (relayout_ms * 1e-3) / 1e9
        relayout = {"achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "bytes_per_step": relayout_bytes_per_step(w), "ms_per_step": relayout_ms}
    kernels = {}
    ring_info = None
    pairs = valid_pairs(w, ins["key_len"])
    sm_hz = (clock_summary.get("sm_mhz") or 0) * 1e6
    for n, ms in calls.items():
        entry = {"ms": ms}
        if n in ("attn_fwd", "ring_chunk_fwd"):
            entry["ms_per_step"] = per_step[n]
            entry["tflops"] = fwd_f / (per_step[n] * 1e-3) / 1e12
            # exact work: 4*d flops and one exponential per visible (query, key) pair
            entry["valid_tflops"] = 4.0 * w.d * pairs / (per_step[n] * 1e-3) / 1e12
            ex2 = pairs / (per_step[n] * 1e-3)
            entry["ex2"] = {"per_s": ex2, "unit": "exp/s"}
            if sm_hz > 0:
                peak_ex2 = MUFU_EX2_PER_CLK_SM * torch.cuda.get_device_properties(
                    device).multi_processor_count * sm_hz
                entry["ex2"].update({"peak": peak_ex2, "frac": ex2 / peak_ex2,
                                     "peak_basis": "32 lanes/clk/SM x SMs x median SM clock"})
        elif n in ("attn_bwd", "ring_chunk_bwd"):
            entry["ms_per_step"] = per_step[n]
            entry["tflops"] = 2.5 * fwd_f / (per_step[n] * 1e-3) / 1e12
            entry["valid_tflops"] = 10.0 * w.d * pairs / (per_step[n] * 1e-3) / 1e12
        elif n.startswith("proj_"):
            # the tcgen05 GEMMs of the projections (forward: one product; backward: the
            # input and the weight gradient)
            M, dim, hd = w.b * w.s, w.h * w.d, w.h * w.d
            f = 2.0 * M * dim * (3 * hd if "qkv" in n else hd) * (2 if n.endswith("_bwd") else 1)
            entry["tflops"] = f / (ms * 1e-3) / 1e12
            entry["frac_of_burst"] = entry["tflops"] / peak_burst
        elif n == "ring_merge":
            entry["ms_per_step"] = per_step[n]
            nbytes = merge_bytes_per_step(w, args.ring)
            gbs = nbytes / (per_step[n] * 1e-3) / 1e9
            entry["gbs"] = gbs
            ring_info = {"chunks": args.ring,
                         "merge": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                   "frac": gbs / hbm, "bytes_per_step": nbytes,
                                   "ms_per_step": per_step[n]}}
        else:
            tensors = 3 if n in ("seq2head_qkv", "head2seq_grads") else 1
            entry["gbs"] = tensors * 2 * tensor_bytes(w) / (ms * 1e-3) / 1e9
        kernels[n] = entry
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)*scale bf16, shapes of the workload)",
        "config": {**config_of(w, args.ring),
                   **({"key_mask": "right padding given as a general per-key mask"}
                      if args.key_mask else {}),
                   **({"fused_relayout": True} if args.fused else {}),
                   **({"layer": "projections included (hidden = h*d); value = (attention + "
                               "projection flops) / time"} if args.layer else {})},
        "pct_bf16_peak": {"burst": value / peak_burst, "sustained": value / peak_sus,
                          "peaks": peak_kind},
        "roofline": {"kernel": (f"sp_attn_bwd over {args.ring} key chunks (statistics + tcgen05 "
                                "main + dQ convert each)") if ring else
                               "sp_attn_bwd (statistics + tcgen05 main + dQ convert)",
                     # the call lasts tens of milliseconds inside a step well under a
                     # second: the burst peak is its denominator, the sustained one beside it
                     "bound": "tensor", "achieved": bwd_tf, "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": bwd_tf / peak_burst,
                     "peak_kind": f"{peak_kind} burst bf16",
                     "frac_sustained": bwd_tf / peak_sus, "peak_sustained": peak_sus,
                     "traffic": traffic,
                     "algorithmic_flops_per_launch": 2.5 * fwd_f},
        "relayout": relayout,
        "kernels": kernels,
        "ring": ring_info,
        "e2e": e2e,
        **({"graph": graph} if graph is not None else {}),
        "gpu_launches": launches_per_step(w, args.ring, args.fused) * args.steps,
        "clocks": clock_summary,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, ins)
    default_run = not (args.ring or args.layer or args.fused or args.key_mask or args.graph or
                       args.heads is not None) and w.name == DEFAULT_WORKLOAD
    if world == 1 and default_run and not args.no_workloads:
        # free the headline's buffers before the other workloads allocate theirs
        ins = step = host_step = host_in = host_out = None
        torch.cuda.empty_cache()
        line["workloads"] = measure_other_workloads(max(args.warmup, 3), device, peaks, local)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workloads.ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads that the default run times after the headline")
    ap.add_argument("--ring", type=int, default=0,
                    help="run the attention blockwise over this many key chunks (ring attention "
                         "on one GPU: chunked forward + merge, chunked backward)")
    ap.add_argument("--layer", action="store_true",
                    help="the whole attention layer: q/k/v and output projections (hidden = "
                         "h*d, synthetic weights) around the step; value counts their flops too")
    ap.add_argument("--fused", action="store_true",
                    help="attention reads and writes the sequence shards directly (the "
                         "regrouping done by the kernels' addressing, no relayout launches)")
    ap.add_argument("--key-mask", action="store_true",
                    help="give the workload's key padding as a general per-key mask "
                         "(the mask path of the kernels) instead of key lengths")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph and replayed")
    ap.add_argument("--heads", type=int, default=None,
                    help="total heads instead of the workload's (same sequence, head dim and "
                         "shard count; for profiling a smaller case of the same kernels)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    w = workloads.WORKLOADS[args.workload]
    if args.heads is not None:
        if args.heads < w.N or args.heads % w.N:
            ap.error(f"--heads must be a multiple of the shard count {w.N}")
        w = dataclasses.replace(w, h=args.heads)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
