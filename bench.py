#!/usr/bin/env python3
"""Benchmark of the grouped-tril masked softmax (forward + backward) on GB300.

One step = the whole hot path over one batch: gtms_forward (mask, scale,
softmax, zero tail) then gtms_backward on its output, both through the C ABI
on inputs already resident in HBM. The default workload is
X[12,64,1000,1000] fp32 ~N(0,1), seq_len ~ U{500..1000}, scale 1, dY ~N(0,1):
the README's A10 shape, and the largest listed single-GPU workload that runs
both directions at S = 1000.

Throughput is effective bandwidth on the bytes the method must move
(e = element bytes, live(L) = L(L+1)/2 kept entries per (b, m) slice):
  forward  e * sum_{b,m} (live(L_b) + S^2)     kept x read + every y written
  backward e * sum_{b,m} (2 live(L_b) + S^2)   kept y, dy read + every dx written

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gtms|reference]
Under torchrun (N > 1) each rank runs its own replica of the workload (rows are
independent; no collective on the data path) and rank 0 prints one JSON line.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "masked-softmax fwd/bwd effective GB/s & % GB300 HBM peak; ms per [B,M,S,S] call"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "s1000_b12"


# ---------------------------------------------------------------------------
# Byte model
# ---------------------------------------------------------------------------

def kept_per_slice(w, L):
    """Kept elements of one (b, m) slice of length L under the workload's mask family."""
    S = w.S
    L = min(max(int(L), 0), S)
    if w.mask_kind == 1:                 # length mask: c < L on rows r < L
        return L * L
    if w.mask_kind == 2:                 # sliding causal window of width win: min(r + 1, win) on rows r < L
        win = min(max(int(w.window), 1), S)
        full = min(L, win)
        return full * (full + 1) // 2 + (L - full) * win
    return L * (L + 1) // 2              # grouped tril: c <= r < L


def required_bytes(w, lens, kept_total=None):
    """(forward bytes, backward bytes) the method must move for one call each: the kept
    elements read (x; y and dy), every output element written, and for an explicit-mask
    workload its uint8 [B, S, S] mask once (the heads share it; kept_total: the mask's
    kept count over all heads)."""
    S, e = w.S, w.elem_bytes
    live = kept_total if kept_total is not None else w.M * sum(kept_per_slice(w, L) for L in lens)
    dense = w.B * w.M * S * S
    mask = w.B * S * S if w.keep_prob > 0 else 0
    fwd = e * (live + dense) + mask
    bwd = e * (2 * live + dense) + mask if w.backward else 0
    return fwd, bwd


def touched_bytes(w, mask):
    """(forward, backward) bytes that the explicit-mask kernels move at 16-byte granularity: every
    16-byte unit of x (of y and dy) that holds a kept element, the uint8 mask once, every output. With
    scattered keep bits most units hold one, so this exceeds the kept-element count of required_bytes,
    and it is the least any kernel that reads whole units can move."""
    import torch

    epu = 16 // w.elem_bytes
    units = int(torch.count_nonzero(mask.view(w.B, w.S, w.S // epu, epu).amax(dim=-1)).item()) * w.M
    dense = w.B * w.M * w.S * w.S * w.elem_bytes
    mask_bytes = w.B * w.S * w.S
    return 16 * units + mask_bytes + dense, 32 * units + mask_bytes + dense


def entry_points(lib, w):
    """The C calls of one step of workload w: fwd(x, y, lens, mask, stream) and
    bwd(y, dy, dx, lens, mask, stream) (pointers as ints; mask used by explicit-mask
    workloads only), with the names of the entry points."""
    B, M, S, code, scale = w.B, w.M, w.S, w.dtype_code, float(w.scale)
    if w.keep_prob > 0:
        return (lambda x, y, lp, mp, sp: lib.gtms_forward_explicit(x, y, mp, B, B, M, S, scale, code, sp),
                lambda y, g, d, lp, mp, sp: lib.gtms_backward_explicit(y, g, d, mp, B, B, M, S, scale, code, sp),
                "gtms_forward_explicit", "gtms_backward_explicit")
    if w.mask_kind:
        k, win = w.mask_kind, w.window
        return (lambda x, y, lp, mp, sp: lib.gtms_forward_masked(x, y, lp, B, M, S, scale, k, win, code, sp),
                lambda y, g, d, lp, mp, sp: lib.gtms_backward_masked(y, g, d, lp, B, M, S, scale, k, win, code, sp),
                "gtms_forward_masked", "gtms_backward_masked")
    return (lambda x, y, lp, mp, sp: lib.gtms_forward(x, y, lp, B, M, S, scale, code, sp),
            lambda y, g, d, lp, mp, sp: lib.gtms_backward(y, g, d, lp, B, M, S, scale, code, sp),
            "gtms_forward", "gtms_backward")


def kernel_label(gtms, w, direction):
    """Name of the kernel a call of workload w launches (same variant table for every mask)."""
    if w.keep_prob > 0:
        return gtms.kernel_name_explicit(direction, w.S, w.dtype_code)
    return gtms.kernel_name_masked(direction, w.S, w.dtype_code, w.mask_kind, w.window)


# ---------------------------------------------------------------------------
# Peaks, traffic records, clocks
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        v = peaks.get("hbm_gbs")
        if isinstance(v, dict):
            v = v.get("value", v.get("burst"))
        if isinstance(v, (int, float)) and v > 0:
            return float(v), "measured"
    except (OSError, ValueError, AttributeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# Source files each kernel family is compiled from (csrc/), for the source hash that keys the
# recorded DRAM traffic: a record stays valid while these files are unchanged.
_COMMON_SOURCES = ("gtms_kernels.cuh", "gtms_dispatch.h", "gtms_launch.cuh")
_FAMILY_SOURCES = (
    ("gtms_attn", ("gtms_kernels.cuh", "gtms_tcgen05.cuh", "gtms_attn_bwd.cuh", "gtms_attn_tma.cuh",
                   "gtms_attn_bwd.cu", "gtms_attn_tma.cu")),
    ("gtms_fwd_explicit", _COMMON_SOURCES + ("gtms_explicit.cuh",)),
    ("gtms_bwd_explicit", _COMMON_SOURCES + ("gtms_explicit.cuh",)),
    ("gtms_fwd_stream", _COMMON_SOURCES + ("gtms_stream.cuh",)),
    ("gtms_bwd_stream", _COMMON_SOURCES + ("gtms_stream.cuh",)),
    ("gtms_fwd_band", _COMMON_SOURCES + ("gtms_band.cuh",)),
    ("gtms_bwd_band", _COMMON_SOURCES + ("gtms_band.cuh",)),
    ("gtms_fwd_staged", _COMMON_SOURCES + ("gtms_staged.cuh", "gtms_tcgen05.cuh")),
)


def kernel_sources(kernel):
    """The csrc files a kernel (by its reported name) is compiled from."""
    for prefix, files in _FAMILY_SOURCES:
        if kernel.startswith(prefix):
            return files
    return _COMMON_SOURCES   # per-row vector, heads and element kernels


def kernel_source_sha(kernel=""):
    """Hash of the sources a kernel is compiled from (kernel_sources)."""
    h = hashlib.sha256()
    for name in sorted(kernel_sources(kernel)):
        p = os.path.join(ROOT, "masked_softmax_attention_gb300", "csrc", name)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none or the kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha(kernel)
    with open(path) as f:
        for line in f:
            if not line.startswith("traffic "):
                continue
            kv = dict(tok.split("=", 1) for tok in line.split()[1:] if "=" in tok)
            if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("source_sha") == sha:
                return int(float(kv["dram_bytes_per_launch"]))
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in a thread."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.error = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as exc:
            self.error = f"nvidia-smi unavailable: {exc}"
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.error:
            return {"error": self.error}
        rows = []
        for t, line in self.samples:
            if t0 <= t <= t1:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 7:
                    rows.append(parts)
        if not rows:
            return {"error": "no nvidia-smi sample inside the timed region"}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------

def oracle_sample(w, lens, slices, device="cpu"):
    """Inputs of `slices` (b, m) slices of workload w, as raw bits, drawn on the CPU."""
    import numpy as np

    import seeded_inputs as si

    picked = [b for b, _ in slices]
    ws = si.Workload(w.name + "_sample", len(picked), 1, w.S, w.dtype, w.scale, x_std=w.x_std,
                     fixed_seq_lens=tuple(int(lens[b]) for b in picked), spike_prob=w.spike_prob,
                     spike_value=w.spike_value, backward=w.backward, seed=w.seed + 7, head_dim=w.head_dim,
                     mask_kind=w.mask_kind, window=w.window, keep_prob=w.keep_prob)
    bits_t = {"f32": (np.uint32, "int32"), "bf16": (np.uint16, "int16"), "f16": (np.uint16, "int16")}[w.dtype]
    import torch

    tview = getattr(torch, bits_t[1])

    def bits(t):
        return t.view(tview).numpy().view(bits_t[0])

    xb = bits(si.make_x(ws, device))
    if ws.head_dim > 0:
        # attention-backward sample: P is the oracle's own (rounded) softmax of x; dO and V as drawn
        import oracle

        lens_s = np.array(ws.fixed_seq_lens, dtype=np.int32)
        pb = oracle.round_to(oracle.forward(xb, lens_s, ws.B, ws.M, ws.S, ws.scale, ws.dtype_code,
                                            threads=os.cpu_count() or 1), ws.dtype_code)
        dout, v = si.make_head_operands(ws, device)
        return ws, pb, (bits(dout), bits(v))
    if ws.keep_prob > 0:   # explicit-mask sample: dy and the sample's own seeded keep mask
        return ws, xb, (bits(si.make_dy(ws, device)), si.make_keep_mask(ws, device).numpy())
    return ws, xb, bits(si.make_dy(ws, device))


def sample_bytes(ws, dyb):
    """Algorithmic bytes of one oracle step over a sample from oracle_sample."""
    kept = int((dyb[1] != 0).sum()) * ws.M if ws.keep_prob > 0 else None
    return step_bytes(ws, ws.fixed_seq_lens, kept)


def step_bytes(w, lens, kept_total=None):
    """Algorithmic bytes of one step: the softmax forward + backward, or for an
    attention-backward workload the kept P read, every dS written, dO and V read."""
    fb, bb = required_bytes(w, lens, kept_total)
    if w.head_dim > 0:
        return fb + 2 * w.B * w.M * w.S * w.head_dim * w.elem_bytes
    return fb + bb


def oracle_step(ws, xb, dyb, threads):
    """One oracle pass over the sample: forward, round, backward, round (all rows); for an
    attention-backward sample, the dS step from (P, dO, V) and its rounding. With several
    threads the rows are cut into chunks and each thread runs the whole pass (rounding
    included) over its chunks, so no step runs on one core while the others wait."""
    import concurrent.futures as cf

    import numpy as np

    import oracle

    lens = np.array(ws.fixed_seq_lens, dtype=np.int32)
    B, M, S, code = ws.B, ws.M, ws.S, ws.dtype_code
    rows = B * M * S
    x_rows = xb.reshape(-1)

    def run(chunk):
        r0, r1 = chunk
        xs = x_rows[r0 * S:r1 * S]
        if ws.head_dim > 0:
            dout, v = dyb
            oracle.round_to(oracle.attn_dscores(xs, dout, v, lens, B, M, S, ws.head_dim, ws.scale, code,
                                                row_begin=r0, row_end=r1), code)
            return
        if ws.keep_prob > 0:
            dy, mask = dyb
            yb = oracle.round_to(oracle.forward_explicit(xs, mask, B, M, S, ws.scale, code, row_begin=r0,
                                                         row_end=r1), code)
            if ws.backward:
                oracle.round_to(oracle.backward_explicit(yb, dy.reshape(-1)[r0 * S:r1 * S], mask, B, M, S,
                                                         ws.scale, code, row_begin=r0, row_end=r1), code)
            return
        kw = dict(row_begin=r0, row_end=r1, mask_kind=ws.mask_kind, window=ws.window)
        yb = oracle.round_to(oracle.forward(xs, lens, B, M, S, ws.scale, code, **kw), code)
        if ws.backward:
            oracle.round_to(oracle.backward(yb, dyb.reshape(-1)[r0 * S:r1 * S], lens, B, M, S, ws.scale, code,
                                            **kw), code)

    if threads <= 1:
        run((0, rows))
        return
    step = -(-rows // (4 * threads))
    chunks = [(r, min(r + step, rows)) for r in range(0, rows, step)]
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, chunks))


def cpu_model():
    """The host CPU's model name (Linux /proc/cpuinfo; Arm hosts report no name, so the part number)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return None
    arm_parts = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd8e": "Arm Neoverse-N3"}
    for key in ("model name", "Model Name", "CPU part"):
        for line in info.splitlines():
            if line.startswith(key):
                v = line.split(":", 1)[1].strip()
                return f"{arm_parts[v]} (CPU part {v})" if v in arm_parts else v
    return None


def cpu_baseline(w, lens, budget_s=12.0):
    """The oracle as it stands, on the host cores, over a bounded sample of the
    workload: groups of (b, m) slices until about budget_s of wall time, on all
    cores; then one group on a single thread."""
    threads = os.cpu_count() or 1
    group = max(1, min(16, w.B * w.M))
    done_slices, total_bytes, total_s, groups = 0, 0, 0.0, 0
    while total_s < budget_s and done_slices < w.B * w.M:
        slices = [((done_slices + i) % w.B, 0) for i in range(group)]
        ws, xb, dyb = oracle_sample(w, lens, slices)
        t0 = time.perf_counter()
        oracle_step(ws, xb, dyb, threads)
        total_s += time.perf_counter() - t0
        total_bytes += sample_bytes(ws, dyb)
        done_slices += group
        groups += 1
    ws, xb, dyb = oracle_sample(w, lens, [(b % w.B, 0) for b in range(min(4, w.B * w.M))])
    t0 = time.perf_counter()
    oracle_step(ws, xb, dyb, 1)
    single = sample_bytes(ws, dyb) / (time.perf_counter() - t0) / 1e9
    return {"value": round(total_bytes / total_s / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "value_1_thread": round(single, 4), "cpu_model": cpu_model(),
            "sample": f"{done_slices} (b,m) slices of {w.name} (S={w.S}, the workload's seq_lens and value "
                      f"distribution, drawn on the CPU) in {groups} groups: {oracle_step_name(w)}, "
                      f"{total_s:.2f} s wall on {threads} threads"}


def oracle_step_name(w):
    return "oracle dS step from (P, dO, V) + round" if w.head_dim > 0 else "oracle forward + round + backward"


def full_kept_total(w):
    """Kept entries of the whole workload's explicit keep mask, over all heads (None for mask families)."""
    if w.keep_prob <= 0:
        return None
    import torch

    import seeded_inputs as si

    return int(torch.count_nonzero(si.make_keep_mask(w, "cpu")).item()) * w.M


def run_reference(args, w, lens):
    """The oracle as the reference arm: K timed steps of a bounded sample each."""
    import numpy as np  # noqa: F401

    threads = os.cpu_count() or 1
    ws, xb, dyb = oracle_sample(w, lens, [(0, 0)])
    for _ in range(args.warmup):
        oracle_step(ws, xb, dyb, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(ws, xb, dyb, threads)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = sample_bytes(ws, dyb) / dt / 1e9
    sample = (f"1 (b,m) slice of {w.name} per step (S={w.S}, seq_len={ws.fixed_seq_lens[0]}, drawn on the "
              f"CPU): {oracle_step_name(w)}")
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": workload_config(w, lens, full_kept_total(w)),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Multi-rank logic (one process per GPU; rows are independent, so each rank
# runs its own replica of the workload and only the step time is reduced)
# ---------------------------------------------------------------------------

def replica_workload(w, rank):
    """Rank r's replica: same shape and distribution, seed offset by rank."""
    import dataclasses

    return w if rank == 0 else dataclasses.replace(w, seed=w.seed + 1000 * rank)


def shard_slices(n_slices, rank, world):
    """Contiguous range [s0, s1) of the B*M (batch, head) slices that rank `rank` of `world`
    runs when one workload is split over the ranks (sizes differ by at most one)."""
    base, extra = divmod(n_slices, world)
    s0 = rank * base + min(rank, extra)
    return s0, s0 + base + (1 if rank < extra else 0)


def shard_workload(w, lens, rank, world):
    """Rank r's part of one workload split over `world` ranks: its range of (b, m) slices
    as a [slices, 1, S, S] workload whose per-slice length is the slice's batch length
    (the heads of a batch share it). Values come from the rank's own seeded draw with the
    workload's distribution; the lengths, and so the bytes, are exactly the workload's."""
    import dataclasses

    s0, s1 = shard_slices(w.B * w.M, rank, world)
    shard_lens = tuple(int(lens[s // w.M]) for s in range(s0, s1))
    return dataclasses.replace(w, name=f"{w.name}_shard{rank}of{world}", B=s1 - s0, M=1, fixed_seq_lens=shard_lens,
                               seq_len_range=None, seed=w.seed + 1000 * rank)


def max_over_ranks(value, dist, device):
    """Largest per-rank value (the step time of the slowest rank)."""
    import torch

    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, dist, device):
    """Total over ranks (each rank's replica has its own seeded lengths, so its own byte count)."""
    import torch

    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_gbs(total_bytes, ms_step):
    """Bytes moved by all ranks in one step over the slowest rank's step time."""
    return total_bytes / (ms_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def workload_config(w, lens, kept_total=None):
    fb, bb = required_bytes(w, lens, kept_total)
    return {"workload": w.name + ": " + w.describe(), "B": w.B, "M": w.M, "S": w.S, "dtype": w.dtype,
            "scale": w.scale, "seq_lens_seeded": [int(v) for v in lens] if len(lens) <= 16 else "see seed",
            "seed": w.seed, **({"head_dim": w.head_dim, "required_bytes_step": step_bytes(w, lens)}
                               if w.head_dim > 0 else {"required_bytes_fwd": fb, "required_bytes_bwd": bb}),
            "l2": "no flush: " + ("P and dS are" if w.head_dim > 0 else "x, y, dy, dx are each")
                  + " larger than the 129 MB L2",
            "parallelism": "one replica per GPU (rows independent, no collective)"}


def run_gpu_attention(args, w, lens, rank, world, local_rank):
    """The attention-backward step dS = scale * P * (dO V^T - rowsum(dO V^T * P)) (one fused launch).
    Algorithmic bytes per (b, m) slice: kept P read once, every dS written, dO and V read once."""
    import torch

    import masked_softmax_attention_gb300 as gtms
    import seeded_inputs as si

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    wr = replica_workload(w, rank)
    lens_r = si.seq_lens(wr)
    lens_d = torch.from_numpy(lens_r).to(dev)
    p = gtms.forward(si.make_x(wr, dev), lens_d, wr.scale)
    dout, v = si.make_head_operands(wr, dev)
    ds = torch.empty_like(p)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fn = gtms.load_library().gtms_attention_softmax_backward
    args_c = (p.data_ptr(), dout.data_ptr(), v.data_ptr(), ds.data_ptr(), lens_d.data_ptr(), wr.B, wr.M, wr.S,
              wr.head_dim, float(wr.scale), wr.dtype_code, status.data_ptr(), stream.cuda_stream)
    for _ in range(args.warmup):
        if fn(*args_c):
            raise RuntimeError("gtms_attention_softmax_backward failed")
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    s_ev.record(stream)
    rc = 0
    for a, b in ev:
        a.record(stream)
        rc |= fn(*args_c)
        b.record(stream)
    e_ev.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if rc or int(status.item()):
        raise RuntimeError("gtms_attention_softmax_backward failed or timed out inside the timed region")
    ms = max_over_ranks(s_ev.elapsed_time(e_ev) / args.steps, dist, dev)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    fb, _ = required_bytes(wr, lens_r)                    # kept P read + every dS written
    nbytes = fb + 2 * wr.B * wr.M * wr.S * wr.head_dim * wr.elem_bytes
    value = whole_job_gbs(sum_over_ranks(nbytes, dist, dev), ms)
    peak, peak_kind = hbm_peak()
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    e2e = None
    if rank == 0 and args.e2e_steps > 0:
        del ds
        torch.cuda.empty_cache()
        e2e = run_e2e_attention_host_resident(args, wr, lens_r, p, dout, v, stream, fn)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, lens)
    if rank == 0:
        kname = f"gtms_attn_dscores_tma_kernel<{wr.dtype},d{wr.head_dim}>"   # device operands take the TMA kernel
        gbs = nbytes / (ms * 1e-3) / 1e9
        print(json.dumps({
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "ms_per_step_median": round(statistics.median(step_ms), 5), "ms_per_step_min": round(min(step_ms), 5),
            "config": {**workload_config(w, lens),
                       "step": "gtms_attention_softmax_backward (dP = dO V^T on tcgen05, fused softmax backward)"},
            "kernels": {"attention_softmax_backward": {"kernel": kname, "ms_per_call": round(ms, 5),
                                                       "required_bytes": nbytes, "achieved_gbs": round(gbs, 2),
                                                       "frac_of_peak": round(gbs / peak, 4)}},
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": recorded_traffic(kname, wr.name),
                         "peak_source": f"{peak_kind} ({'MEASURED_PEAKS.json hbm_gbs' if peak_kind == 'measured' else 'recipe fallback 6.8 TB/s'})",
                         "algorithmic_bytes_per_launch": nbytes},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": clocks, "impl": "gtms"}), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e_attention_host_resident(args, w, lens, p, dout, v, stream, fn):
    """The attention-backward step through the C ABI with P, dO, V and dS in
    pinned host memory, read and written by the kernel over the host link."""
    import torch

    import masked_softmax_attention_gb300 as gtms

    try:
        p_h = torch.empty(p.shape, dtype=p.dtype, pin_memory=True)
        ds_h = torch.empty(p.shape, dtype=p.dtype, pin_memory=True)
        do_h = torch.empty(dout.shape, dtype=dout.dtype, pin_memory=True)
        v_h = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    except RuntimeError as exc:
        return {"error": f"pinned host buffers unavailable: {exc}"}
    p_h.copy_(p)
    do_h.copy_(dout)
    v_h.copy_(v)
    lens_h = torch.from_numpy(lens).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=p.device)
    torch.cuda.synchronize()
    dp = gtms.device_pointer_of_host
    args_c = (dp(p_h.data_ptr()), dp(do_h.data_ptr()), dp(v_h.data_ptr()), dp(ds_h.data_ptr()),
              dp(lens_h.data_ptr()), w.B, w.M, w.S, w.head_dim, float(w.scale), w.dtype_code, status.data_ptr(),
              stream.cuda_stream)
    if fn(*args_c):
        raise RuntimeError("gtms_attention_softmax_backward failed in the end-to-end loop")
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    rc = 0
    for _ in range(args.e2e_steps):
        rc |= fn(*args_c)
    e.record(stream)
    torch.cuda.synchronize()
    if rc or int(status.item()):
        raise RuntimeError("gtms_attention_softmax_backward failed in the end-to-end loop")
    ms = s.elapsed_time(e) / args.e2e_steps
    fb, _ = required_bytes(w, lens)
    dense = w.B * w.M * w.S * w.S * w.elem_bytes
    heads = 2 * w.B * w.M * w.S * w.head_dim * w.elem_bytes
    return {"value": round((fb + heads) / (ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": fb - dense + heads + 4 * w.B, "d2h_bytes_per_step": dense,
            "steps": args.e2e_steps,
            "host_buffers": "pinned, mapped; the kernel reads kept P, dO, V from and writes dS to host memory "
                            "over NVLink-C2C (no staging copy); host operands take the cp.async kernel "
                            f"gtms_attn_dscores_kernel<{w.dtype},d{w.head_dim}>"}


# Workloads timed one after another beside the headline step (rank 0 of a one-GPU
# run): every listed configuration besides the headline one, the S = 4096 point,
# the long rows, the other mask families, the explicit mask and the attention step.
CONFIG_TABLE = ("worked_example", "s1000_b3", "s2048_bf16", "s8192_f16", "s4096_bf16", "s16384_bf16",
                "s32768_bf16", "s65536_bf16", "s65536_f32", "length_s2048_bf16", "window_s2048_bf16",
                "explicit_s2048_bf16", "attn_s2048_bf16", "attn_d128_s2048_f16")
L2_BYTES = 129 * 1000 * 1000


def time_config(args, name, dev, stream, peak):
    """Per-call CUDA-event timings of one workload through the C ABI: W untimed calls,
    then K timed calls of the forward, then of the backward (or of the attention step),
    inputs resident in HBM. Workloads whose tensors do not exceed L2 get an L2 flush
    (a write of twice its size) before every timed call, outside the timed events.
    Returns (entry, [(t0, t1) host windows of the timed loops])."""
    import torch

    import masked_softmax_attention_gb300 as gtms
    import seeded_inputs as si

    w = si.WORKLOADS[name]
    lens = si.seq_lens(w)
    lens_d = torch.from_numpy(lens).to(dev)
    lib = gtms.load_library()
    sp = stream.cuda_stream
    keep = [lens_d]
    calls = []
    status = None
    if w.head_dim > 0:
        p = gtms.forward(si.make_x(w, dev), lens_d, w.scale)
        dout, v = si.make_head_operands(w, dev)
        ds = torch.empty_like(p)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        fn = lib.gtms_attention_softmax_backward
        ca = (p.data_ptr(), dout.data_ptr(), v.data_ptr(), ds.data_ptr(), lens_d.data_ptr(), w.B, w.M, w.S,
              w.head_dim, float(w.scale), w.dtype_code, status.data_ptr(), sp)
        keep += [p, dout, v, ds, status]
        calls.append(("attention_softmax_backward", lambda: fn(*ca), step_bytes(w, lens),
                      f"gtms_attn_dscores_tma_kernel<{w.dtype},d{w.head_dim}>"))
        tensor_bytes = p.numel() * p.element_size()
    else:
        x = si.make_x(w, dev)
        y = torch.empty_like(x)
        mask = si.make_keep_mask(w, dev) if w.keep_prob > 0 else None
        kept_total = int(torch.count_nonzero(mask).item()) * w.M if mask is not None else None
        fwd_c, bwd_c, _, _ = entry_points(lib, w)
        fb, bb = required_bytes(w, lens, kept_total)
        xp, yp, lp = x.data_ptr(), y.data_ptr(), lens_d.data_ptr()
        mp = mask.data_ptr() if mask is not None else None
        keep += [x, y, mask]
        calls.append(("forward", lambda: fwd_c(xp, yp, lp, mp, sp), fb, kernel_label(gtms, w, 0)))
        staged = gtms.kernel_name(2, w.S, w.dtype_code)
        if mask is None and not w.mask_kind and staged != "none":
            # the same forward by the staged kernel (rows brought into shared memory by TMA bulk copies)
            calls.append(("forward_staged", lambda: lib.gtms_forward_staged(xp, yp, lp, w.B, w.M, w.S, float(w.scale),
                                                                            w.dtype_code, sp), fb, staged))
        if w.backward:
            dy = si.make_dy(w, dev)
            dx = torch.empty_like(x)
            dyp, dxp = dy.data_ptr(), dx.data_ptr()
            keep += [dy, dx]
            calls.append(("backward", lambda: bwd_c(yp, dyp, dxp, lp, mp, sp), bb, kernel_label(gtms, w, 1)))
        tensor_bytes = x.numel() * x.element_size()
    flush = None
    if tensor_bytes <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    entry = {"workload": w.name + ": " + w.describe()}
    touched = touched_bytes(w, mask) if w.head_dim == 0 and w.keep_prob > 0 else None
    windows = []
    for label, call, nbytes, kname in calls:
        for _ in range(args.warmup):
            if call():
                raise RuntimeError(f"{name} {label}: libgtms call failed")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        torch.cuda.synchronize()
        t0 = time.time()
        rc = 0
        with torch.cuda.stream(stream):
            for a, b in ev:
                if flush is not None:
                    flush.zero_()
                a.record(stream)
                rc |= call()
                b.record(stream)
        torch.cuda.synchronize()
        windows.append((t0, time.time()))
        if rc:
            raise RuntimeError(f"{name} {label}: libgtms call failed inside the timed loop")
        ms = [a.elapsed_time(b) for a, b in ev]
        mean = statistics.fmean(ms)
        gbs = nbytes / (mean * 1e-3) / 1e9
        entry[label] = {"kernel": kname, "ms_per_call": round(mean, 5),
                        "ms_median": round(statistics.median(ms), 5), "ms_min": round(min(ms), 5),
                        "required_bytes": nbytes, "achieved_gbs": round(gbs, 2),
                        "frac_of_peak": round(gbs / peak, 4)}
        if flush is not None:
            entry[label]["l2"] = "flushed before every timed call (tensors smaller than L2); latency only"
        if touched is not None:   # the same time on the bytes of whole 16-byte units touched
            tb = touched[0 if label == "forward" else 1]
            entry[label]["touched_bytes"] = tb
            entry[label]["frac_of_peak_touched"] = round(tb / (statistics.fmean(ms) * 1e-3) / 1e9 / peak, 4)
    if status is not None and int(status.item()):
        raise RuntimeError(f"{name}: a bounded wait inside the attention kernel ran out")
    del keep, calls, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry, windows


def time_configs(args, dev, stream, peak, sampler):
    """The CONFIG_TABLE workloads (or --configs), one after another, buffers freed between them."""
    names = CONFIG_TABLE if args.configs is None else [n for n in args.configs.split(",") if n]
    out, windows = {}, []
    for name in names:
        entry, win = time_config(args, name, dev, stream, peak)
        out[name] = entry
        windows += win
    if sampler is not None and windows:
        out["clocks"] = sampler.summary(min(t for t, _ in windows), max(t for _, t in windows))
    out["timing"] = (f"CUDA events around each call on the launching stream; {args.warmup} untimed then "
                     f"{args.steps} timed calls per direction; ms_per_call is the mean")
    return out


def run_gpu(args, w, lens, rank, world, local_rank):
    import torch

    import masked_softmax_attention_gb300 as gtms
    import seeded_inputs as si

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    gtms.load_library()
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    if args.split and (w.keep_prob > 0 or w.head_dim > 0):
        raise SystemExit("--split serves the mask-family workloads (seq_lens masks) only")
    wr = shard_workload(w, lens, rank, world) if args.split else replica_workload(w, rank)
    lens_r = si.seq_lens(wr)
    x = si.make_x(wr, dev)
    dy = si.make_dy(wr, dev)
    lens_d = torch.from_numpy(lens_r).to(dev)
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    S, code = wr.S, wr.dtype_code
    mask = si.make_keep_mask(wr, dev) if wr.keep_prob > 0 else None
    kept_total = int(torch.count_nonzero(mask).item()) * wr.M if mask is not None else None
    xp, yp, dyp, dxp, lp = x.data_ptr(), y.data_ptr(), dy.data_ptr(), dx.data_ptr(), lens_d.data_ptr()
    mp = mask.data_ptr() if mask is not None else None
    fwd_c, bwd_c, fwd_name, bwd_name = entry_points(gtms.load_library(), wr)

    def step():
        rc = fwd_c(xp, yp, lp, mp, sp)
        if rc:
            raise gtms.GtmsError(fwd_name, rc)
        if wr.backward:
            rc = bwd_c(yp, dyp, dxp, lp, mp, sp)
            if rc:
                raise gtms.GtmsError(bwd_name, rc)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    start.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        rc = fwd_c(xp, yp, lp, mp, sp)
        ev[k][1].record(stream)
        if wr.backward:
            rc |= bwd_c(yp, dyp, dxp, lp, mp, sp)
        ev[k][2].record(stream)
        if rc:
            raise RuntimeError("libgtms call failed inside the timed region")
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    if dist is not None:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    fwd_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev) if wr.backward else 0.0
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    ms_step = max_over_ranks(total_ms / K, dist, dev)
    clocks = sampler.summary(t_host0, t_host1) if sampler else None

    fb, bb = required_bytes(wr, lens_r, kept_total)
    value = whole_job_gbs(sum_over_ranks(fb + bb, dist, dev), ms_step)

    peak, peak_kind = hbm_peak()
    kern = {}
    for name, nbytes, ms, direction in (("forward", fb, fwd_ms, 0), ("backward", bb, bwd_ms, 1)):
        if nbytes == 0:
            continue
        kname = kernel_label(gtms, wr, direction)
        gbs = nbytes / (ms * 1e-3) / 1e9
        kern[name] = {"kernel": kname, "ms_per_call": round(ms, 5), "required_bytes": nbytes,
                      "achieved_gbs": round(gbs, 2), "frac_of_peak": round(gbs / peak, 4)}
    dom = max(kern, key=lambda k: kern[k]["ms_per_call"])
    dk = kern[dom]
    traffic = recorded_traffic(dk["kernel"], wr.name)
    roofline = {"bound": "hbm", "kernel": dk["kernel"], "achieved": dk["achieved_gbs"], "peak": peak,
                "unit": "GB/s", "frac": dk["frac_of_peak"], "traffic": traffic,
                "peak_source": f"{peak_kind} ({'MEASURED_PEAKS.json hbm_gbs' if peak_kind == 'measured' else 'recipe fallback 6.8 TB/s'})",
                "algorithmic_bytes_per_launch": dk["required_bytes"]}

    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        configs = time_configs(args, dev, stream, peak, sampler)

    e2e = e2e_staged = None
    if args.e2e_steps > 0:
        e2e = run_e2e_host_resident(args, wr, lens_r, dev, stream, fwd_c, bwd_c, mask, kept_total)
        if mask is None and not wr.mask_kind:   # the staged pipeline serves the default op
            e2e_staged = run_e2e(args, wr, lens_r, dev, stream)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, lens)
    if sampler:
        sampler.stop()

    if rank == 0:
        config = workload_config(w, lens, kept_total) if args.split else workload_config(wr, lens_r, kept_total)
        if args.split:
            config["parallelism"] = (f"one workload split over {world} GPU(s): rank r runs a contiguous range of "
                                     "the B*M (batch, head) slices, no collective on the data path")
        line = {"metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
                "scaling": "strong" if args.split else "weak", "vs_baseline": None, "dtype": w.dtype,
                "data": "synthetic", "config": config, "pct_hbm_peak": round(100 * (value / world) / peak, 2),
                "ms_per_step_median": round(statistics.median(step_ms), 5), "ms_per_step_min": round(min(step_ms), 5),
                "kernels": kern, "roofline": roofline, "configs": configs, "cpu_baseline": cpu, "e2e": e2e,
                "e2e_staged": e2e_staged,
                "gpu_launches": K * (2 if wr.backward else 1), "clocks": clocks,
                "impl": "gtms"}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e_host_resident(args, w, lens, dev, stream, fwd_c, bwd_c, mask=None, kept_total=None):
    """The step through the C ABI with every tensor in pinned host memory: the
    kernels read the kept inputs from, and write every output to, host memory
    over the host link (gtms_device_pointer_of_host), no staging copy. An
    explicit keep mask (`mask`, on the device) is copied to pinned memory too."""
    import torch

    import masked_softmax_attention_gb300 as gtms
    import seeded_inputs as si

    try:
        x_h = torch.empty((w.B, w.M, w.S, w.S), dtype=w.torch_dtype, pin_memory=True)
        y_h = torch.empty_like(x_h, pin_memory=True)
        dy_h = torch.empty_like(x_h, pin_memory=True) if w.backward else None
        dx_h = torch.empty_like(x_h, pin_memory=True) if w.backward else None
    except RuntimeError as exc:
        return {"error": f"pinned host buffers unavailable: {exc}"}
    x_h.copy_(si.make_x(w, dev))
    if w.backward:
        dy_h.copy_(si.make_dy(w, dev))
    lens_h = torch.from_numpy(lens).pin_memory()
    mask_h = mask.cpu().pin_memory() if mask is not None else None
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    dp = gtms.device_pointer_of_host
    xp, yp, lp = dp(x_h.data_ptr()), dp(y_h.data_ptr()), dp(lens_h.data_ptr())
    dyp = dp(dy_h.data_ptr()) if w.backward else None
    dxp = dp(dx_h.data_ptr()) if w.backward else None
    mp = dp(mask_h.data_ptr()) if mask_h is not None else None
    sp = stream.cuda_stream

    def step():
        rc = fwd_c(xp, yp, lp, mp, sp)
        if w.backward:
            rc |= bwd_c(yp, dyp, dxp, lp, mp, sp)
        if rc:
            raise RuntimeError("libgtms call failed in the end-to-end loop")

    step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(args.e2e_steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.e2e_steps
    fb, bb = required_bytes(w, lens, kept_total)
    dense = w.B * w.M * w.S * w.S * w.elem_bytes
    mask_reads = w.B * w.M * w.S * w.S if mask is not None else 0   # each row reads its mask row over the link
    kept = fb - dense - (w.B * w.S * w.S if mask is not None else 0)   # kept bytes of one tensor
    h2d = kept + (2 * kept if w.backward else 0) + 4 * w.B + mask_reads * (2 if w.backward else 1)
    d2h = dense * (2 if w.backward else 1)
    return {"value": round((fb + bb) / (ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "host_buffers": "pinned, mapped; kernels read kept x, y, dy from and write y, dx to host memory "
                            "over NVLink-C2C (no staging copy)"}


def run_e2e(args, w, lens, dev, stream):
    """Same step through the public host-buffer API: inputs in pinned host
    memory, H2D of x, dy, seq_lens and D2H of y, dx inside the timed region
    (chunks of batches pipelined over three streams)."""
    import torch

    import seeded_inputs as si
    from masked_softmax_attention_gb300.pipeline import HostPipeline

    try:
        x_h = torch.empty((w.B, w.M, w.S, w.S), dtype=w.torch_dtype, pin_memory=True)
        y_h = torch.empty_like(x_h, pin_memory=True)
        dy_h = torch.empty_like(x_h, pin_memory=True) if w.backward else None
        dx_h = torch.empty_like(x_h, pin_memory=True) if w.backward else None
    except RuntimeError as exc:
        return {"error": f"pinned host buffers unavailable: {exc}"}
    x_h.copy_(si.make_x(w, dev))
    if w.backward:
        dy_h.copy_(si.make_dy(w, dev))
    lens_h = torch.from_numpy(lens).pin_memory()
    torch.cuda.empty_cache()
    pipe = HostPipeline(w.B, w.M, w.S, w.torch_dtype, dev, chunk_batches=args.e2e_chunk, depth=2,
                        backward=w.backward)

    def step():
        pipe.run(x_h, lens_h, w.scale, y_h, dy_h, dx_h)

    step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(args.e2e_steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.e2e_steps
    fb, bb = required_bytes(w, lens)
    h2d, d2h = pipe.bytes_per_call()
    return {"value": round((fb + bb) / (ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "host_buffers": "pinned", "pipeline": f"{args.e2e_chunk} batch(es) per chunk, double-buffered, "
                                                  "3 streams (copy-in, kernels, copy-out)"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gtms", "reference"], default="gtms")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunk", type=int, default=1, help="batches per chunk in the host pipeline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table (CONFIG_TABLE)")
    ap.add_argument("--split", action="store_true",
                    help="split one workload over the ranks (strong scaling) instead of one replica per rank")
    ap.add_argument("--configs", default=None, help="comma-separated workloads for the per-workload table")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    import seeded_inputs as si

    w = si.WORKLOADS[args.workload]
    lens = si.seq_lens(w)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w, lens)
        return
    if w.head_dim > 0:
        run_gpu_attention(args, w, lens, rank, world, local_rank)
    else:
        run_gpu(args, w, lens, rank, world, local_rank)


if __name__ == "__main__":
    main()
