"""Seeded synthetic inputs for the grouped-tril masked softmax workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no mask, no softmax, no rounding rule of its own). It is
the one module that both the CUDA-path tests / bench and the CPU oracle take
inputs from.

Workloads (shapes, dtypes and distributions of the pages' runs):

* ``worked_example`` -- X[3,2,5,5] fp32 ~N(0,1), seq_lens [3,4,5], scale 1,
  forward only: the printed example of the "Attention-Mask-Optimization"
  README (operator behaviour section).
* ``s1000_b3`` -- X[3,64,1000,1000] fp32 ~N(0,1), seq_len ~ U{1..1000},
  scale 1, forward: the README's DevCloud / A10 shape.
* ``s1000_b12`` -- X[12,64,1000,1000] fp32 ~N(0,1), seq_len ~ U{500..1000},
  scale 1, forward + backward with dY ~N(0,1) fp32 (the README's A10 shape).
* ``s2048_bf16`` -- X[32,16,2048,2048] bf16 ~N(0, variance 4),
  seq_len ~ U{1024..2048}, scale 0.125 (head_dim 64), forward + backward with
  dY ~N(0,1) bf16 ("优化ScaledMaskSoftmax算子" section 3.2: batch 32, head_dim 64).
* ``s8192_f16`` -- X[4,16,8192,8192] fp16 ~N(0,1) with an independent 1%
  of entries set to +30, seq_len ~ U{4096..8192}, scale 0.125, forward +
  backward with dY ~N(0,1) fp16 (long rows, overflow stress).
* ``s4096_bf16`` -- X[32,16,4096,4096] bf16 ~N(0, variance 4),
  seq_len ~ U{2048..4096}, scale 0.125, forward + backward: an added S=4096
  measurement point mirroring the ScaledMaskSoftmax article's 4096 row.
* ``s16384_bf16`` -- X[4,8,16384,16384] bf16 ~N(0, variance 4),
  seq_len ~ U{8192..16384}, scale 0.125, ``s32768_bf16`` --
  X[1,4,32768,32768], seq_len ~ U{16384..32768}, and ``s65536_bf16`` /
  ``s65536_f32`` -- X[1,2,65536,65536] bf16 / X[1,1,65536,65536] fp32,
  seq_len ~ U{32768..65536}: added measurement points for rows of 32 KB and
  more (the two-pass stream kernels), up to the longest rows served.
* ``attn_s2048_bf16`` -- the attention-backward step at the ``s2048_bf16``
  shape: P the softmax of X[32,16,2048,2048] (bf16, variance 4,
  seq_len ~ U{1024..2048}, scale 0.125), dO and V [32,16,2048,64] ~ N(0,1).
* ``attn_d128_s2048_f16`` -- the same step in fp16 with head_dim 128: P the
  softmax of X[32,16,2048,2048] (fp16, variance 4, seq_len ~ U{1024..2048},
  scale 0.125), dO and V [32,16,2048,128] ~ N(0,1).
* ``length_s2048_bf16``, ``window_s2048_bf16``, ``explicit_s2048_bf16`` -- the
  ``s2048_bf16`` shape and distribution under the length mask, a sliding causal
  window of width 256, and an explicit uint8 keep mask (``make_keep_mask``:
  each c <= r < seq_len entry kept with probability 1/2).
* ``attn_s2048_b4`` -- ``attn_s2048_bf16`` with 4 batches: a profiler stand-in
  (P and dS 537 MB each, still larger than L2); ``attn_d128_b4`` likewise for
  ``attn_d128_s2048_f16``.
* ``s1000_b2`` -- X[2,64,1000,1000], otherwise like ``s1000_b12``: a small
  stand-in for profiler captures.
* ``s32768_m1`` -- X[1,1,32768,32768], otherwise like ``s32768_bf16`` (same
  seed, same length): one of its four heads, a stand-in for profiler captures.

Every tensor comes from torch's seeded generators (Philox on CUDA, mt19937 on
the CPU), drawn in float32 and cast to the IO dtype with round-to-nearest-even.
The same seed on the same device type gives the same bytes.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2}
TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    M: int
    S: int
    dtype: str
    scale: float
    x_std: float = 1.0
    seq_len_range: tuple | None = None      # inclusive (lo, hi), drawn uniformly per batch
    fixed_seq_lens: tuple | None = None
    spike_prob: float = 0.0                 # probability that an x entry is replaced by spike_value
    spike_value: float = 30.0
    backward: bool = True
    seed: int = 20261202
    head_dim: int = 0                       # > 0: attention-backward step workload (dO, V of this width)
    mask_kind: int = 0                      # 0 grouped tril, 1 length mask, 2 sliding causal window
    window: int = 0                         # band width for mask_kind 2
    keep_prob: float = 0.0                  # > 0: explicit uint8 keep mask (see make_keep_mask)

    @property
    def rows(self) -> int:
        return self.B * self.M * self.S

    @property
    def elems(self) -> int:
        return self.B * self.M * self.S * self.S

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def torch_dtype(self):
        return TORCH_DTYPES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    def describe(self) -> str:
        if self.fixed_seq_lens is not None:
            lens = "seq_lens=" + ",".join(str(v) for v in self.fixed_seq_lens)
        else:
            lens = f"seq_len~U{{{self.seq_len_range[0]}..{self.seq_len_range[1]}}}"
        dist = f"N(0,{self.x_std ** 2:g})"
        if self.spike_prob:
            dist += f"+{self.spike_prob:g}x{self.spike_value:g}"
        if self.head_dim > 0:
            return (f"dS from P=softmax(X[{self.B},{self.M},{self.S},{self.S}] {self.dtype} {dist} {lens} "
                    f"scale={self.scale:g}), dO and V [{self.B},{self.M},{self.S},{self.head_dim}] N(0,1)")
        if self.keep_prob > 0:
            lens += f", explicit uint8 keep mask [B,S,S]: c<=r<L kept with p={self.keep_prob:g}"
        elif self.mask_kind == 1:
            lens += ", length mask (c<L, r<L)"
        elif self.mask_kind == 2:
            lens += f", sliding causal window w={self.window}"
        return (f"X[{self.B},{self.M},{self.S},{self.S}] {self.dtype} {dist} {lens} scale={self.scale:g} "
                f"{'fwd+bwd' if self.backward else 'fwd'}")


WORKLOADS = {
    "worked_example": Workload("worked_example", 3, 2, 5, "f32", 1.0, fixed_seq_lens=(3, 4, 5),
                               backward=False, seed=20261203),
    "s1000_b3": Workload("s1000_b3", 3, 64, 1000, "f32", 1.0, seq_len_range=(1, 1000),
                         backward=False, seed=20261204),
    "s1000_b12": Workload("s1000_b12", 12, 64, 1000, "f32", 1.0, seq_len_range=(500, 1000),
                          seed=20261205),
    "s2048_bf16": Workload("s2048_bf16", 32, 16, 2048, "bf16", 0.125, x_std=2.0,
                           seq_len_range=(1024, 2048), seed=20261206),
    "s8192_f16": Workload("s8192_f16", 4, 16, 8192, "f16", 0.125, seq_len_range=(4096, 8192),
                          spike_prob=0.01, spike_value=30.0, seed=20261207),
    "s4096_bf16": Workload("s4096_bf16", 32, 16, 4096, "bf16", 0.125, x_std=2.0,
                           seq_len_range=(2048, 4096), seed=20261208),
    # rows of 32 KB and more (two-pass stream kernels): added measurement points
    "s16384_bf16": Workload("s16384_bf16", 4, 8, 16384, "bf16", 0.125, x_std=2.0,
                            seq_len_range=(8192, 16384), seed=20261210),
    "s32768_bf16": Workload("s32768_bf16", 1, 4, 32768, "bf16", 0.125, x_std=2.0,
                            seq_len_range=(16384, 32768), seed=20261211),
    "s65536_bf16": Workload("s65536_bf16", 1, 2, 65536, "bf16", 0.125, x_std=2.0,
                            seq_len_range=(32768, 65536), seed=20261217),
    "s65536_f32": Workload("s65536_f32", 1, 1, 65536, "f32", 0.125, x_std=2.0,
                           seq_len_range=(32768, 65536), seed=20261218),
    # attention-backward step (dS from P, dO, V) at the bf16 S = 2048 shape, head_dim 64
    "attn_s2048_bf16": Workload("attn_s2048_bf16", 32, 16, 2048, "bf16", 0.125, x_std=2.0,
                                seq_len_range=(1024, 2048), seed=20261212, head_dim=64),
    # the same step in fp16 with head_dim 128 (the kernel's other ring shape)
    "attn_d128_s2048_f16": Workload("attn_d128_s2048_f16", 32, 16, 2048, "f16", 0.125, x_std=2.0,
                                    seq_len_range=(1024, 2048), seed=20261219, head_dim=128),
    # the other mask families and an explicit keep mask, on the s2048_bf16 shape and distribution
    "length_s2048_bf16": Workload("length_s2048_bf16", 32, 16, 2048, "bf16", 0.125, x_std=2.0,
                                  seq_len_range=(1024, 2048), seed=20261214, mask_kind=1),
    "window_s2048_bf16": Workload("window_s2048_bf16", 32, 16, 2048, "bf16", 0.125, x_std=2.0,
                                  seq_len_range=(1024, 2048), seed=20261215, mask_kind=2, window=256),
    "explicit_s2048_bf16": Workload("explicit_s2048_bf16", 32, 16, 2048, "bf16", 0.125, x_std=2.0,
                                    seq_len_range=(1024, 2048), seed=20261216, keep_prob=0.5),
    # profiling stand-in for attn_s2048_bf16: same distribution, 4 of the 32 batches
    "attn_s2048_b4": Workload("attn_s2048_b4", 4, 16, 2048, "bf16", 0.125, x_std=2.0,
                              seq_len_range=(1024, 2048), seed=20261212, head_dim=64),
    "attn_d128_b4": Workload("attn_d128_b4", 4, 16, 2048, "f16", 0.125, x_std=2.0,
                             seq_len_range=(1024, 2048), seed=20261219, head_dim=128),
    # profiling stand-in for s1000_b12: same distribution, 2 of the 12 batches
    # (2 GB on the device), small enough for a multi-pass ncu capture
    "s1000_b2": Workload("s1000_b2", 2, 64, 1000, "f32", 1.0, seq_len_range=(500, 1000), seed=20261209),
    # profiling stand-in for s32768_bf16: the same seed, so the same length, one of the 4 heads
    # (2.1 GB per tensor)
    "s32768_m1": Workload("s32768_m1", 1, 1, 32768, "bf16", 0.125, x_std=2.0,
                          seq_len_range=(16384, 32768), seed=20261211),
}


def custom(name, B, M, S, dtype, scale=1.0, *, seq_lens=None, seq_len_range=None, x_std=1.0,
           spike_prob=0.0, backward=True, seed=1) -> Workload:
    """A workload of any shape (tests: ragged tails, edge sizes, odd lengths)."""
    if seq_lens is None and seq_len_range is None:
        seq_len_range = (0, S)
    return Workload(name, B, M, S, dtype, scale, x_std=x_std,
                    seq_len_range=None if seq_lens is not None else tuple(seq_len_range),
                    fixed_seq_lens=None if seq_lens is None else tuple(int(v) for v in seq_lens),
                    spike_prob=spike_prob, backward=backward, seed=seed)


def seq_lens(w: Workload) -> np.ndarray:
    """int32 [B]: fixed lengths, or uniform integers in the inclusive range."""
    if w.fixed_seq_lens is not None:
        return np.array(w.fixed_seq_lens, dtype=np.int32)
    g = torch.Generator().manual_seed(w.seed * 4 + 3)
    lo, hi = w.seq_len_range
    return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def _chunks(w: Workload, max_elems: int):
    slices = w.B * w.M
    per = max(1, max_elems // max(1, w.S * w.S))
    for s0 in range(0, slices, per):
        yield s0, min(slices, s0 + per)


def _draw(w: Workload, device, stream_id: int, std: float, spikes: bool, max_chunk_elems: int):
    dev = torch.device(device)
    out = torch.empty((w.B, w.M, w.S, w.S), dtype=w.torch_dtype, device=dev)
    if w.elems == 0:
        return out
    g = torch.Generator(device=dev).manual_seed(w.seed * 4 + stream_id)
    flat = out.view(w.B * w.M, w.S, w.S)
    for s0, s1 in _chunks(w, max_chunk_elems):
        shape = (s1 - s0, w.S, w.S)
        v = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        if spikes and w.spike_prob > 0:
            hit = torch.rand(shape, generator=g, device=dev, dtype=torch.float32) < w.spike_prob
            v.masked_fill_(hit, w.spike_value)
        flat[s0:s1].copy_(v)
    return out


def make_x(w: Workload, device="cpu", max_chunk_elems: int = 1 << 28) -> torch.Tensor:
    """Scores X[B,M,S,S] in the workload's dtype."""
    return _draw(w, device, 0, w.x_std, True, max_chunk_elems)


def make_dy(w: Workload, device="cpu", max_chunk_elems: int = 1 << 28) -> torch.Tensor:
    """Upstream gradient dY[B,M,S,S] ~ N(0,1) in the workload's dtype."""
    return _draw(w, device, 1, 1.0, False, max_chunk_elems)


def make_keep_mask(w: Workload, device="cpu") -> torch.Tensor:
    """uint8 [B, S, S] explicit keep mask: entry (b, r, c) is 1 with probability keep_prob
    where c <= r < seq_len[b], else 0 (independent seeded draws, one batch at a time)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(w.seed * 4 + 7)
    lens = seq_lens(w)
    r = torch.arange(w.S, device=dev)
    causal = r[None, :] <= r[:, None]
    out = torch.empty(w.B, w.S, w.S, dtype=torch.uint8, device=dev)
    for b in range(w.B):
        u = torch.rand(w.S, w.S, generator=g, device=dev)
        live = causal & (r[:, None] < int(lens[b]))
        out[b] = (live & (u < w.keep_prob)).to(torch.uint8)
    return out


def make_head_operands(w: Workload, device="cpu"):
    """dO and V [B, M, S, head_dim] ~ N(0,1) in the workload's dtype (attention-backward workloads)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(w.seed * 4 + 5)
    shape = (w.B, w.M, w.S, w.head_dim)
    dout = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(w.torch_dtype)
    v = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(w.torch_dtype)
    return dout, v


def make_probs(w: Workload, device="cpu", max_chunk_elems: int = 1 << 28) -> torch.Tensor:
    """A stand-in Y[B,M,S,S] ~ U[0,1) for backward edge cases whose values need no structure."""
    dev = torch.device(device)
    out = torch.empty((w.B, w.M, w.S, w.S), dtype=w.torch_dtype, device=dev)
    if w.elems == 0:
        return out
    g = torch.Generator(device=dev).manual_seed(w.seed * 4 + 2)
    flat = out.view(w.B * w.M, w.S, w.S)
    for s0, s1 in _chunks(w, max_chunk_elems):
        flat[s0:s1].copy_(torch.rand((s1 - s0, w.S, w.S), generator=g, device=dev, dtype=torch.float32))
    return out


def sample_slices(w: Workload, count: int) -> list:
    """A fixed, seeded choice of (b, m) slices: first, last, and random others."""
    total = w.B * w.M
    if total <= count:
        return [(s // w.M, s % w.M) for s in range(total)]
    rng = np.random.default_rng(w.seed)
    picks = {0, total - 1}
    while len(picks) < count:
        picks.add(int(rng.integers(0, total)))
    return [(s // w.M, s % w.M) for s in sorted(picks)]
