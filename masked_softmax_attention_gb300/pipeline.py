"""Host-buffer pipeline: scores and gradients live in pinned host memory.

Rows of different batches are independent, so a call over X[B,M,S,S] splits
into chunks of whole batches. Each chunk is copied host -> device on one
stream, passed through ``gtms_forward`` (and ``gtms_backward``) on a second,
and its outputs copied device -> host on a third; double-buffered device
staging lets the copy-in of chunk i+1, the kernels of chunk i and the
copy-out of chunk i-1 run at the same time. Torch supplies only the staging
memory, the streams, the events and the copies; the compute is the two C
calls. Nothing here falls back to a CPU implementation.
"""
from __future__ import annotations

import torch

from . import GTMS_OK, GtmsError, _dtype_code, load_library


class HostPipeline:
    """Reusable device staging for one [B, M, S, S] shape and dtype.

    ``chunk_batches`` batches go through the device at a time, ``depth``
    chunks are staged at once (2 = double buffering).
    """

    def __init__(self, B, M, S, dtype, device, chunk_batches=2, depth=2, backward=True):
        self.B, self.M, self.S, self.dtype = B, M, S, dtype
        self.device = torch.device(device)
        self.chunk = max(1, min(chunk_batches, B))
        self.depth = max(1, depth)
        self.backward = backward
        shape = (self.chunk, M, S, S)
        mk = lambda: torch.empty(shape, dtype=dtype, device=self.device)  # noqa: E731
        self.x = [mk() for _ in range(self.depth)]
        self.y = [mk() for _ in range(self.depth)]
        self.dy = [mk() for _ in range(self.depth)] if backward else None
        self.dx = [mk() for _ in range(self.depth)] if backward else None
        self.lens = torch.empty(B, dtype=torch.int32, device=self.device)
        self.s_in = torch.cuda.Stream(self.device)
        self.s_run = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        ev = lambda: [torch.cuda.Event() for _ in range(self.depth)]  # noqa: E731
        self.ev_in, self.ev_run, self.ev_free = ev(), ev(), ev()
        self.lib = load_library()
        self.code = _dtype_code(self.x[0])

    def bytes_per_call(self):
        """(host->device, device->host) bytes one call moves."""
        e = self.x[0].element_size()
        t = self.B * self.M * self.S * self.S * e
        k = 2 if self.backward else 1
        return k * t + self.B * 4, k * t

    def run(self, x_h, lens_h, scale, y_h, dy_h=None, dx_h=None):
        """Enqueue one forward (+ backward) over the host tensors; returns at once.

        Work is ordered after everything already queued on the current stream,
        and the current stream waits for the last copy-out, so a caller that
        synchronises the current stream sees the host outputs complete.
        """
        cur = torch.cuda.current_stream(self.device)
        M, S = self.M, self.S
        self.s_in.wait_stream(cur)
        with torch.cuda.stream(self.s_in):
            self.lens.copy_(lens_h, non_blocking=True)
        for i, b0 in enumerate(range(0, self.B, self.chunk)):
            b1 = min(self.B, b0 + self.chunk)
            nb, k = b1 - b0, i % self.depth
            with torch.cuda.stream(self.s_in):
                if i >= self.depth:
                    self.s_in.wait_event(self.ev_free[k])
                self.x[k][:nb].copy_(x_h[b0:b1], non_blocking=True)
                if self.backward:
                    self.dy[k][:nb].copy_(dy_h[b0:b1], non_blocking=True)
                self.ev_in[k].record(self.s_in)
            self.s_run.wait_event(self.ev_in[k])
            sp = self.s_run.cuda_stream
            lp = self.lens.data_ptr() + 4 * b0
            rc = self.lib.gtms_forward(self.x[k].data_ptr(), self.y[k].data_ptr(), lp, nb, M, S, float(scale),
                                       self.code, sp)
            if rc != GTMS_OK:
                raise GtmsError("gtms_forward", rc)
            if self.backward:
                rc = self.lib.gtms_backward(self.y[k].data_ptr(), self.dy[k].data_ptr(), self.dx[k].data_ptr(), lp,
                                            nb, M, S, float(scale), self.code, sp)
                if rc != GTMS_OK:
                    raise GtmsError("gtms_backward", rc)
            self.ev_run[k].record(self.s_run)
            self.s_out.wait_event(self.ev_run[k])
            with torch.cuda.stream(self.s_out):
                y_h[b0:b1].copy_(self.y[k][:nb], non_blocking=True)
                if self.backward:
                    dx_h[b0:b1].copy_(self.dx[k][:nb], non_blocking=True)
                self.ev_free[k].record(self.s_out)
        cur.wait_stream(self.s_out)
