"""Host-buffer calls, pipelined over 128-row-aligned chunks.

For inputs and outputs in pinned host memory the work is cut into chunks of
rows, a multiple of 128 each, and three CUDA streams overlap the copy of chunk
i+1 to the device, the producer call on chunk i and the copy of chunk i-1's
codes and scales back.  This works because rows are independent and the
scales of a 128-row tile are one contiguous byte range of the swizzled matrix
(``h3q_scale_offset_of_row_tile`` in include/h3q.h).  Every chunk is computed by
the library's C ABI call on device staging buffers; the staging buffers, the
streams and the events live in a reusable :class:`HostPipeline`.

The frame of each row reaches the chunk calls as a device ``row_frame`` slice,
so chunks need not line up with frames.  Given ``rows_per_frame`` instead, the
row -> frame array (``row // rows_per_frame``) is written on the host once per
(rows, rows_per_frame), copied to the device and kept.
"""
from __future__ import annotations

import numpy as np
import torch

from . import h3q_rmsnorm_adaln_nvfp4, padded_rows


def scale_offset_of_row_tile(row0: int, cols: int) -> int:
    """Byte offset in the swizzled scale matrix of the scales of rows row0.. (row0 % 128 == 0)."""
    if row0 % 128:
        raise ValueError("row0 must be a multiple of 128")
    return row0 // 128 * (cols // 64) * 512


class HostPipeline:
    """Device staging buffers, streams and events for pipelined host-buffer calls
    of up to `max_cols` columns in chunks of `chunk_rows` rows (a multiple of 128).

    A call is ordered after the work queued on the caller's current stream, and
    the caller's current stream is made to wait for the call's last copy back, so
    the outputs may be read after ``torch.cuda.current_stream().synchronize()``.
    """

    def __init__(self, device, max_cols: int, chunk_rows: int = 8192, depth: int = 3):
        if chunk_rows <= 0 or chunk_rows % 128:
            raise ValueError("chunk_rows must be a positive multiple of 128")
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.device = torch.device(device)
        self.chunk_rows, self.depth, self.max_cols = chunk_rows, depth, max_cols
        elems = chunk_rows * max_cols
        new = lambda n, dt: torch.empty(n, dtype=dt, device=self.device)  # noqa: E731
        self.x = [new(elems, torch.bfloat16) for _ in range(depth)]
        self.codes = [new(elems // 2, torch.uint8) for _ in range(depth)]
        self.scales = [new(elems // 16, torch.uint8) for _ in range(depth)]
        self.h2d = torch.cuda.Stream(self.device)
        self.compute = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self.loaded = [torch.cuda.Event() for _ in range(depth)]
        self.computed = [torch.cuda.Event() for _ in range(depth)]
        self.drained = [torch.cuda.Event() for _ in range(depth)]
        self._frames = {}

    def frame_array(self, rows: int, rows_per_frame: int) -> torch.Tensor:
        """Device int32 [rows] holding row // rows_per_frame (kept for reuse)."""
        key = (rows, rows_per_frame)
        if key not in self._frames:
            host = torch.from_numpy((np.arange(rows, dtype=np.int64) // rows_per_frame).astype(np.int32))
            self._frames[key] = host.to(self.device)
        return self._frames[key]

    def _to_device(self, t):
        """t on the device; a copy made here is queued on the H2D stream and marked
        as used by the compute stream so the allocator keeps it until then."""
        if t.device == self.device:
            return t
        d = t.to(self.device, non_blocking=True)
        d.record_stream(self.compute)
        return d

    def rmsnorm_adaln_nvfp4(self, x_host, gamma, mod_table, global_scale, codes_host, scales_host, *,
                            rows_per_frame=None, row_frame=None, eps=1e-6):
        """RMSNorm + AdaLN -> NVFP4 of a contiguous host bf16 [rows, cols] tensor into
        contiguous host codes [rows, cols/2] and scales [pad128(rows), cols/16] (uint8).
        gamma, mod_table, global_scale and row_frame (int32 [rows]) may be host or
        device tensors; host ones are copied once per call."""
        if x_host.dim() != 2 or not x_host.is_contiguous() or x_host.dtype != torch.bfloat16:
            raise ValueError("x_host must be a contiguous bf16 [rows, cols] tensor")
        rows, cols = x_host.shape
        if cols > self.max_cols:
            raise ValueError("cols exceeds the pipeline's max_cols")
        for name, t, shape in (("codes_host", codes_host, (rows, cols // 2)),
                               ("scales_host", scales_host, (padded_rows(rows), cols // 16))):
            if tuple(t.shape) != shape or not t.is_contiguous() or t.dtype != torch.uint8:
                raise ValueError(f"{name} must be contiguous uint8 {shape}")
        if row_frame is None and rows_per_frame is None:
            raise ValueError("give row_frame or rows_per_frame")
        cur = torch.cuda.current_stream(self.device)
        self.h2d.wait_stream(cur)
        with torch.cuda.stream(self.h2d):
            gamma_d = self._to_device(gamma)
            table_d = self._to_device(mod_table)
            gsf_d = self._to_device(global_scale)
            frames = (self._to_device(row_frame) if row_frame is not None
                      else self.frame_array(rows, rows_per_frame))
        params = torch.cuda.Event()
        params.record(self.h2d)
        self.compute.wait_event(params)
        codes_flat, scales_flat = codes_host.view(-1), scales_host.view(-1)
        for i, r0 in enumerate(range(0, rows, self.chunk_rows)):
            s = i % self.depth
            r1 = min(rows, r0 + self.chunk_rows)
            n, nc, ns = r1 - r0, (r1 - r0) * cols // 2, padded_rows(r1 - r0) * cols // 16
            if i >= self.depth:  # slot s: chunk i - depth has read its x
                self.h2d.wait_event(self.computed[s])
            xs = self.x[s][:n * cols].view(n, cols)
            with torch.cuda.stream(self.h2d):
                xs.copy_(x_host[r0:r1], non_blocking=True)
            self.loaded[s].record(self.h2d)
            self.compute.wait_event(self.loaded[s])
            if i >= self.depth:  # slot s: chunk i - depth's outputs have been copied back
                self.compute.wait_event(self.drained[s])
            codes_d = self.codes[s][:nc].view(n, cols // 2)
            scales_d = self.scales[s][:ns].view(padded_rows(n), cols // 16)
            h3q_rmsnorm_adaln_nvfp4(xs, gamma_d, table_d, gsf_d, row_frame=frames[r0:r1], eps=eps,
                                    codes=codes_d, scales=scales_d, stream=self.compute)
            self.computed[s].record(self.compute)
            self.d2h.wait_event(self.computed[s])
            lo = scale_offset_of_row_tile(r0, cols)
            with torch.cuda.stream(self.d2h):
                codes_flat[r0 * cols // 2:r1 * cols // 2].copy_(codes_d.view(-1), non_blocking=True)
                scales_flat[lo:lo + ns].copy_(scales_d.view(-1), non_blocking=True)
            self.drained[s].record(self.d2h)
        cur.wait_stream(self.d2h)
        return codes_host, scales_host
