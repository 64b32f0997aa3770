"""Host-buffer calls: a reusable front end for h3q_rmsnorm_adaln_nvfp4_host.

The library call takes the input and the outputs in host memory and pipelines
the copies with the producer over 128-row-aligned chunks (three staging slots,
the producer on the caller's stream, a library stream for each copy direction;
the scales of a 128-row tile are one contiguous byte range of the swizzled
matrix, ``h3q_scale_offset_of_row_tile`` in include/h3q.h).  :class:`HostPipeline`
keeps the device workspace between calls and moves parameters given as host
tensors (gamma, the modulation table, the global scale, row_frame) to the
device first, on the caller's stream.
"""
from __future__ import annotations

import torch

from . import h3q_rmsnorm_adaln_nvfp4_host, host_workspace_bytes, padded_rows


def scale_offset_of_row_tile(row0: int, cols: int) -> int:
    """Byte offset in the swizzled scale matrix of the scales of rows row0.. (row0 % 128 == 0)."""
    if row0 % 128:
        raise ValueError("row0 must be a multiple of 128")
    return row0 // 128 * (cols // 64) * 512


class HostPipeline:
    """Pipelined host-buffer calls of up to `max_cols` columns in chunks of
    `chunk_rows` rows (a multiple of 128), three staging slots in the library.

    A call is ordered after the work queued on the caller's current stream, and
    that stream waits for the call's last copy back, so the outputs may be read
    after ``torch.cuda.current_stream().synchronize()``.
    """

    depth = 3  # the library's staging slots

    def __init__(self, device, max_cols: int, chunk_rows: int = 2048):
        if chunk_rows <= 0 or chunk_rows % 128:
            raise ValueError("chunk_rows must be a positive multiple of 128")
        self.device = torch.device(device)
        self.chunk_rows, self.max_cols = chunk_rows, max_cols
        self._workspace = None

    def workspace(self, rows: int, cols: int, with_frames: bool) -> torch.Tensor:
        """The device workspace for a call, grown when a call needs more."""
        need = host_workspace_bytes(self.chunk_rows, cols, rows, with_frames)
        if self._workspace is None or self._workspace.numel() < need:
            self._workspace = None
            self._workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._workspace

    def _to_device(self, t):
        return t if t.device == self.device else t.to(self.device, non_blocking=True)

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
        with torch.cuda.stream(cur):
            gamma_d = self._to_device(gamma)
            table_d = self._to_device(mod_table)
            gsf_d = self._to_device(global_scale)
            frames_d = None if row_frame is None else self._to_device(row_frame)
        ws = self.workspace(rows, cols, frames_d is None)
        return h3q_rmsnorm_adaln_nvfp4_host(x_host, gamma_d, table_d, gsf_d, codes_host, scales_host, ws,
                                            row_frame=frames_d, rows_per_frame=rows_per_frame, eps=eps,
                                            chunk_rows=self.chunk_rows, stream=cur)
