"""Helpers for the GPU parity tests: move tensors to the oracle and compare bytes.

Parity is bit for bit: codes, scale bytes (at their swizzled offsets, padding
rows zero), dequantized values and row statistics must equal the oracle's.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

THREADS = max(1, min(16, os.cpu_count() or 1))


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy array of its bit patterns (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def gsf_tensor(value: float, device) -> torch.Tensor:
    return torch.tensor([value], dtype=torch.float32, device=device)


def fill(t: torch.Tensor, byte: int = 0xAB) -> torch.Tensor:
    """Pre-fill an output with a sentinel so that unwritten bytes show."""
    t.view(torch.uint8).fill_(byte)
    return t


def check_rows(codes_gpu: torch.Tensor, scales_gpu: torch.Tensor, rows_idx, cols: int,
               codes_ref: np.ndarray, sf_ref: np.ndarray, what: str) -> None:
    """Compare the listed rows: codes [n, cols/2] and logical scales [n, cols/16]."""
    rows_idx = np.asarray(rows_idx, dtype=np.int64)
    idx = torch.as_tensor(rows_idx, device=codes_gpu.device)
    got_codes = codes_gpu.index_select(0, idx).cpu().numpy()
    bad = np.nonzero((got_codes != codes_ref).any(1))[0]
    assert bad.size == 0, f"{what}: codes differ in rows {rows_idx[bad[:8]].tolist()}"
    offs = oracle.scale_offsets(rows_idx, cols)
    flat = scales_gpu.view(-1)
    got_sf = flat.index_select(0, torch.as_tensor(offs.ravel(), device=flat.device)).cpu().numpy()
    got_sf = got_sf.reshape(offs.shape)
    bad = np.nonzero((got_sf != sf_ref).any(1))[0]
    assert bad.size == 0, f"{what}: scales differ in rows {rows_idx[bad[:8]].tolist()}"


def check_padding(scales_gpu: torch.Tensor, rows: int, cols: int, what: str) -> None:
    pad = oracle.padded_rows(rows)
    if pad == rows:
        return
    offs = oracle.scale_offsets(np.arange(rows, pad), cols).ravel()
    flat = scales_gpu.view(-1)
    got = flat.index_select(0, torch.as_tensor(offs, device=flat.device)).cpu().numpy()
    assert (got == 0).all(), f"{what}: padding rows of the scale matrix are not zero"


def check_full(codes_gpu, scales_gpu, rows, cols, codes_ref, sf_ref, what):
    """Every byte of both outputs equals the oracle (scales swizzled, padding zero)."""
    assert np.array_equal(codes_gpu.cpu().numpy(), codes_ref), f"{what}: codes differ"
    want = oracle.swizzle_scales(sf_ref, rows, cols)
    got = scales_gpu.cpu().numpy().ravel()
    if not np.array_equal(got, want):
        diff = np.nonzero(got != want)[0]
        raise AssertionError(f"{what}: {diff.size} scale bytes differ, first at {diff[:8].tolist()}")
