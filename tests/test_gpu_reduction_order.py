"""The kernels' RMS statistics on the hand-derived rows of tests/golden/rstd_order.txt.

Each row there is built so that the canonical order of the sum of squares gives
different bits from a plausible slip (a sequential sum, another lane map, a
reversed butterfly, ...), and its rstd is derived by hand.  Through the C ABI:
the AdaLN producer at the rows' width (4,096 columns: the 128-thread kernel)
must return those rstd bits exactly; the same rows widened with zeros to 7,168
(the 448-thread block kernel), 8,192 and 16,384 columns (the generic kernel)
keep the same sum of squares, and their rstd must equal the oracle's; the
residual fold, fed the rows as its fp32 residual with o = 0, must return the
hand-derived bits too.
"""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
from test_oracle_reduction_order import RECORDS

pytestmark = pytest.mark.gpu

ROWS = [r for r in RECORDS if r["kind"] == "row"]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _bf16_rows(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def _adaln_rstd(dev, x_bits: np.ndarray, eps: float) -> np.ndarray:
    rows, cols = x_bits.shape
    x = _bf16_rows(x_bits, dev)
    gamma = torch.ones(cols, dtype=torch.bfloat16, device=dev)
    table = torch.zeros((1, 2, cols), dtype=torch.bfloat16, device=dev)
    rstd = torch.full((rows,), float("nan"), dtype=torch.float32, device=dev)
    gsf = torch.ones(1, dtype=torch.float32, device=dev)
    h3q.h3q_rmsnorm_adaln_nvfp4(x, gamma, table, gsf, rows_per_frame=rows, eps=eps, row_rstd=rstd)
    return rstd.cpu().numpy().view(np.uint32)


def _stack(records, cols):
    """The records' rows widened with zeros to `cols`, then again in reverse order
    (so each row is met at two positions in the kernels' row steps)."""
    recs = list(records) + list(reversed(records))
    x = np.zeros((len(recs), cols), np.uint16)
    for i, r in enumerate(recs):
        x[i, :r["n"]] = r["bf16"]
    return recs, x


@pytest.mark.parametrize("eps_bits", [0x00000000, 0x34000000])
def test_adaln_rstd_is_the_hand_derived_one(dev, eps_bits):
    recs = [r for r in ROWS if r["eps"].view(np.uint32) == eps_bits]
    assert recs
    recs, x = _stack(recs, 4096)
    eps = float(np.array([eps_bits], np.uint32).view(np.float32)[0])
    got = _adaln_rstd(dev, x, eps)
    for i, r in enumerate(recs):
        assert got[i] == r["rstd"], f"{r['name']} (row {i}): rstd {got[i]:#010x} != {r['rstd']:#010x}"


@pytest.mark.parametrize("cols", [7168, 8192, 16384])
def test_adaln_rstd_of_widened_rows_is_the_oracle(dev, cols):
    for eps in (0.0, float(np.float32(2.0 ** -23)), 1e-6):
        recs, x = _stack(ROWS, cols)
        got = _adaln_rstd(dev, x, eps)
        for i, r in enumerate(recs):
            want = np.float32(oracle.row_rstd(x[i], eps)).view(np.uint32)
            assert got[i] == want, f"{r['name']} at {cols} columns, eps {eps}: {got[i]:#010x} != {want:#010x}"
            # widening adds exact zeros: the sum of squares is the row's own
            assert np.float32(oracle.sumsq_bf16(x[i])).view(np.uint32) == r["ss"]


def test_residual_fold_rstd_is_the_hand_derived_one(dev):
    recs = [r for r in RECORDS if r["kind"] in ("row", "f32row")]
    rows, cols = len(recs), 4096
    h = torch.from_numpy(np.stack([r["values"] for r in recs])).to(dev)
    o = torch.zeros((rows, cols), dtype=torch.bfloat16, device=dev)
    gate = torch.zeros((1, cols), dtype=torch.bfloat16, device=dev)
    gamma = torch.ones(cols, dtype=torch.bfloat16, device=dev)
    table = torch.zeros((1, 2, cols), dtype=torch.bfloat16, device=dev)
    gsf = torch.ones(1, dtype=torch.float32, device=dev)
    for r in recs:
        assert r["eps"] in (np.float32(0.0), np.float32(2.0 ** -23))
    for eps in (0.0, float(np.float32(2.0 ** -23))):
        rstd = torch.full((rows,), float("nan"), dtype=torch.float32, device=dev)
        h_run = h.clone()
        h3q.h3q_residual_rmsnorm_adaln_nvfp4(h_run, o, gate, gamma, table, gsf, rows_per_frame=rows,
                                             eps=eps, row_rstd=rstd)
        got = rstd.cpu().numpy().view(np.uint32)
        assert torch.equal(h_run, h), "the fold with o = 0 changed h"
        for i, r in enumerate(recs):
            want = np.float32(oracle.row_rstd_f32(r["values"], eps)).view(np.uint32)
            assert got[i] == want, f"{r['name']}, eps {eps}: {got[i]:#010x} != {want:#010x}"
            if r["rstd"] is not None and np.float32(eps) == r["eps"]:
                assert got[i] == r["rstd"], f"{r['name']}: {got[i]:#010x} != hand-derived {r['rstd']:#010x}"
