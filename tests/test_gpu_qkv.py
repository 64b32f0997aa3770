"""GPU parity of the QKV epilogue (bias + per-head RMSNorm + partial rotate-half
RoPE on q and k, bias on v) through the C ABI: every output bf16 of
q, k and v equals the oracle's, over head dims 64/128/256, rotary widths 0 to
HD, odd head counts (a half-filled warp), strided views of one packed
projection, and every row of the 65,280-token workload the benchmark times."""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from parity import THREADS, bits, fill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _run(w, interleaved=False):
    rows = w["q"].shape[0]
    outs = [fill(torch.empty((rows, w["heads"], w["head_dim"]), dtype=torch.bfloat16,
                             device=w["q"].device)) for _ in range(3)]
    return h3q.h3q_qkv_epilogue(w["q"], w["k"], w["v"], w["biases"], w["cos"], w["sin"], w["heads"],
                                w["eps"], outs=outs, interleaved=interleaved)


def _oracle(w, idx=None, interleaved=False):
    """The oracle's q, k, v outputs (rows `idx` only, when given)."""
    def sel(t):
        if t is None:
            return None
        return bits(t if idx is None else t.index_select(0, idx))

    cos, sin = sel(w["cos"]), sel(w["sin"])
    out = []
    for i, name in enumerate("qkv"):
        out.append(oracle.qkv_epilogue_rows(sel(w[name]), bits(w["biases"][i]), w["heads"], cos, sin,
                                            w["eps"], is_v=(name == "v"), threads=THREADS,
                                            interleaved=interleaved))
    return out


def _check(got, want, what):
    for name, g, r in zip("qkv", got, want):
        g = bits(g)
        bad = np.argwhere(g != r)
        assert bad.size == 0, f"{what}: {name} differs at {bad[:4].tolist()} ({g[tuple(bad[0])]:#06x} vs " \
                              f"{r[tuple(bad[0])]:#06x})"


@pytest.mark.parametrize("rows,heads,hd,rot,packed", [
    (1, 1, 128, 64, True), (37, 56, 128, 64, True), (130, 3, 128, 128, False), (64, 5, 128, 16, True),
    (50, 2, 128, 0, True), (41, 7, 64, 32, True), (29, 4, 64, 64, False), (33, 3, 256, 96, True),
    (17, 2, 256, 256, False), (300, 24, 128, 48, True)])
def test_shapes(dev, rows, heads, hd, rot, packed):
    w = workloads.qkv_inputs(dev, rows=rows, heads=heads, head_dim=hd, rot=rot, seed=rows + heads + rot,
                             packed=packed)
    _check(_run(w), _oracle(w), f"qkv {rows}x{heads}x{hd} rot {rot}")


@pytest.mark.parametrize("rows,heads,hd,rot,packed", [
    (1, 1, 128, 64, True), (37, 56, 128, 128, True), (41, 7, 64, 32, False), (17, 3, 256, 96, True),
    (300, 24, 128, 16, True)])
def test_interleaved_pairs(dev, rows, heads, hd, rot, packed):
    """RoPE on the pairs (2j, 2j+1) (the FlashRT page's fused RMSNorm + RoPE kernel)."""
    w = workloads.qkv_inputs(dev, rows=rows, heads=heads, head_dim=hd, rot=rot, seed=rows + 7 * heads,
                             packed=packed)
    _check(_run(w, interleaved=True), _oracle(w, interleaved=True), f"qkv interleaved {rows}x{heads}x{hd}")


def test_full_workload_interleaved_sampled_rows(dev):
    w = workloads.qkv_inputs(dev, seed=8)
    got = _run(w, interleaved=True)
    torch.cuda.synchronize()
    idx = workloads.sample_rows(w["q"].shape[0], random=512).to(dev)
    _check([g.index_select(0, idx) for g in got], _oracle(w, idx, interleaved=True), "qkv interleaved full")


def test_eps_and_large_values(dev):
    """A large eps (the rstd then depends on it) and inputs with a wide range: heads
    whose squares underflow to zero or to subnormals, heads of large values, heads
    whose sum of squares overflows to infinity (rstd 0), and all-zero heads."""
    w = workloads.qkv_inputs(dev, rows=64, heads=8, head_dim=128, rot=64, seed=11)
    q = w["q"].clone()
    for h, factor in enumerate((1e-30, 1e-19, 1e15, 1e30, 0.0)):
        q[:, h * 128:(h + 1) * 128] = q[:, h * 128:(h + 1) * 128] * factor
    w["q"] = q
    w["eps"] = 0.25
    _check(_run(w), _oracle(w), "qkv eps 0.25, wide range")


def test_full_workload_every_row(dev):
    """The 65,280-token x 56 x 128 (ROT 64) workload from one packed projection, in
    the configuration the benchmark times: every output bf16 of q, k and v against
    the oracle, in chunks of 8,192 rows."""
    w = workloads.qkv_inputs(dev)
    got = _run(w)
    torch.cuda.synchronize()
    rows = w["q"].shape[0]
    step = 8192
    for r0 in range(0, rows, step):
        idx = torch.arange(r0, min(rows, r0 + step), device=dev)
        _check([g.index_select(0, idx) for g in got], _oracle(w, idx), f"qkv 65280x56x128 rows {r0}..")


def test_past_2_31_elements_the_pages_regression_shape(dev):
    """8,500,000 tokens x 2 heads x 128 per tensor (2.176e9 elements, the shape of
    the FastVideo commit log's int64 fix for the q/k norm + partial RoPE kernel):
    the first and last 256 rows and 512 random rows of q, k and v equal the
    oracle's (the last rows sit past element 2^31)."""
    rows = 8_500_000
    w = workloads.qkv_inputs(dev, rows=rows, heads=2, head_dim=128, rot=64, seed=31)
    assert w["q"].shape[0] * w["q"].shape[1] > 2 ** 31
    got = _run(w)
    torch.cuda.synchronize()
    idx = workloads.sample_rows(rows, random=512).to(dev)
    _check([g.index_select(0, idx) for g in got], _oracle(w, idx), "qkv 8.5M x 2 x 128")
    del w, got
    torch.cuda.empty_cache()
