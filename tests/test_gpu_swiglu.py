"""GPU parity of the SwiGLU -> NVFP4 producer (b), through the C ABI."""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from parity import THREADS, bits, check_full, check_padding, check_rows, fill, gsf_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _oracle_gsf(gate, up):
    _, _, y = oracle.swiglu_rows(bits(gate), bits(up), None, want_y=True, threads=THREADS)
    return oracle.global_scale(float(np.abs(oracle.bf16_value(y)).max()))


def _run(dev, gate, up, gsf):
    rows, cols = gate.shape
    codes = fill(torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((h3q.padded_rows(rows), cols // 16), dtype=torch.uint8, device=dev))
    return h3q.h3q_swiglu_nvfp4(gate, up, gsf_tensor(gsf, dev), codes, scales)


@pytest.mark.parametrize("rows,cols", [(1, 64), (131, 320), (128, 512), (300, 18944), (257, 1600)])
def test_shapes(dev, rows, cols):
    gate, up = workloads.swiglu_inputs(dev, rows=rows, cols=cols, seed=rows + cols)
    gsf = _oracle_gsf(gate, up)
    codes, scales = _run(dev, gate, up, gsf)
    co, so, _ = oracle.swiglu_rows(bits(gate), bits(up), gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, f"swiglu {rows}x{cols}")
    check_padding(scales, rows, cols, f"swiglu {rows}x{cols}")


def test_extreme_gates_take_the_general_exponential(dev):
    """Gates beyond +-87 (exp overflow / subnormal range / the +-89, -104 limits),
    mixed into a row with ordinary values."""
    rows, cols = 96, 1024
    gate, up = workloads.swiglu_inputs(dev, rows=rows, cols=cols, seed=99)
    special = torch.tensor([87.5, 88.0, 88.5, 88.75, 89.0, 89.5, 90.0, 100.0, 104.0, 104.5, 200.0,
                            -87.5, -88.0, -88.5, -88.75, -89.0, -89.5, -90.0, -100.0, -104.0,
                            -104.5, -200.0, -1e30, 1e30, 3.0e38, -3.0e38, 86.9, -86.9],
                           dtype=torch.bfloat16, device=dev)
    gen = torch.Generator(device="cpu").manual_seed(4)
    pos = torch.randperm(rows * cols, generator=gen)[:2000].to(dev)
    g_sp = special[torch.arange(2000, device=dev) % special.numel()]
    gate.view(-1)[pos] = g_sp
    # keep y = silu(g) * u moderate so the calibrated global scale resolves every block
    up.view(-1)[pos] = (0.75 / g_sp.float().abs().clamp(min=1.0)).to(torch.bfloat16)
    up.view(-1)[pos[:200]] = 0
    gsf = _oracle_gsf(gate, up)
    codes, scales = _run(dev, gate, up, gsf)
    co, so, _ = oracle.swiglu_rows(bits(gate), bits(up), gsf)
    check_full(codes, scales, rows, cols, co, so, "swiglu extreme gates")


def test_every_bf16_gate(dev):
    """Every finite bf16 value as a gate against a fixed up of 1 and of -3."""
    vals = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    vals = vals[np.isfinite(vals)]
    cols = 1024
    n = -(-vals.size // cols) * cols
    g = np.zeros(n, np.float32)
    g[: vals.size] = vals
    gate = torch.from_numpy(g.reshape(-1, cols)).to(torch.bfloat16).to(dev)
    # fixed global scales: 1 resolves ordinary magnitudes, 1e-30 the huge ones
    # (with saturation to inf above), 1e30 the tiny ones
    for u, gsf in ((1.0, 1.0), (-3.0, 1.0), (1.0, 1e-30), (1.0, 1e30)):
        up = torch.full_like(gate, u)
        codes, scales = _run(dev, gate, up, gsf)
        co, so, _ = oracle.swiglu_rows(bits(gate), bits(up), gsf, threads=THREADS)
        check_full(codes, scales, gate.shape[0], cols, co, so, f"every gate, up={u}, gsf={gsf}")


def test_table_window_every_gate_and_its_edges(dev):
    """Every bf16 gate the per-CTA SiLU table holds (2^-25 <= |g| <= 127.5, both
    signs; above 87 its entries come from the general exponential) laid out so
    that whole warps take the table path, then the same rows with one gate per
    warp just outside the window (2^-25 minus one bf16 step, 127.5 plus one step),
    which sends those warps to the direct computation."""
    mags = np.arange(0x3300, 0x4300, dtype=np.uint16)
    gates = np.concatenate([mags, mags | np.uint16(0x8000)])
    rows, cols = 12, 8192
    gen = np.random.default_rng(7)
    g_bits = gates[gen.permutation(rows * cols) % gates.size].reshape(rows, cols)
    assert set(np.unique(g_bits)) == set(gates.tolist())
    up = workloads.swiglu_inputs(dev, rows=rows, cols=cols, seed=21)[1]
    for edge in (None, 0x32FF, 0x4300, 0xC300, 0xB2FF):
        gb = g_bits.copy()
        if edge is not None:
            gb[:, ::512] = edge  # one gate in every 512-column segment
        gate = torch.from_numpy(gb.view(np.int16)).view(torch.bfloat16).to(dev)
        gsf = _oracle_gsf(gate, up)
        codes, scales = _run(dev, gate, up, gsf)
        co, so, _ = oracle.swiglu_rows(bits(gate), bits(up), gsf, threads=THREADS)
        check_full(codes, scales, rows, cols, co, so, f"swiglu table window edge={edge}")


def test_packed_gate_up_projection_views(dev):
    """gate and up as the two halves of one [rows, 2F] projection (ld = 2F)."""
    rows, f = 200, 1536
    proj = workloads.swiglu_inputs(dev, rows=rows, cols=2 * f, seed=5)[0]
    gate, up = proj[:, :f], proj[:, f:]
    gsf = _oracle_gsf(gate, up)
    codes, scales = h3q.h3q_swiglu_nvfp4(gate, up, gsf_tensor(gsf, dev))
    co, so, _ = oracle.swiglu_rows(bits(gate), bits(up), gsf, threads=THREADS)
    check_full(codes, scales, rows, f, co, so, "packed projection")


def test_full_65280x18944_every_row(dev):
    """The 65,280 x 18,944 workload, gate and up ~ N(0, 1.5^2); gsf from a
    calibration pass of the oracle over 2,048 rows of the same seed; every byte of
    the codes and of the swizzled scales against the oracle."""
    gate, up = workloads.swiglu_inputs(dev)
    rows, cols = gate.shape
    calib = torch.arange(0, rows, rows // 2048, device=dev)[:2048]
    gsf = _oracle_gsf(gate.index_select(0, calib), up.index_select(0, calib))
    codes, scales = _run(dev, gate, up, gsf)
    co, so, _ = oracle.swiglu_rows(bits(gate), bits(up), gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, "swiglu 65280x18944")
