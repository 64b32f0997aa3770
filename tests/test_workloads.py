"""The seeded input generators: shapes, determinism and the planted structure."""
import torch

import workloads


def test_tiny_adaln_shapes_and_determinism():
    a = workloads.tiny_adaln_inputs("cpu")
    b = workloads.tiny_adaln_inputs("cpu")
    assert a["x"].shape == (64, 256) and a["gamma"].shape == (256,)
    assert a["table"].shape == (4, 2, 256) and a["rows_per_frame"] == 16
    assert all(a[k].dtype == torch.bfloat16 for k in ("x", "gamma", "table"))
    assert all(torch.equal(a[k], b[k]) for k in ("x", "gamma", "table"))
    assert abs(a["gamma"].float().mean().item() - 1.0) < 0.05


def test_quantize_inputs_planted_blocks():
    x = workloads.quantize_inputs("cpu", rows=64, cols=1024, zero_frac=0.01, outlier_frac=0.01)
    blocks = x.view(-1, 16).float()
    n = blocks.shape[0]
    zero = (blocks == 0).all(1).sum().item()
    outl = (blocks == 1000.0).any(1).sum().item()
    assert zero >= round(0.01 * n) and outl == round(0.01 * n)
    assert ((blocks == 1000.0).sum(1) <= 1).all()


def test_swiglu_and_attention_shapes():
    g, u = workloads.swiglu_inputs("cpu", rows=10, cols=128)
    assert g.shape == u.shape == (10, 128) and not torch.equal(g, u)
    a = workloads.attention_output("cpu", tokens=7, heads=2, head_dim=64)
    assert a.shape == (7, 128)


def test_sample_rows():
    s = workloads.sample_rows(1000, head=10, tail=10, random=50)
    assert s[0] == 0 and s[-1] == 999 and len(set(s.tolist())) == len(s)
    assert workloads.sample_rows(5).tolist() == [0, 1, 2, 3, 4]


def test_qkv_inputs_layout():
    w = workloads.qkv_inputs("cpu", rows=9, heads=3, head_dim=64, rot=32)
    assert w["q"].shape == w["k"].shape == w["v"].shape == (9, 192)
    assert w["q"].stride(0) == 3 * 192 and w["k"].data_ptr() - w["q"].data_ptr() == 192 * 2
    assert all(b.shape == (192,) for b in w["biases"])
    c, s = w["cos"].float(), w["sin"].float()
    assert c.shape == s.shape == (9, 32)
    assert torch.equal(c[:, :16], c[:, 16:]) and torch.equal(s[:, :16], s[:, 16:])  # halves share theta
    assert (c * c + s * s - 1).abs().max() < 0.02
    u = workloads.qkv_inputs("cpu", rows=9, heads=3, head_dim=64, rot=32, packed=False)
    assert u["q"].is_contiguous() and torch.equal(u["k"], w["k"])
    assert workloads.qkv_inputs("cpu", rows=2, heads=1, rot=0)["cos"] is None


def test_swiglu_packed_inputs_are_value_first():
    gate, up = workloads.swiglu_inputs("cpu", rows=5, cols=64)
    o, bias = workloads.swiglu_packed_inputs("cpu", rows=5, cols=64)
    assert o.shape == (5, 128) and bias.shape == (128,)
    assert torch.equal(o[:, :64], up) and torch.equal(o[:, 64:], gate)
    assert torch.equal(bias, workloads.swiglu_packed_inputs("cpu", rows=5, cols=64)[1])
