"""The producers inside a captured CUDA graph: every call only validates on the
host and launches on the caller's stream (no allocation, no synchronisation),
so a step of the AdaLN, SwiGLU, quantize, residual-fold, QKV-epilogue and
dynamic-scale calls captures into one graph.  Replays produce the same bytes as
eager calls, and replaying after the inputs change in place recomputes from the
new inputs.  The no-scratch dynamic quantize launches its quantize as a
programmatic dependent of the abs-max pass; captured, that becomes a graph edge,
also when the call is the process's first of it (its per-device lookups then
happen during the capture)."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _step(w, outs, stream):
    """One step of every producer, writing into the preallocated `outs`."""
    a, s, r, q, d = w["adaln"], w["swiglu"], w["residual"], w["qkv"], w["dyn"]
    h3q.h3q_rmsnorm_adaln_nvfp4(a["x"], a["gamma"], a["table"], w["gsf"], rows_per_frame=a["rows_per_frame"],
                                eps=a["eps"], codes=outs["a_codes"], scales=outs["a_scales"], stream=stream)
    h3q.h3q_swiglu_nvfp4(s[0], s[1], w["gsf"], outs["s_codes"], outs["s_scales"], stream=stream)
    h3q.h3q_quantize_nvfp4(w["attn"], w["gsf"], outs["q_codes"], outs["q_scales"], stream=stream)
    outs["h"].copy_(r["h"])  # the fold writes h in place: start each step from the same residual
    h3q.h3q_residual_rmsnorm_adaln_nvfp4(outs["h"], r["o"], r["gate"], r["gamma"], r["table"], w["gsf"],
                                         bias=r["bias"], rows_per_frame=r["rows_per_frame"], eps=r["eps"],
                                         codes=outs["r_codes"], scales=outs["r_scales"], stream=stream)
    h3q.h3q_qkv_epilogue(q["q"], q["k"], q["v"], q["biases"], q["cos"], q["sin"], q["heads"], q["eps"],
                         outs=[outs["qo"], outs["ko"], outs["vo"]], stream=stream)
    outs["amax"].zero_()
    h3q.h3q_rmsnorm_adaln_amax(d["x"], d["gamma"], d["table"], rows_per_frame=d["rows_per_frame"], eps=d["eps"],
                               amax=outs["amax"], stream=stream)
    h3q.h3q_global_scale_from_amax(outs["amax"], outs["dyn_gsf"], stream=stream)
    h3q.h3q_rmsnorm_adaln_nvfp4(d["x"], d["gamma"], d["table"], outs["dyn_gsf"], rows_per_frame=d["rows_per_frame"],
                                eps=d["eps"], codes=outs["d_codes"], scales=outs["d_scales"], stream=stream)
    h3q.h3q_quantize_nvfp4_dynamic(w["attn"], global_scale=outs["qd_gsf"], codes=outs["qd_codes"],
                                   scales=outs["qd_scales"], stream=stream)


def _buffers(w, dev):
    def nv(rows, cols):
        return (torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev),
                torch.empty((h3q.padded_rows(rows), cols // 16), dtype=torch.uint8, device=dev))

    outs = {}
    outs["a_codes"], outs["a_scales"] = nv(*w["adaln"]["x"].shape)
    outs["s_codes"], outs["s_scales"] = nv(*w["swiglu"][0].shape)
    outs["q_codes"], outs["q_scales"] = nv(*w["attn"].shape)
    outs["r_codes"], outs["r_scales"] = nv(*w["residual"]["o"].shape)
    outs["d_codes"], outs["d_scales"] = nv(*w["dyn"]["x"].shape)
    outs["qd_codes"], outs["qd_scales"] = nv(*w["attn"].shape)
    outs["qd_gsf"] = torch.zeros(1, dtype=torch.float32, device=dev)
    outs["h"] = torch.empty_like(w["residual"]["h"])
    q = w["qkv"]
    for name in ("qo", "ko", "vo"):
        outs[name] = torch.empty((q["q"].shape[0], q["heads"], q["head_dim"]), dtype=torch.bfloat16, device=dev)
    outs["amax"] = torch.zeros(1, dtype=torch.float32, device=dev)
    outs["dyn_gsf"] = torch.zeros(1, dtype=torch.float32, device=dev)
    return outs


def test_producers_in_a_captured_graph(dev):
    w = {
        "adaln": workloads.adaln_inputs(dev, rows=1000, frames=1, rows_per_frame=1000, seed=41),
        "swiglu": workloads.swiglu_inputs(dev, rows=300, cols=1024, seed=42),
        "attn": workloads.attention_output(dev, tokens=700, seed=43),
        "residual": workloads.residual_inputs(dev, rows=400, cols=2048, frames=2, rows_per_frame=200, seed=44),
        "qkv": workloads.qkv_inputs(dev, rows=123, heads=4, seed=45),
        "dyn": workloads.adaln_inputs(dev, rows=500, frames=1, rows_per_frame=500, seed=46),
        "gsf": torch.tensor([30.0], dtype=torch.float32, device=dev),
    }
    side = torch.cuda.Stream(dev)
    eager = _buffers(w, dev)
    with torch.cuda.stream(side):
        _step(w, eager, side)  # also fills the library's per-kernel launch caches
    side.synchronize()

    outs = _buffers(w, dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        _step(w, outs, side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for k in eager:
        assert torch.equal(outs[k].view(torch.uint8), eager[k].view(torch.uint8)), f"graph replay differs: {k}"

    # change inputs in place: a replay recomputes from them
    w["attn"].mul_(-1)
    w["dyn"]["x"].mul_(2)
    graph.replay()
    with torch.cuda.stream(side):
        _step(w, eager, side)
    torch.cuda.synchronize()
    for k in ("q_codes", "q_scales", "d_codes", "d_scales", "dyn_gsf", "qd_codes", "qd_scales", "qd_gsf"):
        assert torch.equal(outs[k].view(torch.uint8), eager[k].view(torch.uint8)), f"replay after update: {k}"


_FIRST_CALL_CAPTURED = textwrap.dedent("""
    import torch
    import nvfp4_activation_quantize_gb300 as h3q
    import workloads
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    x = workloads.attention_output(dev, tokens=1000, seed=47)
    codes = torch.empty((1000, x.shape[1] // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((h3q.padded_rows(1000), x.shape[1] // 16), dtype=torch.uint8, device=dev)
    gsf = torch.zeros(1, dtype=torch.float32, device=dev)
    side = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):  # the process's first call of the entry point
        h3q.h3q_quantize_nvfp4_dynamic(x, global_scale=gsf, codes=codes, scales=scales, stream=side)
    graph.replay()
    torch.cuda.synchronize()
    c, s, g = h3q.h3q_quantize_nvfp4_dynamic(x)
    torch.cuda.synchronize()
    assert torch.equal(codes, c) and torch.equal(scales, s) and torch.equal(gsf, g), "replay differs"
    x.mul_(0.25)
    graph.replay()
    c, s, g = h3q.h3q_quantize_nvfp4_dynamic(x)
    torch.cuda.synchronize()
    assert torch.equal(codes, c) and torch.equal(scales, s) and torch.equal(gsf, g), "replay after update"
    print("ok")
""")


def test_dynamic_quantize_first_called_inside_a_capture(dev):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([root, os.path.join(root, "tests")]))
    res = subprocess.run([sys.executable, "-c", _FIRST_CALL_CAPTURED], cwd=root, env=env, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout[-2000:] + res.stderr[-2000:]
