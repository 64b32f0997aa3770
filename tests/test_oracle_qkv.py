"""The oracle's QKV epilogue against what fixes it independently:
the bias add in numpy binary32 with torch's bf16 rounding; the per-head rstd
equal to the AdaLN oracle's row rstd on the same 128 values (for a row of HD
columns the two canonical orders coincide) and within 1e-6 of binary64; the
rotate-half RoPE, op by op in numpy with torch's bf16 rounding, on the normed
values; the pass-through of the values beyond ROT."""
import numpy as np
import pytest
import torch

import oracle

HD = 128


def _bf16(values) -> np.ndarray:
    return torch.as_tensor(np.asarray(values, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def _r(values) -> np.ndarray:
    """fp32 values rounded to bf16 (as fp32)."""
    return _val(_bf16(values))


def _inputs(n, heads, rot, seed):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((n, heads * HD)) * 3)
    b = _bf16(rng.standard_normal(heads * HD) * 0.2)
    ang = rng.uniform(0, 2 * np.pi, (n, rot // 2))
    cos = _bf16(np.concatenate([np.cos(ang), np.cos(ang)], 1))
    sin = _bf16(np.concatenate([np.sin(ang), np.sin(ang)], 1))
    return x, b, cos, sin


def test_v_gets_the_bias_only():
    x, b, cos, sin = _inputs(9, 4, 64, 1)
    out = oracle.qkv_epilogue_rows(x, b, 4, cos, sin, 1e-6, is_v=True)
    want = _bf16(_val(x) + _val(b)[None, :]).reshape(9, 4, HD)
    assert np.array_equal(out, want)


def _normed(x, b, heads, n):
    """The normed heads through the oracle itself, with cos = 1 and sin = 0 (the
    rotation then leaves n unchanged: n + 0)."""
    ones = _bf16(np.ones((n, 16)))
    zeros = _bf16(np.zeros((n, 16)))
    return oracle.qkv_epilogue_rows(x, b, heads, ones, zeros, 1e-6, is_v=False)


def test_head_rstd_is_the_adaln_row_rstd_of_the_head():
    n, heads = 6, 3
    x, b, _, _ = _inputs(n, heads, 64, 2)
    xb = _bf16(_val(x) + _val(b)[None, :])          # x' = bf16(x + b)
    normed = _val(_normed(x, b, heads, n).reshape(n, heads * HD))
    for r in range(n):
        for h in range(heads):
            head = xb[r, h * HD:(h + 1) * HD][None, :]
            rstd = oracle.adaln_rows(head, _bf16(np.ones(HD)), _bf16(np.zeros((1, 2, HD))), [0], 1e-6,
                                     None)[2][0]
            want = _r(_val(head[0]) * np.float32(rstd))
            got = normed[r, h * HD:(h + 1) * HD]
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
            exact = 1 / np.sqrt((_val(head[0]).astype(np.float64) ** 2).mean() + np.float64(np.float32(1e-6)))
            assert abs(rstd - exact) / exact <= 1e-6


@pytest.mark.parametrize("rot", [16, 64, 128])
def test_rotate_half_rope_op_by_op(rot):
    n, heads = 5, 2
    x, b, cos, sin = _inputs(n, heads, rot, rot)
    nrm = _val(_normed(x, b, heads, n))                         # [n, heads, HD]
    out = _val(oracle.qkv_epilogue_rows(x, b, heads, cos, sin, 1e-6, is_v=False))
    c, s = _val(cos)[:, None, :], _val(sin)[:, None, :]
    first = nrm[..., :rot]
    rotated = np.concatenate([-first[..., rot // 2:], first[..., :rot // 2]], -1)
    want = _r(_r(first * c) + _r(rotated * s))
    assert np.array_equal(out[..., :rot].view(np.uint32), want.view(np.uint32))
    assert np.array_equal(out[..., rot:].view(np.uint32), nrm[..., rot:].view(np.uint32))


def test_no_tables_is_the_norm_without_a_rotation():
    """ROT = 0 (no cos/sin tables) leaves every normed value as it is: the same as
    ROT = 16 with cos = 1 and sin = 0 (n * 1 + r * 0 = n exactly)."""
    n, heads = 7, 3
    x, b, _, _ = _inputs(n, heads, 64, 12)
    got = oracle.qkv_epilogue_rows(x, b, heads, None, None, 1e-6, is_v=False)
    assert np.array_equal(got, _normed(x, b, heads, n))


@pytest.mark.parametrize("rot", [16, 64, 128])
def test_interleaved_rope_op_by_op(rot):
    """Pairs (2j, 2j+1) rotated together: r_2j = -n_2j+1, r_2j+1 = n_2j."""
    n, heads = 5, 2
    x, b, cos, sin = _inputs(n, heads, rot, rot + 1)
    nrm = _val(_normed(x, b, heads, n))
    out = _val(oracle.qkv_epilogue_rows(x, b, heads, cos, sin, 1e-6, is_v=False, interleaved=True))
    c, s = _val(cos)[:, None, :], _val(sin)[:, None, :]
    first = nrm[..., :rot]
    rotated = np.empty_like(first)
    rotated[..., 0::2] = -first[..., 1::2]
    rotated[..., 1::2] = first[..., 0::2]
    want = _r(_r(first * c) + _r(rotated * s))
    assert np.array_equal(out[..., :rot].view(np.uint32), want.view(np.uint32))
    assert np.array_equal(out[..., rot:].view(np.uint32), nrm[..., rot:].view(np.uint32))


def test_interleaved_is_rotate_half_in_permuted_coordinates():
    """Interleaved RoPE on a head equals rotate-half RoPE on the head with its first
    ROT values permuted (element 2j -> j, 2j+1 -> j + ROT/2) and cos/sin permuted the
    same way, permuted back: the norm is order-independent only in exact arithmetic,
    so the heads here are built so every partial sum is exact (values in {0, +-1, +-2})."""
    n, heads, rot = 4, 3, 64
    rng = np.random.default_rng(21)
    x = _bf16(rng.choice([-2.0, -1.0, 0.0, 1.0, 2.0], size=(n, heads * HD)))
    b = _bf16(np.zeros(heads * HD))
    _, _, cos, sin = _inputs(n, heads, rot, 22)
    perm = np.concatenate([np.arange(0, rot, 2), np.arange(1, rot, 2), np.arange(rot, HD)])
    xp = x.reshape(n, heads, HD)[..., perm].reshape(n, heads * HD)
    cp, sp = cos[:, perm[:rot]], sin[:, perm[:rot]]
    half = oracle.qkv_epilogue_rows(xp, b, heads, cp, sp, 1e-6, is_v=False)
    inter = oracle.qkv_epilogue_rows(x, b, heads, cos, sin, 1e-6, is_v=False, interleaved=True)
    back = np.empty_like(half)
    back[..., perm] = half
    assert np.array_equal(back, inter)
