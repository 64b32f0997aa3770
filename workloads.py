"""Seeded synthetic inputs for the NVFP4 activation producers.

Shared by the tests, the smoke check and the benchmark; holds none of the
method's arithmetic (no normalisation, no SiLU, no quantize, no scale
formula).  Every tensor is drawn from a ``torch.Generator`` on the requested
device, in fp32, and rounded to bf16.  Shapes follow the workloads the pages
describe for MiniMax-H3 video DiT serving:

* hidden width 7,168 = 56 heads x 128 (the attention-output shape of the
  FastVideo commit log's int64 fix: 56 x 128 per token);
* 65,280 tokens = 32 latent frames x 2,040 tokens (544 x 960 at 16x spatial
  downsampling is 34 x 60 = 2,040 tokens per frame), row -> frame = row // 2,040;
* FFN width 18,944 for the SwiGLU producer (and the FFN-up GEMM: 7,168 ->
  2 x 18,944, value/gate-paired weight rows);
* 300,000 tokens for the attention output crosses 2^31 elements (the pages'
  boundary for 56 x 128 is 299,593 tokens).

No public dataset is involved; these stand in for the pages' private prompts.
"""
from __future__ import annotations

import torch

HIDDEN = 7168
FFN = 18944
TOKENS = 65280
FRAMES = 32
TOKENS_PER_FRAME = 2040
ATTN_TOKENS = 300_000

_CHUNK_ELEMS = 1 << 27  # fp32 scratch per draw: 512 MiB at most


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(rows: int, cols: int, gen, device, std: float = 1.0, mean: float = 0.0,
                 col_scale: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 [rows, cols] ~ mean + std * N(0, 1) (optionally times a per-column factor),
    drawn in row chunks so the fp32 scratch stays bounded."""
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    step = max(1, _CHUNK_ELEMS // max(cols, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        z = torch.randn((r1 - r0, cols), generator=gen, device=device, dtype=torch.float32)
        if col_scale is not None:
            z.mul_(col_scale)
        if std != 1.0:
            z.mul_(std)
        if mean != 0.0:
            z.add_(mean)
        out[r0:r1].copy_(z)
        del z
    return out


def adaln_inputs(device, rows: int = TOKENS, cols: int = HIDDEN, frames: int = FRAMES,
                 rows_per_frame: int = TOKENS_PER_FRAME, seed: int = 3,
                 channel_lognormal_sigma: float = 0.5, table_std: float = 0.3) -> dict:
    """RMSNorm + AdaLN producer inputs.

    x ~ N(0, 1) * s_j with per-channel s_j ~ LogNormal(0, channel_lognormal_sigma)
    (0 disables it), gamma ~ N(1, 0.1), modulation table [frames, 2, cols] ~
    N(0, table_std) ([t, 0] shift, [t, 1] scale), eps 1e-6.
    """
    gen = _gen(device, seed)
    col_scale = None
    if channel_lognormal_sigma:
        col_scale = torch.exp(channel_lognormal_sigma *
                              torch.randn(cols, generator=gen, device=device, dtype=torch.float32))
    x = _normal_bf16(rows, cols, gen, device, col_scale=col_scale)
    gamma = _normal_bf16(1, cols, gen, device, std=0.1, mean=1.0).reshape(cols)
    table = _normal_bf16(frames * 2, cols, gen, device, std=table_std).reshape(frames, 2, cols)
    return {"x": x, "gamma": gamma, "table": table, "rows_per_frame": rows_per_frame, "eps": 1e-6}


def residual_inputs(device, rows: int = TOKENS, cols: int = HIDDEN, frames: int = FRAMES,
                    rows_per_frame: int = TOKENS_PER_FRAME, seed: int = 6, bias: bool = True) -> dict:
    """Residual fold + RMSNorm + AdaLN inputs: the fp32 residual h ~ 4 * N(0, 1) * s_j
    with per-channel s_j ~ LogNormal(0, 0.5), the MLP output o ~ N(0, 1) (bf16), a bias
    ~ N(0, 0.1) (bf16, or None), the gate table [frames, cols] ~ N(0, 0.3), gamma ~
    N(1, 0.1) and the modulation table [frames, 2, cols] ~ N(0, 0.3); eps 1e-6."""
    gen = _gen(device, seed)
    col_scale = torch.exp(0.5 * torch.randn(cols, generator=gen, device=device, dtype=torch.float32))
    h = torch.empty((rows, cols), dtype=torch.float32, device=device)
    step = max(1, _CHUNK_ELEMS // max(cols, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        h[r0:r1] = torch.randn((r1 - r0, cols), generator=gen, device=device) * col_scale * 4.0
    o = _normal_bf16(rows, cols, gen, device)
    b = _normal_bf16(1, cols, gen, device, std=0.1).reshape(cols) if bias else None
    gate = _normal_bf16(frames, cols, gen, device, std=0.3)
    gamma = _normal_bf16(1, cols, gen, device, std=0.1, mean=1.0).reshape(cols)
    table = _normal_bf16(frames * 2, cols, gen, device, std=0.3).reshape(frames, 2, cols)
    return {"h": h, "o": o, "bias": b, "gate": gate, "gamma": gamma, "table": table,
            "rows_per_frame": rows_per_frame, "eps": 1e-6}


def tiny_adaln_inputs(device, seed: int = 1) -> dict:
    """The tiny bit-exactness case: x [64, 256] ~ N(0, 1), gamma ~ N(1, 0.1),
    table [4, 2, 256] ~ N(0, 0.2), row -> frame = row // 16, eps 1e-6."""
    return adaln_inputs(device, rows=64, cols=256, frames=4, rows_per_frame=16, seed=seed,
                        channel_lognormal_sigma=0.0, table_std=0.2)


def quantize_inputs(device, rows: int = 8192, cols: int = HIDDEN, seed: int = 2,
                    dof: int = 3, scale: float = 2.0, zero_frac: float = 0.001,
                    outlier_frac: float = 0.001, outlier: float = 1000.0) -> torch.Tensor:
    """Standalone quantize input: Student-t(dof) x scale, with a fraction of the
    16-element blocks all zero and another fraction holding one +outlier element
    at a random position."""
    gen = _gen(device, seed)
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    step = max(1, _CHUNK_ELEMS // (cols * (dof + 1)))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        z = torch.randn((dof + 1, r1 - r0, cols), generator=gen, device=device)
        chi2 = (z[1:] * z[1:]).sum(0).div_(dof)
        x[r0:r1].copy_(z[0].div_(chi2.sqrt_()).mul_(scale))
        del z, chi2
    blocks = rows * cols // 16
    n_zero = int(round(blocks * zero_frac))
    n_out = int(round(blocks * outlier_frac))
    if n_zero + n_out:
        pick = torch.randperm(blocks, generator=gen, device=device)[: n_zero + n_out]
        flat = x.view(blocks, 16)
        flat[pick[:n_zero]] = 0
        pos = torch.randint(0, 16, (n_out,), generator=gen, device=device)
        flat[pick[n_zero:], pos] = outlier
    return x


def swiglu_inputs(device, rows: int = TOKENS, cols: int = FFN, seed: int = 4,
                  std: float = 1.5) -> tuple[torch.Tensor, torch.Tensor]:
    """gate, up bf16 [rows, cols] ~ N(0, std^2)."""
    gen = _gen(device, seed)
    gate = _normal_bf16(rows, cols, gen, device, std=std)
    up = _normal_bf16(rows, cols, gen, device, std=std)
    return gate, up


def swiglu_packed_inputs(device, rows: int = TOKENS, cols: int = FFN, seed: int = 4, std: float = 1.5,
                         bias_std: float = 0.2) -> tuple[torch.Tensor, torch.Tensor]:
    """The value-first packed projection o [rows, 2 * cols] = [up | gate] with the
    values of swiglu_inputs(seed), and its bias [2 * cols] ~ N(0, bias_std^2)
    (drawn from seed + 100)."""
    gate, up = swiglu_inputs(device, rows=rows, cols=cols, seed=seed, std=std)
    o = torch.cat([up, gate], 1)
    del gate, up
    bias = _normal_bf16(1, 2 * cols, _gen(device, seed + 100), device, std=bias_std).reshape(2 * cols)
    return o, bias


def attention_output(device, tokens: int = ATTN_TOKENS, heads: int = 56, head_dim: int = 128,
                     seed: int = 5) -> torch.Tensor:
    """Attention output bf16 [1, tokens, heads, head_dim] ~ N(0, 1), returned as the
    [tokens, heads * head_dim] view that is quantized along its last axis."""
    gen = _gen(device, seed)
    return _normal_bf16(tokens, heads * head_dim, gen, device)


def qkv_inputs(device, rows: int = TOKENS, heads: int = 56, head_dim: int = 128, rot: int = 64,
               seed: int = 7, packed: bool = True) -> dict:
    """QKV epilogue inputs: the projection output [rows, 3 * heads * head_dim] bf16 ~
    N(0, 1) * s_j with per-channel s_j ~ LogNormal(0, 0.5) (q, k and v are its three
    column slices when `packed`, else three contiguous tensors of the same values),
    biases [heads * head_dim] ~ N(0, 0.1), and cos/sin [rows, rot] bf16 of an angle
    theta ~ U(0, 2 pi) per row and pair, the pair's two halves sharing the angle
    (the rotate-half table layout); eps 1e-6."""
    import math

    gen = _gen(device, seed)
    d = heads * head_dim
    col_scale = torch.exp(0.5 * torch.randn(3 * d, generator=gen, device=device, dtype=torch.float32))
    proj = _normal_bf16(rows, 3 * d, gen, device, col_scale=col_scale)
    if packed:
        q, k, v = proj[:, :d], proj[:, d:2 * d], proj[:, 2 * d:]
    else:
        q, k, v = (proj[:, i * d:(i + 1) * d].contiguous() for i in range(3))
        del proj
    biases = tuple(_normal_bf16(1, d, gen, device, std=0.1).reshape(d) for _ in range(3))
    cos = sin = None
    if rot:
        theta = torch.rand((rows, rot // 2), generator=gen, device=device) * (2 * math.pi)
        cos = torch.cat([theta.cos(), theta.cos()], 1).to(torch.bfloat16)
        sin = torch.cat([theta.sin(), theta.sin()], 1).to(torch.bfloat16)
    return {"q": q, "k": k, "v": v, "biases": biases, "cos": cos, "sin": sin, "heads": heads,
            "head_dim": head_dim, "rot": rot, "eps": 1e-6}


def ffn_up_inputs(device, rows: int = TOKENS, hidden: int = HIDDEN, ffn: int = FFN, seed: int = 8,
                  w_std: float | None = None) -> dict:
    """The FFN-up projection's bf16 operands before their NVFP4 quantize: the
    activation x [rows, hidden] ~ N(0, 1) * s_j with per-channel s_j ~
    LogNormal(0, 0.5) (a normed, modulated hidden state), and the weight
    w [2 * ffn, hidden] ~ N(0, w_std^2), w_std = 1 / sqrt(hidden) by default,
    its rows interleaved as (value, gate) pairs: row 2j the value and row 2j+1
    the gate of output j.  (Random-init weights; no checkpoint is involved.)"""
    g = _gen(device, seed)
    s = torch.exp(torch.randn(hidden, generator=g, device=device) * 0.5)
    x = _normal_bf16(rows, hidden, g, device, col_scale=s)
    std = hidden ** -0.5 if w_std is None else w_std
    w = _normal_bf16(2 * ffn, hidden, g, device, std=std)
    return {"x": x, "w": w}


def sample_rows(rows: int, head: int = 256, tail: int = 256, random: int = 4096,
                seed: int = 0) -> torch.Tensor:
    """Row indices for sampled checks on full-size outputs: the first `head`, the
    last `tail` and `random` others, sorted and unique (CPU int64)."""
    g = torch.Generator().manual_seed(seed)
    parts = [torch.arange(min(head, rows)), torch.arange(max(0, rows - tail), rows)]
    if rows > 0 and random:
        parts.append(torch.randint(0, rows, (random,), generator=g))
    return torch.unique(torch.cat(parts))
