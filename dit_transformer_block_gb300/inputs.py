"""Seeded synthetic inputs shaped like the packed audio-video DiT workload.

This module only draws random numbers and lays out positions; it holds none of
the block's arithmetic. Both the CUDA path and the CPU oracle take its output.

Workload shape (from the vLLM-Omni H3 blog, section 3.1): one packed sequence
of text, audio and video tokens, L valid rows inside an aligned buffer of S
rows (58,758 in 58,816), hidden width 5,376. Weights and activations are drawn
here because no trained checkpoint is used.

Recipe (fixed draw order per seed, torch.Generator, float32 draws rounded to
bf16 where the tensor is bf16):
    x ~ N(0,1), W_qkv, W_o, W_gu, W_down ~ N(0, 0.02), g_q, g_k ~ 1 + N(0, 0.1),
    mod [6, D] ~ N(0, 0.1) float32, then N(0,1) garbage for the pad rows.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class BlockShape:
    S: int          # buffer rows (aligned)
    L: int          # valid rows
    D: int          # hidden width = H * Dh
    H: int          # heads
    Dh: int         # head dim
    F: int          # SwiGLU inner width
    axis_dims: tuple = (128, 0, 0)
    theta: float = 1e4
    eps_ln: float = 1e-6
    eps_qk: float = 1e-6
    pos_kind: str = "1d"   # "1d" or "3d"
    grid: tuple = (31, 24, 79)   # (t, h, w) latent grid of the video tokens ("3d")
    n_tail: int = 22             # trailing audio/text tokens ("3d")


# Tiny single block: 250 valid tokens in a 256 buffer, 1D RoPE.
TINY = BlockShape(S=256, L=250, D=512, H=4, Dh=128, F=1536)
# The packed 10 s workload: 58,758 valid of 58,816, 42 x 128 heads, 3-axis RoPE.
FULL = BlockShape(S=58816, L=58758, D=5376, H=42, Dh=128, F=14336,
                  axis_dims=(32, 48, 48), pos_kind="3d")


def positions_1d(S: int, L: int) -> torch.Tensor:
    """[S, 3] int32: (p, 0, 0) for p < L, zeros in the pad rows."""
    pos = torch.zeros(S, 3, dtype=torch.int32)
    pos[:L, 0] = torch.arange(L, dtype=torch.int32)
    return pos


def positions_3d(S: int, L: int, grid=(31, 24, 79), n_tail: int = 22) -> torch.Tensor:
    """[S, 3] int32 (t, h, w) positions of a packed video + audio/text sequence.

    The first L - n_tail tokens walk the latent grid in (t, h, w) row-major
    order (truncated when the grid holds more cells than that); the n_tail
    trailing tokens carry t = h = w = T + i, i.e. they continue after the
    last temporal index. Pad rows are zero.
    """
    T, Hh, W = grid
    n_vid = L - n_tail
    assert 0 <= n_vid <= T * Hh * W
    idx = torch.arange(n_vid, dtype=torch.int64)
    pos = torch.zeros(S, 3, dtype=torch.int32)
    pos[:n_vid, 0] = (idx // (Hh * W)).to(torch.int32)
    pos[:n_vid, 1] = ((idx // W) % Hh).to(torch.int32)
    pos[:n_vid, 2] = (idx % W).to(torch.int32)
    tail = torch.arange(n_tail, dtype=torch.int32) + T
    pos[n_vid:L, 0] = tail
    pos[n_vid:L, 1] = tail
    pos[n_vid:L, 2] = tail
    return pos


def positions(shape: BlockShape) -> torch.Tensor:
    if shape.pos_kind == "3d":
        return positions_3d(shape.S, shape.L, shape.grid, shape.n_tail)
    return positions_1d(shape.S, shape.L)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(g, shape, std=1.0, mean=0.0, device="cpu", dtype=torch.bfloat16):
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def block_inputs(shape: BlockShape, seed: int, device="cpu") -> dict:
    """All inputs of one block forward. bf16 tensors except resid/mod/gains (fp32).

    x is drawn N(0,1) as bf16 and handed to the block as the FP32 residual
    stream (an exact upcast). Pad rows of x are overwritten with fresh N(0,1)
    garbage drawn last, which no valid output may depend on.
    """
    g = _gen(seed, device)
    S, L, D, F, Dh = shape.S, shape.L, shape.D, shape.F, shape.Dh
    x = _randn(g, (S, D), device=device)
    w_qkv = _randn(g, (3 * D, D), 0.02, device=device)
    w_o = _randn(g, (D, D), 0.02, device=device)
    w_gu = _randn(g, (2 * F, D), 0.02, device=device)
    w_down = _randn(g, (D, F), 0.02, device=device)
    q_gain = _randn(g, (Dh,), 0.1, 1.0, device=device, dtype=torch.float32)
    k_gain = _randn(g, (Dh,), 0.1, 1.0, device=device, dtype=torch.float32)
    mod = _randn(g, (6, D), 0.1, device=device, dtype=torch.float32)
    if S > L:
        x[L:] = _randn(g, (S - L, D), device=device)
    return dict(resid=x.float(), w_qkv=w_qkv, w_o=w_o, w_gu=w_gu, w_down=w_down,
                q_gain=q_gain, k_gain=k_gain, mod=mod,
                pos=positions(shape).to(device))


def qk_inputs(S: int, L: int, H: int, Dh: int, seed: int, device="cpu") -> dict:
    """q, k ~ N(0,1) bf16 [S, H, Dh] (pad rows included), gains ~ 1 + N(0, 0.1)."""
    g = _gen(seed, device)
    q = _randn(g, (S, H, Dh), device=device)
    k = _randn(g, (S, H, Dh), device=device)
    q_gain = _randn(g, (Dh,), 0.1, 1.0, device=device, dtype=torch.float32)
    k_gain = _randn(g, (Dh,), 0.1, 1.0, device=device, dtype=torch.float32)
    return dict(q=q, k=k, q_gain=q_gain, k_gain=k_gain)


def attention_inputs(S: int, L: int, H: int, Dh: int, seed: int, device="cpu") -> dict:
    """q, k drawn N(0,1) and rescaled to unit root-mean-square per (row, head)
    (the distribution normalised Q/K have), v ~ N(0,1); all bf16 [S, H, Dh]."""
    g = _gen(seed, device)

    def unit_rms(t):
        return t / t.pow(2).mean(dim=-1, keepdim=True).sqrt()

    q = unit_rms(torch.randn(S, H, Dh, generator=g, device=device)).to(torch.bfloat16)
    k = unit_rms(torch.randn(S, H, Dh, generator=g, device=device)).to(torch.bfloat16)
    v = torch.randn(S, H, Dh, generator=g, device=device).to(torch.bfloat16)
    return dict(q=q, k=k, v=v)


def frame_local_attention_inputs(S: int, L: int, H: int, Dh: int, frame: int, seed: int,
                                 device="cpu", strength: float = 16.0) -> dict:
    """Attention inputs with frame locality (tokens of one frame attend mostly
    to each other): rows are grouped into frames of `frame` consecutive rows;
    every (frame, head) draws a random unit direction e, and q = n_q +
    strength * e, k = n_k + strength * e with n_q, n_k ~ N(0,1) per channel;
    v ~ N(0,1); all bf16 [S, H, Dh]. At strength 16 and Dh = 128 a query's
    logits against its own frame sit about 30 base-2 units above those
    against other frames (softmax scale Dh^-1/2)."""
    g = _gen(seed, device)
    nf = (S + frame - 1) // frame
    e = torch.randn(nf, H, Dh, generator=g, device=device)
    e = e / e.norm(dim=-1, keepdim=True)
    ef = e.repeat_interleave(frame, dim=0)[:S] * strength
    q = (torch.randn(S, H, Dh, generator=g, device=device) + ef).to(torch.bfloat16)
    k = (torch.randn(S, H, Dh, generator=g, device=device) + ef).to(torch.bfloat16)
    v = torch.randn(S, H, Dh, generator=g, device=device).to(torch.bfloat16)
    return dict(q=q, k=k, v=v)


def swiglu_inputs(S: int, F: int, seed: int, device="cpu") -> dict:
    """gate_up ~ N(0, 1.5^2) bf16 [S, 2F] (the spread of an FFN up-projection)."""
    g = _gen(seed, device)
    return dict(gate_up=_randn(g, (S, 2 * F), 1.5, device=device))


def mod_inputs(S: int, D: int, seed: int, device="cpu") -> dict:
    """resid ~ N(0,1) fp32 [S, D], delta ~ N(0,1) bf16, mod [6, D] ~ N(0, 0.1)."""
    g = _gen(seed, device)
    resid = torch.randn(S, D, generator=g, device=device)
    delta = _randn(g, (S, D), device=device)
    mod = _randn(g, (6, D), 0.1, device=device, dtype=torch.float32)
    return dict(resid=resid, delta=delta, mod=mod)
