"""CPU oracle for the joint audio-video DiT block forward (test infrastructure).

This module is TEST INFRASTRUCTURE. Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it. The product path (the CUDA
library and its Python binding) never calls it and shares no code with it.

It is a plain, slow, obviously correct restatement of what the block computes,
written in NumPy with every intermediate in float64. Values are rounded to
bfloat16 (round to nearest, ties to even) only where the block hands a bf16
tensor from one step to the next, and the FP32 residual stream is rounded to
float32 where it is stored. Every function cites the passage of the source
pages it follows. The pages are:

  [vLLM-Omni H3 blog] "vLLM-Omni 上的 MiniMax H3：从系统级优化到基于 FastVideo
      FastH3 的实时服务" (the Chinese blog post), sections 3.1 and 3.2.
  [H3 blog PR] "MiniMax H3 on vLLM-Omni: From System-Wide Optimization to
      Real-Time Serving with FastVideo's FastH3" (the English PR thread).

What the pages fix: one packed sequence of text, audio and video tokens whose
first L rows are valid inside an aligned buffer of S rows (58,758 in 58,816);
attention takes the valid length and does no work on the tail padding; the
hidden state is 5,376 wide; the small fused ops are per-head Q/K RMSNorm with
RoPE, FP32 modulation + normalisation + residual, and SwiGLU in place of a
separate SiLU and multiply (blog section 3.1, section 3.2). The pages print no
equations, so the formulas below are the plainest readings, listed here:

  * modulation norm: LayerNorm without affine over the hidden axis, eps 1e-6,
    h = LN(r) * (1 + scale) + shift; residual r <- r + gate * y.
  * modulation vector [6, D] FP32 in the order (shift, scale, gate) for the
    attention branch, then (shift, scale, gate) for the FFN branch.
  * Q/K norm: RMSNorm per head over head_dim, x / sqrt(mean(x^2) + eps) * g,
    one FP32 gain vector of length head_dim for Q and one for K.
  * RMSNorm first, then RoPE.
  * RoPE: head_dim is split into axis sections (d_0, d_1, d_2) for positions
    (t, h, w); inside section a the pair (o_a + 2j, o_a + 2j + 1) is rotated by
    angle pos_a * theta^(-2j / d_a) (interleaved pairs, section-local exponent).
  * QKV weight rows are [q | k | v], each head-major; the FFN up weight rows
    are [gate | up]; no biases.
  * attention: softmax(q k^T * scale) v over keys [0, L), bidirectional;
    output rows >= L are not produced.
  * SwiGLU: u = SiLU(g) * v with SiLU(g) = g / (1 + exp(-g)).

Parity pins: every function here is checked in tests/test_oracle_pins.py
against closed forms, invariants, library routines on special cases and brute
force on tiny inputs; none is unpinned.
"""
from __future__ import annotations

import numpy as np

# bf16 has 8 significant bits (1 implicit + 7 stored) and the exponent range
# of float32: the smallest normal is 2^-126, subnormals step in 2^-133.
_BF16_SIG_BITS = 8
_BF16_MIN_QUANTUM_EXP = -133
_BF16_MAX = float.fromhex("0x1.fep127")


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    Written from the definition of the format: a finite x = m * 2^e with
    0.5 <= |m| < 1 is rounded to a multiple of the quantum 2^(e - 8) (never
    finer than the subnormal step 2^-133); np.rint rounds half to even.
    Scaling by a power of two is exact, so the only rounding is the one asked
    for. Values beyond the largest bf16 become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    finite = np.isfinite(x) & (x != 0)
    _, e = np.frexp(x[finite])
    q = np.maximum(e - _BF16_SIG_BITS, _BF16_MIN_QUANTUM_EXP).astype(np.float64)
    scale = np.exp2(q)
    r = np.rint(x[finite] / scale) * scale
    r = np.where(np.abs(r) > _BF16_MAX, np.sign(r) * np.inf, r)
    out[finite] = r
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def round_f32(x) -> np.ndarray:
    """Round float64 values to float32 (numpy's cast is round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# a1: FP32 modulation + normalisation + residual
# [vLLM-Omni H3 blog] section 3.2: "FP32 modulation, normalisation and residual"
# merged into one op (#6281, #6878); [H3 blog PR] fused-ops summary.
# ---------------------------------------------------------------------------

def layer_norm(x, eps: float) -> np.ndarray:
    """LayerNorm without affine over the last axis: (x - mean) / sqrt(var + eps)."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def mod_norm_residual(resid, delta=None, gate=None, shift=None, scale=None,
                      eps: float = 1e-6):
    """One modulation/normalisation/residual step on the FP32 residual stream.

    resid [rows, D] float32 values; delta [rows, D] bf16 values or None;
    gate, shift, scale [D] float32 values or None.
      r' = r + gate * delta          (when delta is given), stored as float32
      h  = LN(r') * (1 + scale) + shift  (when shift/scale are given), bf16
    Returns (r', h) with h None when no norm output is asked for.
    """
    r = np.asarray(resid, dtype=np.float64)
    if delta is not None:
        r = round_f32(r + np.asarray(gate, np.float64)[None, :] * np.asarray(delta, np.float64))
    h = None
    if scale is not None:
        n = layer_norm(r, eps)
        h = round_bf16(n * (1.0 + np.asarray(scale, np.float64)[None, :])
                       + np.asarray(shift, np.float64)[None, :])
    return r, h


# ---------------------------------------------------------------------------
# a2: per-head Q/K RMSNorm + rotary position embedding
# [vLLM-Omni H3 blog] section 3.2: Q/K RMSNorm fused with RoPE (#5990);
# section 3.1: rank-local RoPE rows built from each token's positions.
# ---------------------------------------------------------------------------

def rms_norm(x, gain, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = (x * x).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gain, np.float64)


def rope_angles(pos, axis_dims, theta: float) -> np.ndarray:
    """Rotation angle of every pair: [rows, head_dim // 2], float64.

    pos [rows, 3] integer positions (t, h, w); axis_dims (d_0, d_1, d_2) with
    even entries summing to head_dim. Pair j of section a turns by
    pos_a * theta^(-2j / d_a).
    """
    pos = np.asarray(pos, dtype=np.float64)
    cols = []
    for a, d in enumerate(axis_dims):
        if d == 0:
            continue
        j = np.arange(d // 2, dtype=np.float64)
        omega = theta ** (-2.0 * j / d)
        cols.append(pos[:, a:a + 1] * omega[None, :])
    return np.concatenate(cols, axis=1)


def rope_apply(x, phi) -> np.ndarray:
    """Rotate interleaved pairs (2i, 2i+1) of x[..., head_dim] by phi[..., head_dim//2].

    x has shape [rows, heads, head_dim] and phi [rows, head_dim // 2] (the
    same angles for every head of a token).
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def qk_norm_rope(x, gain, pos, axis_dims, theta: float, eps: float) -> np.ndarray:
    """RMSNorm per head, then RoPE, rounded to bf16. x [rows, heads, head_dim]."""
    n = rms_norm(x, gain, eps)
    return round_bf16(rope_apply(n, rope_angles(pos, axis_dims, theta)))


# ---------------------------------------------------------------------------
# a3: dense bidirectional attention over the valid length
# [vLLM-Omni H3 blog] section 3.1: the attention backend receives the valid
# sequence length and the structural tail padding is removed, so keys >= L
# take no part and padded rows get no output.
# ---------------------------------------------------------------------------

def softmax(z, axis=-1) -> np.ndarray:
    """Numerically stable softmax (max subtracted), float64."""
    z = np.asarray(z, dtype=np.float64)
    z = z - z.max(axis=axis, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=axis, keepdims=True)


def attention(q, k, v, L: int, scale: float, rows=None) -> np.ndarray:
    """softmax(q k^T * scale) v per head over keys [0, L).

    q, k, v [S, heads, head_dim] (bf16 values). rows: query row indices to
    evaluate (default: all of [0, L)). Returns [len(rows), heads, head_dim]
    rounded to bf16.
    """
    if rows is None:
        rows = np.arange(L)
    rows = np.asarray(rows)
    q = np.asarray(q, np.float64)[rows]
    k = np.asarray(k, np.float64)[:L]
    v = np.asarray(v, np.float64)[:L]
    out = np.empty(q.shape, dtype=np.float64)
    for h in range(q.shape[1]):
        p = softmax((q[:, h, :] @ k[:, h, :].T) * scale, axis=-1)
        out[:, h, :] = p @ v[:, h, :]
    return round_bf16(out)


# ---------------------------------------------------------------------------
# a4: block projections  (the matrix multiplies the small ops sit around,
# [vLLM-Omni H3 blog] section 3.2; hidden width 5,376 from section 3.1)
# ---------------------------------------------------------------------------

def linear(x, w) -> np.ndarray:
    """x @ w^T with bf16-valued operands, float64 accumulation, bf16 result."""
    return round_bf16(np.asarray(x, np.float64) @ np.asarray(w, np.float64).T)


# ---------------------------------------------------------------------------
# a5: SwiGLU  ([vLLM-Omni H3 blog] section 3.2: fused SwiGLU replaces the
# separate SiLU and multiply launches, #6283)
# ---------------------------------------------------------------------------

def silu(g) -> np.ndarray:
    g = np.asarray(g, np.float64)
    return g / (1.0 + np.exp(-g))


def swiglu(gu) -> np.ndarray:
    """gu [rows, 2F] = [g | v]  ->  SiLU(g) * v, rounded to bf16, [rows, F]."""
    gu = np.asarray(gu, np.float64)
    F = gu.shape[-1] // 2
    return round_bf16(silu(gu[..., :F]) * gu[..., F:])


# ---------------------------------------------------------------------------
# a6: the whole block, steps in the order of the fused-op list
# ([vLLM-Omni H3 blog] sections 3.1-3.2)
# ---------------------------------------------------------------------------

def unpack_mod(mod):
    """mod [6, D] -> (shift1, scale1, gate1, shift2, scale2, gate2)."""
    mod = np.asarray(mod, np.float64)
    return tuple(mod[i] for i in range(6))


def block_forward(resid, mod, w_qkv, w_o, w_gu, w_down, q_gain, k_gain, pos,
                  *, L: int, heads: int, head_dim: int, axis_dims, theta: float,
                  eps_ln: float = 1e-6, eps_qk: float = 1e-6, rows=None,
                  kv_chunk: int = 4096, return_intermediates: bool = False):
    """Forward pass of one DiT block for query rows `rows` (default all < L).

    resid [S, D] float32 residual stream; mod [6, D]; weights bf16-valued
    [3D, D], [D, D], [2F, D], [D, F]; gains [head_dim]; pos [S, 3].
    Keys and values are formed for all L valid rows (every query row attends
    to all of them); everything after attention is row-local, so only the
    asked-for rows are carried through. Returns the updated residual rows
    [len(rows), D] (float32 values) and, optionally, a dict of the
    intermediates for those rows.
    """
    D = heads * head_dim
    if rows is None:
        rows = np.arange(L)
    rows = np.asarray(rows)
    sh1, sc1, g1, sh2, sc2, g2 = unpack_mod(mod)
    r_all = np.asarray(resid, np.float64)[:L]
    w_qkv = np.asarray(w_qkv, np.float64)
    scale = 1.0 / np.sqrt(head_dim)

    # keys and values for every valid row, in row chunks to bound memory
    k_all = np.empty((L, heads, head_dim))
    v_all = np.empty((L, heads, head_dim))
    w_k = w_qkv[D:2 * D]
    w_v = w_qkv[2 * D:3 * D]
    for c0 in range(0, L, kv_chunk):
        c1 = min(L, c0 + kv_chunk)
        _, h1c = mod_norm_residual(r_all[c0:c1], shift=sh1, scale=sc1, eps=eps_ln)
        kc = linear(h1c, w_k).reshape(c1 - c0, heads, head_dim)
        k_all[c0:c1] = qk_norm_rope(kc, k_gain, pos[c0:c1], axis_dims, theta, eps_qk)
        v_all[c0:c1] = linear(h1c, w_v).reshape(c1 - c0, heads, head_dim)

    r = r_all[rows]
    _, h1 = mod_norm_residual(r, shift=sh1, scale=sc1, eps=eps_ln)
    q = linear(h1, w_qkv[0:D]).reshape(len(rows), heads, head_dim)
    q = qk_norm_rope(q, q_gain, np.asarray(pos)[rows], axis_dims, theta, eps_qk)
    q_full = np.zeros((L, heads, head_dim))
    q_full[rows] = q
    a = attention(q_full, k_all, v_all, L, scale, rows=rows).reshape(len(rows), D)
    o = linear(a, w_o)
    r, h2 = mod_norm_residual(r, o, g1, sh2, sc2, eps=eps_ln)
    gu = linear(h2, w_gu)
    u = swiglu(gu)
    f = linear(u, w_down)
    r, _ = mod_norm_residual(r, f, g2, eps=eps_ln)
    if return_intermediates:
        return r, dict(h1=h1, q=q, k=k_all[rows], v=v_all[rows], a=a, o=o,
                       h2=h2, gu=gu, u=u, f=f)
    return r
