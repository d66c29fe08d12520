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
    The split-half layout pairs (o_a + j, o_a + d_a/2 + j) instead, with the
    same angle for pair j; it is the interleaved rotation under a fixed
    permutation of each section's channels.
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

import math

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
        r = round_f32(r + _per_row(gate) * np.asarray(delta, np.float64))
    h = None
    if scale is not None:
        n = layer_norm(r, eps)
        h = round_bf16(n * (1.0 + _per_row(scale)) + _per_row(shift))
    return r, h


def _per_row(v) -> np.ndarray:
    """A modulation vector [D] (same for every row) or one per row [rows, D]."""
    v = np.asarray(v, np.float64)
    return v[None, :] if v.ndim == 1 else v


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


def rope_pairs(axis_dims, pairing: str = "interleaved"):
    """Channel indices (first, second) of every rotated pair, in the pair order
    of rope_angles (section a, then pair j inside it).

    interleaved: (o_a + 2j, o_a + 2j + 1); half: (o_a + j, o_a + d_a/2 + j),
    o_a being the first channel of section a.
    """
    first, second = [], []
    o = 0
    for d in axis_dims:
        for j in range(d // 2):
            if pairing == "interleaved":
                first.append(o + 2 * j)
                second.append(o + 2 * j + 1)
            elif pairing == "half":
                first.append(o + j)
                second.append(o + d // 2 + j)
            else:
                raise ValueError(pairing)
        o += d
    return np.array(first), np.array(second)


def rope_apply(x, phi, axis_dims=None, pairing: str = "interleaved") -> np.ndarray:
    """Rotate the pairs of x[..., head_dim] by phi[..., head_dim//2].

    x has shape [rows, heads, head_dim] and phi [rows, head_dim // 2] (the
    same angles for every head of a token). Interleaved pairs (2i, 2i+1) by
    default; pairing="half" rotates the split-half pairs of rope_pairs
    (axis_dims needed).
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    if pairing == "interleaved":
        x0 = x[..., 0::2]
        x1 = x[..., 1::2]
        out = np.empty_like(x)
        out[..., 0::2] = x0 * c - x1 * s
        out[..., 1::2] = x0 * s + x1 * c
        return out
    first, second = rope_pairs(axis_dims, pairing)
    x0 = x[..., first]
    x1 = x[..., second]
    out = np.empty_like(x)
    out[..., first] = x0 * c - x1 * s
    out[..., second] = x0 * s + x1 * c
    return out


def qk_norm_rope(x, gain, pos, axis_dims, theta: float, eps: float,
                 pairing: str = "interleaved") -> np.ndarray:
    """RMSNorm per head, then RoPE, rounded to bf16. x [rows, heads, head_dim]."""
    n = rms_norm(x, gain, eps)
    return round_bf16(rope_apply(n, rope_angles(pos, axis_dims, theta), axis_dims, pairing))


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
    """mod [6, D] -> (shift1, scale1, gate1, shift2, scale2, gate2).
    mod [rows, 6, D] (one modulation per row) -> six [rows, D] arrays."""
    mod = np.asarray(mod, np.float64)
    return tuple(mod[..., i, :] for i in range(6))


def modulation_rows(mod, seg, rows):
    """Modulation of the given rows. mod [6, D] applies to every token; with
    seg [S] (the token-group index of every row, e.g. video vs audio tokens
    that follow their own sigma schedule, or conditioning vs noisy tokens;
    vLLM-Omni H3 blog, section 1 Fig. 1, and the H3 blog PR's dual
    video/audio schedules) mod is a table [G, 6, D] and row i uses
    mod[seg[i]]. Returns [6, D] or [len(rows), 6, D]."""
    mod = np.asarray(mod, np.float64)
    if seg is None:
        return mod
    return mod[np.asarray(seg)[np.asarray(rows)]]


def block_forward(resid, mod, w_qkv, w_o, w_gu, w_down, q_gain, k_gain, pos,
                  *, L: int, heads: int, head_dim: int, axis_dims, theta: float,
                  eps_ln: float = 1e-6, eps_qk: float = 1e-6, rows=None,
                  kv_chunk: int = 4096, return_intermediates: bool = False, seg=None,
                  fp8: bool = False, fp8_attention: bool = False,
                  rope_pairing: str = "interleaved"):
    """Forward pass of one DiT block for query rows `rows` (default all < L).

    resid [S, D] float32 residual stream; mod [6, D]; weights bf16-valued
    [3D, D], [D, D], [2F, D], [D, F]; gains [head_dim]; pos [S, 3].
    Keys and values are formed for all L valid rows (every query row attends
    to all of them); everything after attention is row-local, so only the
    asked-for rows are carried through. Returns the updated residual rows
    [len(rows), D] (float32 values) and, optionally, a dict of the
    intermediates for those rows. seg: optional token-group index per row,
    with mod a table [G, 6, D] (see modulation_rows). fp8: the four
    projections run as online FP8 (weights and inputs quantised per row,
    see quantize_fp8_rows / linear_fp8). rope_pairing: see rope_pairs.
    """
    qw_cache = {}

    def proj(x, w):
        if not fp8:
            return linear(x, w)
        key = id(w)
        if key not in qw_cache:
            qw_cache[key] = quantize_fp8_rows(w)
        qx, sx = quantize_fp8_rows(x)
        qw, sw = qw_cache[key]
        return linear_fp8(qx, sx, qw, sw)

    D = heads * head_dim
    if rows is None:
        rows = np.arange(L)
    rows = np.asarray(rows)
    sh1, sc1, g1, sh2, sc2, g2 = unpack_mod(modulation_rows(mod, seg, rows))
    r_all = np.asarray(resid, np.float64)[:L]
    w_qkv = np.asarray(w_qkv, np.float64)
    scale = 1.0 / np.sqrt(head_dim)

    # keys and values for every valid row, in row chunks to bound memory
    k_all = np.empty((L, heads, head_dim))
    v_all = np.empty((L, heads, head_dim))
    w_k = w_qkv[D:2 * D]
    w_v = w_qkv[2 * D:3 * D]
    # FP8 attention scales Q per 128-row tile, so every row's q is needed then
    q_all = np.zeros((L, heads, head_dim)) if fp8_attention else None
    w_q = w_qkv[0:D]
    for c0 in range(0, L, kv_chunk):
        c1 = min(L, c0 + kv_chunk)
        shc, scc = unpack_mod(modulation_rows(mod, seg, np.arange(c0, c1)))[:2]
        _, h1c = mod_norm_residual(r_all[c0:c1], shift=shc, scale=scc, eps=eps_ln)
        if fp8_attention:
            qc = proj(h1c, w_q).reshape(c1 - c0, heads, head_dim)
            q_all[c0:c1] = qk_norm_rope(qc, q_gain, pos[c0:c1], axis_dims, theta, eps_qk,
                                          rope_pairing)
        kc = proj(h1c, w_k).reshape(c1 - c0, heads, head_dim)
        k_all[c0:c1] = qk_norm_rope(kc, k_gain, pos[c0:c1], axis_dims, theta, eps_qk,
                                      rope_pairing)
        v_all[c0:c1] = proj(h1c, w_v).reshape(c1 - c0, heads, head_dim)

    r = r_all[rows]
    _, h1 = mod_norm_residual(r, shift=sh1, scale=sc1, eps=eps_ln)
    q = proj(h1, w_q).reshape(len(rows), heads, head_dim)
    q = qk_norm_rope(q, q_gain, np.asarray(pos)[rows], axis_dims, theta, eps_qk, rope_pairing)
    if fp8_attention:
        q_full = q_all
    else:
        q_full = np.zeros((L, heads, head_dim))
        q_full[rows] = q
    if fp8_attention:
        ops = sage_quantize(q_full, k_all, v_all, L)
        a = attention_sage(ops, L, scale, rows=rows).reshape(len(rows), D)
    else:
        a = attention(q_full, k_all, v_all, L, scale, rows=rows).reshape(len(rows), D)
    o = proj(a, w_o)
    r, h2 = mod_norm_residual(r, o, g1, sh2, sc2, eps=eps_ln)
    gu = proj(h2, w_gu)
    u = swiglu(gu)
    f = proj(u, w_down)
    r, _ = mod_norm_residual(r, f, g2, eps=eps_ln)
    if return_intermediates:
        return r, dict(h1=h1, q=q, k=k_all[rows], v=v_all[rows], a=a, o=o,
                       h2=h2, gu=gu, u=u, f=f)
    return r


def stack_forward(resid, mods, weights, q_gains, k_gains, pos, *, L: int, heads: int,
                  head_dim: int, axis_dims, theta: float, eps_ln: float = 1e-6,
                  eps_qk: float = 1e-6, seg=None, rope_pairing: str = "interleaved"):
    """Blocks applied one after another to the whole residual stream (all
    rows < L); the denoiser runs its transformer blocks in sequence for every
    forward (vLLM-Omni H3 blog, section 5: FastH3's forwards). mods[b] and
    (w_qkv, w_o, w_gu, w_down) = weights[b] belong to block b."""
    r = np.asarray(resid, np.float64).copy()
    for b in range(len(mods)):
        w_qkv, w_o, w_gu, w_down = weights[b]
        r[:L] = block_forward(r, mods[b], w_qkv, w_o, w_gu, w_down, q_gains[b], k_gains[b], pos,
                              L=L, heads=heads, head_dim=head_dim, axis_dims=axis_dims,
                              theta=theta, eps_ln=eps_ln, eps_qk=eps_qk, seg=seg,
                              rope_pairing=rope_pairing)
    return r[:L]


# ---------------------------------------------------------------------------
# GPU output preparation ([vLLM-Omni H3 blog] section 3.4: decoded FP32
# BCTHW frames become contiguous uint8 BTHWC before transfer, a quarter of the
# bytes). The pages give no formula; the reading here is the usual decoder
# convention: x in [-1, 1] maps to round(clamp(x / 2 + 1/2, 0, 1) * 255) with
# round-half-to-even, every step in float32 (the precision both sides use for
# this integer decision), no fused multiply-add.
# ---------------------------------------------------------------------------

def frames_to_u8(frames) -> np.ndarray:
    """frames [B, C, T, H, W] float32 -> [B, T, H, W, C] uint8."""
    x = np.asarray(frames, dtype=np.float32)
    t = (x * np.float32(0.5)).astype(np.float32) + np.float32(0.5)
    t = np.clip(t, np.float32(0.0), np.float32(1.0)).astype(np.float32)
    v = np.rint((t * np.float32(255.0)).astype(np.float32))
    return np.ascontiguousarray(np.moveaxis(v.astype(np.uint8), 1, -1))


# ---------------------------------------------------------------------------
# Online FP8 projections ([vLLM-Omni H3 blog] section 4.3, "online FP8": the
# eligible linear layers' weights are quantised to FP8 once at load time with
# their scales, and their activations are quantised online). The pages give
# no scaling granularity; the reading here is per-row absmax scaling to
# FP8 E4M3 (max 448): each weight row (output channel) and each activation
# row (token) gets its own float32 scale. Every step that decides a code is
# taken in float32 on both sides:
#   amax = max |x|,  inv = 448 / amax (0 when amax == 0),  code = e4m3(x * inv)
#   scale = amax / 448  (dequantised value = code * scale)
# and the product is y = bf16( (sum_k qa[i,k] qw[j,k]) * sa[i] * sw[j] ).
# ---------------------------------------------------------------------------

_E4M3_MAX = 448.0


def round_e4m3(x) -> np.ndarray:
    """Round float64 values to FP8 E4M3 (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; no infinities), nearest-even, saturating to +-448.
    Normal numbers have 4 significant bits; below 2^-6 the step is 2^-9."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    _, e = np.frexp(x[nz])
    q = np.maximum(e - 4, -9).astype(np.float64)
    step = np.exp2(q)
    r = np.rint(x[nz] / step) * step
    out[nz] = np.clip(r, -_E4M3_MAX, _E4M3_MAX)
    return out


def quantize_fp8_rows(x):
    """Per-row absmax quantisation of x [rows, K] (bf16 values) to E4M3.
    Returns (codes as float64 values [rows, K], scales float32 values [rows])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=1)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, np.float32(_E4M3_MAX) / amax, np.float32(0)).astype(np.float32)
    prod = (x32 * inv[:, None]).astype(np.float32)
    codes = round_e4m3(prod.astype(np.float64))
    scale = (amax / np.float32(_E4M3_MAX)).astype(np.float32)
    return codes, scale.astype(np.float64)


def linear_fp8(qx, sx, qw, sw) -> np.ndarray:
    """bf16( (qx @ qw^T) * sx[:, None] * sw[None, :] ), float64 accumulation."""
    acc = np.asarray(qx, np.float64) @ np.asarray(qw, np.float64).T
    return round_bf16(acc * np.asarray(sx, np.float64)[:, None] * np.asarray(sw, np.float64)[None, :])


# ---------------------------------------------------------------------------
# Skip-Softmax ([vLLM-Omni H3 blog] section 4.3: the attention backend can
# skip the softmax and P x V work of tiles the QK scores show to be
# negligible, decided per tile). Reading: keys are taken in tiles of 128 from
# key 0 and queries in tiles of 128 from row 0; a key tile is skipped for a
# query tile when, for every query row of that tile, the tile's largest
# scaled score lies more than log2(1/eps) below the row's running maximum
# (in base-2 units, over the key tiles already kept). eps = 0 never skips and
# is dense attention.
# ---------------------------------------------------------------------------

def attention_skip(q, k, v, L: int, scale: float, eps: float, tile: int = 128):
    """Attention with tile-level skipping; returns (out [L, H, Dh] bf16 values,
    kept [n_qtiles, H, n_ktiles] bool)."""
    q = np.asarray(q, np.float64)[:L]
    k = np.asarray(k, np.float64)[:L]
    v = np.asarray(v, np.float64)[:L]
    H = q.shape[1]
    nq = (L + tile - 1) // tile
    nk = (L + tile - 1) // tile
    out = np.empty_like(q)
    kept = np.ones((nq, H, nk), bool)
    thresh = np.inf if eps <= 0 else np.log2(1.0 / eps)
    for h in range(H):
        s = (q[:, h, :] @ k[:, h, :].T) * scale / np.log(2.0)  # base-2 logits
        for qi in range(nq):
            r0, r1 = qi * tile, min(L, (qi + 1) * tile)
            m = np.full(r1 - r0, -np.inf)
            keep_cols = []
            for kj in range(nk):
                c0, c1 = kj * tile, min(L, (kj + 1) * tile)
                tmax = s[r0:r1, c0:c1].max(axis=1)
                if np.all(tmax < m - thresh):
                    kept[qi, h, kj] = False
                    continue
                m = np.maximum(m, tmax)
                keep_cols.append(np.arange(c0, c1))
            cols = np.concatenate(keep_cols)
            z = s[r0:r1][:, cols]
            p = np.exp2(z - z.max(axis=1, keepdims=True))
            out[r0:r1, h, :] = (p / p.sum(axis=1, keepdims=True)) @ v[cols, h, :]
    return round_bf16(out), kept


# ---------------------------------------------------------------------------
# FP8 ("SAGE") attention ([vLLM-Omni H3 blog] section 4.3, Fig. 6: the
# attention backend can quantise Q, K, P and V to FP8 for the QK and PV
# products). The pages give no scaling scheme; the reading here treats every
# one of the four operands the same way, with absmax scaling into E4M3's full
# range (inv = 448 / amax, code = e4m3(x * inv), scale = amax / 448, every
# step in float32):
#   * K is first smoothed by subtracting its per-(head, channel) mean over the
#     L valid keys (their correctly rounded sum, math.fsum, divided by L in
#     double and rounded to float32, so that the mean depends on the values
#     alone and not on an order of summation; softmax is unchanged because
#     each row's scores move by one constant);
#   * Q and the smoothed K are quantised per (128-row tile, head) block, V per
#     (head, channel) over the valid keys;
#   * scores = (Q codes . K codes) * sq * sk; the softmax weights are
#     p = 2^(z - max z) with the exact row maximum, so every row of P has
#     absmax exactly 1 and is quantised as 448 * p (scale 1 / 448);
#   * the row sum uses the unrounded p; O = (P codes . V codes) * sv / 448 /
#     sum p.
# ---------------------------------------------------------------------------

def _absmax_codes(x32, axis):
    """float32 block -> (E4M3 code values, float32 scale), absmax over `axis`."""
    amax = np.max(np.abs(x32), axis=axis, keepdims=True)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, np.float32(_E4M3_MAX) / amax, np.float32(0)).astype(np.float32)
    codes = round_e4m3((x32 * inv).astype(np.float32).astype(np.float64))
    scale = (amax / np.float32(_E4M3_MAX)).astype(np.float32)
    return codes, scale


def sage_quantize(q, k, v, L: int, tile: int = 128):
    """FP8 operands of SAGE attention. q, k, v [S, H, Dh] bf16 values.
    Returns dict: qc [L,H,Dh], sq [nt,H], kc, sk [nt,H], vc, sv [H,Dh] and
    k_mean [H,Dh] (float32 values: math.fsum of the valid keys / L, rounded
    to float32)."""
    q = np.asarray(q, np.float32)[:L]
    k = np.asarray(k, np.float32)[:L]
    v = np.asarray(v, np.float32)[:L]
    H, Dh = q.shape[1], q.shape[2]
    cols = np.ascontiguousarray(np.asarray(k, np.float64).reshape(L, H * Dh).T)
    k_mean = round_f32(np.array([math.fsum(c.tolist()) for c in cols]).reshape(H, Dh) / L)
    ks = (k - k_mean.astype(np.float32)[None]).astype(np.float32)
    nt = (L + tile - 1) // tile
    qc = np.empty((L, H, Dh)); kc = np.empty((L, H, Dh))
    sq = np.empty((nt, H), np.float32); sk = np.empty((nt, H), np.float32)
    for t in range(nt):
        r0, r1 = t * tile, min(L, (t + 1) * tile)
        c, s = _absmax_codes(q[r0:r1], axis=(0, 2))
        qc[r0:r1], sq[t] = c, s[0, :, 0]
        c, s = _absmax_codes(ks[r0:r1], axis=(0, 2))
        kc[r0:r1], sk[t] = c, s[0, :, 0]
    vc, sv = _absmax_codes(v, axis=0)
    return dict(qc=qc, sq=sq, kc=kc, sk=sk, vc=vc, sv=sv[0], k_mean=k_mean)


def _sage_logits(ops, h, rows, L, scale, tile):
    """Base-2 logits z = (Q codes . K codes) * sq * sk * scale / ln 2 of head h
    for the given query rows against the L valid keys, float64 [len(rows), L]."""
    qc, kc = ops["qc"], ops["kc"]
    sq = ops["sq"].astype(np.float64)
    sk = ops["sk"].astype(np.float64)
    key_tile = np.arange(L) // tile
    s = (qc[rows, h, :] @ kc[:L, h, :].T) * sq[rows // tile, h][:, None] * sk[key_tile, h][None, :]
    return s * scale / np.log(2.0)


def _sage_weights(ops, h, rows, L, scale, tile):
    """Softmax weights p = 2^(z - max z) of head h for the given query rows
    (exact row maximum), float64 [len(rows), L]."""
    z = _sage_logits(ops, h, rows, L, scale, tile)
    return np.exp2(z - z.max(axis=1, keepdims=True))


def attention_sage(ops, L: int, scale: float, rows=None, tile: int = 128):
    """FP8 attention from sage_quantize's operands, for query rows `rows`."""
    if rows is None:
        rows = np.arange(L)
    rows = np.asarray(rows)
    vc = ops["vc"]
    sv = ops["sv"].astype(np.float64)
    H, Dh = vc.shape[1], vc.shape[2]
    out = np.empty((len(rows), H, Dh))
    for h in range(H):
        p = _sage_weights(ops, h, rows, L, scale, tile)
        pc = round_e4m3(_E4M3_MAX * p)
        out[:, h, :] = (pc @ vc[:L, h, :]) * sv[h][None, :] / (_E4M3_MAX * p.sum(axis=1, keepdims=True))
    return round_bf16(out)


def _sage_skip_tiles(ops, L, scale, eps, tile):
    """Skip-Softmax on the FP8 logits ([vLLM-Omni H3 blog] section 4.3, Fig. 6:
    Skip-Softmax uses the QK result to leave out whole softmax and P x V
    tiles; the tile rule is the one of attention_skip): for each 128-row query
    tile and head, walk the key tiles in order, keeping for every row the
    maximum logit over the tiles kept so far; a key tile is left out when
    every row's maximum logit in it lies more than log2(1/eps) below that
    running maximum (eps = 0: nothing is left out; the first key tile is
    always kept). Yields (h, query tile index, rows, kept tile mask, kept key
    columns, logits of the rows against the kept keys)."""
    H = ops["vc"].shape[1]
    nq = nk = (L + tile - 1) // tile
    thresh = np.inf if eps <= 0 else np.log2(1.0 / eps)
    for h in range(H):
        for qi in range(nq):
            rows = np.arange(qi * tile, min(L, (qi + 1) * tile))
            z = _sage_logits(ops, h, rows, L, scale, tile)
            m = np.full(len(rows), -np.inf)
            keep = np.zeros(nk, bool)
            for kj in range(nk):
                c0, c1 = kj * tile, min(L, (kj + 1) * tile)
                tmax = z[:, c0:c1].max(axis=1)
                if np.all(tmax < m - thresh):
                    continue
                keep[kj] = True
                m = np.maximum(m, tmax)
            cols = np.flatnonzero(np.repeat(keep, tile)[:L])
            yield h, qi, rows, keep, cols, z[:, cols]


def attention_sage_skip(ops, L: int, scale: float, eps: float, tile: int = 128):
    """SAGE attention with Skip-Softmax: the key tiles _sage_skip_tiles keeps
    go through attention_sage's steps (weights against the row maximum of the
    kept keys, E4M3 codes of 448 p, the sum of the unrounded weights); the
    left-out tiles take no part. Returns (out [L, H, Dh] bf16 values,
    kept [n_qtiles, H, n_ktiles] bool)."""
    vc = ops["vc"]
    sv = ops["sv"].astype(np.float64)
    H, Dh = vc.shape[1], vc.shape[2]
    nt = (L + tile - 1) // tile
    out = np.empty((L, H, Dh))
    kept = np.zeros((nt, H, nt), bool)
    for h, qi, rows, keep, cols, z in _sage_skip_tiles(ops, L, scale, eps, tile):
        kept[qi, h] = keep
        p = np.exp2(z - z.max(axis=1, keepdims=True))
        pc = round_e4m3(_E4M3_MAX * p)
        out[rows, h, :] = ((pc @ vc[cols, h, :]) * sv[h][None, :]
                           / (_E4M3_MAX * p.sum(axis=1, keepdims=True)))
    return round_bf16(out), kept


def sage_skip_error_terms(ops, L: int, scale: float, eps: float, tile: int = 128):
    """sage_error_terms over the key tiles attention_sage_skip keeps, for
    every valid row: (a1, a0, v2, u2), each [L, H, Dh] float64."""
    vc = ops["vc"]
    sv = ops["sv"].astype(np.float64)
    H, Dh = vc.shape[1], vc.shape[2]
    a1 = np.empty((L, H, Dh)); a0 = np.empty_like(a1)
    v2 = np.empty_like(a1); u2 = np.empty_like(a1)
    for h, qi, rows, keep, cols, z in _sage_skip_tiles(ops, L, scale, eps, tile):
        p = np.exp2(z - z.max(axis=1, keepdims=True))
        tot = p.sum(axis=1, keepdims=True)
        w = np.abs(vc[cols, h, :] * sv[h][None, :])
        a1[rows, h, :] = (p @ w) / tot
        a0[rows, h, :] = w.sum(axis=0)[None, :] / tot
        v2[rows, h, :] = ((p * p) @ (w * w)) / (tot * tot)
        u2[rows, h, :] = (w * w).sum(axis=0)[None, :] / (tot * tot)
    return a1, a0, v2, u2


def sage_error_terms(ops, L: int, scale: float, rows=None, tile: int = 128):
    """Per-element sums that bound how far two correct FP8 evaluations of
    attention_sage may differ when they quantise P at different scales
    (their E4M3 roundings of the same weight then differ): with
    w = V codes * sv (the dequantised V) and p the exact weights,
      a1[i,h,d] = sum_k p_k |w_kd| / sum_k p_k
      a0[i,h,d] = sum_k |w_kd| / sum_k p_k
      v2[i,h,d] = sum_k p_k^2 w_kd^2 / (sum_k p_k)^2
      u2[i,h,d] = sum_k w_kd^2 / (sum_k p_k)^2
    Returns (a1, a0, v2, u2), each [len(rows), H, Dh] float64."""
    if rows is None:
        rows = np.arange(L)
    rows = np.asarray(rows)
    vc = ops["vc"]
    sv = ops["sv"].astype(np.float64)
    H, Dh = vc.shape[1], vc.shape[2]
    a1 = np.empty((len(rows), H, Dh)); a0 = np.empty_like(a1)
    v2 = np.empty_like(a1); u2 = np.empty_like(a1)
    for h in range(H):
        p = _sage_weights(ops, h, rows, L, scale, tile)
        tot = p.sum(axis=1, keepdims=True)
        w = np.abs(vc[:L, h, :] * sv[h][None, :])
        a1[:, h, :] = (p @ w) / tot
        a0[:, h, :] = w.sum(axis=0)[None, :] / tot
        v2[:, h, :] = ((p * p) @ (w * w)) / (tot * tot)
        u2[:, h, :] = (w * w).sum(axis=0)[None, :] / (tot * tot)
    return a1, a0, v2, u2
