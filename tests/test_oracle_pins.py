"""Pins for the CPU oracle: closed forms, invariants, library special cases and
brute force on tiny inputs. None of these compares the oracle with itself.

Each check lives in a `check_*` helper that takes the oracle module, so the
planted-mistake tests at the bottom can run the same checks against a copy of
the oracle with one deliberate error and confirm that some check fails.
"""
import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


def rng(seed=0):
    return np.random.default_rng(seed)


def bf16_values(a):
    """Round arbitrary float64 data to bf16 with torch (a library cast), for inputs."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


# ------------------------------------------------------------------ rounding
def check_round_bf16(o):
    g = GOLD["bf16_ties"]
    assert np.array_equal(o.round_bf16(np.array(g["x"])), np.array(g["y"]))
    # library pin: torch's float32 -> bfloat16 cast (round to nearest even)
    x = rng(1).standard_normal(20000).astype(np.float32) * np.float32(3.0)
    x = np.concatenate([x, np.float32([0.0, -0.0, 1e-39, -3e-40, 3.3e38, 1.0e-30])])
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o.round_bf16(x.astype(np.float64)), ref)
    # every bf16-valued input maps to itself
    assert np.array_equal(o.round_bf16(ref), ref)


def test_round_bf16():
    check_round_bf16(O)


# ---------------------------------------------------------- a1 modulation
def check_layer_norm(o):
    g = GOLD["layer_norm_1234"]
    y = o.layer_norm(np.array([g["x"]]), g["eps"])[0]
    assert np.allclose(y * math.sqrt(5.0), g["y_times_sqrt5"], rtol=0, atol=1e-14)
    x = rng(2).standard_normal((7, 96)) * 3 + 1.5
    y = o.layer_norm(x, 0.0)
    assert np.allclose(y.mean(-1), 0, atol=1e-13)
    assert np.allclose(y.var(-1), 1, atol=1e-12)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (96,), eps=1e-6).numpy()
    assert np.allclose(o.layer_norm(x, 1e-6), ref, rtol=1e-12, atol=1e-12)


def check_mod_norm_residual(o):
    r = rng(3).standard_normal((5, 64)).astype(np.float32).astype(np.float64)
    delta = bf16_values(rng(4).standard_normal((5, 64)))
    zeros = np.zeros(64)
    # gate = 0: the residual comes back bit for bit
    r2, _ = o.mod_norm_residual(r, delta, zeros)
    assert np.array_equal(r2, r)
    # the residual add is r + gate * delta (float32 store); small exact values
    gate = np.full(64, 0.5)
    d = np.full((5, 64), 2.0)
    r3, _ = o.mod_norm_residual(r, d, gate)
    assert np.array_equal(r3, (r + 1.0).astype(np.float32).astype(np.float64))
    # scale = shift = 0: plain LayerNorm, rounded to bf16
    _, h = o.mod_norm_residual(r, shift=zeros, scale=zeros, eps=1e-6)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(r), (64,), eps=1e-6)
    assert np.all(np.abs(h - ref.numpy()) <= 2.0 ** -8 * np.abs(ref.numpy()))
    # scale = -1: the normalised term vanishes and h is exactly shift
    g = GOLD["modulate_scale_minus_one"]
    shift = np.tile(np.array(g["shift"]), 16)
    _, h = o.mod_norm_residual(r, shift=shift, scale=-np.ones(64))
    assert np.array_equal(h, np.broadcast_to(shift, h.shape))
    # scale doubles the normalised term: (1 + 1) * LN
    _, h1 = o.mod_norm_residual(r, shift=zeros, scale=np.ones(64))
    assert np.allclose(h1, 2 * o.layer_norm(r, 1e-6), rtol=2 ** -8, atol=0)


def test_layer_norm():
    check_layer_norm(O)


def test_mod_norm_residual():
    check_mod_norm_residual(O)


# ------------------------------------------------------ a2 RMSNorm + RoPE
def check_rms_norm(o):
    g = GOLD["rms_norm_3_4"]
    y = o.rms_norm(np.array([g["x"]]), np.array(g["gain"]), 0.0)[0]
    assert np.allclose(y * 5 / math.sqrt(2), g["y_times_5_over_sqrt2"], atol=1e-14)
    x = rng(5).standard_normal((6, 3, 128)) * 4
    ones = np.ones(128)
    y = o.rms_norm(x, ones, 0.0)
    assert np.allclose(np.sqrt((y * y).mean(-1)), 1.0, atol=1e-13)
    assert np.allclose(o.rms_norm(7.5 * x, ones, 0.0), y, atol=1e-13)
    gain = 1 + 0.1 * rng(6).standard_normal(128)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(gain), eps=1e-6)
    assert np.allclose(o.rms_norm(x, gain, 1e-6), ref.numpy(), rtol=1e-12, atol=1e-12)


def check_rope(o):
    g = GOLD["rope_angles_4_2_2"]
    phi = o.rope_angles(np.array([g["pos"]]), g["axis_dims"], g["theta"])[0]
    assert np.allclose(phi, g["phi"], rtol=1e-14, atol=0)
    q = GOLD["rope_quarter_turn"]
    y = o.rope_apply(np.array(q["x"]).reshape(1, 1, 4), np.array([q["phi"]]))
    assert np.allclose(y.reshape(-1), q["y"], atol=1e-15)
    # section-local exponent for the 32/48/48 split: pair 8 of the h section
    phi = o.rope_angles(np.array([[0, 1, 0]]), (32, 48, 48), 1e4)[0]
    assert math.isclose(phi[16 + 8], 1e4 ** (-16 / 48), rel_tol=1e-14)
    assert np.all(phi[:16] == 0) and np.all(phi[40:] == 0)
    x = rng(7).standard_normal((9, 2, 128))
    pos = rng(8).integers(0, 80, size=(9, 3))
    phi = o.rope_angles(pos, (32, 48, 48), 1e4)
    y = o.rope_apply(x, phi)
    # norm of every pair is preserved
    assert np.allclose(np.hypot(y[..., 0::2], y[..., 1::2]),
                       np.hypot(x[..., 0::2], x[..., 1::2]), atol=1e-13)
    # turning back by -phi restores the input; position 0 is the identity
    assert np.allclose(o.rope_apply(y, -phi), x, atol=1e-13)
    assert np.array_equal(o.rope_apply(x, np.zeros_like(phi)), x)
    # complex-number form: (x0 + i x1) * exp(i phi)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * phi)[:, None, :]
    assert np.allclose(y[..., 0::2], z.real, atol=1e-13)
    assert np.allclose(y[..., 1::2], z.imag, atol=1e-13)
    # relative-position property: <R(q,m), R(k,n)> depends on m - n only
    qv = rng(9).standard_normal((1, 1, 128))
    kv = rng(10).standard_normal((1, 1, 128))
    def dot(m, n):
        pm = o.rope_angles(np.array([[m, 2 * m, 3]]), (32, 48, 48), 1e4)
        pn = o.rope_angles(np.array([[n, 2 * n, 3]]), (32, 48, 48), 1e4)
        return float((o.rope_apply(qv, pm) * o.rope_apply(kv, pn)).sum())
    assert math.isclose(dot(5, 2), dot(40, 37), rel_tol=1e-11, abs_tol=1e-11)
    assert not math.isclose(dot(5, 2), dot(5, 3), rel_tol=1e-6)


def check_rope_half(o):
    # worked example, one 4-channel section: pairs (0, 2) and (1, 3); a quarter
    # turn of pair 0 maps (x0, x2) = (1, 3) to (-3, 1), pair 1 stays
    y = o.rope_apply(np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 4), np.array([[np.pi / 2, 0.0]]),
                     (4, 0, 0), "half")
    assert np.allclose(y.reshape(-1), [-3.0, 2.0, 1.0, 4.0], atol=1e-15)
    # sections two channels wide: both layouts pair (o, o + 1)
    x = rng(60).standard_normal((3, 2, 6))
    phi = rng(61).standard_normal((3, 3))
    assert np.array_equal(o.rope_apply(x, phi, (2, 2, 2), "half"), o.rope_apply(x, phi))
    for dims in ((32, 48, 48), (128, 0, 0), (16, 0, 112)):
        x = rng(62).standard_normal((5, 3, 128))
        pos = rng(63).integers(0, 90, size=(5, 3))
        phi = o.rope_angles(pos, dims, 1e4)
        y = o.rope_apply(x, phi, dims, "half")
        # the split-half layout is the interleaved one under a per-section
        # permutation: interleaved slot o+2j <- half slot o+j, o+2j+1 <- o+d/2+j
        perm = []
        base = 0
        for d in dims:
            for j in range(d // 2):
                perm += [base + j, base + d // 2 + j]
            base += d
        perm = np.array(perm)
        assert np.allclose(y[..., perm], o.rope_apply(x[..., perm], phi), atol=1e-13)
        # pair by pair (explicit loop): norm kept, angle added
        base = 0
        p = 0
        for d in dims:
            for j in range(d // 2):
                a, b = base + j, base + d // 2 + j
                z0 = complex(x[0, 1, a], x[0, 1, b]) * complex(math.cos(phi[0, p]), math.sin(phi[0, p]))
                assert math.isclose(y[0, 1, a], z0.real, abs_tol=1e-13)
                assert math.isclose(y[0, 1, b], z0.imag, abs_tol=1e-13)
                p += 1
            base += d
        # turning back restores the input
        assert np.allclose(o.rope_apply(y, -phi, dims, "half"), x, atol=1e-13)


def check_qk_norm_rope(o):
    # norm first, then rope: with all positions 0 the result is the rounded RMSNorm
    x = bf16_values(rng(11).standard_normal((4, 3, 128)))
    gain = 1 + 0.1 * rng(12).standard_normal(128)
    pos0 = np.zeros((4, 3), np.int64)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(gain), eps=1e-6)
    y0 = o.qk_norm_rope(x, gain, pos0, (32, 48, 48), 1e4, 1e-6)
    assert np.all(np.abs(y0 - ref.numpy()) <= 2.0 ** -8 * np.abs(ref.numpy()))
    # the output row has RMS equal to the RMS of the gain-scaled unit vector:
    # with gain = 1 the rotated row keeps unit RMS (up to bf16 rounding)
    pos = rng(13).integers(0, 60, size=(4, 3))
    y = o.qk_norm_rope(x, np.ones(128), pos, (32, 48, 48), 1e4, 0.0)
    assert np.allclose(np.sqrt((y * y).mean(-1)), 1.0, atol=4e-3)


def test_rms_norm():
    check_rms_norm(O)


def test_rope():
    check_rope(O)


def test_rope_half():
    check_rope_half(O)


def test_qk_norm_rope():
    check_qk_norm_rope(O)


# ---------------------------------------------------------- a3 attention
def check_attention(o):
    g = GOLD["attention_two_keys"]
    q = np.zeros((3, 1, 2)); q[0, 0] = [1, 0]
    k = np.zeros((3, 1, 2)); k[1, 0] = [1, 0]; k[2, 0] = [50, 0]
    v = np.zeros((3, 1, 2)); v[0, 0] = [4, 0]; v[1, 0] = [0, 8]; v[2, 0] = [99, 99]
    out = o.attention(q, k, v, L=2, scale=g["scale"], rows=[0])
    assert np.allclose(out[0, 0], g["out"], atol=1e-15)
    r = rng(14)
    S, L, H, Dh = 40, 33, 2, 16
    q = bf16_values(r.standard_normal((S, H, Dh)))
    k = bf16_values(r.standard_normal((S, H, Dh)))
    v = bf16_values(r.standard_normal((S, H, Dh)))
    out = o.attention(q, k, v, L, 0.25)
    # library pin: scaled_dot_product_attention in float64 on the valid rows
    t = lambda a: torch.from_numpy(a[:L]).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=0.25)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy(), rtol=2 ** -8, atol=1e-12)
    # brute force, one element by explicit loops
    i, h, d = 7, 1, 3
    logits = [sum(q[i, h, c] * k[j, h, c] for c in range(Dh)) * 0.25 for j in range(L)]
    m = max(logits)
    w = [math.exp(x - m) for x in logits]
    val = sum(w[j] * v[j, h, d] for j in range(L)) / sum(w)
    assert abs(out[i, h, d] - val) <= 2 ** -8 * abs(val) + 1e-15
    # rows sum to one: constant V passes through unchanged
    assert np.array_equal(o.attention(q, k, np.ones_like(v), L, 0.25), np.ones((L, H, Dh)))
    # identical keys: the output is the mean of V
    kk = np.broadcast_to(k[:1], k.shape).copy()
    assert np.allclose(o.attention(q, kk, v, L, 0.25), O.round_bf16(v[:L].mean(0, keepdims=True)).repeat(L, 0),
                       atol=1e-15)
    # one dominant logit selects that value row
    kd = np.zeros_like(k); kd[5] = 1.0
    qd = np.ones_like(q)
    assert np.allclose(o.attention(qd, kd, v, L, 100.0), np.broadcast_to(v[5], (L, H, Dh)), atol=1e-15)
    # pad rows of K, V do not matter; a row subset equals the full result
    k2, v2 = k.copy(), v.copy(); k2[L:] = 1e3; v2[L:] = -7
    assert np.array_equal(o.attention(q, k2, v2, L, 0.25), out)
    assert np.array_equal(o.attention(q, k, v, L, 0.25, rows=[3, 30, 0]), out[[3, 30, 0]])


def test_attention():
    check_attention(O)


# ------------------------------------------------------ a4 / a5 GEMM, SwiGLU
def check_linear(o):
    r = rng(15)
    x = r.integers(-8, 9, size=(5, 12)).astype(np.float64)
    w = r.integers(-8, 9, size=(7, 12)).astype(np.float64)
    exact = np.array([[sum(x[i, c] * w[j, c] for c in range(12)) for j in range(7)] for i in range(5)])
    assert np.array_equal(o.linear(x, w), exact)   # |values| < 2^8: bf16-exact
    x = bf16_values(r.standard_normal((6, 20)))
    w = bf16_values(r.standard_normal((3, 20)))
    ref = torch.from_numpy(x) @ torch.from_numpy(w).T
    assert np.all(np.abs(o.linear(x, w) - ref.numpy()) <= 2.0 ** -8 * np.abs(ref.numpy()))


def check_swiglu(o):
    g = GOLD["silu_points"]
    assert np.allclose(o.silu(np.array(g["g"])), g["silu"], rtol=1e-15, atol=0)
    assert math.isclose(o.silu(np.array([40.0]))[0], 40.0, rel_tol=1e-15)
    assert abs(o.silu(np.array([-40.0]))[0]) < 1e-15
    r = rng(16)
    gu = bf16_values(r.standard_normal((5, 24)) * 2)
    ref = torch.nn.functional.silu(torch.from_numpy(gu[:, :12])) * torch.from_numpy(gu[:, 12:])
    assert np.allclose(o.swiglu(gu), ref.numpy(), rtol=2 ** -8, atol=1e-30)
    # halves are [gate | up]: gate 0 zeroes the output whatever the up half holds
    gu0 = gu.copy(); gu0[:, :12] = 0
    assert np.array_equal(o.swiglu(gu0), np.zeros((5, 12)))


def test_linear():
    check_linear(O)


def test_swiglu():
    check_swiglu(O)


# ------------------------------------------------------------ a6 the block
def tiny_block(shape=None, seed=0):
    shape = shape or I.BlockShape(S=24, L=21, D=64, H=2, Dh=32, F=96, axis_dims=(16, 8, 8),
                                  pos_kind="3d", grid=(2, 3, 4), n_tail=3)
    inp = I.block_inputs(shape, seed)
    n = {k: (v.double().numpy() if torch.is_tensor(v) and v.is_floating_point() else v.numpy())
         for k, v in inp.items()}
    return shape, n


def run_block(o, shape, n, rows=None, inter=False, seg=None, **over):
    args = dict(n)
    args.update(over)
    return o.block_forward(args["resid"], args["mod"], args["w_qkv"], args["w_o"], args["w_gu"],
                           args["w_down"], args["q_gain"], args["k_gain"], args["pos"],
                           L=shape.L, heads=shape.H, head_dim=shape.Dh,
                           axis_dims=shape.axis_dims, theta=shape.theta, rows=rows,
                           return_intermediates=inter, seg=seg)


def torch_block(shape, n, mod_rows=None):
    """The block written with torch float64 library routines (layer_norm,
    rms_norm, scaled_dot_product_attention, silu) and a complex-number RoPE,
    with bf16 rounding at the same hand-off points. Returns every hand-off.
    mod_rows: optional per-row modulation [L, 6, D] instead of n["mod"]."""
    T = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    rb = lambda t: t.float().to(torch.bfloat16).double()
    L, D, H, Dh = shape.L, shape.D, shape.H, shape.Dh
    r = T(n["resid"])[:L]
    m6 = T(n["mod"] if mod_rows is None else mod_rows)
    mod = [m6[..., i, :] for i in range(6)]
    ln = lambda x: torch.nn.functional.layer_norm(x, (D,), eps=1e-6)
    h1 = rb(ln(r) * (1 + mod[1]) + mod[0])
    qkv = rb(h1 @ T(n["w_qkv"]).T)
    q, k, v = (qkv[:, i * D:(i + 1) * D].reshape(L, H, Dh) for i in range(3))
    pos = T(n["pos"])[:L]
    ang = []
    for a, d in enumerate(shape.axis_dims):
        if d:
            ang.append(pos[:, a:a + 1] * shape.theta ** (-torch.arange(0, d, 2, dtype=torch.float64) / d))
    ang = torch.cat(ang, 1)[:, None, :]
    def rope(x):
        z = torch.complex(x[..., 0::2], x[..., 1::2]) * torch.polar(torch.ones_like(ang), ang)
        return torch.stack([z.real, z.imag], -1).reshape(x.shape)
    q = rb(rope(torch.nn.functional.rms_norm(q, (Dh,), T(n["q_gain"]), eps=1e-6)))
    k = rb(rope(torch.nn.functional.rms_norm(k, (Dh,), T(n["k_gain"]), eps=1e-6)))
    a = torch.nn.functional.scaled_dot_product_attention(q.permute(1, 0, 2), k.permute(1, 0, 2),
                                                         v.permute(1, 0, 2))
    a = rb(a.permute(1, 0, 2).reshape(L, D))
    o = rb(a @ T(n["w_o"]).T)
    r = (r + mod[2] * o).float().double()
    h2 = rb(ln(r) * (1 + mod[4]) + mod[3])
    gu = rb(h2 @ T(n["w_gu"]).T)
    F = gu.shape[1] // 2
    u = rb(torch.nn.functional.silu(gu[:, :F]) * gu[:, F:])
    f = rb(u @ T(n["w_down"]).T)
    r = (r + mod[5] * f).float().double()
    out = dict(h1=h1, q=q, k=k, v=v, a=a, o=o, h2=h2, gu=gu, u=u, f=f, r=r)
    return {key: val.numpy() for key, val in out.items()}


def close_bf16(x, ref):
    """bf16 hand-off agreement: elementwise 2e-2 * max(1, |ref|), rel-L2 1e-2."""
    x, ref = np.asarray(x).reshape(ref.shape), np.asarray(ref)
    ok_el = np.all(np.abs(x - ref) <= 2e-2 * np.maximum(1.0, np.abs(ref)))
    ok_l2 = np.linalg.norm(x - ref) <= 1e-2 * np.linalg.norm(ref)
    return ok_el and ok_l2


def check_block(o):
    shape, n = tiny_block()
    out, mids = run_block(o, shape, n, inter=True)
    ref = torch_block(shape, n)
    for key in ("h1", "q", "k", "v", "a", "o", "h2", "gu", "u", "f"):
        assert close_bf16(mids[key], ref[key]), key
    assert close_bf16(out, ref["r"])
    # the residual increment (gate1 * o + gate2 * f) is small next to the
    # residual itself, so compare it on its own
    r_in = n["resid"][:shape.L]
    assert close_bf16(out - r_in, ref["r"] - r_in), "residual increment"
    # zero output projections leave the residual untouched
    z = run_block(o, shape, n, w_o=np.zeros_like(n["w_o"]), w_down=np.zeros_like(n["w_down"]))
    assert np.array_equal(z, n["resid"][:shape.L])
    # zero gates too
    mod0 = n["mod"].copy(); mod0[2] = 0; mod0[5] = 0
    assert np.array_equal(run_block(o, shape, n, mod=mod0), n["resid"][:shape.L])
    # pad-row garbage does not reach valid rows
    r2 = n["resid"].copy(); r2[shape.L:] = 1e4
    p2 = n["pos"].copy(); p2[shape.L:] = 77
    assert np.array_equal(run_block(o, shape, n, resid=r2, pos=p2), out)
    # a subset of rows equals the same rows of the full evaluation
    rows = [17, 2, 0]
    assert np.array_equal(run_block(o, shape, n, rows=rows), out[rows])


def test_block():
    check_block(O)


def check_segmented_block(o):
    shape, n = tiny_block()
    out = run_block(o, shape, n)
    # one table and every token in group 0 is the per-sample case, bit for bit
    assert np.array_equal(run_block(o, shape, n, mod=n["mod"][None], seg=np.zeros(shape.S, int)),
                          out)
    g = rng(41)
    seg = g.integers(0, 2, shape.S)
    # two identical tables: the grouping does not matter
    assert np.array_equal(run_block(o, shape, n, mod=np.stack([n["mod"], n["mod"]]), seg=seg),
                          out)
    # two different tables against the torch composition with per-row modulation
    mod2 = np.stack([n["mod"], 0.3 * g.standard_normal(n["mod"].shape)])
    out2, mids = run_block(o, shape, n, mod=mod2, seg=seg, inter=True)
    ref = torch_block(shape, n, mod_rows=mod2[seg[:shape.L]])
    for key in ("h1", "q", "k", "a", "o", "h2", "u", "f"):
        assert close_bf16(mids[key], ref[key]), key
    r_in = n["resid"][:shape.L]
    assert close_bf16(out2 - r_in, ref["r"] - r_in), "segmented increment"
    # relabelling the groups (tables swapped, ids flipped) changes nothing
    assert np.array_equal(run_block(o, shape, n, mod=mod2[::-1].copy(), seg=1 - seg), out2)


def test_segmented_block():
    check_segmented_block(O)


def test_stack_is_two_torch_blocks():
    shape, n = tiny_block()
    _, n2 = tiny_block(seed=9)
    out = O.stack_forward(n["resid"], [n["mod"], n2["mod"]],
                          [(n[k] for k in ("w_qkv", "w_o", "w_gu", "w_down")),
                           (n2[k] for k in ("w_qkv", "w_o", "w_gu", "w_down"))],
                          [n["q_gain"], n2["q_gain"]], [n["k_gain"], n2["k_gain"]], n["pos"],
                          L=shape.L, heads=shape.H, head_dim=shape.Dh, axis_dims=shape.axis_dims,
                          theta=shape.theta)
    r1 = torch_block(shape, n)["r"]
    nb = dict(n2)
    nb["resid"] = np.concatenate([r1, n["resid"][shape.L:]])
    nb["pos"] = n["pos"]
    r2 = torch_block(shape, nb)["r"]
    assert close_bf16(out, r2)
    assert close_bf16(out - r1, r2 - r1), "second block's increment"


# --------------------------------------------- planted mistakes are caught
def _mutant(**repl):
    m = types.ModuleType("oracle_mutant")
    m.__dict__.update({k: v for k, v in O.__dict__.items() if not k.startswith("__")})
    m.__dict__["__builtins__"] = O.__dict__["__builtins__"]  # numpy's keyword calls need them
    for name, fn in repl.items():
        m.__dict__[name] = fn
    # functions look their helpers up in their own globals: rebind them
    for k, v in list(m.__dict__.items()):
        if isinstance(v, types.FunctionType) and k not in repl:
            m.__dict__[k] = types.FunctionType(v.__code__, m.__dict__, v.__name__, v.__defaults__,
                                               v.__closure__)
            m.__dict__[k].__kwdefaults__ = v.__kwdefaults__
    return m


def _rope_wrong_sign(x, phi, *args):
    return O.rope_apply(x, -phi, *args)


def _rope_half_whole_head(x, phi, axis_dims=None, pairing="interleaved"):
    # split-half pairs taken across the whole head instead of per section
    if pairing == "interleaved":
        return O.rope_apply(x, phi)
    return _rope_half_split(x, phi)


def _rope_half_split(x, phi, *args):
    x = np.asarray(x, np.float64)
    h = x.shape[-1] // 2
    c, s = np.cos(phi)[:, None, :], np.sin(phi)[:, None, :]
    out = np.empty_like(x)
    out[..., :h] = x[..., :h] * c - x[..., h:] * s
    out[..., h:] = x[..., :h] * s + x[..., h:] * c
    return out


def _angles_global_exponent(pos, axis_dims, theta):
    hd = sum(axis_dims)
    pos = np.asarray(pos, np.float64)
    cols = []
    for a, d in enumerate(axis_dims):
        if d:
            j = np.arange(d // 2)
            cols.append(pos[:, a:a + 1] * theta ** (-2.0 * j / hd))
    return np.concatenate(cols, 1)


def _mod_no_one_plus(resid, delta=None, gate=None, shift=None, scale=None, eps=1e-6):
    r = np.asarray(resid, np.float64)
    if delta is not None:
        r = O.round_f32(r + gate[None] * delta)
    h = None if scale is None else O.round_bf16(O.layer_norm(r, eps) * scale[None] + shift[None])
    return r, h


def _swiglu_swapped(gu):
    F = gu.shape[-1] // 2
    return O.round_bf16(O.silu(gu[..., F:]) * gu[..., :F])


def _ln_no_center(x, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt((x * x).mean(-1, keepdims=True) + eps)


def _attn_no_max_mask(q, k, v, L, scale, rows=None):
    return O.attention(q, k, v, k.shape[0], scale, rows=rows if rows is not None else np.arange(L))


def _softmax_wrong_axis(z, axis=-1):
    return O.softmax(z, axis=0)


def _unpack_shift_scale_swapped(mod):
    sh1, sc1, g1, sh2, sc2, g2 = O.unpack_mod(mod)
    return sc1, sh1, g1, sc2, sh2, g2


def _unpack_gates_swapped(mod):
    sh1, sc1, g1, sh2, sc2, g2 = O.unpack_mod(mod)
    return sh1, sc1, g2, sh2, sc2, g1


def _modulation_rows_shifted(mod, seg, rows):
    mod = np.asarray(mod, np.float64)
    if seg is None:
        return mod
    return mod[np.roll(np.asarray(seg), 1)[np.asarray(rows)]]


def _rms_no_eps_mean(x, gain, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps) * np.asarray(gain, np.float64)


@pytest.mark.parametrize("name,mut,checks", [
    ("rope sign", dict(rope_apply=_rope_wrong_sign), ["check_rope"]),
    ("rope half-split pairing", dict(rope_apply=_rope_half_split), ["check_rope"]),
    ("rope global exponent", dict(rope_angles=_angles_global_exponent), ["check_rope"]),
    ("split-half pairs across the head", dict(rope_apply=_rope_half_whole_head),
     ["check_rope_half"]),
    ("modulation without 1+", dict(mod_norm_residual=_mod_no_one_plus), ["check_mod_norm_residual"]),
    ("swiglu halves swapped", dict(swiglu=_swiglu_swapped), ["check_swiglu"]),
    ("layernorm not centred", dict(layer_norm=_ln_no_center), ["check_layer_norm"]),
    ("attention keys past L", dict(attention=_attn_no_max_mask), ["check_attention"]),
    ("softmax over queries", dict(softmax=_softmax_wrong_axis), ["check_attention"]),
    ("block with swapped rope", dict(rope_apply=_rope_wrong_sign), ["check_block"]),
    ("block with swapped swiglu", dict(swiglu=_swiglu_swapped), ["check_block"]),
    ("modulation shift/scale order", dict(unpack_mod=_unpack_shift_scale_swapped), ["check_block"]),
    ("modulation gates swapped", dict(unpack_mod=_unpack_gates_swapped), ["check_block"]),
    ("rmsnorm sum instead of mean", dict(rms_norm=_rms_no_eps_mean), ["check_rms_norm"]),
    ("segment of the wrong row", dict(modulation_rows=_modulation_rows_shifted),
     ["check_segmented_block"]),
])
def test_planted_mistake_is_caught(name, mut, checks):
    m = _mutant(**mut)
    for c in checks:
        with pytest.raises(AssertionError):
            globals()[c](m)


# ------------------------------------------------- GPU output preparation
def check_frames_to_u8(o):
    # closed-form points: -1 -> 0, 1 -> 255, 0 -> round(127.5) = 128 (half to
    # even), out-of-range values clamp, NaN-free inputs only
    x = np.array([-1.0, 1.0, 0.0, -3.0, 2.5, 0.5, -0.5], np.float32).reshape(1, 1, 1, 1, 7)
    assert o.frames_to_u8(x).reshape(-1).tolist() == [0, 255, 128, 0, 255, 191, 64]
    # layout: channel moves last, every other axis keeps its order
    g = rng(50)
    f = g.uniform(-1, 1, size=(2, 3, 4, 5, 6)).astype(np.float32)
    u = o.frames_to_u8(f)
    assert u.shape == (2, 4, 5, 6, 3) and u.dtype == np.uint8
    b, c, t, h, w = 1, 2, 3, 4, 5
    one = o.frames_to_u8(f[b:b + 1, c:c + 1, t:t + 1, h:h + 1, w:w + 1]).reshape(())
    assert u[b, t, h, w, c] == one
    # library pin: torch float32 arithmetic on the same steps
    tt = torch.from_numpy(f)
    ref = ((tt * 0.5 + 0.5).clamp(0, 1) * 255).round().to(torch.uint8).permute(0, 2, 3, 4, 1)
    assert np.array_equal(u, ref.contiguous().numpy())
    # monotone in x
    ramp = np.linspace(-1.2, 1.2, 10001, dtype=np.float32).reshape(1, 1, 1, 1, -1)
    assert np.all(np.diff(o.frames_to_u8(ramp).reshape(-1).astype(int)) >= 0)


def test_frames_to_u8():
    check_frames_to_u8(O)


def _frames_wrong_axis(frames):
    x = np.asarray(frames, np.float32)
    v = np.rint(np.clip(x * np.float32(0.5) + np.float32(0.5), 0, 1) * np.float32(255))
    return np.ascontiguousarray(np.moveaxis(v.astype(np.uint8), 2, -1))


def _frames_truncating(frames):
    x = np.asarray(frames, np.float32)
    v = np.floor(np.clip(x * np.float32(0.5) + np.float32(0.5), 0, 1) * np.float32(255))
    return np.ascontiguousarray(np.moveaxis(v.astype(np.uint8), 1, -1))


@pytest.mark.parametrize("mut", [_frames_wrong_axis, _frames_truncating])
def test_planted_output_prep_mistake_is_caught(mut):
    with pytest.raises(AssertionError):
        check_frames_to_u8(_mutant(frames_to_u8=mut))


# ------------------------------------------------------ online FP8 projections
def check_fp8(o):
    # hand-derived E4M3 points: 1 + 1/16 ties to 1 (even), 1 + 3/16 ties to
    # 1.25 (even), 2^-10 ties to 0, 3 * 2^-10 ties to 2^-8, 500 saturates to 448
    pts = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 500.0, -500.0, 2.0 ** -9, 240.0])
    assert o.round_e4m3(pts).tolist() == [1.0, 1.25, 0.0, 2.0 ** -8, 448.0, -448.0, 2.0 ** -9,
                                          240.0]
    # library pin: torch's float32 -> float8_e4m3fn cast inside the finite range
    x = (rng(60).standard_normal(20000) * 50).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(o.round_e4m3(x.astype(np.float64)), ref)
    # per-row absmax: the row maximum maps to +-448 exactly, a zero row to 0
    xs = bf16_values(rng(61).standard_normal((5, 64)) * 3)
    xs[3] = 0
    q, s = o.quantize_fp8_rows(xs)
    am = np.abs(xs).max(1)
    for i in (0, 1, 2, 4):
        assert np.max(np.abs(q[i])) == 448.0
        assert s[i] == np.float32(np.float32(am[i]) / np.float32(448))
    assert np.all(q[3] == 0) and s[3] == 0
    # dequantisation error is at most half an E4M3 step (relative 2^-4) per value
    err = np.abs(q * s[:, None] - xs)
    assert np.all(err <= np.abs(xs) * 2.0 ** -4 + s[:, None] * 2.0 ** -9 + 1e-12)
    # the product: integer codes with unit scales give the exact integer product
    qa = rng(62).integers(-4, 5, size=(4, 32)).astype(np.float64)
    qb = rng(63).integers(-4, 5, size=(6, 32)).astype(np.float64)
    exact = np.array([[sum(qa[i, k] * qb[j, k] for k in range(32)) for j in range(6)]
                      for i in range(4)])
    assert np.array_equal(o.linear_fp8(qa, np.ones(4), qb, np.ones(6)), exact)
    # the row and column scales multiply the product
    sa, sb = np.array([1, 2, 4, 0.5]), np.array([1, 1, 2, 2, 8, 0.25])
    assert np.array_equal(o.linear_fp8(qa, sa, qb, sb),
                          o.round_bf16(exact * sa[:, None] * sb[None, :]))


def test_fp8():
    check_fp8(O)


def _e4m3_truncating(x):
    x = np.asarray(x, np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    _, e = np.frexp(x[nz])
    step = np.exp2(np.maximum(e - 4, -9).astype(np.float64))
    out[nz] = np.clip(np.trunc(x[nz] / step) * step, -448, 448)
    return out


def _linear_fp8_no_row_scale(qx, sx, qw, sw):
    acc = np.asarray(qx, np.float64) @ np.asarray(qw, np.float64).T
    return O.round_bf16(acc * np.asarray(sw, np.float64)[None, :])


@pytest.mark.parametrize("mut", [dict(round_e4m3=_e4m3_truncating),
                                 dict(linear_fp8=_linear_fp8_no_row_scale)])
def test_planted_fp8_mistake_is_caught(mut):
    with pytest.raises(AssertionError):
        check_fp8(_mutant(**mut))


def test_fp8_block_close_to_bf16_block():
    # the FP8 block differs from the BF16 block only by the E4M3 rounding of the
    # four projection operands (relative step 2^-4): its hand-offs stay within
    # a few percent of the BF16 ones, and integer-valued weights and inputs that
    # E4M3 holds exactly give the same projections
    shape, n = tiny_block()
    out, mids = run_block(O, shape, n, inter=True)
    out8, mids8 = O.block_forward(n["resid"], n["mod"], n["w_qkv"], n["w_o"], n["w_gu"],
                                  n["w_down"], n["q_gain"], n["k_gain"], n["pos"], L=shape.L,
                                  heads=shape.H, head_dim=shape.Dh, axis_dims=shape.axis_dims,
                                  theta=shape.theta, return_intermediates=True, fp8=True)
    for key in ("q", "a", "o", "u", "f"):
        assert rel_l2_(mids8[key], mids[key]) < 0.08, key
    assert 0 < rel_l2_(mids8["f"], mids["f"])  # the FP8 path is really taken
    r_in = n["resid"][:shape.L]
    assert rel_l2_(out8 - r_in, out - r_in) < 0.08


def rel_l2_(x, ref):
    return float(np.linalg.norm(np.asarray(x) - np.asarray(ref)) / np.linalg.norm(ref))


def check_attention_skip(o):
    r = rng(70)
    S = L = 384
    H = 2
    q = bf16_values(r.standard_normal((S, H, 16)))
    k = bf16_values(r.standard_normal((S, H, 16)))
    v = bf16_values(r.standard_normal((S, H, 16)))
    dense = o.attention(q, k, v, L, 0.25)
    # eps = 0 keeps every tile and is dense attention
    out0, kept0 = o.attention_skip(q, k, v, L, 0.25, 0.0)
    assert kept0.all() and np.allclose(out0, dense, rtol=2 ** -8, atol=1e-12)
    # a key tile pushed far below every score is skipped for every query tile,
    # and the result is attention over the other keys
    k2 = k.copy()
    q2 = np.abs(q) + 0.5
    k2[128:256] = -np.abs(k2[128:256]) - 8.0
    out, kept = o.attention_skip(q2, k2, v, L, 0.25, 2.0 ** -20)
    assert (~kept[:, :, 1]).all() and kept[:, :, [0, 2]].all()
    keep = np.r_[0:128, 256:384]
    sub = np.empty((L, H, 16))
    for h in range(H):
        z = (q2[:, h] @ k2[keep, h].T) * 0.25
        sub[:, h] = torch.softmax(torch.from_numpy(z), dim=1).numpy() @ v[keep, h]
    assert np.allclose(out, sub, rtol=2 ** -7, atol=1e-12)
    # the first key tile is never skipped (no running maximum yet)
    k3 = k.copy()
    k3[:128] = -np.abs(k3[:128]) - 8.0
    _, kept3 = o.attention_skip(q2, k3, v, L, 0.25, 2.0 ** -20)
    assert kept3[:, :, 0].all()


def test_attention_skip():
    check_attention_skip(O)


def check_sage(o):
    r = rng(80)
    S = L = 300
    H, Dh = 2, 32
    q = bf16_values(r.standard_normal((S, H, Dh)))
    k = bf16_values(r.standard_normal((S, H, Dh)) + 3.0)  # a large common offset
    v = bf16_values(r.standard_normal((S, H, Dh)))
    ops = o.sage_quantize(q, k, v, L)
    # smoothing removes the per-channel mean of the valid keys, a float32 value
    assert np.allclose(ops["k_mean"], k.mean(0), rtol=2 ** -23, atol=0)
    assert np.array_equal(ops["k_mean"], ops["k_mean"].astype(np.float32).astype(np.float64))
    # dequantised operands are within half an E4M3 step of the originals
    for c, s, x, kind in ((ops["qc"], ops["sq"], q, "q"), (ops["kc"], ops["sk"],
                          k - ops["k_mean"][None], "k")):
        deq = c * np.repeat(s.astype(np.float64), 128, axis=0)[:L][:, :, None]
        assert np.all(np.abs(deq - x) <= np.abs(x) * 2.0 ** -4 + 2.0 ** -9 * np.max(np.abs(x)) + 1e-12), kind
    deq_v = ops["vc"] * ops["sv"][None].astype(np.float64)
    assert np.all(np.abs(deq_v - v) <= np.abs(v) * 2.0 ** -4 + 2.0 ** -9 * np.abs(v).max(0) + 1e-12)
    # smoothing is exact in the score: subtracting a per-channel constant from
    # every key moves each query row's scores by one constant, which softmax
    # ignores
    s_full = q[:, 0] @ k[:, 0].T
    s_smooth = q[:, 0] @ (k[:, 0] - ops["k_mean"][0]).T
    d = s_full - s_smooth
    assert np.allclose(d, d[:, :1], atol=1e-9)
    # the FP8 result stays close to dense attention: per-element E4M3 noise on
    # P and V is about 2^-4 / sqrt(3) each, ~5 % of the output for random V
    scale = Dh ** -0.5
    dense = o.attention(q, k, v, L, scale)
    out = o.attention_sage(ops, L, scale)
    assert np.linalg.norm(out - dense) / np.linalg.norm(dense) < 0.1
    # all scores 0 (q = 0): every weight is exactly 1, whose code 448 is exact,
    # so the output is the mean of the dequantised V rows
    opu = o.sage_quantize(np.zeros_like(q), k, v, L)
    deq_v = opu["vc"] * opu["sv"][None].astype(np.float64)
    assert np.allclose(o.attention_sage(opu, L, scale),
                       o.round_bf16(deq_v.mean(0))[None].repeat(L, 0), rtol=2 ** -8, atol=1e-12)
    # one key far above the others: its weight is 1 (code 448, exact), every
    # other weight underflows, so the output is that key's dequantised V row
    kd = np.zeros_like(k)
    kd[7] = 8.0
    opd = o.sage_quantize(np.ones_like(q), kd, v, L)
    deq_vd = opd["vc"] * opd["sv"][None].astype(np.float64)
    assert np.allclose(o.attention_sage(opd, L, 1.0),
                       np.broadcast_to(o.round_bf16(deq_vd[7]), (L, H, Dh)), rtol=2 ** -8,
                       atol=1e-12)
    # hand-built operands (attention_sage takes any values): one query, scale
    # ln 2 so that the base-2 logit is the plain dot product. Key 0 has logit
    # 0.3 (the row maximum, not an integer); keys 1..7 sit log2(270/448)
    # below it, so their weight is 270/448 and its code rounds 270 down to 256
    # (E4M3 step 32 in [256, 512); 272 would be the tie). Key 0's V row is
    # (1, 0) and the others' (0, 1):
    #   out = (448 * (1, 0) + 7 * 256 * (0, 1)) / (448 * (1 + 7 * 270 / 448))
    #       = (448, 1792) / 2338
    n = 8
    hand = dict(qc=np.ones((n, 1, 1)), sq=np.ones((1, 1), np.float32),
                kc=np.full((n, 1, 1), 0.3 + math.log2(270 / 448)),
                sk=np.ones((1, 1), np.float32),
                vc=np.zeros((n, 1, 2)), sv=np.ones((1, 2), np.float32))
    hand["kc"][0] = 0.3
    hand["vc"][0, 0, 0] = 1.0
    hand["vc"][1:, 0, 1] = 1.0
    got = o.attention_sage(hand, n, math.log(2.0), rows=np.array([0]))
    assert np.array_equal(got[0, 0], bf16_values([448 / 2338, 1792 / 2338])), got
    # two keys a whole binade apart (logits 0.3 and -0.7): weights 1 and 1/2,
    # codes 448 and 224, both exact: out = (w0 + w1 / 2) / (3 / 2)
    two = dict(hand, kc=np.array([[[0.3]], [[-0.7]]]), vc=np.array([[[2.0, -1.0]], [[4.0, 8.0]]]),
               sv=np.array([[0.25, 0.5]], np.float32))
    got = o.attention_sage(two, 2, math.log(2.0), rows=np.array([0]))
    assert np.array_equal(got[0, 0], bf16_values([(0.5 + 0.5) / 1.5, (-0.5 + 2.0) / 1.5])), got


def test_sage():
    check_sage(O)


def test_sage_error_terms():
    # the sums of sage_error_terms from the definition, through the library's
    # softmax: with s = softmax of the natural-log logits, p / sum p = s and
    # sum p = 1 / max s (the largest weight is exactly 1)
    r = rng(81)
    L, H, Dh = 37, 2, 8
    q = bf16_values(r.standard_normal((L, H, Dh)))
    k = bf16_values(r.standard_normal((L, H, Dh)))
    v = bf16_values(r.standard_normal((L, H, Dh)))
    ops = O.sage_quantize(q, k, v, L, tile=16)
    rows = np.array([0, 5, 36])
    a1, a0, v2, u2 = O.sage_error_terms(ops, L, 0.3, rows=rows, tile=16)
    for h in range(H):
        for n, i in enumerate(rows):
            zq = ops["qc"][i, h] * float(ops["sq"][i // 16, h])
            logits = [float(zq @ ops["kc"][j, h]) * float(ops["sk"][j // 16, h]) * 0.3
                      for j in range(L)]
            sm = torch.softmax(torch.tensor(logits, dtype=torch.float64), 0).numpy()
            w = np.abs(ops["vc"][:, h, :] * ops["sv"][h].astype(np.float64))
            tot = 1.0 / sm.max()
            assert np.allclose(a1[n, h], sm @ w, rtol=1e-12)
            assert np.allclose(a0[n, h], w.sum(0) / tot, rtol=1e-12)
            assert np.allclose(v2[n, h], (sm * sm) @ (w * w), rtol=1e-12)
            assert np.allclose(u2[n, h], (w * w).sum(0) / tot ** 2, rtol=1e-12)


def _sage_no_smoothing(q, k, v, L, tile=128):
    ops = O.sage_quantize(q, k, v, L, tile)
    ops2 = O.sage_quantize(q, k, v, L, tile)
    ops2["k_mean"] = np.zeros_like(ops["k_mean"])
    return ops2


def _sage_p_unscaled(ops, L, scale, rows=None, tile=128):
    rows = np.arange(L) if rows is None else np.asarray(rows)
    vc, sv = ops["vc"], ops["sv"].astype(np.float64)
    out = np.empty((len(rows),) + vc.shape[1:])
    for h in range(vc.shape[1]):
        p = O._sage_weights(ops, h, rows, L, scale, tile)
        out[:, h, :] = (O.round_e4m3(p) @ vc[:L, h, :]) * sv[h][None, :] / p.sum(1, keepdims=True)
    return O.round_bf16(out)


def _sage_sum_of_codes(ops, L, scale, rows=None, tile=128):
    rows = np.arange(L) if rows is None else np.asarray(rows)
    vc, sv = ops["vc"], ops["sv"].astype(np.float64)
    out = np.empty((len(rows),) + vc.shape[1:])
    for h in range(vc.shape[1]):
        pc = O.round_e4m3(448.0 * O._sage_weights(ops, h, rows, L, scale, tile))
        out[:, h, :] = (pc @ vc[:L, h, :]) * sv[h][None, :] / pc.sum(1, keepdims=True)
    return O.round_bf16(out)


def _sage_weights_ceil_max(ops, h, rows, L, scale, tile):
    # weights against the next integer above the row maximum, at half scale
    # (224 * 2^(z - ceil max z) after the 448 of attention_sage)
    qc, kc = ops["qc"], ops["kc"]
    key_tile = np.arange(L) // tile
    s = (qc[rows, h, :] @ kc[:L, h, :].T) * ops["sq"].astype(np.float64)[rows // tile, h][:, None] \
        * ops["sk"].astype(np.float64)[key_tile, h][None, :]
    z = s * scale / np.log(2.0)
    return 0.5 * np.exp2(z - np.ceil(z.max(axis=1, keepdims=True)))


@pytest.mark.parametrize("mut", [dict(sage_quantize=_sage_no_smoothing),
                                 dict(attention_sage=_sage_p_unscaled),
                                 dict(attention_sage=_sage_sum_of_codes),
                                 dict(_sage_weights=_sage_weights_ceil_max)])
def test_planted_sage_mistake_is_caught(mut):
    with pytest.raises(AssertionError):
        check_sage(_mutant(**mut))


# ------------------------------------------- SAGE attention with Skip-Softmax
def _hand_ops(logits, tile=128):
    """SAGE operands whose base-2 logits (at scale ln 2) are given directly:
    logits [R, L] for R query rows, one head. Head dim 2: q = (1, b_i),
    k = (a_j, c_j) so that z_ij = a_j + b_i c_j; here b_i c_j carries the
    per-row part (zero unless a pin sets it). V codes are a fixed ramp."""
    R, L = logits.shape
    nt = (max(R, L) + tile - 1) // tile
    qc = np.zeros((max(R, L), 1, 2)); qc[:, 0, 0] = 1.0
    kc = np.zeros((L, 1, 2)); kc[:, 0, 0] = logits[0]
    extra = logits - logits[0][None, :]
    rows, cols = np.nonzero(extra)
    for i, j in zip(rows, cols):  # one per-row exception per key at most
        qc[i, 0, 1] = 1.0
        kc[j, 0, 1] = extra[i, j]
    vc = np.zeros((L, 1, 3))
    vc[:, 0, 0] = np.arange(L) % 7 - 3.0
    vc[:, 0, 1] = np.arange(L) % 5 - 2.0
    vc[:, 0, 2] = 1.0
    return dict(qc=qc, sq=np.ones((nt, 1), np.float32), kc=kc, sk=np.ones((nt, 1), np.float32),
                vc=vc, sv=np.ones((1, 3), np.float32))


def check_sage_skip(o):
    r = rng(90)
    # eps = 0 leaves nothing out: exactly attention_sage
    L, H, Dh = 300, 2, 32
    q = bf16_values(r.standard_normal((L, H, Dh)))
    k = bf16_values(r.standard_normal((L, H, Dh)))
    v = bf16_values(r.standard_normal((L, H, Dh)))
    ops = o.sage_quantize(q, k, v, L)
    out0, kept0 = o.attention_sage_skip(ops, L, Dh ** -0.5, 0.0)
    assert kept0.all() and np.array_equal(out0, o.attention_sage(ops, L, Dh ** -0.5))
    t0 = o.sage_skip_error_terms(ops, L, Dh ** -0.5, 0.0)
    for x, y in zip(t0, o.sage_error_terms(ops, L, Dh ** -0.5)):
        assert np.allclose(x, y, rtol=1e-12, atol=0)
    # hand-built logits (scale ln 2: the logit is the dot product): three key
    # tiles; tiles 0 and 2 in [0, 1], tile 1 in [-5.5, -4.6], i.e. 5.6 or
    # more below the running maximum of the kept tiles (tile 0's maximum is
    # above 0.99). eps = 1/16 (threshold 4) leaves tile 1 out for every query
    # tile (a threshold of log2(16) / ln 2 = 5.77 would keep it), and the
    # result is attention_sage over the other 256 keys; the left-out weights
    # (up to 2^-5.6) are large enough that counting them would move the output
    # by more than 1 %.
    L = 384
    base = np.concatenate([r.uniform(0, 1, 128), r.uniform(-5.5, -4.6, 128), r.uniform(0, 1, 128)])
    assert base[:128].max() - base[128:256].max() < 5.77
    logits = np.repeat(base[None], L, axis=0)
    ops = _hand_ops(logits)
    out, kept = o.attention_sage_skip(ops, L, math.log(2.0), 2.0 ** -4)
    assert np.array_equal(kept, np.repeat(np.array([[[True, False, True]]]), 3, axis=0))
    keep = np.r_[0:128, 256:384]
    red = dict(ops, kc=ops["kc"][keep], vc=ops["vc"][keep], sk=ops["sk"][[0, 2]])
    want = o.attention_sage(red, 256, math.log(2.0), rows=np.arange(L))
    assert np.allclose(out, want, rtol=2 ** -8, atol=1e-12)
    # the V rows of the left-out tile do not matter; in dense attention they do
    vc_v = ops["vc"].copy()
    vc_v[128:256] = 50.0
    ops_v = dict(ops, vc=vc_v)
    assert np.array_equal(o.attention_sage_skip(ops_v, L, math.log(2.0), 2.0 ** -4)[0], out)
    assert np.max(np.abs(o.attention_sage(ops_v, L, math.log(2.0)) - out)) > 0.1
    # the error terms are those of the kept keys
    terms = o.sage_skip_error_terms(ops, L, math.log(2.0), 2.0 ** -4)
    for x, y in zip(terms, o.sage_error_terms(red, 256, math.log(2.0), rows=np.arange(L))):
        assert np.allclose(x, y, rtol=1e-9, atol=0)
    # the threshold is log2(1/eps): tile 1 exactly 3.5 below tile 0's maximum
    # (its own maximum; every row the same) is kept at eps = 1/16
    base_b = base.copy()
    base_b[128:256] = base[:128].max() - 3.5
    _, kept_b = o.attention_sage_skip(_hand_ops(np.repeat(base_b[None], L, axis=0)), L,
                                      math.log(2.0), 2.0 ** -4)
    assert kept_b.all()
    # a tile is left out only when every row of the query tile falls below:
    # row 5 sees key 200 at logit 4, so query tile 0 keeps key tile 1
    logits_c = logits.copy()
    logits_c[5, 200] = 4.0
    _, kept_c = o.attention_sage_skip(_hand_ops(logits_c), L, math.log(2.0), 2.0 ** -4)
    assert kept_c[0, 0, 1] and not kept_c[1, 0, 1] and not kept_c[2, 0, 1]
    # the first key tile is always kept, however far below the later ones
    base_d = base[[*range(128, 256), *range(0, 128), *range(256, 384)]]
    _, kept_d = o.attention_sage_skip(_hand_ops(np.repeat(base_d[None], L, axis=0)), L,
                                      math.log(2.0), 2.0 ** -4)
    assert kept_d[:, :, 0].all() and kept_d[:, :, 1:].all()


def test_sage_skip():
    check_sage_skip(O)


def _skip_tiles_natural_log(ops, L, scale, eps, tile):
    # threshold ln(1/eps) instead of log2(1/eps)
    yield from O._sage_skip_tiles(ops, L, scale, eps ** math.log(2.0), tile)


def _skip_tiles_log_ratio(ops, L, scale, eps, tile):
    # threshold log2(1/eps) / ln 2 (the logits' base mixed up the other way)
    yield from O._sage_skip_tiles(ops, L, scale, eps ** (1 / math.log(2.0)), tile)


def _skip_tiles_any_row(ops, L, scale, eps, tile):
    # leave a tile out when ANY row falls below (instead of every row)
    H = ops["vc"].shape[1]
    nt = (L + tile - 1) // tile
    thresh = np.inf if eps <= 0 else np.log2(1.0 / eps)
    for h in range(H):
        for qi in range(nt):
            rows = np.arange(qi * tile, min(L, (qi + 1) * tile))
            z = O._sage_logits(ops, h, rows, L, scale, tile)
            m = np.full(len(rows), -np.inf)
            keep = np.zeros(nt, bool)
            for kj in range(nt):
                tmax = z[:, kj * tile:min(L, (kj + 1) * tile)].max(axis=1)
                if np.any(tmax < m - thresh):
                    continue
                keep[kj] = True
                m = np.maximum(m, tmax)
            cols = np.flatnonzero(np.repeat(keep, tile)[:L])
            yield h, qi, rows, keep, cols, z[:, cols]


def _sage_skip_sum_all(ops, L, scale, eps, tile=128):
    # the row sum over every key, left-out tiles included
    vc, sv = ops["vc"], ops["sv"].astype(np.float64)
    nt = (L + tile - 1) // tile
    out = np.empty((L,) + vc.shape[1:])
    kept = np.zeros((nt, vc.shape[1], nt), bool)
    for h, qi, rows, keep, cols, z in O._sage_skip_tiles(ops, L, scale, eps, tile):
        kept[qi, h] = keep
        zall = O._sage_logits(ops, h, rows, L, scale, tile)
        p = np.exp2(z - z.max(axis=1, keepdims=True))
        pall = np.exp2(zall - z.max(axis=1, keepdims=True))
        out[rows, h, :] = (O.round_e4m3(448.0 * p) @ vc[cols, h, :]) * sv[h][None, :] \
            / (448.0 * pall.sum(axis=1, keepdims=True))
    return O.round_bf16(out), kept


@pytest.mark.parametrize("mut", [dict(_sage_skip_tiles=_skip_tiles_natural_log),
                                 dict(_sage_skip_tiles=_skip_tiles_log_ratio),
                                 dict(_sage_skip_tiles=_skip_tiles_any_row),
                                 dict(attention_sage_skip=_sage_skip_sum_all)])
def test_planted_sage_skip_mistake_is_caught(mut):
    with pytest.raises(AssertionError):
        check_sage_skip(_mutant(**mut))
