"""Online FP8 projections on tcgen05 (kind::f8f6f4) against the oracle:
per-row E4M3 codes and scales bit for bit (an integer decision both sides take
in float32), FP8 GEMMs within the bf16 tolerances, the FP8 block on every row
of the tiny block and on sampled rows at full size."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, assert_close_block, np64, rel_l2, sample_rows

pytestmark = pytest.mark.gpu
dev = "cuda"
SENT = -7.25


def codes_to_values(q):
    return q.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()


def quantize(h3lib, x):
    q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    s = torch.empty(x.shape[0], dtype=torch.float32, device=dev)
    h3lib.quantize_fp8_rows(x, q, s)
    h3lib.check_device_error()
    return q, s


@pytest.mark.parametrize("R,K", [(7, 8), (250, 512), (64, 5376), (33, 14336), (5, 16384)])
def test_quantize_matches_oracle_bitwise(h3lib, R, K):
    g = torch.Generator(device=dev)
    g.manual_seed(R + K)
    x = (torch.randn(R, K, generator=g, device=dev) * 3).to(torch.bfloat16)
    x[0, : K // 2] = 0  # a partly zero row
    if R > 2:
        x[2] = 0         # an all-zero row
    q, s = quantize(h3lib, x)
    qr, sr = O.quantize_fp8_rows(np64(x))
    assert np.array_equal(codes_to_values(q), qr)
    assert np.array_equal(s.double().cpu().numpy(), sr)


def test_linear_fp8_exact_small_integers(h3lib):
    # codes of small integers with unit scales: every product and partial sum
    # is an exact integer in FP32 and bf16 holds the result exactly
    S, N, K = 256, 256, 128
    g = torch.Generator(device="cpu")
    g.manual_seed(11)
    xa = torch.randint(-2, 3, (S, K), generator=g).float()
    xb = torch.randint(-2, 3, (N, K), generator=g).float()
    qa = xa.to(torch.float8_e4m3fn).view(torch.uint8).to(dev)
    qb = xb.to(torch.float8_e4m3fn).view(torch.uint8).to(dev)
    ones_a = torch.ones(S, device=dev)
    ones_b = torch.ones(N, device=dev)
    y = torch.full((S, N), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear_fp8(qa, ones_a, qb, ones_b, y)
    h3lib.check_device_error()
    assert torch.equal(y.double().cpu(), xa.double() @ xb.double().T)


@pytest.mark.parametrize("S,L,N,K", [(256, 250, 256, 128), (300, 257, 768, 512),
                                     (58816, 58758, 16128, 5376)])
def test_linear_fp8(h3lib, S, L, N, K):
    g = torch.Generator(device=dev)
    g.manual_seed(N)
    x = torch.randn(S, K, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    qx, sx = quantize(h3lib, x)
    qw, sw = quantize(h3lib, w)
    y = torch.full((S, N), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear_fp8(qx, sx, qw, sw, y, L)
    h3lib.check_device_error()
    rows = np.arange(L) if L < 1000 else sample_rows(L, 128, 5)
    tr = torch.from_numpy(rows).to(dev)
    ref = O.linear_fp8(codes_to_values(qx[tr]), np64(sx[tr]), codes_to_values(qw), np64(sw))
    assert_close_bf16(np64(y[tr]), ref, "linear_fp8")
    assert bool((y[L:] == SENT).all())


def test_linear_swiglu_fp8_matches_unfused(h3lib):
    S, L, F, K = 256, 250, 1536, 512
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    x = torch.randn(S, K, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(2 * F, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    qx, sx = quantize(h3lib, x)
    qw, sw = quantize(h3lib, w)
    gu = torch.empty(S, 2 * F, dtype=torch.bfloat16, device=dev)
    u1 = torch.full((S, F), SENT, dtype=torch.bfloat16, device=dev)
    u2 = torch.full((S, F), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear_fp8(qx, sx, qw, sw, gu, L)
    h3lib.swiglu(gu, u1, L)
    h3lib.linear_swiglu_fp8(qx, sx, qw, sw, u2, L)
    h3lib.check_device_error()
    assert torch.equal(u1, u2)


def run_fp8_block(h3lib, shape, inp):
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)
    w8 = h3lib.quantize_block_weights_fp8(inp)
    ws = torch.empty(h3lib.block_workspace_bytes_fp8(cfg), dtype=torch.uint8, device=dev)
    out = inp["resid"].clone()
    h3lib.block_forward_fp8(cfg, w8, out, inp["mod"], inp["pos"], ws)
    h3lib.check_device_error()
    return out


def check_fp8_block(out_rows, shape, inp, rows, elementwise=True):
    """elementwise=False: the whole-block comparison at full size is held to
    relative L2 only. Upstream bf16 hand-offs may legitimately differ in their
    last bit between two correct evaluations; across an FP8 quantisation that
    can move a row's absmax scale or an E4M3 code by a whole step (2^-3
    relative), which no bf16-level elementwise bound covers. The strict FP8
    parity is the stage tests above: bit-exact codes and scales, and the FP8
    GEMM given identical codes."""
    n = {k: np64(v) if v.is_floating_point() else v.cpu().numpy() for k, v in inp.items()}
    ref, mids = O.block_forward(n["resid"], n["mod"], n["w_qkv"], n["w_o"], n["w_gu"],
                                n["w_down"], n["q_gain"], n["k_gain"], n["pos"], L=shape.L,
                                heads=shape.H, head_dim=shape.Dh, axis_dims=shape.axis_dims,
                                theta=shape.theta, rows=rows, return_intermediates=True, fp8=True)
    if elementwise:
        assert_close_block(np64(out_rows), ref, mids["f"], mids["o"], n["mod"][2], n["mod"][5],
                           n["resid"][rows], "fp8 block")
        return
    x = np64(out_rows)
    r_in = n["resid"][rows]
    assert rel_l2(x, ref) <= 1e-2, rel_l2(x, ref)
    # the increment gate1 * o + gate2 * f comes straight out of FP8 projections:
    # an upstream relative difference d between two correct evaluations flips
    # an E4M3 code with probability about d / 2^-4, each flip moving one
    # operand by up to 2^-3, so a projection output moves by about
    # 2^-3 * sqrt(d / 2^-4); d <= 1e-2 (the attention-output tolerance) gives
    # 5e-2
    assert rel_l2(x - r_in, ref - r_in) <= 5e-2, rel_l2(x - r_in, ref - r_in)


def test_fp8_block_tiny(h3lib):
    shape = I.TINY
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=0).items()}
    out = run_fp8_block(h3lib, shape, inp)
    check_fp8_block(out[:shape.L], shape, inp, np.arange(shape.L))
    assert torch.equal(out[shape.L:], inp["resid"][shape.L:])


@pytest.mark.slow
def test_fp8_block_full_size_sampled(h3lib):
    shape = I.FULL
    inp = I.block_inputs(shape, seed=3, device=dev)
    out = run_fp8_block(h3lib, shape, inp)
    rows = sample_rows(shape.L, 256, 9)
    check_fp8_block(out[torch.from_numpy(rows).to(dev)], shape, inp, rows, elementwise=False)


def run_fp8_block_attn(h3lib, shape, inp):
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)
    w8 = h3lib.quantize_block_weights_fp8(inp)
    ws = torch.empty(h3lib.block_workspace_bytes_fp8(cfg), dtype=torch.uint8, device=dev)
    out = inp["resid"].clone()
    h3lib.block_forward_fp8(cfg, w8, out, inp["mod"], inp["pos"], ws, fp8_attention=True)
    h3lib.check_device_error()
    return out


@pytest.mark.parametrize("full", [False, pytest.param(True, marks=pytest.mark.slow)])
def test_fp8_block_with_fp8_attention(h3lib, full):
    """FP8 projections and FP8 (SAGE) attention together, against the oracle's
    block with the same options; relative L2 on the output and the increment
    (the same tolerances and reasons as the FP8 full-size block)."""
    shape = I.FULL if full else I.TINY
    inp = (I.block_inputs(shape, seed=3, device=dev) if full else
           {k: v.to(dev) for k, v in I.block_inputs(shape, seed=0).items()})
    out = run_fp8_block_attn(h3lib, shape, inp)
    rows = sample_rows(shape.L, 128, 13) if full else np.arange(shape.L)
    n = {k: np64(v) if v.is_floating_point() else v.cpu().numpy() for k, v in inp.items()}
    ref = O.block_forward(n["resid"], n["mod"], n["w_qkv"], n["w_o"], n["w_gu"], n["w_down"],
                          n["q_gain"], n["k_gain"], n["pos"], L=shape.L, heads=shape.H,
                          head_dim=shape.Dh, axis_dims=shape.axis_dims, theta=shape.theta,
                          rows=rows, fp8=True, fp8_attention=True)
    x = np64(out[torch.from_numpy(rows).to(dev)])
    r_in = n["resid"][rows]
    assert rel_l2(x, ref) <= 1e-2, rel_l2(x, ref)
    assert rel_l2(x - r_in, ref - r_in) <= 5e-2, rel_l2(x - r_in, ref - r_in)
