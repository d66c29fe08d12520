"""GPU parity of the HBM-bound kernels (SwiGLU, Q/K RMSNorm+RoPE,
modulation/LayerNorm/residual) against the CPU oracle, called through the
C-ABI. Small cases compare every element; the full packed-sequence sizes
compare seeded row samples."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, assert_close_f32, np64, sample_rows

pytestmark = pytest.mark.gpu
SENT = -7.25  # bf16-exact sentinel for pad rows of outputs
dev = "cuda"


@pytest.mark.parametrize("S,L,F", [(256, 250, 1536), (64, 1, 8), (130, 129, 24), (40, 33, 14336)])
def test_swiglu_small(h3lib, S, L, F):
    gu = I.swiglu_inputs(S, F, seed=11)["gate_up"].to(dev)
    out = torch.full((S, F), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.swiglu(gu, out, L)
    h3lib.check_device_error()
    assert_close_bf16(np64(out[:L]), O.swiglu(np64(gu[:L])), "swiglu")
    assert bool((out[L:] == SENT).all()), "pad rows written"


def test_swiglu_full_size(h3lib):
    S, L, F = 58816, 58758, 14336
    gu = I.swiglu_inputs(S, F, seed=12, device=dev)["gate_up"]
    out = torch.full((S, F), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.swiglu(gu, out, L)
    h3lib.check_device_error()
    rows = torch.from_numpy(sample_rows(L, 512, 13)).to(dev)
    assert_close_bf16(np64(out[rows]), O.swiglu(np64(gu[rows])), "swiglu full")
    assert bool((out[L:] == SENT).all())


def run_qk(h3lib, S, L, H, axis_dims, pos, seed, rows=None, pairing=0):
    inp = I.qk_inputs(S, L, H, 128, seed, device=dev)
    q0, k0 = inp["q"].clone(), inp["k"].clone()
    q, k = inp["q"], inp["k"]
    h3lib.qk_norm_rope(q, k, inp["q_gain"], inp["k_gain"], pos.to(dev), axis_dims, L, 1e4, 1e-6,
                       pairing=pairing)
    h3lib.check_device_error()
    rows = np.arange(L) if rows is None else rows
    tr = torch.from_numpy(rows).to(dev)
    p = pos.numpy()[rows]
    for name, x0, x, g in (("q", q0, q, inp["q_gain"]), ("k", k0, k, inp["k_gain"])):
        ref = O.qk_norm_rope(np64(x0[tr]), np64(g), p, axis_dims, 1e4, 1e-6,
                             ("interleaved", "half")[pairing])
        assert_close_bf16(np64(x[tr]), ref, f"qk_norm_rope {name}")
        assert torch.equal(x[L:], x0[L:]), "pad rows written"


@pytest.mark.parametrize("S,L,H", [(256, 250, 4), (8, 1, 2), (70, 65, 3)])
def test_qk_norm_rope_1d(h3lib, S, L, H):
    run_qk(h3lib, S, L, H, (128, 0, 0), I.positions_1d(S, L), seed=21)


def test_qk_norm_rope_3d_small(h3lib):
    S, L = 200, 190
    pos = I.positions_3d(S, L, grid=(3, 5, 12), n_tail=22)
    run_qk(h3lib, S, L, 5, (32, 48, 48), pos, seed=22)


@pytest.mark.parametrize("S,L,H,axis", [(256, 250, 4, (32, 48, 48)), (70, 65, 3, (128, 0, 0)),
                                         (200, 190, 5, (16, 64, 48)), (8, 1, 2, (0, 96, 32))])
def test_qk_norm_rope_split_half(h3lib, S, L, H, axis):
    pos = I.positions_3d(S, L, grid=(3, 5, 12), n_tail=max(0, L - 180))
    run_qk(h3lib, S, L, H, axis, pos, seed=24, pairing=1)


def test_qk_norm_rope_split_half_full_size(h3lib):
    S, L, H = 58816, 58758, 42
    run_qk(h3lib, S, L, H, (32, 48, 48), I.positions_3d(S, L), seed=25,
           rows=sample_rows(L, 512, 25), pairing=1)


def test_qk_norm_rope_full_size(h3lib):
    S, L, H = 58816, 58758, 42
    pos = I.positions_3d(S, L)
    run_qk(h3lib, S, L, H, (32, 48, 48), pos, seed=1, rows=sample_rows(L, 512, 1))


def test_qk_norm_rope_long_1d_positions(h3lib):
    # 1D positions up to ~58k: the angle is reduced in FP64 on the device
    S, L, H = 58816, 58758, 2
    run_qk(h3lib, S, L, H, (128, 0, 0), I.positions_1d(S, L), seed=23,
           rows=sample_rows(L, 256, 23))


def run_mnr(h3lib, S, L, D, mode, seed, rows=None):
    inp = I.mod_inputs(S, D, seed, device=dev)
    resid, delta, mod = inp["resid"], inp["delta"], inp["mod"]
    r0 = resid.clone()
    normed = torch.full((S, D), SENT, dtype=torch.bfloat16, device=dev)
    use_delta = mode in ("both", "residual")
    use_norm = mode in ("both", "norm")
    h3lib.mod_norm_residual(resid, delta if use_delta else None, mod[2] if use_delta else None,
                            mod[0] if use_norm else None, mod[1] if use_norm else None,
                            normed if use_norm else None, L, eps=1e-6)
    h3lib.check_device_error()
    rows = np.arange(L) if rows is None else rows
    tr = torch.from_numpy(rows).to(dev)
    m = np64(mod)
    r_ref, h_ref = O.mod_norm_residual(
        np64(r0[tr]), np64(delta[tr]) if use_delta else None, m[2] if use_delta else None,
        m[0] if use_norm else None, m[1] if use_norm else None, eps=1e-6)
    assert_close_f32(np64(resid[tr]), r_ref, "resid")
    if use_norm:
        assert_close_bf16(np64(normed[tr]), h_ref, "normed")
        assert bool((normed[L:] == SENT).all())
    assert torch.equal(resid[L:], r0[L:]), "pad rows of resid written"


@pytest.mark.parametrize("mode", ["norm", "both", "residual"])
@pytest.mark.parametrize("S,L,D", [(256, 250, 512), (7, 5, 5376), (3, 3, 8), (9, 9, 8192)])
def test_mod_norm_residual_small(h3lib, S, L, D, mode):
    run_mnr(h3lib, S, L, D, mode, seed=31)


@pytest.mark.parametrize("mode", ["norm", "both", "residual"])
def test_mod_norm_residual_full_size(h3lib, mode):
    S, L, D = 58816, 58758, 5376
    run_mnr(h3lib, S, L, D, mode, seed=32, rows=sample_rows(L, 512, 32))


def test_gate_zero_leaves_residual_bitwise(h3lib):
    S, L, D = 64, 60, 512
    inp = I.mod_inputs(S, D, 33, device=dev)
    r0 = inp["resid"].clone()
    h3lib.mod_norm_residual(inp["resid"], inp["delta"], torch.zeros(D, device=dev), L=L)
    h3lib.check_device_error()
    assert torch.equal(inp["resid"], r0)


@pytest.mark.parametrize("S,L,D,G", [(256, 250, 512, 3), (64, 61, 5376, 2),
                                     (58816, 58758, 5376, 2)])
def test_mod_norm_residual_segmented(h3lib, S, L, D, G):
    inp = I.mod_inputs(S, D, seed=34, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(35)
    table = (torch.randn(G, 6, D, generator=g, device=dev) * 0.1).contiguous()
    seg = torch.randint(0, G, (S,), generator=g, device=dev, dtype=torch.int32)
    resid, delta = inp["resid"], inp["delta"]
    r0 = resid.clone()
    normed = torch.full((S, D), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.mod_norm_residual_seg(resid, table, seg, delta=delta, gate_idx=2, shift_idx=3,
                                scale_idx=4, normed=normed, L=L)
    h3lib.check_device_error()
    rows = np.arange(L) if L < 1000 else sample_rows(L, 512, 36)
    tr = torch.from_numpy(rows).to(dev)
    m = O.modulation_rows(np64(table), seg.cpu().numpy(), rows)
    r_ref, h_ref = O.mod_norm_residual(np64(r0[tr]), np64(delta[tr]), m[:, 2], m[:, 3], m[:, 4])
    assert_close_f32(np64(resid[tr]), r_ref, "resid (segmented)")
    assert_close_bf16(np64(normed[tr]), h_ref, "normed (segmented)")
    assert torch.equal(resid[L:], r0[L:]) and bool((normed[L:] == SENT).all())
