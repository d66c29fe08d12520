"""GPU parity of the whole block (h3_block_forward through the C-ABI)
against the oracle: every row of the tiny block, a seeded 512-row sample of
the full packed-sequence block, determinism and pad invariance."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_block, np64, sample_rows

pytestmark = pytest.mark.gpu
dev = "cuda"


def gpu_block(h3lib, shape, inp):
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)
    ws = torch.empty(h3lib.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    resid = inp["resid"].clone()
    h3lib.block_forward(cfg, inp, resid, inp["mod"], inp["pos"], ws)
    h3lib.check_device_error()
    return resid


def check_block(out_rows, shape, inp, rows=None, what="block"):
    """Compares GPU output rows with the oracle's, with the block tolerance."""
    n = {k: np64(v) if v.is_floating_point() else v.cpu().numpy() for k, v in inp.items()}
    ref, mids = O.block_forward(n["resid"], n["mod"], n["w_qkv"], n["w_o"], n["w_gu"],
                                n["w_down"], n["q_gain"], n["k_gain"], n["pos"], L=shape.L,
                                heads=shape.H, head_dim=shape.Dh, axis_dims=shape.axis_dims,
                                theta=shape.theta, eps_ln=shape.eps_ln, eps_qk=shape.eps_qk,
                                rows=rows, return_intermediates=True)
    r_in = n["resid"][:shape.L] if rows is None else n["resid"][rows]
    assert_close_block(np64(out_rows), ref, mids["f"], mids["o"], n["mod"][2], n["mod"][5], r_in,
                       what)


SMALL = [I.TINY,
         I.BlockShape(S=384, L=321, D=768, H=6, Dh=128, F=2048, axis_dims=(32, 48, 48),
                      pos_kind="3d", grid=(2, 10, 16), n_tail=22),
         I.BlockShape(S=64, L=1, D=256, H=2, Dh=128, F=256)]


@pytest.mark.parametrize("shape", SMALL, ids=["tiny", "ragged3d", "one_row"])
def test_block_small(h3lib, shape):
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=0).items()}
    out = gpu_block(h3lib, shape, inp)
    check_block(out[:shape.L], shape, inp)
    assert torch.equal(out[shape.L:], inp["resid"][shape.L:]), "pad rows written"


def test_block_deterministic_and_pad_invariant(h3lib):
    shape = I.TINY
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=1).items()}
    a = gpu_block(h3lib, shape, inp)
    b = gpu_block(h3lib, shape, inp)
    assert torch.equal(a, b)
    inp2 = dict(inp)
    r2 = inp["resid"].clone()
    r2[shape.L:] = 1e4
    p2 = inp["pos"].clone()
    p2[shape.L:] = 999
    inp2["resid"], inp2["pos"] = r2, p2
    c = gpu_block(h3lib, shape, inp2)
    assert torch.equal(a[:shape.L], c[:shape.L])


@pytest.mark.slow
def test_block_full_size_sampled(h3lib):
    shape = I.FULL
    inp = I.block_inputs(shape, seed=3, device=dev)
    out = gpu_block(h3lib, shape, inp)
    rows = sample_rows(shape.L, 512, 3)
    check_block(out[torch.from_numpy(rows).to(dev)], shape, inp, rows, "block full")
    assert torch.equal(out[shape.L:], inp["resid"][shape.L:])


@pytest.mark.slow
@pytest.mark.parametrize("L", [29034, 87846])
def test_block_stack_length_sweep(h3lib, L):
    """A stack of blocks with independent seeded weights at the short and long
    packed lengths (buffers padded to a multiple of 64): each block is checked
    on sampled rows against the oracle given the GPU's own input to that
    block; the 29,034-row case runs four blocks, the 87,846-row case one."""
    S = (L + 63) // 64 * 64
    shape = I.BlockShape(S=S, L=L, D=5376, H=42, Dh=128, F=14336, axis_dims=(32, 48, 48),
                         pos_kind="3d", grid=(47, 24, 79) if L > 60000 else (16, 24, 79))
    blocks = 4 if L < 60000 else 1
    x = None
    for b in range(blocks):
        inp = I.block_inputs(shape, seed=4 + b + (0 if L < 60000 else 10), device=dev)
        if x is not None:
            inp["resid"] = x
        out = gpu_block(h3lib, shape, inp)
        rows = sample_rows(L, 128, 40 + b)
        check_block(out[torch.from_numpy(rows).to(dev)], shape, inp, rows, f"block {b} L={L}")
        assert torch.equal(out[L:], inp["resid"][L:])
        x = out
