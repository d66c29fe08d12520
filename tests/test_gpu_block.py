"""GPU parity of the whole block (h3_block_forward through the C-ABI)
against the oracle: every row of the tiny block, a seeded 512-row sample of
the full packed-sequence block, determinism and pad invariance."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, np64, sample_rows

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


def oracle_block(shape, inp, rows=None):
    n = {k: np64(v) if v.is_floating_point() else v.cpu().numpy() for k, v in inp.items()}
    return O.block_forward(n["resid"], n["mod"], n["w_qkv"], n["w_o"], n["w_gu"], n["w_down"],
                           n["q_gain"], n["k_gain"], n["pos"], L=shape.L, heads=shape.H,
                           head_dim=shape.Dh, axis_dims=shape.axis_dims, theta=shape.theta,
                           eps_ln=shape.eps_ln, eps_qk=shape.eps_qk, rows=rows)


SMALL = [I.TINY,
         I.BlockShape(S=384, L=321, D=768, H=6, Dh=128, F=2048, axis_dims=(32, 48, 48),
                      pos_kind="3d", grid=(2, 10, 16), n_tail=22),
         I.BlockShape(S=64, L=1, D=256, H=2, Dh=128, F=256)]


@pytest.mark.parametrize("shape", SMALL, ids=["tiny", "ragged3d", "one_row"])
def test_block_small(h3lib, shape):
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=0).items()}
    out = gpu_block(h3lib, shape, inp)
    ref = oracle_block(shape, inp)
    assert_close_bf16(np64(out[:shape.L]), ref, "block")
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
    ref = oracle_block(shape, inp, rows=rows)
    assert_close_bf16(np64(out[torch.from_numpy(rows).to(dev)]), ref, "block full")
    assert torch.equal(out[shape.L:], inp["resid"][shape.L:])
