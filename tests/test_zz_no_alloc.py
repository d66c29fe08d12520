"""The allocation-free block entry point, checked against the workspace one.

h3_block_forward_noalloc is for callers that cannot allocate device memory,
for example a host program whose device memory all belongs to a framework's
pool and which may not call cudaMalloc itself. Instead of a caller workspace
it uses a fixed 32 MiB array inside the library. These tests call it through
the C ABI twice in a row and compare each result with h3_block_forward's
(same bf16 tolerances as the other block tests), and check that a block too
large for the array is refused on the host.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, np64

pytestmark = pytest.mark.gpu
dev = "cuda"


def test_noalloc_matches_workspace_entry_point_twice(h3lib):
    shape = I.TINY
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=5).items()}
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)
    assert h3lib.block_workspace_bytes(cfg) <= h3lib.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(h3lib.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    ref = inp["resid"].clone()
    h3lib.block_forward(cfg, inp, ref, inp["mod"], inp["pos"], ws)
    h3lib.check_device_error()
    for _ in range(2):
        out = inp["resid"].clone()
        h3lib.block_forward_noalloc(cfg, inp, out, inp["mod"], inp["pos"])
        h3lib.check_device_error()
        assert_close_bf16(np64(out[:shape.L]), np64(ref[:shape.L]), "no-alloc block")
        assert torch.equal(out[shape.L:], inp["resid"][shape.L:]), "pad rows written"


def test_noalloc_refuses_block_larger_than_its_array(h3lib):
    shape = I.FULL
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims)
    fake = 4096  # never dereferenced: the size check comes first
    w = h3lib.BlockWeights(fake, fake, fake, fake, fake, fake)
    st = h3lib.lib().h3_block_forward_noalloc(ctypes.byref(cfg), ctypes.byref(w),
                                              ctypes.c_void_p(fake), ctypes.c_void_p(fake),
                                              ctypes.c_void_p(fake), None)
    assert st == 4 and "scratch" in h3lib.last_error()
