"""The allocation-free block entry point, checked against the workspace one.

h3_block_forward_noalloc is for callers that cannot allocate device memory,
for example a host program whose device memory all belongs to a framework's
pool and which may not call cudaMalloc itself. Instead of a caller workspace
it uses a fixed 32 MiB array inside the library. These tests call it through
the C ABI twice in a row and require each result to equal h3_block_forward's
bit for bit (the same kernels run on the same inputs), with a block of another
shape run through the same array in between so that stale scratch contents
would show, check that the calls leave the device's free memory unchanged,
and check that a block too large for the array is refused on the host.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from dit_transformer_block_gb300 import inputs as I

pytestmark = pytest.mark.gpu
dev = "cuda"


def _block(h3lib, shape, seed):
    inp = {k: v.to(dev) for k, v in I.block_inputs(shape, seed=seed).items()}
    cfg = h3lib.block_config(shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F,
                             shape.axis_dims, shape.theta, shape.eps_ln, shape.eps_qk)
    assert h3lib.block_workspace_bytes(cfg) <= h3lib.NOALLOC_SCRATCH_BYTES
    return inp, cfg


def test_noalloc_matches_workspace_entry_point_twice(h3lib):
    shape = I.TINY
    inp, cfg = _block(h3lib, shape, seed=5)
    # a second shape (more rows, another FFN width) that fills more of the
    # array, run through it between the two calls under test
    other = I.BlockShape(S=640, L=600, D=512, H=4, Dh=128, F=2048)
    inp2, cfg2 = _block(h3lib, other, seed=6)
    assert h3lib.block_workspace_bytes(cfg2) > h3lib.block_workspace_bytes(cfg)
    ws = torch.empty(h3lib.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    ref = inp["resid"].clone()
    h3lib.block_forward(cfg, inp, ref, inp["mod"], inp["pos"], ws)
    h3lib.check_device_error()
    # the other shape's own workspace run (every kernel is loaded before the
    # free memory is read)
    ws2 = torch.empty(h3lib.block_workspace_bytes(cfg2), dtype=torch.uint8, device=dev)
    ref2 = inp2["resid"].clone()
    h3lib.block_forward(cfg2, inp2, ref2, inp2["mod"], inp2["pos"], ws2)
    h3lib.check_device_error()
    outs = [inp["resid"].clone() for _ in range(2)]
    out2 = inp2["resid"].clone()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for i, out in enumerate(outs):
        h3lib.block_forward_noalloc(cfg, inp, out, inp["mod"], inp["pos"])
        h3lib.check_device_error()
        if i == 0:
            h3lib.block_forward_noalloc(cfg2, inp2, out2, inp2["mod"], inp2["pos"])
            h3lib.check_device_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    for out in outs:
        assert torch.equal(out, ref), "no-alloc block differs from the workspace block"
    assert torch.equal(out2, ref2), "no-alloc block of the second shape differs"


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
