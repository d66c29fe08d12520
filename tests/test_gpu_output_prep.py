"""GPU output preparation (FP32 BCTHW frames -> uint8 BTHWC) against the
oracle, bit for bit: the uint8 code is an integer decision both sides take
in float32 with the same rounding steps."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O

pytestmark = pytest.mark.gpu
dev = "cuda"


def run(h3lib, f):
    B, C, T, H, W = f.shape
    out = torch.full((B, T, H, W, C), 77, dtype=torch.uint8, device=dev)
    h3lib.frames_to_u8(f, out)
    h3lib.check_device_error()
    return out


@pytest.mark.parametrize("shape", [(1, 3, 2, 3, 8), (2, 3, 5, 7, 4), (1, 1, 1, 4, 4),
                                   (3, 5, 2, 2, 6), (1, 16, 1, 1, 4)])
def test_frames_to_u8_small(h3lib, shape):
    g = torch.Generator(device="cpu")
    g.manual_seed(sum(shape))
    f = (torch.rand(*shape, generator=g) * 2.6 - 1.3).to(dev)  # includes clamped values
    assert np.array_equal(run(h3lib, f).cpu().numpy(), O.frames_to_u8(f.cpu().numpy()))


def test_frames_to_u8_special_values(h3lib):
    vals = torch.tensor([-1.0, 1.0, 0.0, -3.0, 2.5, 0.5, -0.5, 1e-8, -1e-8, 0.99607843],
                        dtype=torch.float32)
    # every float32 whose code sits on a rounding boundary of the map
    k = torch.arange(256, dtype=torch.float32)
    ties = ((k + 0.5) / 255.0) * 2.0 - 1.0
    f = torch.cat([vals, ties, torch.zeros(2)]).reshape(1, 1, 1, 1, -1).to(dev)
    assert f.shape[-1] % 4 == 0
    assert np.array_equal(run(h3lib, f).cpu().numpy(), O.frames_to_u8(f.cpu().numpy()))


def test_frames_to_u8_ten_second_clip(h3lib):
    # the 10 s, 1344 x 768, 24 fps clip of the workload: 243 frames
    B, C, T, H, W = 1, 3, 243, 768, 1344
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    f = torch.randn(B, C, T, H, W, generator=g, device=dev).mul_(0.6).clamp_(-1.2, 1.2)
    out = run(h3lib, f)
    for t0 in (0, 121, 241):
        ref = O.frames_to_u8(f[:, :, t0:t0 + 2].cpu().numpy())
        assert np.array_equal(out[:, t0:t0 + 2].cpu().numpy(), ref)
