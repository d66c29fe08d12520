"""GPU parity of the tcgen05 projection GEMMs (and the fused SwiGLU
epilogue) against the oracle, called through the C-ABI."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from helpers import assert_close_bf16, np64, sample_rows

pytestmark = pytest.mark.gpu
SENT = -7.25
dev = "cuda"


def make(S, N, K, seed, device=dev):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(S, K, generator=g, device=device).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return x, w


def test_linear_exact_small_integers(h3lib):
    # integer operands with |sum| < 256: every product and sum is exact in FP32
    # and the result is exactly representable in bf16, so the GEMM must be exact
    S, L, N, K = 256, 256, 256, 128
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    x = torch.randint(-1, 2, (S, K), generator=g).to(torch.bfloat16).to(dev)
    w = torch.randint(-1, 2, (N, K), generator=g).to(torch.bfloat16).to(dev)
    y = torch.full((S, N), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear(x, w, y, L)
    h3lib.check_device_error()
    ref = x.double().cpu() @ w.double().cpu().T
    assert torch.equal(y.double().cpu(), ref)


@pytest.mark.parametrize("S,L,N,K", [(256, 250, 256, 64), (256, 250, 1536, 512),
                                     (300, 257, 512, 1536), (128, 1, 256, 64),
                                     (1000, 999, 768, 320)])
def test_linear_small(h3lib, S, L, N, K):
    x, w = make(S, N, K, seed=N + K)
    y = torch.full((S, N), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear(x, w, y, L)
    h3lib.check_device_error()
    assert_close_bf16(np64(y[:L]), O.linear(np64(x[:L]), np64(w)), "linear")
    assert bool((y[L:] == SENT).all()), "pad rows written"


@pytest.mark.parametrize("N,K", [(16128, 5376), (5376, 5376), (5376, 14336)])
def test_linear_full_size_sampled(h3lib, N, K):
    S, L = 58816, 58758
    x, w = make(S, N, K, seed=7)
    y = torch.full((S, N), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear(x, w, y, L)
    h3lib.check_device_error()
    rows = torch.from_numpy(sample_rows(L, 256, N)).to(dev)
    assert_close_bf16(np64(y[rows]), O.linear(np64(x[rows]), np64(w)), "linear full")
    assert bool((y[L:] == SENT).all())


@pytest.mark.parametrize("S,L,F,K", [(256, 250, 1536, 512), (130, 129, 128, 64)])
def test_linear_swiglu_matches_unfused_and_oracle(h3lib, S, L, F, K):
    x, w = make(S, 2 * F, K, seed=F)
    gu = torch.full((S, 2 * F), SENT, dtype=torch.bfloat16, device=dev)
    u1 = torch.full((S, F), SENT, dtype=torch.bfloat16, device=dev)
    u2 = torch.full((S, F), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear(x, w, gu, L)
    h3lib.swiglu(gu, u1, L)
    h3lib.linear_swiglu(x, w, u2, L)
    h3lib.check_device_error()
    assert torch.equal(u1, u2), "fused epilogue differs from linear + swiglu"
    ref = O.swiglu(O.linear(np64(x[:L]), np64(w)))
    assert_close_bf16(np64(u2[:L]), ref, "linear_swiglu")


def test_linear_swiglu_full_size_sampled(h3lib):
    S, L, F, K = 58816, 58758, 14336, 5376
    x, w = make(S, 2 * F, K, seed=9)
    u = torch.full((S, F), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear_swiglu(x, w, u, L)
    h3lib.check_device_error()
    rows = torch.from_numpy(sample_rows(L, 128, 9)).to(dev)
    ref = O.swiglu(O.linear(np64(x[rows]), np64(w)))
    assert_close_bf16(np64(u[rows]), ref, "linear_swiglu full")
    assert bool((u[L:] == SENT).all())


def test_linear_deterministic(h3lib):
    x, w = make(512, 1024, 512, seed=3)
    y1 = torch.empty(512, 1024, dtype=torch.bfloat16, device=dev)
    y2 = torch.empty_like(y1)
    h3lib.linear(x, w, y1)
    h3lib.linear(x, w, y2)
    h3lib.check_device_error()
    assert torch.equal(y1, y2)
