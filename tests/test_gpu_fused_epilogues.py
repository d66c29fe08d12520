"""GPU parity of the fused GEMM epilogues, called through the C-ABI:
  * h3_rope_table against the oracle's RoPE angles;
  * h3_linear_qk_norm_rope against h3_linear + h3_qk_norm_rope and against
    the oracle (projection, then per-head RMSNorm + RoPE);
  * h3_linear_residual against h3_linear + the residual step of
    h3_mod_norm_residual (bit for bit) and against the oracle."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, bf16_ulp, np64, sample_rows

pytestmark = pytest.mark.gpu
SENT = -7.25
dev = "cuda"


def make(S, N, K, seed):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn(S, K, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    return x, w, g


@pytest.mark.parametrize("kind", ["1d", "3d"])
def test_rope_table_matches_oracle_angles(h3lib, kind):
    S, L = 58816, 58758
    if kind == "1d":
        pos, axis = I.positions_1d(S, L), (128, 0, 0)
    else:
        pos, axis = I.positions_3d(S, L), (32, 48, 48)
    tab = torch.full((S, 64, 2), SENT, dtype=torch.float32, device=dev)
    h3lib.rope_table(pos.to(dev), axis, tab, L, theta=1e4)
    h3lib.check_device_error()
    rows = sample_rows(L, 1024, 31)
    phi = O.rope_angles(pos.numpy()[rows], axis, 1e4)
    t = tab[torch.from_numpy(rows).to(dev)].double().cpu().numpy()
    # FP32 sin/cos of an argument reduced to [-pi, pi] in FP64: a few FP32 ulps
    assert np.abs(t[..., 0] - np.cos(phi)).max() < 1e-6
    assert np.abs(t[..., 1] - np.sin(phi)).max() < 1e-6
    assert bool((tab[L:] == SENT).all()), "pad rows written"


def qkv_case(S, L, H, K, axis, pos, seed):
    D = H * 128
    x, w, g = make(S, 3 * D, K, seed)
    qg = (1.0 + 0.1 * torch.randn(128, generator=g, device=dev)).float()
    kg = (1.0 + 0.1 * torch.randn(128, generator=g, device=dev)).float()
    return x, w, qg, kg


@pytest.mark.parametrize("S,L,H,K,kind,pairing", [
    (256, 250, 4, 512, "3d", 0), (130, 129, 2, 64, "1d", 0), (1000, 999, 6, 320, "3d", 0),
    (256, 250, 4, 512, "3d", 1), (130, 129, 2, 64, "1d", 1), (300, 290, 2, 128, "3d16", 1)])
def test_linear_qk_norm_rope_matches_unfused_and_oracle(h3lib, S, L, H, K, kind, pairing):
    D = H * 128
    if kind == "1d":
        pos, axis = I.positions_1d(S, L), (128, 0, 0)
    else:
        pos = I.positions_3d(S, L, grid=(3, 5, 12), n_tail=max(0, L - 180))
        axis = (32, 48, 48) if kind == "3d" else (16, 64, 48)
    x, w, qg, kg = qkv_case(S, L, H, K, axis, pos, seed=H + K)
    tab = torch.empty(S, 64, 2, dtype=torch.float32, device=dev)
    h3lib.rope_table(pos.to(dev), axis, tab, L)
    un = torch.full((S, 3 * D), SENT, dtype=torch.bfloat16, device=dev)
    fu = torch.full((S, 3 * D), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear(x, w, un, L)
    raw = un.clone()
    q, k = un[:, :D].view(S, H, 128), un[:, D:2 * D].view(S, H, 128)
    # q, k are strided views of the qkv buffer: run the unfused kernel on copies
    qc, kc = q.contiguous(), k.contiguous()
    h3lib.qk_norm_rope(qc, kc, qg, kg, pos.to(dev), axis, L, 1e4, 1e-6, pairing=pairing)
    h3lib.linear_qk_norm_rope(x, w, fu, qg, kg, tab, axis, L, eps=1e-6, pairing=pairing)
    h3lib.check_device_error()
    # v columns: the plain product, bit for bit
    assert torch.equal(fu[:, 2 * D:], raw[:, 2 * D:])
    # q, k: same arithmetic up to the order of the sum of squares and of the
    # FP32 contractions inside the rotation -> at most one bf16 step apart at
    # the scale of the rotated pair (whose norm the rotation keeps; an output
    # near zero from cancellation may differ at that scale), and rarely
    for name, f, u in (("q", fu[:L, :D], qc[:L].view(L, D)), ("k", fu[:L, D:2 * D], kc[:L].view(L, D))):
        d = (f.float() - u.float()).abs().view(L, D // 2, 2)
        norm = u.float().view(L, D // 2, 2).norm(dim=-1, keepdim=True)
        step = (norm * 2.0 ** -7).clamp_min(2.0 ** -133)
        assert bool((d <= step).all()), f"{name}: fused and unfused differ by more than one bf16 step"
        assert float((d > 0).float().mean()) < 1e-3, f"{name}: too many one-step differences"
    # against the oracle: projection rounded to bf16, then RMSNorm + RoPE
    ref_qkv = O.linear(np64(x[:L]), np64(w))
    p = pos.numpy()[:L]
    lay = ("interleaved", "half")[pairing]
    for name, lo, gain in (("q", 0, qg), ("k", D, kg)):
        ref = O.qk_norm_rope(ref_qkv[:, lo:lo + D].reshape(L, H, 128), np64(gain), p, axis, 1e4,
                             1e-6, lay)
        assert_close_bf16(np64(fu[:L, lo:lo + D]).reshape(L, H, 128), ref, f"fused {name}")
    assert_close_bf16(np64(fu[:L, 2 * D:]), ref_qkv[:, 2 * D:], "fused v")
    assert bool((fu[L:] == SENT).all()), "pad rows written"


def test_linear_qk_norm_rope_full_size_sampled(h3lib):
    S, L, H, K = 58816, 58758, 42, 5376
    D = H * 128
    pos, axis = I.positions_3d(S, L), (32, 48, 48)
    x, w, qg, kg = qkv_case(S, L, H, K, axis, pos, seed=17)
    tab = torch.empty(S, 64, 2, dtype=torch.float32, device=dev)
    h3lib.rope_table(pos.to(dev), axis, tab, L)
    fu = torch.full((S, 3 * D), SENT, dtype=torch.bfloat16, device=dev)
    h3lib.linear_qk_norm_rope(x, w, fu, qg, kg, tab, axis, L, eps=1e-6)
    h3lib.check_device_error()
    rows = sample_rows(L, 128, 19)
    tr = torch.from_numpy(rows).to(dev)
    ref_qkv = O.linear(np64(x[tr]), np64(w))
    for name, lo, gain in (("q", 0, qg), ("k", D, kg)):
        ref = O.qk_norm_rope(ref_qkv[:, lo:lo + D].reshape(len(rows), H, 128), np64(gain),
                             pos.numpy()[rows], axis, 1e4, 1e-6)
        assert_close_bf16(np64(fu[tr, lo:lo + D]).reshape(len(rows), H, 128), ref,
                          f"fused {name} full")
    assert_close_bf16(np64(fu[tr, 2 * D:]), ref_qkv[:, 2 * D:], "fused v full")
    assert bool((fu[L:] == SENT).all())


@pytest.mark.parametrize("S,L,N,K", [(256, 250, 512, 1536), (130, 129, 256, 64),
                                     (1000, 999, 768, 320)])
def test_linear_residual_matches_unfused_and_oracle(h3lib, S, L, N, K):
    x, w, g = make(S, N, K, seed=N + 3 * K)
    r0 = torch.randn(S, N, generator=g, device=dev)
    gate = torch.randn(N, generator=g, device=dev)
    y = torch.empty(S, N, dtype=torch.bfloat16, device=dev)
    r_un, r_fu = r0.clone(), r0.clone()
    h3lib.linear(x, w, y, L)
    h3lib.mod_norm_residual(r_un, y, gate, None, None, None, L)
    h3lib.linear_residual(x, w, r_fu, gate, L)
    h3lib.check_device_error()
    assert torch.equal(r_fu, r_un), "fused residual differs from linear + residual step"
    f_ref = O.linear(np64(x[:L]), np64(w))
    r_ref, _ = O.mod_norm_residual(np64(r0[:L]), f_ref, np64(gate), None, None, eps=1e-6)
    # FP32 residual tolerance, plus one bf16 step of f times the gate where the
    # FP32-accumulated product rounds to the other neighbour of the FP64 one
    bound = 1e-5 * np.maximum(1.0, np.abs(r_ref)) + np.abs(np64(gate)) * bf16_ulp(f_ref)
    assert bool((np.abs(np64(r_fu[:L]) - r_ref) <= bound).all()), "linear_residual vs oracle"
    assert torch.equal(r_fu[L:], r0[L:]), "pad rows of resid written"


def test_linear_residual_zero_gate_is_bitwise_identity(h3lib):
    S, L, N, K = 512, 500, 512, 256
    x, w, g = make(S, N, K, seed=77)
    r0 = torch.randn(S, N, generator=g, device=dev)
    r = r0.clone()
    h3lib.linear_residual(x, w, r, torch.zeros(N, device=dev), L)
    h3lib.check_device_error()
    assert torch.equal(r, r0)
