"""GPU parity of the tcgen05 valid-length attention against the oracle,
called through the C-ABI, plus closed-form cases and pad invariance."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, np64, sample_rows

pytestmark = pytest.mark.gpu
SENT = -7.25
dev = "cuda"


def run(h3lib, q, k, v, L):
    S = q.shape[0]
    o = torch.full_like(q, SENT)
    h3lib.attention_varlen(q, k, v, o, L)
    h3lib.check_device_error()
    assert bool((o[L:] == SENT).all()), "pad rows written"
    return o


@pytest.mark.parametrize("S,L,H", [(256, 250, 4), (128, 1, 2), (128, 127, 2), (128, 128, 2),
                                   (256, 129, 2), (640, 600, 3)])
def test_attention_small(h3lib, S, L, H):
    inp = I.attention_inputs(S, L, H, 128, seed=S + L, device=dev)
    o = run(h3lib, inp["q"], inp["k"], inp["v"], L)
    ref = O.attention(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), L, 128 ** -0.5)
    assert_close_bf16(np64(o[:L]), ref, "attention")


def test_attention_large_logits(h3lib):
    # un-normalised q, k (logit spread ~ 10): exercises the running-max rescale
    S, L, H = 512, 500, 2
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    q = (torch.randn(S, H, 128, generator=g, device=dev) * 3).to(torch.bfloat16)
    k = (torch.randn(S, H, 128, generator=g, device=dev) * 3).to(torch.bfloat16)
    v = torch.randn(S, H, 128, generator=g, device=dev).to(torch.bfloat16)
    o = run(h3lib, q, k, v, L)
    ref = O.attention(np64(q), np64(k), np64(v), L, 128 ** -0.5)
    assert_close_bf16(np64(o[:L]), ref, "attention large logits")


def test_attention_identical_keys_give_mean_of_v(h3lib):
    S, L, H = 384, 300, 2
    inp = I.attention_inputs(S, L, H, 128, seed=5, device=dev)
    k = inp["k"][:1].expand(S, H, 128).contiguous()
    o = run(h3lib, inp["q"], k, inp["v"], L)
    mean = np64(inp["v"][:L]).mean(0)
    assert_close_bf16(np64(o[:L]), np.broadcast_to(mean, (L, H, 128)), "mean of V")


def test_attention_pad_rows_do_not_matter(h3lib):
    S, L, H = 384, 333, 2
    inp = I.attention_inputs(S, L, H, 128, seed=6, device=dev)
    o1 = run(h3lib, inp["q"], inp["k"], inp["v"], L)
    k2, v2, q2 = inp["k"].clone(), inp["v"].clone(), inp["q"].clone()
    k2[L:] = 30.0
    v2[L:] = -1000.0
    q2[L:] = float("nan")
    o2 = run(h3lib, q2, k2, v2, L)
    assert torch.equal(o1[:L], o2[:L])
    # growing the buffer leaves the valid rows unchanged too
    S3 = S + 128
    pad = lambda t: torch.cat([t, torch.randn(128, H, 128, device=dev).to(t.dtype)])
    o3 = run(h3lib, pad(inp["q"]), pad(inp["k"]), pad(inp["v"]), L)
    assert torch.equal(o1[:L], o3[:L])


def test_attention_deterministic(h3lib):
    inp = I.attention_inputs(1024, 1000, 2, 128, seed=7, device=dev)
    o1 = run(h3lib, inp["q"], inp["k"], inp["v"], 1000)
    o2 = run(h3lib, inp["q"], inp["k"], inp["v"], 1000)
    assert torch.equal(o1, o2)


@pytest.mark.slow
def test_attention_full_size_sampled(h3lib):
    S, L, H = 58816, 58758, 42
    inp = I.attention_inputs(S, L, H, 128, seed=2, device=dev)
    o = run(h3lib, inp["q"], inp["k"], inp["v"], L)
    rows = sample_rows(L, 512, 2)
    ref = O.attention(np64(inp["q"][:L]), np64(inp["k"][:L]), np64(inp["v"][:L]), L, 128 ** -0.5,
                      rows=rows)
    assert_close_bf16(np64(o[torch.from_numpy(rows).to(dev)]), ref, "attention full")


def test_skip_softmax_eps_zero_is_dense_bitwise(h3lib):
    S, L, H = 640, 600, 3
    inp = I.attention_inputs(S, L, H, 128, seed=8, device=dev)
    o1 = run(h3lib, inp["q"], inp["k"], inp["v"], L)
    o2 = torch.full_like(o1, SENT)
    kept = torch.full(((L + 127) // 128, H), -1, dtype=torch.int32, device=dev)
    h3lib.attention_varlen_skip(inp["q"], inp["k"], inp["v"], o2, L, skip_eps=0.0, kept=kept)
    h3lib.check_device_error()
    assert torch.equal(o1, o2)
    assert bool((kept == -1).all())  # the counts are written only when eps > 0


def test_skip_softmax_skips_the_tile_the_rule_names(h3lib):
    # scores in base-2 units (softmax scale ln 2): key tile 0 scores 20, tile 1
    # scores 18.5 (1.5 below the running max: skipped at eps = 1/2), tile 2
    # scores 19.5 (kept); every query row is the same, so the decision is the
    # same for every row and tile 1's keys would carry real weight if kept
    S = L = 384
    H = 1
    q = torch.zeros(S, H, 128)
    q[:, 0, 0] = 1.0
    k = torch.zeros(S, H, 128)
    k[:128, 0, 0] = 20.0
    k[128:256, 0, 0] = 18.5
    k[256:, 0, 0] = 19.5
    g = torch.Generator().manual_seed(9)
    v = torch.randn(S, H, 128, generator=g)
    v[128:256] += 1.0  # makes the skipped tile's weight visible in the output
    q, k, v = (t.to(torch.bfloat16).to(dev) for t in (q, k, v))
    scale = float(np.log(2.0))
    o_skip = torch.full_like(q, SENT)
    h3lib.attention_varlen_skip(q, k, v, o_skip, L, scale=scale, skip_eps=0.5)
    h3lib.check_device_error()
    ref, kept = O.attention_skip(np64(q), np64(k), np64(v), L, scale, 0.5)
    assert kept[:, 0].tolist() == [[True, False, True]] * 3
    assert_close_bf16(np64(o_skip[:L]), ref, "skip-softmax")
    kept_gpu = torch.full((3, H), -1, dtype=torch.int32, device=dev)
    h3lib.attention_varlen_skip(q, k, v, o_skip, L, scale=scale, skip_eps=0.5, kept=kept_gpu)
    h3lib.check_device_error()
    assert kept_gpu.cpu().tolist() == [[2]] * 3
    o_dense = torch.full_like(q, SENT)
    h3lib.attention_varlen(q, k, v, o_dense, L, scale=scale)
    h3lib.check_device_error()
    assert (o_skip.float() - o_dense.float()).abs().max().item() > 0.05


def test_skip_softmax_random_data_matches_dense_within_eps(h3lib):
    S, L, H = 2048, 2000, 2
    inp = I.attention_inputs(S, L, H, 128, seed=10, device=dev)
    o = torch.full_like(inp["q"], SENT)
    h3lib.attention_varlen_skip(inp["q"], inp["k"], inp["v"], o, L, skip_eps=2.0 ** -20)
    h3lib.check_device_error()
    ref = O.attention(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), L, 128 ** -0.5)
    assert_close_bf16(np64(o[:L]), ref, "skip-softmax random")


@pytest.mark.parametrize("S,L,eps_log2", [(2048, 2000, 4), (1024, 1024, 2), (1408, 1300, 6)])
def test_skip_softmax_random_data_matches_oracle_rule(h3lib, S, L, eps_log2):
    """Random keys and queries with a shared direction whose per-key-tile
    weight varies, so that whole tiles fall far below the running maximum and
    many tiles are really skipped: the kept-tile counts equal the oracle's (the
    kernel applies the exact running maximum of the kept tiles, as the oracle
    does), the output matches attention over the kept tiles element by
    element, and it differs from dense attention. The ragged last query tile's
    pad rows take no part in the vote."""
    H = 2
    g = torch.Generator().manual_seed(S + eps_log2)
    q = torch.randn(S, H, 128, generator=g)
    k = torch.randn(S, H, 128, generator=g)
    v = torch.randn(S, H, 128, generator=g)
    q[:, :, 0] += 8.0
    nk = (S + 127) // 128
    b = torch.randn(nk, H, generator=g) * 8.0
    k[:, :, 0] += b.repeat_interleave(128, dim=0)[:S]
    q, k, v = (t.to(torch.bfloat16).to(dev) for t in (q, k, v))
    eps = 2.0 ** -eps_log2
    nq = (L + 127) // 128
    kept_gpu = torch.full((nq, H), -1, dtype=torch.int32, device=dev)
    o = torch.full_like(q, SENT)
    h3lib.attention_varlen_skip(q, k, v, o, L, skip_eps=eps, kept=kept_gpu)
    h3lib.check_device_error()
    assert bool((o[L:] == SENT).all())
    ref, kept = O.attention_skip(np64(q), np64(k), np64(v), L, 128 ** -0.5, eps)
    want = kept.sum(axis=2)
    assert want.sum() < nq * H * ((L + 127) // 128)  # tiles really are skipped
    assert np.array_equal(kept_gpu.cpu().numpy(), want)
    assert_close_bf16(np64(o[:L]), ref, "skip-softmax, oracle rule")
    dense = O.attention(np64(q), np64(k), np64(v), L, 128 ** -0.5)
    assert np.max(np.abs(ref - dense)) > 0


def test_skip_softmax_frame_local_inputs(h3lib):
    """The frame-local inputs of the Skip-Softmax measurement (frames of
    1,024 rows) at 4,096 rows: about half of the key tiles are left out, the
    kept counts equal the oracle's and the output is within bf16 tolerance of
    the oracle's attention over the kept tiles."""
    S = L = 4096
    H = 2
    loc = I.frame_local_attention_inputs(S, L, H, 128, frame=1024, seed=5, device=dev)
    eps = 1e-3
    nq = L // 128
    kept_gpu = torch.full((nq, H), -1, dtype=torch.int32, device=dev)
    o = torch.full_like(loc["q"], SENT)
    h3lib.attention_varlen_skip(loc["q"], loc["k"], loc["v"], o, L, skip_eps=eps, kept=kept_gpu)
    h3lib.check_device_error()
    ref, kept = O.attention_skip(np64(loc["q"]), np64(loc["k"]), np64(loc["v"]), L,
                                 128 ** -0.5, eps)
    want = kept.sum(axis=2)
    assert 0.3 < want.sum() / (nq * H * nq) < 0.8
    assert np.array_equal(kept_gpu.cpu().numpy(), want)
    assert_close_bf16(np64(o[:L]), ref, "skip-softmax, frame-local")
