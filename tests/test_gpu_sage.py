"""SAGE-style FP8 attention against the oracle.

The oracle quantises the bf16 inputs itself (sage_quantize); every E4M3 code,
every scale and the K mean (FP64 sums on both sides, rounded once to float32)
must match it bit for bit, at small sizes and at the full 58,758-row size.
The FP8 attention output is then compared with the oracle's attention_sage on
the oracle's own operands within the tolerance derived from the E4M3 step of
the softmax weights (helpers.assert_close_sage): the kernel quantises P
against an integer running maximum, the oracle against the exact one.
"""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_sage, np64, rel_l2, sample_rows

pytestmark = pytest.mark.gpu
dev = "cuda"
SENT = -7.25
SCALE = 128 ** -0.5


def decode(q):
    return q.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()


def assert_ops_equal(ops, ref, L):
    """GPU codes and scales against the oracle's, bit for bit."""
    got = dict(qc=decode(ops["qc"][:L]), kc=decode(ops["kc"][:L]), vc=decode(ops["vc"][:L]),
               sq=np64(ops["sq"]), sk=np64(ops["sk"]), sv=np64(ops["sv"]),
               k_mean=np64(ops["k_mean"]))
    for key in ("k_mean", "sq", "sk", "sv", "qc", "kc", "vc"):
        want = np.asarray(ref[key], np.float64).reshape(got[key].shape)
        bad = int(np.sum(got[key] != want))
        assert bad == 0, f"{key}: {bad} of {want.size} values differ"


@pytest.mark.parametrize("S,L,H", [(256, 250, 4), (640, 600, 3), (128, 1, 2), (1152, 1100, 2)])
def test_sage_codes_and_attention(h3lib, S, L, H):
    inp = I.attention_inputs(S, L, H, 128, seed=S + H, device=dev)
    q, k, v = inp["q"], inp["k"], inp["v"]
    k = (k.float() + 0.75).to(torch.bfloat16)  # a common offset the smoothing removes
    ops = h3lib.sage_quantize(q, k, v, L)
    h3lib.check_device_error()
    ref_ops = O.sage_quantize(np64(q), np64(k), np64(v), L)
    assert_ops_equal(ops, ref_ops, L)
    o = torch.full_like(q, SENT)
    h3lib.attention_fp8(ops, o, L)
    h3lib.check_device_error()
    ref = O.attention_sage(ref_ops, L, SCALE)
    terms = O.sage_error_terms(ref_ops, L, SCALE)
    assert_close_sage(np64(o[:L]), ref, terms, L)
    assert bool((o[L:] == SENT).all())
    dense = O.attention(np64(q), np64(k), np64(v), L, SCALE)
    assert rel_l2(np64(o[:L]), dense) < 0.1


def test_sage_all_scores_equal_gives_mean_of_v(h3lib):
    """q = 0: every score is 0, every weight is exactly representable (224 in
    the kernel, 448 in the oracle), so both give the mean of the dequantised V
    rows: equal up to the FP32 accumulation order, within one bf16 step."""
    S, L, H = 384, 300, 2
    inp = I.attention_inputs(S, L, H, 128, seed=9, device=dev)
    q = torch.zeros_like(inp["q"])
    ops = h3lib.sage_quantize(q, inp["k"], inp["v"], L)
    ref_ops = O.sage_quantize(np64(q), np64(inp["k"]), np64(inp["v"]), L)
    assert_ops_equal(ops, ref_ops, L)
    o = torch.full_like(q, SENT)
    h3lib.attention_fp8(ops, o, L)
    h3lib.check_device_error()
    ref = O.attention_sage(ref_ops, L, SCALE)
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    assert np.all(np.abs(np64(o[:L]) - ref) <= step)


@pytest.mark.slow
def test_sage_full_size_sampled(h3lib):
    S, L, H = 58816, 58758, 42
    inp = I.attention_inputs(S, L, H, 128, seed=2, device=dev)
    ops = h3lib.sage_quantize(inp["q"], inp["k"], inp["v"], L)
    o = torch.full_like(inp["q"], SENT)
    h3lib.attention_fp8(ops, o, L)
    h3lib.check_device_error()
    ref_ops = O.sage_quantize(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), L)
    assert_ops_equal(ops, ref_ops, L)
    rows = sample_rows(L, 256, 12)
    ref = O.attention_sage(ref_ops, L, SCALE, rows=rows)
    terms = O.sage_error_terms(ref_ops, L, SCALE, rows=rows)
    assert_close_sage(np64(o[torch.from_numpy(rows).to(dev)]), ref, terms, L, "sage full size")
    assert bool((o[L:] == SENT).all())


def test_sage_skip_eps_zero_is_attention_fp8_bitwise(h3lib):
    S, L, H = 640, 600, 3
    inp = I.attention_inputs(S, L, H, 128, seed=31, device=dev)
    ops = h3lib.sage_quantize(inp["q"], inp["k"], inp["v"], L)
    o_ref = torch.full_like(inp["q"], SENT)
    h3lib.attention_fp8(ops, o_ref, L)
    o = torch.full_like(inp["q"], SENT)
    kept = torch.full(((L + 127) // 128, H), -1, dtype=torch.int32, device=dev)
    h3lib.attention_fp8_skip(ops, o, L, skip_eps=0.0, kept=kept)
    h3lib.check_device_error()
    assert torch.equal(o, o_ref)
    assert bool((kept == -1).all())  # left untouched at eps = 0


@pytest.mark.parametrize("S,L,eps_log2", [(2048, 2000, 4), (1024, 1024, 2), (1408, 1300, 6)])
def test_sage_skip_matches_oracle_rule(h3lib, S, L, eps_log2):
    """Queries and keys with a shared direction whose per-key-tile weight
    varies, so that whole tiles fall far below the running maximum: the
    GPU's codes equal the oracle's, its kept-tile counts equal those of
    oracle.attention_sage_skip, its output is within the SAGE tolerance of
    the oracle's (error terms over the kept keys), and it differs from the
    unskipped FP8 attention. Pad rows are not written."""
    H = 2
    g = torch.Generator().manual_seed(S + 7 * eps_log2)
    q = torch.randn(S, H, 128, generator=g)
    k = torch.randn(S, H, 128, generator=g)
    v = torch.randn(S, H, 128, generator=g)
    q[:, :, 0] += 8.0
    nk = (S + 127) // 128
    b = torch.randn(nk, H, generator=g) * 8.0
    k[:, :, 0] += b.repeat_interleave(128, dim=0)[:S]
    q, k, v = (t.to(torch.bfloat16).to(dev) for t in (q, k, v))
    ops = h3lib.sage_quantize(q, k, v, L)
    ref_ops = O.sage_quantize(np64(q), np64(k), np64(v), L)
    assert_ops_equal(ops, ref_ops, L)
    eps = 2.0 ** -eps_log2
    nq = (L + 127) // 128
    kept_gpu = torch.full((nq, H), -1, dtype=torch.int32, device=dev)
    o = torch.full_like(q, SENT)
    h3lib.attention_fp8_skip(ops, o, L, skip_eps=eps, kept=kept_gpu)
    h3lib.check_device_error()
    assert bool((o[L:] == SENT).all())
    ref, kept = O.attention_sage_skip(ref_ops, L, SCALE, eps)
    want = kept.sum(axis=2)
    assert want.sum() < nq * H * nq  # tiles really are skipped
    assert np.array_equal(kept_gpu.cpu().numpy(), want)
    terms = O.sage_skip_error_terms(ref_ops, L, SCALE, eps)
    assert_close_sage(np64(o[:L]), ref, terms, L, "sage + skip-softmax")
    full = O.attention_sage(ref_ops, L, SCALE)
    assert np.max(np.abs(ref - full)) > 0


@pytest.mark.parametrize("S,L", [(128, 1), (256, 250), (1152, 1100)])
def test_sage_skip_small_and_ragged(h3lib, S, L):
    """Small and ragged lengths at a real threshold: codes, kept counts and
    output against the oracle (nothing or little is skipped on these
    unit-RMS inputs)."""
    H = 2
    inp = I.attention_inputs(S, L, H, 128, seed=S + 3, device=dev)
    ops = h3lib.sage_quantize(inp["q"], inp["k"], inp["v"], L)
    ref_ops = O.sage_quantize(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), L)
    assert_ops_equal(ops, ref_ops, L)
    eps = 2.0 ** -3
    nq = (L + 127) // 128
    kept_gpu = torch.full((nq, H), -1, dtype=torch.int32, device=dev)
    o = torch.full_like(inp["q"], SENT)
    h3lib.attention_fp8_skip(ops, o, L, skip_eps=eps, kept=kept_gpu)
    h3lib.check_device_error()
    assert bool((o[L:] == SENT).all())
    ref, kept = O.attention_sage_skip(ref_ops, L, SCALE, eps)
    assert np.array_equal(kept_gpu.cpu().numpy(), kept.sum(axis=2))
    assert_close_sage(np64(o[:L]), ref, O.sage_skip_error_terms(ref_ops, L, SCALE, eps), L,
                      "sage + skip, small")


def test_sage_skip_frame_local_inputs(h3lib):
    """The frame-local inputs of the Skip-Softmax measurement (frames of
    1,024 rows), at 4,096 rows: about half of the key tiles are left out;
    kept counts equal the oracle's and the output is within the SAGE
    tolerance over the kept keys."""
    S = L = 4096
    H = 2
    loc = I.frame_local_attention_inputs(S, L, H, 128, frame=1024, seed=5, device=dev)
    ops = h3lib.sage_quantize(loc["q"], loc["k"], loc["v"], L)
    ref_ops = O.sage_quantize(np64(loc["q"]), np64(loc["k"]), np64(loc["v"]), L)
    assert_ops_equal(ops, ref_ops, L)
    eps = 1e-3
    nq = L // 128
    kept_gpu = torch.full((nq, H), -1, dtype=torch.int32, device=dev)
    o = torch.full_like(loc["q"], SENT)
    h3lib.attention_fp8_skip(ops, o, L, skip_eps=eps, kept=kept_gpu)
    h3lib.check_device_error()
    ref, kept = O.attention_sage_skip(ref_ops, L, SCALE, eps)
    want = kept.sum(axis=2)
    assert 0.3 < want.sum() / (nq * H * nq) < 0.8
    assert np.array_equal(kept_gpu.cpu().numpy(), want)
    assert_close_sage(np64(o[:L]), ref, O.sage_skip_error_terms(ref_ops, L, SCALE, eps), L,
                      "sage + skip, frame-local")
