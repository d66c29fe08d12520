"""SAGE-style FP8 attention against the oracle: the E4M3 codes and scales bit
for bit (quantising with the GPU's own K mean, a float32 sum whose rounding
order the oracle does not share), the K mean to float32 accuracy, and the FP8
attention within the bf16 tolerances given identical operands."""
import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
from helpers import assert_close_bf16, np64, rel_l2, sample_rows

pytestmark = pytest.mark.gpu
dev = "cuda"
SENT = -7.25


def decode(q):
    return q.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()


def gpu_ops_as_oracle(ops, L):
    return dict(qc=decode(ops["qc"][:L]), kc=decode(ops["kc"][:L]), vc=decode(ops["vc"][:L]),
                sq=np64(ops["sq"]).astype(np.float32), sk=np64(ops["sk"]).astype(np.float32),
                sv=np64(ops["sv"]).astype(np.float32), k_mean=np64(ops["k_mean"]))


@pytest.mark.parametrize("S,L,H", [(256, 250, 4), (640, 600, 3), (128, 1, 2)])
def test_sage_codes_and_attention(h3lib, S, L, H):
    inp = I.attention_inputs(S, L, H, 128, seed=S + H, device=dev)
    q, k, v = inp["q"], inp["k"], inp["v"]
    k = (k.float() + 0.75).to(torch.bfloat16)  # a common offset the smoothing removes
    ops = h3lib.sage_quantize(q, k, v, L)
    h3lib.check_device_error()
    mean64 = np64(k[:L]).mean(0)
    assert np.allclose(np64(ops["k_mean"]), mean64, rtol=1e-6, atol=1e-7)
    ref_ops = O.sage_quantize(np64(q), np64(k), np64(v), L, k_mean=np64(ops["k_mean"]))
    g = gpu_ops_as_oracle(ops, L)
    for key in ("qc", "kc", "vc", "sq", "sk", "sv"):
        assert np.array_equal(g[key], ref_ops[key]), key
    o = torch.full_like(q, SENT)
    h3lib.attention_fp8(ops, o, L)
    h3lib.check_device_error()
    ref = O.attention_sage(g, L, 128 ** -0.5)
    assert_close_bf16(np64(o[:L]), ref, "sage attention")
    assert bool((o[L:] == SENT).all())
    dense = O.attention(np64(q), np64(k), np64(v), L, 128 ** -0.5)
    assert rel_l2(np64(o[:L]), dense) < 0.1


@pytest.mark.slow
def test_sage_full_size_sampled(h3lib):
    S, L, H = 58816, 58758, 42
    inp = I.attention_inputs(S, L, H, 128, seed=2, device=dev)
    ops = h3lib.sage_quantize(inp["q"], inp["k"], inp["v"], L)
    o = torch.full_like(inp["q"], SENT)
    h3lib.attention_fp8(ops, o, L)
    h3lib.check_device_error()
    rows = sample_rows(L, 256, 12)
    g = gpu_ops_as_oracle(ops, L)
    ref = O.attention_sage(g, L, 128 ** -0.5, rows=rows)
    assert_close_bf16(np64(o[torch.from_numpy(rows).to(dev)]), ref, "sage attention full")
    assert bool((o[L:] == SENT).all())
