"""The FP8 attention tolerance (helpers.assert_close_sage) on the CPU.

A second correct FP8 evaluation that quantises the softmax weights against an
integer running maximum (224 * 2^(z - m), m within [max z - 1, ceil(max z)],
as an online one-pass kernel has to) must pass against the oracle, and
evaluations with a real mistake must fail (the E4M3 rounding of P alone
moves an output by a few percent, so the comparison resolves mistakes of
about 10 % and more in relative L2). The alternative evaluations below
are written here, in the test, from that description; they are not part of
the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle.h3_oracle as O
from helpers import assert_close_sage


def bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).double().numpy()


def integer_max_eval(ops, L, scale, tile=128, use_floor=False, drop_tile=None, v_scale=1.0):
    """FP8 attention with P against the integer reference m = ceil(max z), or
    floor(max z) when use_floor (both lie in [max z - 1, ceil(max z)]).
    drop_tile / v_scale plant a mistake (a key tile left out, a wrong V scale)."""
    qc, kc, vc = ops["qc"], ops["kc"], ops["vc"]
    sq, sk = ops["sq"].astype(np.float64), ops["sk"].astype(np.float64)
    sv = ops["sv"].astype(np.float64) * v_scale
    H = qc.shape[1]
    keys = np.arange(L)
    if drop_tile is not None:
        keys = keys[keys // tile != drop_tile]
    out = np.empty((L, H, qc.shape[2]))
    for h in range(H):
        s = (qc[:L, h] @ kc[keys, h].T) * sq[np.arange(L) // tile, h][:, None] \
            * sk[keys // tile, h][None, :]
        z = s * scale / math.log(2.0)
        zmax = z.max(axis=1, keepdims=True)
        m = np.floor(zmax) if use_floor else np.ceil(zmax)
        p = 224.0 * np.exp2(z - m)
        pc = e4m3(p)
        out[:, h] = (pc @ vc[keys, h]) * sv[h][None, :] / p.sum(axis=1, keepdims=True)
    return bf16(out)


def case(L, H, seed, q_scale=1.0):
    r = np.random.default_rng(seed)
    q = bf16(r.standard_normal((L, H, 128)) * q_scale)
    k = bf16(r.standard_normal((L, H, 128)) + 0.5)
    v = bf16(r.standard_normal((L, H, 128)))
    return O.sage_quantize(q, k, v, L)


@pytest.mark.parametrize("L,H,seed,qs", [(300, 2, 1, 1.0), (600, 1, 2, 0.2), (250, 2, 3, 2.0)])
def test_integer_maximum_evaluation_passes(L, H, seed, qs):
    ops = case(L, H, seed, qs)
    scale = 128 ** -0.5
    ref = O.attention_sage(ops, L, scale)
    terms = O.sage_error_terms(ops, L, scale)
    for use_floor in (False, True):
        alt = integer_max_eval(ops, L, scale, use_floor=use_floor)
        assert np.any(alt != ref)  # the two really round differently
        assert_close_sage(alt, ref, terms, L)


@pytest.mark.parametrize("mistake", [dict(drop_tile=1), dict(drop_tile=4), dict(v_scale=1.25)])
def test_planted_mistake_fails(mistake):
    L, H = 600, 2
    ops = case(L, H, 4, 1.0)
    scale = 128 ** -0.5
    ref = O.attention_sage(ops, L, scale)
    terms = O.sage_error_terms(ops, L, scale)
    with pytest.raises(AssertionError):
        assert_close_sage(integer_max_eval(ops, L, scale, **mistake), ref, terms, L)
