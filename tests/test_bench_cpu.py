"""bench.py's host-side pieces on the CPU: the work model, the oracle samples
of the CPU baseline (on a small shape), and the job arithmetic."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dit_transformer_block_gb300 import inputs as I  # noqa: E402

SMALL = I.BlockShape(S=320, L=300, D=256, H=2, Dh=128, F=512, axis_dims=(32, 48, 48),
                     pos_kind="3d", grid=(2, 12, 12), n_tail=22)


def test_block_work_counts_the_pages_workload():
    w = bench.block_work(58816, 58758, 5376, 42, 128, 14336)
    assert abs(w["attn_flop"] - 74.24e12) / 74.24e12 < 1e-3
    assert abs(w["gemm_flop"] - 40.76e12) / 40.76e12 < 1e-3


def test_job_value_divides_by_replicas():
    assert bench.job_value(80.0, 1) == 80.0
    assert bench.job_value(80.0, 4) == 20.0


def test_oracle_samples_run_and_extrapolate():
    bench._KV_CACHE.clear()
    ms, desc, secs, parts = bench.oracle_sample(SMALL, n_kv=64, n_q=8, seed=1)
    assert ms > 0 and secs > 0 and "extrapolated" in desc
    # the extrapolation is L times the per-row costs of the two stages
    assert np.isclose(parts["kv_all_rows_ms_extrapolated"], parts["kv_ms"] / 64 * SMALL.L,
                      rtol=0.02, atol=0.2)
    qk_ms, qk_all = bench.oracle_qk_rows(SMALL, n=16)
    assert qk_ms > 0 and np.isclose(qk_all, qk_ms * SMALL.L / 16)
    at_ms, at_all = bench.oracle_attention_rows(SMALL, n=16)
    assert at_ms > 0 and np.isclose(at_all, at_ms * SMALL.L / 16)
