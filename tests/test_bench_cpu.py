"""bench.py's host-side pieces on the CPU: the work model, the oracle samples
of the CPU baseline (on a small shape), the job arithmetic, and the gate that
reports a committed ncu traffic figure only while its kernel code is
unchanged."""
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


def test_code_hash_ignores_comments_and_blank_lines_only():
    src = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    same = "// a header comment\nint f(int x) {\n\n  return x + 1;   \n}\n"
    other = "int f(int x) {\n  return x + 2;  // one more\n}\n"
    assert bench.code_sha256(src) == bench.code_sha256(same)
    assert bench.code_sha256(src) != bench.code_sha256(other)


def test_profile_traffic_only_while_the_kernel_code_is_unchanged(tmp_path, monkeypatch):
    csrc = tmp_path / "dit_transformer_block_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("__global__ void k() {}  // kernel\n")
    (csrc / "k.cuh").write_text("constexpr int N = 4;\n")
    files = ("k.cu", "k.cuh")
    prefix = bench.code_sha256("__global__ void k() {}\nconstexpr int N = 4;\n")[:16]
    (tmp_path / "profiles" / "p.md").write_text(
        f"text\n\ndram_bytes_per_launch: 123456\nsource_sha256: {prefix}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic(files, "p.md") == 123456.0
    # a comment-only edit keeps the figure; a code edit makes it stale
    (csrc / "k.cu").write_text("// reworded\n__global__ void k() {}  // the kernel\n")
    assert bench.profile_traffic(files, "p.md") == 123456.0
    (csrc / "k.cuh").write_text("constexpr int N = 8;\n")
    assert bench.profile_traffic(files, "p.md") is None
    assert bench.profile_traffic(files, "missing.md") is None
