#!/usr/bin/env python
"""Benchmark of one joint audio-video DiT block forward on GB300.

A step is one pass of the whole block (modulation + LN, QKV projection, Q/K
RMSNorm + RoPE, valid-length attention, output projection, residual +
modulation + LN, gate/up projection with SwiGLU, down projection, residual)
over the packed sequence of 58,758 valid tokens in a 58,816-token buffer
(hidden 5376, 42 x 128 heads, SwiGLU inner 14336, 3-axis RoPE 32/48/48), the
workload of the vLLM-Omni MiniMax H3 blog, section 3.1.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0). With N > 1 (torchrun), every rank runs its own
replica of the block on its own GPU ("replicas only": the block has no
exchange step on one GPU) and the time is the maximum over ranks.
--impl reference times the CPU oracle (plain NumPy FP64) on a bounded sample
of the same workload, extrapolated to one block.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DiT block fwd ms & attention TFLOP/s at 58,758-token packed seq; % of BF16 peak"
WORKLOAD = ("full DiT block forward: packed sequence L=58758 valid of S=58816, D=5376, "
            "42 heads x 128, SwiGLU F=14336, 3-axis RoPE 32/48/48")


def args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the FP8 block, block-stack and output-prep measurements")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ----------------------------------------------------------------- work model
def block_work(S, L, D, H, Dh, F):
    """Algorithmic FLOPs and bytes of one block (valid rows only)."""
    attn = 4.0 * L * L * H * Dh
    gemm = 2.0 * L * D * (3 * D) + 2.0 * L * D * D + 2.0 * L * D * (2 * F) + 2.0 * L * F * D
    # bytes of the HBM-bound stages as launched: the first modulated LayerNorm
    # (plus the RoPE table: positions in, 64 (cos, sin) pairs out per row) and
    # the middle residual + LayerNorm; Q/K RMSNorm + RoPE, SwiGLU and the last
    # residual update run in GEMM epilogues
    mnr = L * D * (4 + 2) + L * D * (4 + 2 + 4 + 2)
    rope = L * (12 + 64 * 8)
    return dict(attn_flop=attn, gemm_flop=gemm, elementwise_bytes=mnr + rope)


def stage_work(S, L, D, H, Dh, F):
    """Per stage of the block: (bound, algorithmic work, unit of the rate).
    GEMMs count 2MNK, attention 4 L^2 H Dh, HBM-bound stages their minimum
    bytes read + written (rows < L only)."""
    return [
        ("hbm", L * D * (4 + 2) + L * (12 + 64 * 8), "GB/s"),   # r -> h1; pos -> RoPE table
        ("tensor", 2.0 * L * D * 3 * D, "TFLOP/s"),              # QKV + Q/K RMSNorm + RoPE
        ("tensor", 4.0 * L * L * H * Dh, "TFLOP/s"),             # attention
        ("tensor", 2.0 * L * D * D, "TFLOP/s"),                  # out
        ("hbm", L * D * (4 + 2 + 4 + 2), "GB/s"),                # r, o -> r, h2
        ("tensor", 2.0 * L * D * 2 * F, "TFLOP/s"),              # gate/up + SwiGLU
        ("tensor", 2.0 * L * F * D, "TFLOP/s"),                  # down + residual
    ]


# -------------------------------------------------------------- clock sampler
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ------------------------------------------------------------ across ranks
def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks of the default
    process group (identity with one rank). Each rank runs its own replica of
    the block, so the job's time is the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_value(step_ms: float, world: int) -> float:
    """Whole-job ms per block forward: N replicas finish N blocks per step."""
    return step_ms / world


# ----------------------------------------------------------- CPU baseline leg
_KV_CACHE = {}


def oracle_sample(shape, n_kv=8192, n_q=96, seed=3):
    """Times the oracle on a bounded sample of one block and extrapolates.

    Sample: the key/value stage (LayerNorm + K and V projections + K
    RMSNorm/RoPE) for n_kv rows, and the per-query path (LayerNorm, Q
    projection, Q RMSNorm/RoPE, attention over all L keys, output projection,
    residual + LayerNorm, gate/up projection, SwiGLU, down projection,
    residual) for n_q rows. One block = L x (t_kv / n_kv + t_q / n_q).
    The full-length keys/values the query rows attend to are drawn once per
    process (untimed); their cost is what the timed K/V stage measures.
    """
    import numpy as np
    import torch

    import oracle.h3_oracle as O
    from dit_transformer_block_gb300 import inputs as I

    g = torch.Generator().manual_seed(seed)
    D, H, Dh, F, L = shape.D, shape.H, shape.Dh, shape.F, shape.L
    bf = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(torch.bfloat16).double().numpy()
    w_qkv = bf(3 * D, D, std=0.02)
    w_o = bf(D, D, std=0.02)
    w_gu = bf(2 * F, D, std=0.02)
    w_down = bf(D, F, std=0.02)
    gain = 1 + 0.1 * torch.randn(Dh, generator=g).double().numpy()
    mod = 0.1 * torch.randn(6, D, generator=g).double().numpy()
    pos = I.positions_3d(shape.S, L).numpy()
    x_kv = bf(n_kv, D)
    x_q = bf(n_q, D)
    k_all, v_all = _kv(shape)

    t0 = time.perf_counter()
    for c0 in range(0, n_kv, 2048):
        c1 = min(n_kv, c0 + 2048)
        _, h = O.mod_norm_residual(x_kv[c0:c1], shift=mod[0], scale=mod[1])
        k = O.linear(h, w_qkv[D:2 * D]).reshape(c1 - c0, H, Dh)
        O.qk_norm_rope(k, gain, pos[c0:c1], shape.axis_dims, shape.theta, shape.eps_qk)
        O.linear(h, w_qkv[2 * D:])
    t_kv = time.perf_counter() - t0

    t0 = time.perf_counter()
    r = x_q
    _, h1 = O.mod_norm_residual(r, shift=mod[0], scale=mod[1])
    q = O.linear(h1, w_qkv[:D]).reshape(n_q, H, Dh)
    q = O.qk_norm_rope(q, gain, pos[L - n_q:L], shape.axis_dims, shape.theta, shape.eps_qk)
    qf = np.zeros((L, H, Dh))
    rows = np.arange(L - n_q, L)
    qf[rows] = q
    a = O.attention(qf, k_all, v_all, L, Dh ** -0.5, rows=rows).reshape(n_q, D)
    o = O.linear(a, w_o)
    r, h2 = O.mod_norm_residual(r, o, mod[2], mod[3], mod[4])
    u = O.swiglu(O.linear(h2, w_gu))
    f = O.linear(u, w_down)
    O.mod_norm_residual(r, f, mod[5])
    t_q = time.perf_counter() - t0
    ms = L * (t_kv / n_kv + t_q / n_q) * 1e3
    desc = (f"oracle (NumPy FP64) on the key/value stage of {n_kv} rows and the full query path "
            f"of {n_q} rows of the L={L} block, extrapolated linearly to all rows")
    return ms, desc, t_kv + t_q, dict(kv_rows=n_kv, kv_ms=round(t_kv * 1e3, 1),
                                       kv_all_rows_ms_extrapolated=round(t_kv / n_kv * L * 1e3, 1),
                                       query_rows=n_q, query_ms=round(t_q * 1e3, 1),
                                       query_all_rows_ms_extrapolated=round(t_q / n_q * L * 1e3, 1))


def oracle_qk_rows(shape, n=512, seed=1):
    """Oracle Q/K RMSNorm + RoPE on n seeded rows of the full-size workload
    (all 42 heads, q and k); returns (ms for the n rows, ms extrapolated
    linearly to all L rows)."""
    import numpy as np
    import torch

    import oracle.h3_oracle as O
    from dit_transformer_block_gb300 import inputs as I

    L, H, Dh = shape.L, shape.H, shape.Dh
    g = torch.Generator().manual_seed(seed)
    rows = np.sort(np.random.default_rng(seed).choice(L, n, replace=False))
    q = torch.randn(n, H, Dh, generator=g).to(torch.bfloat16).double().numpy()
    k = torch.randn(n, H, Dh, generator=g).to(torch.bfloat16).double().numpy()
    gain = 1 + 0.1 * torch.randn(Dh, generator=g).double().numpy()
    pos = I.positions_3d(shape.S, L).numpy()[rows]
    t0 = time.perf_counter()
    for x in (q, k):
        O.qk_norm_rope(x, gain, pos, shape.axis_dims, shape.theta, shape.eps_qk)
    ms = (time.perf_counter() - t0) * 1e3
    return ms, ms * L / n


def oracle_attention_rows(shape, n=512, seed=2):
    """Oracle attention for n seeded query rows over all L keys of the
    full-size workload (42 heads); returns (ms for the n rows, ms extrapolated
    linearly to all L rows). The keys and values are drawn once per process,
    untimed (they are this configuration's inputs)."""
    import numpy as np

    import oracle.h3_oracle as O

    L, H, Dh = shape.L, shape.H, shape.Dh
    k_all, v_all = _kv(shape)
    rows = np.sort(np.random.default_rng(seed).choice(L, n, replace=False))
    q = np.zeros((L, H, Dh))
    q[rows] = k_all[rows[::-1]]  # unit-RMS-like rows; their values do not change the cost
    t0 = time.perf_counter()
    O.attention(q, k_all, v_all, L, Dh ** -0.5, rows=rows)
    ms = (time.perf_counter() - t0) * 1e3
    return ms, ms * L / n


def _kv(shape):
    """Full-length bf16-valued keys and values, drawn once per process."""
    import torch
    key = (shape.L, shape.H, shape.Dh)
    if key not in _KV_CACHE:
        gk = torch.Generator().manual_seed(12345)
        kv = lambda: torch.randn(*key, generator=gk).to(torch.bfloat16).double().numpy()
        _KV_CACHE[key] = (kv(), kv())
    return _KV_CACHE[key]


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                low = line.lower()
                if low.startswith("model name") or low.startswith("hardware"):
                    return line.split(":", 1)[1].strip()
                if low.startswith("cpu part"):
                    import platform
                    return f"{platform.machine()} CPU part {line.split(':', 1)[1].strip()}"
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


_TINY_CODE = """
import time, numpy as np, torch
import oracle.h3_oracle as O
from dit_transformer_block_gb300 import inputs as I
sh = I.TINY
n = {k: v.double().numpy() if v.is_floating_point() else v.numpy()
     for k, v in I.block_inputs(sh, seed=0).items()}
best = 1e9
for _ in range(3):
    t0 = time.perf_counter()
    O.block_forward(n["resid"], n["mod"], n["w_qkv"], n["w_o"], n["w_gu"], n["w_down"],
                    n["q_gain"], n["k_gain"], n["pos"], L=sh.L, heads=sh.H, head_dim=sh.Dh,
                    axis_dims=sh.axis_dims, theta=sh.theta)
    best = min(best, time.perf_counter() - t0)
print(best * 1e3)
"""


def oracle_tiny_ms(threads=None):
    """Whole oracle block on the 256-row configuration (every row), best of
    three, in a child process so that the BLAS thread count can be fixed."""
    env = dict(os.environ)
    if threads is not None:
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[v] = str(threads)
    out = subprocess.run([sys.executable, "-c", _TINY_CODE], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    if out.returncode != 0:
        return None
    return round(float(out.stdout.strip().splitlines()[-1]), 2)


def cpu_cores():
    try:
        import numpy  # noqa: F401
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ------------------------------------------------------------------ extras
def measure_extras(h3, torch, shape, inp, cfg, ws, stream, pk):
    """Rows beyond the BF16 block, timed after the main measurement with CUDA
    events on the launching stream (3 warm-up launches each):
      qk_norm_rope  Q/K RMSNorm + RoPE alone on its full-size workload, both
                    channel pairings (GB/s against the copy bandwidth)
      attention     attention alone on its full-size workload (unit-RMS q, k)
      sage_quantize, attention_fp8   the FP8 (SAGE) operands and attention on
                    the same inputs
      skip_softmax  Skip-Softmax (BF16 and with SAGE FP8) on the same inputs
                    and on frame-local inputs, with the kept-tile fraction
      fp8_block     the block with online FP8 projections
      stack4        4 blocks in one h3_stack_forward call (fused boundaries)
      frames_to_u8  output preparation of the 10 s, 1344 x 768 clip"""
    def timeit(fn, n):
        for _ in range(3):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(n):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        h3.check_device_error()
        return s.elapsed_time(e) / n

    out = {}
    from dit_transformer_block_gb300 import inputs as I
    S, L, H = shape.S, shape.L, shape.H
    # Q/K RMSNorm + RoPE alone (q, k ~ N(0,1) [58816, 42, 128], 3-axis RoPE,
    # seed 1): 8 bytes per (row, head, channel) read + written for q and k
    qk = I.qk_inputs(S, L, H, 128, seed=1, device=inp["resid"].device)
    pos = I.positions_3d(S, L).to(inp["resid"].device)
    qk_bytes = L * H * 128 * 2 * 2 * 2
    out["qk_norm_rope"] = {"workload": "q, k ~ N(0,1) bf16 [58816, 42, 128], 58,758 valid, "
                           "3-axis RoPE 32/48/48, seed 1", "bytes": qk_bytes}
    for name, pairing in (("interleaved", 0), ("split_half", 1)):
        ms = timeit(lambda: h3.qk_norm_rope(qk["q"], qk["k"], qk["q_gain"], qk["k_gain"], pos,
                                            shape.axis_dims, L=L, pairing=pairing), 20)
        gbs = qk_bytes / ms / 1e6
        out["qk_norm_rope"][name] = {"ms": round(ms, 4), "achieved_gbs": round(gbs, 1),
                                     "frac_hbm": round(gbs / pk["hbm"], 3)}
    del qk
    # attention alone (q, k unit-RMS, v ~ N(0,1), [58816, 42, 128], seed 2)
    at = I.attention_inputs(S, L, H, 128, seed=2, device=inp["resid"].device)
    o_at = torch.empty_like(at["q"])
    flop = 4.0 * L * L * H * 128
    ms = timeit(lambda: h3.attention_varlen(at["q"], at["k"], at["v"], o_at, L), 3)
    tf = flop / ms / 1e9
    out["attention"] = {"workload": "q, k unit-RMS, v ~ N(0,1) bf16 [58816, 42, 128], 58,758 "
                        "valid, seed 2", "ms": round(ms, 3), "tflops": round(tf, 1),
                        "frac_bf16_sustained": round(tf / pk["bf16_sustained"], 3),
                        "frac_bf16_burst": round(tf / pk["bf16"], 3)}
    ops = h3.sage_quantize(at["q"], at["k"], at["v"], L)
    ms = timeit(lambda: h3.sage_quantize(at["q"], at["k"], at["v"], L), 5)
    out["sage_quantize"] = {"ms": round(ms, 3),
                            "achieved_gbs": round(L * H * 128 * 9 / ms / 1e6, 1)}
    ms = timeit(lambda: h3.attention_fp8(ops, o_at, L), 3)
    out["attention_fp8"] = {"ms": round(ms, 3), "tflops_dense_equivalent": round(flop / ms / 1e9, 1)}
    # Skip-Softmax (eps 1e-3) on the same inputs (no tile falls far enough
    # below to be left out: the cost of the vote), then on frame-local inputs
    # (frames of 1,024 rows, seed 5) with and without it, BF16 and FP8
    nq = (L + 127) // 128
    kept = torch.empty(nq, H, dtype=torch.int32, device=o_at.device)
    eps = 1e-3
    skip = {"eps": eps}
    ms = timeit(lambda: h3.attention_fp8_skip(ops, o_at, L, skip_eps=eps, kept=kept), 3)
    skip["fp8_unit_rms"] = {"ms": round(ms, 3),
                            "kept_fraction": round(kept.sum().item() / (nq * H * nq), 4)}
    ms = timeit(lambda: h3.attention_varlen_skip(at["q"], at["k"], at["v"], o_at, L,
                                                 skip_eps=eps, kept=kept), 3)
    skip["bf16_unit_rms"] = {"ms": round(ms, 3),
                             "kept_fraction": round(kept.sum().item() / (nq * H * nq), 4)}
    del at, ops
    loc = I.frame_local_attention_inputs(S, L, H, 128, frame=1024, seed=5,
                                         device=inp["resid"].device)
    skip["workload_local"] = ("q = n + 16 e, k = n' + 16 e (n, n' ~ N(0,1), e a random unit "
                              "direction per 1,024-row frame and head), v ~ N(0,1), bf16 "
                              "[58816, 42, 128], seed 5")
    ms = timeit(lambda: h3.attention_varlen(loc["q"], loc["k"], loc["v"], o_at, L), 3)
    skip["bf16_local_dense_ms"] = round(ms, 3)
    ms = timeit(lambda: h3.attention_varlen_skip(loc["q"], loc["k"], loc["v"], o_at, L,
                                                 skip_eps=eps, kept=kept), 3)
    skip["bf16_local"] = {"ms": round(ms, 3),
                          "kept_fraction": round(kept.sum().item() / (nq * H * nq), 4)}
    ops = h3.sage_quantize(loc["q"], loc["k"], loc["v"], L)
    ms = timeit(lambda: h3.attention_fp8(ops, o_at, L), 3)
    skip["fp8_local_dense_ms"] = round(ms, 3)
    ms = timeit(lambda: h3.attention_fp8_skip(ops, o_at, L, skip_eps=eps, kept=kept), 3)
    skip["fp8_local"] = {"ms": round(ms, 3),
                         "kept_fraction": round(kept.sum().item() / (nq * H * nq), 4)}
    out["skip_softmax"] = skip
    del loc, o_at, ops, kept
    r = inp["resid"].clone()
    w8 = h3.quantize_block_weights_fp8(inp)
    ws8 = torch.empty(h3.block_workspace_bytes_fp8(cfg), dtype=torch.uint8, device=r.device)
    ms = timeit(lambda: h3.block_forward_fp8(cfg, w8, r, inp["mod"], inp["pos"], ws8), 3)
    out["fp8_block"] = {"ms": round(ms, 3), "note": "four projections in FP8 E4M3 with per-row "
                        "scales; attention and elementwise steps as in the BF16 block"}
    ms = timeit(lambda: h3.block_forward_fp8(cfg, w8, r, inp["mod"], inp["pos"], ws8,
                                             fp8_attention=True), 3)
    out["fp8_block_fp8_attention"] = {"ms": round(ms, 3), "note": "FP8 projections and FP8 "
                                      "(SAGE-style) attention"}
    del ws8, w8
    mods = torch.stack([inp["mod"]] * 4).contiguous()
    ms = timeit(lambda: h3.stack_forward(cfg, [inp] * 4, r, mods, inp["pos"], ws), 1)
    out["stack4"] = {"ms_per_block": round(ms / 4, 3)}
    # length sweep of a 4-block stack (independent seeded weights per block),
    # buffers padded to a multiple of 64: ms per block and TFLOP/s vs length
    del ws
    sweep = []
    for L_s, grid in ((29034, (16, 24, 79)), (58758, (31, 24, 79)), (87846, (47, 24, 79))):
        S_s = (L_s + 63) // 64 * 64
        sh = I.BlockShape(S=S_s, L=L_s, D=shape.D, H=shape.H, Dh=shape.Dh, F=shape.F,
                          axis_dims=shape.axis_dims, pos_kind="3d", grid=grid)
        blocks = [I.block_inputs(sh, seed=4 + b, device=r.device) for b in range(4)]
        cfg_s = h3.block_config(sh.S, sh.L, sh.D, sh.H, sh.Dh, sh.F, sh.axis_dims)
        ws_s = torch.empty(h3.block_workspace_bytes(cfg_s), dtype=torch.uint8, device=r.device)
        mods = torch.stack([b["mod"] for b in blocks]).contiguous()
        rs = blocks[0]["resid"].clone()
        ms = timeit(lambda: h3.stack_forward(cfg_s, blocks, rs, mods, blocks[0]["pos"], ws_s), 1)
        w = block_work(sh.S, sh.L, sh.D, sh.H, sh.Dh, sh.F)
        sweep.append({"L": L_s, "S": S_s, "ms_per_block": round(ms / 4, 3),
                      "tflops": round((w["attn_flop"] + w["gemm_flop"]) / (ms / 4) / 1e9, 1)})
        del blocks, ws_s, rs, mods
    out["length_sweep_stack4"] = sweep
    f = torch.randn(1, 3, 243, 768, 1344, device=r.device).clamp_(-1.2, 1.2)
    o = torch.empty(1, 243, 768, 1344, 3, dtype=torch.uint8, device=r.device)
    ms = timeit(lambda: h3.frames_to_u8(f, o), 5)
    gbs = f.numel() * 5 / ms / 1e6
    out["frames_to_u8"] = {"ms": round(ms, 3), "achieved_gbs": round(gbs, 1),
                           "frac_hbm": round(gbs / pk["hbm"], 3),
                           "workload": "243 x 768 x 1344 RGB frames (FP32 in, uint8 out)"}
    return out


# ------------------------------------------------------------ reference arm
def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from dit_transformer_block_gb300 import inputs as I
    shape = I.FULL
    times = []
    desc = ""
    for i in range(a.warmup + a.steps):
        ms, desc, _, _ = oracle_sample(shape, n_kv=2048, n_q=24, seed=100 + i)
        if i >= a.warmup:
            times.append(ms)
    value = statistics.mean(times)
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "ms",
            "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": round(value, 1), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": round(value, 1), "unit": "ms", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 1), "unit": "ms", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def profile_traffic(kernel_files, profile_md: str):
    """DRAM bytes per launch recorded in a committed ncu summary, if the
    kernel sources it was taken from (their texts joined in the order given)
    are unchanged."""
    p = os.path.join(ROOT, "profiles", profile_md)
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{16,64})", text)
    if not m or not h:
        return None
    src = "\n".join(open(os.path.join(ROOT, "dit_transformer_block_gb300", "csrc", f)).read()
                    for f in kernel_files)
    if not code_sha256(src).startswith(h.group(1)):
        return None
    return float(m.group(1))


# the dense attention kernel's sources, for the recorded DRAM traffic
ATTENTION_SOURCES = ("h3_attention.cu", "h3_attn_common.cuh")


def code_sha256(src: str) -> str:
    """SHA-256 of a CUDA source with its // comments, trailing blanks and
    empty lines removed, so that only a change of the code itself makes a
    recorded counter stale."""
    lines = []
    for line in src.splitlines():
        line = re.sub(r"//.*$", "", line).rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def run_ours(a):
    import torch
    import torch.distributed as dist

    from dit_transformer_block_gb300 import build, h3
    from dit_transformer_block_gb300 import inputs as I

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    h3.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    shape = I.FULL
    S, L, D, H, Dh, F = shape.S, shape.L, shape.D, shape.H, shape.Dh, shape.F
    inp = I.block_inputs(shape, seed=3 + rank, device=dev)
    cfg = h3.block_config(S, L, D, H, Dh, F, shape.axis_dims, shape.theta, shape.eps_ln,
                          shape.eps_qk)
    ws = torch.empty(h3.block_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    weights = h3.block_weights(inp)
    resid = inp["resid"].clone()
    stream = torch.cuda.current_stream()

    nev = h3.BLOCK_STAGES + 1
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(a.steps)]
    for row in events:  # create the event handles before they are handed to the library
        for e in row:
            e.record(stream)

    for _ in range(a.warmup):
        h3.block_forward(cfg, weights, resid, inp["mod"], inp["pos"], ws)
    h3.check_device_error()

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_uuid(torch, local)) as clocks:
        time.sleep(0.3)
        t_start.record(stream)
        for k in range(a.steps):
            h3.block_forward(cfg, weights, resid, inp["mod"], inp["pos"], ws, events=events[k])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    h3.check_device_error()
    if not bool(torch.isfinite(resid[:L]).all()):
        raise RuntimeError("non-finite block output")
    total_ms = t_start.elapsed_time(t_end)
    stage_ms = [statistics.mean(events[k][i].elapsed_time(events[k][i + 1])
                                for k in range(a.steps)) for i in range(h3.BLOCK_STAGES)]
    step_ms = total_ms / a.steps
    per_step = sorted(events[k][0].elapsed_time(events[k][h3.BLOCK_STAGES])
                      for k in range(a.steps))
    red = max_over_ranks([step_ms] + stage_ms, device=dev)
    step_ms, stage_ms = red[0], red[1:]

    # ---- end to end through the C-ABI with host buffers: every step uploads
    # its residual, modulation and positions from pinned memory and downloads
    # the updated residual. All copies run in order on one copy stream (an
    # upload and a download running at the same time slowed each other down
    # several-fold on this host link), three device buffer sets: step k+3's
    # upload is queued right behind step k's download and has two block
    # times to land (single uploads sometimes took 40+ ms instead of 6); the
    # timed region spans the first upload to the last download.
    NBUF = 3
    pin = lambda t: t.detach().to("cpu").pin_memory()
    h_one = (pin(inp["resid"]), pin(inp["mod"]), pin(inp["pos"]))
    h_in = [h_one] * NBUF  # every buffer set uploads the same host data
    h_one_out = torch.empty_like(h_one[0]).pin_memory()
    h_out = [h_one_out] * NBUF
    d_buf = [(torch.empty_like(inp["resid"]), torch.empty_like(inp["mod"]),
              torch.empty_like(inp["pos"])) for _ in range(NBUF)]
    h2d = sum(t.numel() * t.element_size() for t in h_in[0])
    d2h = h_out[0].numel() * 4
    copy_s = torch.cuda.Stream()
    comp_s = torch.cuda.Stream()  # not the legacy default stream, which would serialise the copies

    def e2e_run(n, timeline=False):
        ev = lambda: torch.cuda.Event(enable_timing=timeline)
        up0 = [ev() for _ in range(n)]
        up = [ev() for _ in range(n)]
        c0 = [ev() for _ in range(n)]
        done = [ev() for _ in range(n)]
        dn0 = [ev() for _ in range(n)]
        down = [ev() for _ in range(n)]
        host = []  # host seconds spent enqueueing: upload, block, download

        def upload(k):  # on copy_s, into buffer set k % NBUF
            up0[k].record(copy_s)
            for d, h in zip(d_buf[k % NBUF], h_in[k % NBUF]):
                d.copy_(h, non_blocking=True)
            up[k].record(copy_s)

        with torch.cuda.stream(copy_s):
            for k in range(min(n, NBUF)):
                upload(k)
        for k in range(n):
            b = k % NBUF
            h0 = time.perf_counter()
            comp_s.wait_event(up[k])
            c0[k].record(comp_s)
            h3.block_forward(cfg, weights, d_buf[b][0], d_buf[b][1], d_buf[b][2], ws,
                             stream=comp_s)
            done[k].record(comp_s)
            h1 = time.perf_counter()
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(done[k])
                dn0[k].record(copy_s)
                h_out[b].copy_(d_buf[b][0], non_blocking=True)
                down[k].record(copy_s)
                h2 = time.perf_counter()
                if k + NBUF < n:
                    upload(k + NBUF)  # buffer set b: its download is queued just before
            host.append((time.perf_counter() - h2, h1 - h0, h2 - h1))
        torch.cuda.synchronize()
        if not timeline:
            return None
        mean = lambda xs: round(statistics.mean(xs), 3) if xs else None
        return {
            "upload_ms": mean([up0[k].elapsed_time(up[k]) for k in range(n)]),
            "compute_ms": mean([c0[k].elapsed_time(done[k]) for k in range(n)]),
            "download_ms": mean([dn0[k].elapsed_time(down[k]) for k in range(n)]),
            # idle time of the compute stream between consecutive blocks
            "compute_gap_ms": mean([done[k - 1].elapsed_time(c0[k]) for k in range(1, n)]),
            # first upload start to last download end, on the device
            "span_ms": round(up0[0].elapsed_time(down[n - 1]), 3),
            # host time spent in the calls that enqueue each part of a step
            "host_enqueue_ms": {name: mean([1e3 * h[i] for h in host])
                                for i, name in enumerate(("upload", "block", "download"))},
            # device times (ms from the first upload) of four middle steps:
            # upload start/end, block start/end, download start/end
            "schedule_ms": {str(k): [round(up0[0].elapsed_time(e[k]), 2)
                                     for e in (up0, up, c0, done, dn0, down)]
                            for k in range(n // 2, min(n, n // 2 + 4))},
        }

    e2e_run(2)
    barrier()
    t0 = time.perf_counter()
    e2e_run(a.e2e_steps)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / a.e2e_steps
    barrier()
    e2e_ms = max_over_ranks([e2e_ms], device=dev)[0]
    e2e_timeline = e2e_run(a.e2e_steps, timeline=True)
    h3.check_device_error()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    pk = peaks()
    work = block_work(S, L, D, H, Dh, F)
    attn_ms = stage_ms[2]
    gemm_ms = stage_ms[1] + stage_ms[3] + stage_ms[5] + stage_ms[6]
    ew_ms = stage_ms[0] + stage_ms[4]
    attn_tf = work["attn_flop"] / attn_ms / 1e9
    gemm_tf = work["gemm_flop"] / gemm_ms / 1e9
    traffic = profile_traffic(ATTENTION_SOURCES, "attention_pair_small_case.md")
    stages_roofline = {}
    for name, t, (bound, amount, unit) in zip(h3.STAGE_NAMES, stage_ms,
                                              stage_work(S, L, D, H, Dh, F)):
        rate = amount / t / (1e9 if unit == "TFLOP/s" else 1e6)
        peak = pk["bf16_sustained"] if bound == "tensor" else pk["hbm"]
        stages_roofline[name] = {"bound": bound, "achieved": round(rate, 1), "unit": unit,
                                 "peak": peak, "frac": round(rate / peak, 3)}
    extras = None if a.no_extras else measure_extras(h3, torch, shape, inp, cfg, ws, stream, pk)
    cpu = None
    if not a.no_cpu_baseline and world == 1:
        ms, desc, secs, parts = oracle_sample(shape, n_kv=4096, n_q=512)
        qk_ms, qk_all = oracle_qk_rows(shape)
        at_ms, at_all = oracle_attention_rows(shape)
        cpu = {"value": round(ms, 1), "unit": "ms", "cores": cpu_cores(), "kind": "oracle",
               "sample": desc + f" ({secs:.1f} s of CPU work)", "cpu_model": cpu_model(),
               "per_config": {
                   "qk_norm_rope": {"rows": 512, "ms": round(qk_ms, 1),
                                    "all_rows_ms_extrapolated": round(qk_all, 1)},
                   "attention": {"rows": 512, "ms": round(at_ms, 1),
                                 "all_rows_ms_extrapolated": round(at_all, 1)},
                   "block": parts},
               "tiny_block_ms": {"all_threads": oracle_tiny_ms(),
                                 "one_thread": oracle_tiny_ms(1),
                                 "workload": "whole oracle block, 256-row configuration "
                                             "(L=250, D=512, 4 heads, F=1536), every row"}}
    value = job_value(step_ms, world)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "ms", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(step_ms, 3),
        "ms_per_step_median": round(statistics.median(per_step), 3),
        "ms_per_step_min": round(per_step[0], 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded: x~N(0,1), W~N(0,0.02) bf16; FP32 residual and modulation)",
        "config": {"workload": WORKLOAD, "S": S, "L": L, "D": D, "heads": H, "head_dim": Dh,
                   "ffn": F, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (no flush between steps)"},
        "attention_ms": round(attn_ms, 3), "attention_tflops": round(attn_tf, 1),
        "attention_frac_bf16_peak": round(attn_tf / pk["bf16_sustained"], 3),
        "gemm_ms": round(gemm_ms, 3), "gemm_tflops": round(gemm_tf, 1),
        "gemm_frac_bf16_peak": round(gemm_tf / pk["bf16_sustained"], 3),
        "elementwise_ms": round(ew_ms, 3),
        "elementwise_gbs": round(work["elementwise_bytes"] / ew_ms / 1e6, 1),
        "stages_ms": {n: round(t, 3) for n, t in zip(h3.STAGE_NAMES, stage_ms)},
        "stages_roofline": stages_roofline,
        "roofline": {"bound": "tensor", "kernel": "attention_pair_kernel",
                     "achieved": round(attn_tf, 1), "peak": pk["bf16_sustained"],
                     "unit": "TFLOP/s", "frac": round(attn_tf / pk["bf16_sustained"], 3),
                     "traffic": traffic,
                     "peak_source": f"{pk['source']} bf16 sustained (kernel timed inside a long step)"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_ms, 3), "unit": "ms", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": h3.BLOCK_LAUNCHES * a.steps,
        "e2e_note": (f"{a.e2e_steps} steps timed from the first upload to the last download "
                     "(pipeline fill and drain included); uploads and downloads in order on one "
                     "copy stream beside the compute stream, three buffer sets: copies overlap "
                     "compute"),
        "e2e_timeline": e2e_timeline,
        "clocks": clocks.summary(),
        "extras": extras,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    a = args()
    if a.impl == "reference":
        return run_reference(a)
    return run_ours(a)


if __name__ == "__main__":
    sys.exit(main())
