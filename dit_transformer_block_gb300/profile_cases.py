"""Small, fixed cases for ncu captures of the library's kernels.

    python -m dit_transformer_block_gb300.profile_cases [attention] [gemm] [elementwise] [fp8] [sage]

Each selected kernel runs twice on inputs larger than L2 (129 MB) but a few
hundred MB in total, so that an `ncu --set full -k <kernel> -s 1 -c 1`
capture of the second launch ends within a minute or two:
  attention   S = L = 16384, 42 heads x 128 (q, k, v, o: 704 MB)
  gemm        M = 8192, N = 16128, K = 5376 (the QKV projection shape; 520 MB),
              plain and with Q/K RMSNorm + RoPE in the epilogue (after its RoPE
              table), then the down projection shape M = 8192, N = 5376,
              K = 14336 with the residual update in the epilogue (565 MB)
  elementwise qk_norm_rope on 16384 x 42 x 128 (interleaved, then split-half
              pairs), SwiGLU on 16384 x 2 x 14336,
              modulation/LN/residual on 16384 x 5376
  fp8         FP8 GEMM (QKV shape, M = 8192), per-row FP8 quantisation of
              8192 x 5376, SAGE quantisation and FP8 attention at S = L = 16384
  sage        SAGE quantisation alone (K mean, V absmax, Q/K tile and V codes)
              at S = L = 16384, 42 heads
"""
from __future__ import annotations

import sys

import torch

from dit_transformer_block_gb300 import build, h3


def main(argv):
    which = set(argv) or {"attention", "gemm", "elementwise", "fp8", "sage"}
    build.build()
    h3.lib()
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    rnd = lambda *s, std=1.0: (torch.randn(*s, generator=g, device=dev) * std).to(torch.bfloat16)
    runs = []
    if "attention" in which:
        S = 16384
        q, k, v = rnd(S, 42, 128), rnd(S, 42, 128), rnd(S, 42, 128)
        o = torch.empty_like(q)
        runs.append(lambda: h3.attention_varlen(q, k, v, o, S))
    if "gemm" in which:
        M, N, K = 8192, 16128, 5376
        x, w = rnd(M, K), rnd(N, K, std=0.02)
        y = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        runs.append(lambda: h3.linear(x, w, y, M))
        from dit_transformer_block_gb300 import inputs as I
        pos = I.positions_3d(M, M, grid=(31, 24, 79), n_tail=22).to(dev)
        tab = torch.empty(M, 64, 2, device=dev)
        gains = torch.ones(128, device=dev)
        runs.append(lambda: h3.rope_table(pos, (32, 48, 48), tab, M))
        runs.append(lambda: h3.linear_qk_norm_rope(x, w, y, gains, gains, tab, (32, 48, 48), M))
        xd, wd = rnd(M, 14336), rnd(5376, 14336, std=0.02)
        rd = torch.randn(M, 5376, generator=g, device=dev)
        gate = torch.randn(5376, generator=g, device=dev) * 0.1
        runs.append(lambda: h3.linear_residual(xd, wd, rd, gate, M))
    if "elementwise" in which:
        S = 16384
        qq, kk = rnd(S, 42, 128), rnd(S, 42, 128)
        ones = torch.ones(128, device=dev)
        pos = torch.zeros(S, 3, dtype=torch.int32, device=dev)
        gu = rnd(S, 2 * 14336)
        u = torch.empty(S, 14336, device=dev, dtype=torch.bfloat16)
        r = torch.randn(S, 5376, generator=g, device=dev)
        d = rnd(S, 5376)
        hh = torch.empty(S, 5376, device=dev, dtype=torch.bfloat16)
        mod = torch.randn(6, 5376, generator=g, device=dev) * 0.1
        runs.append(lambda: h3.qk_norm_rope(qq, kk, ones, ones, pos, (32, 48, 48), S))
        runs.append(lambda: h3.qk_norm_rope(qq, kk, ones, ones, pos, (32, 48, 48), S, pairing=1))
        runs.append(lambda: h3.swiglu(gu, u, S))
        runs.append(lambda: h3.mod_norm_residual(r, d, mod[2], mod[3], mod[4], hh, S))
    if "fp8" in which:
        M, N, K = 8192, 16128, 5376
        x8, w8 = rnd(M, K), rnd(N, K, std=0.02)
        qx = torch.empty(M, K, dtype=torch.uint8, device=dev)
        sx = torch.empty(M, device=dev)
        qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
        sw = torch.empty(N, device=dev)
        h3.quantize_fp8_rows(w8, qw, sw)
        y8 = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        runs.append(lambda: h3.quantize_fp8_rows(x8, qx, sx))
        runs.append(lambda: h3.linear_fp8(qx, sx, qw, sw, y8, M))
        S = 16384
        qa, ka, va = rnd(S, 42, 128), rnd(S, 42, 128), rnd(S, 42, 128)
        oa = torch.empty_like(qa)
        ops = h3.sage_quantize(qa, ka, va, S)
        runs.append(lambda: h3.attention_fp8(ops, oa, S))
    if "sage" in which:
        S = 16384
        qs, ks, vs = rnd(S, 42, 128), rnd(S, 42, 128), rnd(S, 42, 128)
        runs.append(lambda: h3.sage_quantize(qs, ks, vs, S))
    for _ in range(2):
        for fn in runs:
            fn()
    torch.cuda.synchronize()
    h3.check_device_error()
    print("ok")


if __name__ == "__main__":
    main(sys.argv[1:])
