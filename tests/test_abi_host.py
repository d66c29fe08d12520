"""Host-side checks of the C-ABI library: it builds, loads without a GPU,
exports every function include/h3block.h declares, and rejects bad
arguments on the host with the documented status before any launch."""
import ctypes
import os

import pytest

from dit_transformer_block_gb300 import build as B
from dit_transformer_block_gb300 import h3


@pytest.fixture(scope="module")
def lib():
    B.build()
    return h3.lib()


def test_exports_every_declared_function(lib):
    names = h3.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(h3._SIGS), "binding and header disagree"


def test_version_and_status_strings(lib):
    assert lib.h3_version() >> 16 == 1
    for code, name in h3.STATUS.items():
        assert lib.h3_status_string(code).decode() == name


NULL = None
P = ctypes.c_void_p(4096)       # 16-byte aligned fake device address (never dereferenced)
PM = ctypes.c_void_p(4096 + 2)  # misaligned


def st(lib, fn, *args):
    return getattr(lib, fn)(*args)


def test_attention_argument_errors(lib):
    f = "h3_attention_varlen"
    assert st(lib, f, P, P, P, P, 10, 11, 2, 128, 0.1, NULL) == 1     # L > S
    assert "L=11" in h3.last_error(), h3.last_error()
    assert st(lib, f, P, P, P, P, 10, -1, 2, 128, 0.1, NULL) == 1     # L < 0
    assert st(lib, f, NULL, P, P, P, 10, 5, 2, 128, 0.1, NULL) == 1   # null q
    assert st(lib, f, P, P, P, P, 10, 5, 2, 64, 0.1, NULL) == 2       # head_dim
    assert st(lib, f, P, PM, P, P, 10, 5, 2, 128, 0.1, NULL) == 3     # misaligned
    assert st(lib, f, P, P, P, P, 10, 0, 2, 128, 0.1, NULL) == 0      # empty: no-op
    assert h3.last_error() == ""


def test_skip_and_fp8_attention_argument_errors(lib):
    f = "h3_attention_varlen_skip"
    eps = ctypes.c_float
    assert st(lib, f, P, P, P, P, 10, 5, 2, 128, ctypes.c_float(0.1), eps(1.0), NULL, NULL) == 1
    assert "skip_eps" in h3.last_error(), h3.last_error()
    assert st(lib, f, P, P, P, P, 10, 5, 2, 128, ctypes.c_float(0.1), eps(-0.5), NULL, NULL) == 1
    assert st(lib, f, P, P, P, P, 10, 11, 2, 128, ctypes.c_float(0.1), eps(0.1), NULL, NULL) == 1
    assert st(lib, f, P, P, P, P, 10, 0, 2, 128, ctypes.c_float(0.1), eps(0.1), NULL, NULL) == 0
    g = "h3_attention_fp8_skip"
    args = (P, P, P, P, P, P, P)  # codes, scales, o
    assert st(lib, g, *args, 10, 5, 2, 128, ctypes.c_float(0.1), eps(1.0), NULL, NULL) == 1
    assert "skip_eps" in h3.last_error(), h3.last_error()
    assert st(lib, g, *args, 10, 11, 2, 128, ctypes.c_float(0.1), eps(0.1), NULL, NULL) == 1
    assert st(lib, g, NULL, *args[1:], 10, 5, 2, 128, ctypes.c_float(0.1), eps(0.1), NULL,
              NULL) == 1                                                   # null codes
    assert st(lib, g, *args, 10, 5, 2, 64, ctypes.c_float(0.1), eps(0.1), NULL, NULL) == 2
    assert st(lib, g, PM, *args[1:], 10, 5, 2, 128, ctypes.c_float(0.1), eps(0.1), NULL,
              NULL) == 3                                                   # misaligned codes
    assert st(lib, g, *args, 10, 5, 2, 128, ctypes.c_float(0.1), eps(0.1),
              ctypes.c_void_p(4096 + 2), NULL) == 3                        # misaligned counts
    assert st(lib, g, *args, 10, 0, 2, 128, ctypes.c_float(0.1), eps(0.1), NULL, NULL) == 0
    assert h3.last_error() == ""


def test_elementwise_argument_errors(lib):
    assert st(lib, "h3_swiglu", P, P, 4, 5, 16, NULL) == 1
    assert st(lib, "h3_swiglu", P, P, 4, 4, 12, NULL) == 2
    assert st(lib, "h3_swiglu", PM, P, 4, 4, 16, NULL) == 3
    assert st(lib, "h3_swiglu", P, P, 4, 0, 16, NULL) == 0
    ax = (ctypes.c_int * 3)(32, 48, 48)
    axp = ctypes.cast(ax, ctypes.c_void_p)
    bad = (ctypes.c_int * 3)(32, 48, 40)
    badp = ctypes.cast(bad, ctypes.c_void_p)
    f = "h3_qk_norm_rope"
    assert st(lib, f, P, P, P, P, P, axp, 8, 9, 2, 128, 1e4, 1e-6, NULL) == 1
    assert st(lib, f, P, P, P, P, P, badp, 8, 8, 2, 128, 1e4, 1e-6, NULL) == 1
    assert "sum" in h3.last_error()
    assert st(lib, f, P, P, P, P, P, axp, 8, 8, 2, 96, 1e4, 1e-6, NULL) == 2
    assert st(lib, f, P, P, P, P, NULL, axp, 8, 8, 2, 128, 1e4, 1e-6, NULL) == 1
    f = "h3_mod_norm_residual"
    assert st(lib, f, P, NULL, NULL, NULL, NULL, NULL, 8, 8, 64, 1e-6, NULL) == 1  # nothing to do
    assert st(lib, f, P, P, NULL, NULL, NULL, NULL, 8, 8, 64, 1e-6, NULL) == 1     # no gate
    assert st(lib, f, P, NULL, NULL, P, NULL, P, 8, 8, 64, 1e-6, NULL) == 1        # no scale
    assert st(lib, f, P, P, P, NULL, NULL, NULL, 8, 8, 60, 1e-6, NULL) == 2
    assert st(lib, f, P, P, P, NULL, NULL, NULL, 8, 8, 8200, 1e-6, NULL) == 2
    assert st(lib, f, PM, P, P, NULL, NULL, NULL, 8, 8, 64, 1e-6, NULL) == 3


def test_linear_argument_errors(lib):
    assert st(lib, "h3_linear", P, P, P, 8, 8, 200, 64, NULL) == 2
    assert st(lib, "h3_linear", P, P, P, 8, 8, 256, 60, NULL) == 2
    assert st(lib, "h3_linear", P, P, PM, 8, 8, 256, 64, NULL) == 3
    assert st(lib, "h3_linear", P, P, P, 8, 9, 256, 64, NULL) == 1
    assert st(lib, "h3_linear_swiglu", P, P, P, 8, 8, 100, 64, NULL) == 2
    gain = ctypes.c_void_p(4096)
    ax = ctypes.cast((ctypes.c_int * 3)(32, 48, 48), ctypes.c_void_p)
    f = "h3_linear_qk_norm_rope"
    assert st(lib, f, P, P, P, gain, gain, P, ax, 0, 8, 8, 3, 64, 1e-6, NULL) == 2     # odd H
    assert st(lib, f, P, P, P, gain, gain, P, ax, 0, 8, 8, 2, 60, 1e-6, NULL) == 2     # K % 64
    assert st(lib, f, P, P, P, gain, gain, NULL, ax, 0, 8, 8, 2, 64, 1e-6, NULL) == 1  # no table
    assert st(lib, f, P, P, PM, gain, gain, P, ax, 0, 8, 8, 2, 64, 1e-6, NULL) == 3
    assert st(lib, f, P, P, P, gain, gain, P, ax, 0, 8, 8, 2, 64, -1.0, NULL) == 1     # eps < 0
    assert st(lib, f, P, P, P, gain, gain, P, ax, 2, 8, 8, 2, 64, 1e-6, NULL) == 1     # pairing
    # split-half pairs need every section a multiple of 16: 32/48/48 is, 40/40/48 is not
    ax40 = ctypes.cast((ctypes.c_int * 3)(40, 40, 48), ctypes.c_void_p)
    assert st(lib, f, P, P, P, gain, gain, P, ax40, 1, 8, 8, 2, 64, 1e-6, NULL) == 2
    f = "h3_qk_norm_rope_layout"
    assert st(lib, f, P, P, P, P, P, ax40, 8, 8, 2, 128, 1e4, 1e-6, 1, NULL) == 2
    assert st(lib, f, P, P, P, P, P, ax, 8, 8, 2, 128, 1e4, 1e-6, 3, NULL) == 1
    f = "h3_linear_residual"
    assert st(lib, f, P, P, P, P, 8, 8, 200, 64, NULL) == 2
    assert st(lib, f, P, P, P, NULL, 8, 8, 256, 64, NULL) == 1                 # no gate
    assert st(lib, f, P, P, PM, P, 8, 8, 256, 64, NULL) == 3
    assert st(lib, f, P, P, P, P, 8, 9, 256, 64, NULL) == 1                    # L > S


def test_rope_table_argument_errors(lib):
    f = "h3_rope_table"
    ax = (ctypes.c_int * 3)(32, 48, 48)
    bad = (ctypes.c_int * 3)(32, 48, 46)
    odd = (ctypes.c_int * 3)(33, 47, 48)
    A = lambda a: ctypes.cast(a, ctypes.c_void_p)
    assert st(lib, f, P, A(bad), 8, 8, 1e4, P, NULL) == 1
    assert st(lib, f, P, A(odd), 8, 8, 1e4, P, NULL) == 1
    assert st(lib, f, P, A(ax), 8, 8, 0.0, P, NULL) == 1
    assert st(lib, f, NULL, A(ax), 8, 8, 1e4, P, NULL) == 1
    assert st(lib, f, P, A(ax), 8, 8, 1e4, PM, NULL) == 3
    assert st(lib, f, P, A(ax), 8, 0, 1e4, P, NULL) == 0                      # L == 0: nothing


def test_block_config_and_workspace(lib):
    cfg = h3.block_config(256, 250, 512, 4, 128, 1536, (128, 0, 0))
    n = lib.h3_block_workspace_bytes(ctypes.byref(cfg))
    # h, attn, proj [S, D] + qkv [S, 3D] + ffn [S, F], bf16, and the RoPE
    # table [S, 64] (cos, sin) float32, 256-byte aligned slices
    assert n == 256 * 2 * (512 * 6 + 1536) + 256 * 64 * 8
    bad = h3.block_config(256, 250, 500, 4, 128, 1536, (128, 0, 0))
    assert lib.h3_block_workspace_bytes(ctypes.byref(bad)) == 0
    assert "D=" in h3.last_error()
    w = h3.BlockWeights(4096, 4096, 4096, 4096, 4096, 4096)
    f = lib.h3_block_forward
    assert f(ctypes.byref(cfg), ctypes.byref(w), P, P, P, P, n - 1, NULL) == 4
    assert f(ctypes.byref(cfg), ctypes.byref(w), P, P, P, NULL, n, NULL) == 4
    assert f(ctypes.byref(cfg), ctypes.byref(w), P, P, P, ctypes.c_void_p(4096 + 16), n, NULL) == 3
    assert f(ctypes.byref(cfg), None, P, P, P, P, n, NULL) == 1
    cfg0 = h3.block_config(256, 0, 512, 4, 128, 1536, (128, 0, 0))
    assert f(ctypes.byref(cfg0), ctypes.byref(w), P, P, P, P, n, NULL) == 0


def test_product_path_does_not_import_the_oracle():
    import sys
    import subprocess
    code = ("import sys; import dit_transformer_block_gb300.h3 as h; "
            "import dit_transformer_block_gb300.build; "
            "assert not any(m.startswith('oracle') for m in sys.modules), 'oracle imported'")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       cwd=str(__import__('pathlib').Path(__file__).resolve().parents[1]))
    assert r.returncode == 0, r.stderr


def test_stack_and_segmented_argument_errors(lib):
    cfg = h3.block_config(256, 250, 512, 4, 128, 1536, (128, 0, 0))
    n = lib.h3_block_workspace_bytes(ctypes.byref(cfg))
    w = (h3.BlockWeights * 2)(h3.BlockWeights(4096, 4096, 4096, 4096, 4096, 4096),
                              h3.BlockWeights(4096, 4096, 4096, 4096, 4096, 4096))
    f = lib.h3_stack_forward
    assert f(ctypes.byref(cfg), w, 0, P, P, 1, NULL, P, P, n, NULL) == 1      # no blocks
    assert f(ctypes.byref(cfg), w, 2, P, P, 2, NULL, P, P, n, NULL) == 1      # groups w/o seg
    assert f(ctypes.byref(cfg), w, 2, P, P, 0, P, P, P, n, NULL) == 1         # zero groups
    assert f(ctypes.byref(cfg), w, 2, P, P, 1, NULL, P, P, n - 1, NULL) == 4  # workspace
    w[1].w_o = None
    assert f(ctypes.byref(cfg), w, 2, P, P, 1, NULL, P, P, n, NULL) == 1      # NULL weight
    g = lib.h3_mod_norm_residual_seg
    assert g(P, P, P, NULL, NULL, NULL, 2, 512, NULL, 8, 8, 64, 1e-6, NULL) == 1  # no seg
    assert g(P, P, P, NULL, NULL, P, 2, 32, NULL, 8, 8, 64, 1e-6, NULL) == 1    # stride < D
    assert g(P, P, P, NULL, NULL, P, 2, 66, NULL, 8, 8, 64, 1e-6, NULL) == 3    # stride % 4
    assert g(P, P, P, NULL, NULL, P, 0, 512, NULL, 8, 8, 64, 1e-6, NULL) == 1   # no groups


def test_stage_tables_agree_with_the_header():
    # the binding's stage count and names, the bench's per-stage work model and
    # the header's H3_BLOCK_STAGES describe the same stages
    import re
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hdr = open(os.path.join(root, "include", "h3block.h")).read()
    n = int(re.search(r"#define H3_BLOCK_STAGES (\d+)", hdr).group(1))
    assert h3.BLOCK_STAGES == n == len(h3.STAGE_NAMES)
    work = bench.stage_work(58816, 58758, 5376, 42, 128, 14336)
    assert len(work) == n
    # the tensor-bound stages carry the GEMM and attention FLOPs exactly
    bw = bench.block_work(58816, 58758, 5376, 42, 128, 14336)
    tensor = sum(w for b, w, _ in work if b == "tensor")
    assert abs(tensor - (bw["gemm_flop"] + bw["attn_flop"])) < 1e-6 * tensor


def test_recorded_traffic_hash_ignores_comments():
    import bench
    code = "int f() {\n  return 1;  // one\n}\n"
    assert bench.code_sha256(code) == bench.code_sha256("// header\nint f() {\n\n  return 1;\n}")
    assert bench.code_sha256(code) != bench.code_sha256("int f() {\n  return 2;\n}\n")


def test_binding_argument_counts_match_the_header():
    # every prototype's parameter count equals the ctypes signature's, so a
    # header change that the binding missed fails here rather than on a GPU
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "h3block.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = {}
    for m in re.finditer(r"(h3_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        args = m.group(2).strip()
        n = 0 if args in ("", "void") else len([a for a in args.split(",") if a.strip()])
        protos[m.group(1)] = n
    assert set(protos) == set(h3._SIGS)
    for name, (_, argtypes) in h3._SIGS.items():
        assert len(argtypes) == protos[name], (name, len(argtypes), protos[name])


def test_noalloc_scratch_size_matches_the_header():
    # the binding's NOALLOC_SCRATCH_BYTES is the header's H3_NOALLOC_SCRATCH_BYTES
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hdr = open(os.path.join(root, "include", "h3block.h")).read()
    m = re.search(r"#define H3_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", hdr)
    assert m, "H3_NOALLOC_SCRATCH_BYTES not found in the header"
    assert h3.NOALLOC_SCRATCH_BYTES == int(m.group(1)) * int(m.group(2)) * int(m.group(3))
