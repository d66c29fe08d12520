"""ctypes binding of libh3block.so (argument marshalling only).

Every function takes torch tensors that already live on the current CUDA
device, passes their data pointers and sizes to the C entry point of the same
name (h3_<name>) and raises H3Error when the call returns a non-OK status.
All compute happens in the library's kernels; there is no fallback: if the
library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libh3block.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "h3block.h")

H3_OK = 0
STATUS = {0: "H3_OK", 1: "H3_ERR_INVALID_ARG", 2: "H3_ERR_UNSUPPORTED", 3: "H3_ERR_MISALIGNED",
          4: "H3_ERR_WORKSPACE", 5: "H3_ERR_CUDA", 6: "H3_ERR_TIMEOUT"}


class H3Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"h3_{fn}: {STATUS.get(status, status)}: {msg}")
        self.status = status
        self.msg = msg


class BlockConfig(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int), ("L", ctypes.c_int), ("D", ctypes.c_int), ("H", ctypes.c_int),
                ("Dh", ctypes.c_int), ("F", ctypes.c_int), ("axis_dims", ctypes.c_int * 3),
                ("theta", ctypes.c_float), ("eps_ln", ctypes.c_float), ("eps_qk", ctypes.c_float),
                ("rope_pairing", ctypes.c_int)]


class BlockWeightsFp8(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("s_qkv", ctypes.c_void_p),
                ("w_o", ctypes.c_void_p), ("s_o", ctypes.c_void_p),
                ("w_gu", ctypes.c_void_p), ("s_gu", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("q_gain", ctypes.c_void_p), ("k_gain", ctypes.c_void_p)]


class BlockWeights(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("w_gu", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("q_gain", ctypes.c_void_p),
                ("k_gain", ctypes.c_void_p)]


_P, _I, _F, _U64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
_SIGS = {
    "h3_version": (_I, []),
    "h3_last_error": (ctypes.c_char_p, []),
    "h3_status_string": (ctypes.c_char_p, [_I]),
    "h3_check_device_error": (_I, [_P]),
    "h3_set_wait_timeout_ns": (None, [_U64]),
    "h3_mod_norm_residual": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _F, _P]),
    "h3_qk_norm_rope": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _F, _P]),
    "h3_attention_varlen": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _F, _P]),
    "h3_swiglu": (_I, [_P, _P, _I, _I, _I, _P]),
    "h3_sage_scratch_bytes": (_SZ, [_I, _I]),
    "h3_sage_quantize": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                              _P]),
    "h3_attention_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P]),
    "h3_attention_fp8_skip": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _F, _P, _P]),
    "h3_attention_varlen_skip": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _F, _F, _P, _P]),
    "h3_linear": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "h3_linear_swiglu": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "h3_rope_table": (_I, [_P, _P, _I, _I, _F, _P, _P]),
    "h3_linear_qk_norm_rope": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "h3_qk_norm_rope_layout": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _F, _I, _P]),
    "h3_linear_residual": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "h3_block_workspace_bytes": (_SZ, [ctypes.POINTER(BlockConfig)]),
    "h3_block_forward": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights), _P, _P,
                              _P, _P, _SZ, _P]),
    "h3_block_forward_events": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights),
                                     _P, _P, _P, _P, _SZ, _P, ctypes.POINTER(_P), _I]),
    "h3_block_forward_noalloc": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights),
                                      _P, _P, _P, _P]),
    "h3_debug_wait_timeout": (_I, [_U64, _P]),
    "h3_mod_norm_residual_seg": (_I, [_P, _P, _P, _P, _P, _P, _I, ctypes.c_int64, _P, _I, _I, _I,
                                      _F, _P]),
    "h3_frames_to_u8": (_I, [_P, _P, _I, _I, _I, _I, _I, _P]),
    "h3_quantize_fp8_rows": (_I, [_P, _P, _P, _I, _I, _P]),
    "h3_linear_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "h3_linear_swiglu_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "h3_block_workspace_bytes_fp8": (_SZ, [ctypes.POINTER(BlockConfig)]),
    "h3_block_forward_fp8": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeightsFp8),
                                  _P, _P, _P, _I, _P, _SZ, _P]),
    "h3_stack_forward": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights), _I, _P,
                              _P, _I, _P, _P, _P, _SZ, _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libh3block.so (built by dit_transformer_block_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m "
                               "dit_transformer_block_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/h3block.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_0-9]+\*?\s+\*?(h3_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def last_error() -> str:
    return lib().h3_last_error().decode()


def _check(fn: str, status: int):
    if status != H3_OK:
        raise H3Error(fn, status, last_error())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def version() -> int:
    return lib().h3_version()


def set_wait_timeout_ns(ns: int):
    lib().h3_set_wait_timeout_ns(int(ns))


def check_device_error(stream=None):
    _check("check_device_error", lib().h3_check_device_error(_s(stream)))


def debug_wait_timeout(ns: int, stream=None):
    _check("debug_wait_timeout", lib().h3_debug_wait_timeout(int(ns), _s(stream)))


def mod_norm_residual(resid, delta=None, gate=None, shift=None, scale=None, normed=None, L=None,
                      eps=1e-6, stream=None):
    """resid [S,D] f32 in/out; optional delta [S,D] bf16 + gate [D]; optional normed [S,D] bf16."""
    _need(resid, torch.float32, "resid")
    _need(delta, torch.bfloat16, "delta")
    _need(normed, torch.bfloat16, "normed")
    S, D = resid.shape
    L = S if L is None else L
    _check("mod_norm_residual", lib().h3_mod_norm_residual(
        _p(resid), _p(delta), _p(gate), _p(shift), _p(scale), _p(normed), S, L, D, eps, _s(stream)))


def mod_norm_residual_seg(resid, table, seg, delta=None, gate_idx=None, shift_idx=None,
                          scale_idx=None, normed=None, L=None, eps=1e-6, stream=None):
    """mod_norm_residual with token-group modulation: table [G, 6, D] f32,
    seg [S] int32; row i uses table[seg[i], idx] for the gate/shift/scale
    indices given (0..5), e.g. gate_idx=2, shift_idx=3, scale_idx=4."""
    _need(resid, torch.float32, "resid")
    _need(table, torch.float32, "table")
    _need(seg, torch.int32, "seg")
    S, D = resid.shape
    G = table.shape[0]
    L = S if L is None else L
    row = lambda i: None if i is None else ctypes.c_void_p(table[0, i].data_ptr())
    _check("mod_norm_residual_seg", lib().h3_mod_norm_residual_seg(
        _p(resid), _p(delta), row(gate_idx), row(shift_idx), row(scale_idx), _p(seg), G, 6 * D,
        _p(normed), S, L, D, eps, _s(stream)))


def qk_norm_rope(q, k, q_gain, k_gain, pos, axis_dims, L=None, theta=1e4, eps=1e-6, stream=None,
                 pairing=0):
    """In-place per-head RMSNorm + RoPE of q, k [S,H,Dh] bf16 (pairing 0:
    interleaved pairs, 1: split-half pairs per section)."""
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(pos, torch.int32, "pos")
    S, H, Dh = q.shape
    L = S if L is None else L
    ax = ctypes.cast((ctypes.c_int * 3)(*axis_dims), ctypes.c_void_p)
    if pairing == 0:
        _check("qk_norm_rope", lib().h3_qk_norm_rope(
            _p(q), _p(k), _p(q_gain), _p(k_gain), _p(pos), ax, S, L, H, Dh, theta, eps,
            _s(stream)))
    else:
        _check("qk_norm_rope_layout", lib().h3_qk_norm_rope_layout(
            _p(q), _p(k), _p(q_gain), _p(k_gain), _p(pos), ax, S, L, H, Dh, theta, eps, pairing,
            _s(stream)))


def attention_varlen(q, k, v, o, L=None, scale=None, stream=None):
    """o[:L] = softmax(q k^T * scale) v over keys < L; all [S,H,Dh] bf16."""
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need(t, torch.bfloat16, n)
    S, H, Dh = q.shape
    L = S if L is None else L
    scale = Dh ** -0.5 if scale is None else scale
    _check("attention_varlen", lib().h3_attention_varlen(
        _p(q), _p(k), _p(v), _p(o), S, L, H, Dh, scale, _s(stream)))


def attention_varlen_skip(q, k, v, o, L=None, scale=None, skip_eps=0.0, kept=None, stream=None):
    """attention_varlen with Skip-Softmax tile skipping (skip_eps = 0: dense).
    kept (optional): int32 [ceil(L/128), H], receives the key tiles kept per
    (query tile, head)."""
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need(t, torch.bfloat16, n)
    S, H, Dh = q.shape
    L = S if L is None else L
    scale = Dh ** -0.5 if scale is None else scale
    if kept is not None:
        _need(kept, torch.int32, "kept")
        if tuple(kept.shape) != ((L + 127) // 128, H):
            raise ValueError(f"kept must be [{(L + 127) // 128}, {H}]")
    _check("attention_varlen_skip", lib().h3_attention_varlen_skip(
        _p(q), _p(k), _p(v), _p(o), S, L, H, Dh, scale, skip_eps, _p(kept), _s(stream)))


def sage_quantize(q, k, v, L=None, stream=None) -> dict:
    """FP8 operands for attention_fp8 (allocated here, from torch): codes qc,
    kc, vc (uint8 [S, H, Dh]), scales sq, sk ([ceil(L/128), H]), sv and
    k_mean ([H, Dh])."""
    S, H, Dh = q.shape
    L = S if L is None else L
    dev = q.device
    nt = max(1, (L + 127) // 128)
    out = dict(qc=torch.zeros(S, H, Dh, dtype=torch.uint8, device=dev),
               kc=torch.zeros(S, H, Dh, dtype=torch.uint8, device=dev),
               vc=torch.zeros(S, H, Dh, dtype=torch.uint8, device=dev),
               sq=torch.zeros(nt, H, device=dev), sk=torch.zeros(nt, H, device=dev),
               sv=torch.zeros(H, Dh, device=dev), k_mean=torch.zeros(H, Dh, device=dev))
    nbytes = lib().h3_sage_scratch_bytes(L, H)
    scratch = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _check("sage_quantize", lib().h3_sage_quantize(
        _p(q), _p(k), _p(v), S, L, H, Dh, _p(out["qc"]), _p(out["kc"]), _p(out["vc"]),
        _p(out["sq"]), _p(out["sk"]), _p(out["sv"]), _p(out["k_mean"]), _p(scratch), nbytes,
        _s(stream)))
    return out


def attention_fp8(ops: dict, o, L=None, scale=None, stream=None):
    """FP8 attention on sage_quantize's operands into o [S, H, Dh] bf16."""
    S, H, Dh = o.shape
    L = S if L is None else L
    scale = Dh ** -0.5 if scale is None else scale
    _check("attention_fp8", lib().h3_attention_fp8(
        _p(ops["qc"]), _p(ops["kc"]), _p(ops["vc"]), _p(ops["sq"]), _p(ops["sk"]),
        _p(ops["sv"]), _p(o), S, L, H, Dh, scale, _s(stream)))


def attention_fp8_skip(ops: dict, o, L=None, scale=None, skip_eps=0.0, kept=None, stream=None):
    """attention_fp8 with Skip-Softmax tile skipping on the FP8 logits
    (skip_eps = 0: attention_fp8 bit for bit). kept (optional): int32
    [ceil(L/128), H], receives the key tiles kept per (query tile, head)."""
    S, H, Dh = o.shape
    L = S if L is None else L
    scale = Dh ** -0.5 if scale is None else scale
    if kept is not None:
        _need(kept, torch.int32, "kept")
        if tuple(kept.shape) != ((L + 127) // 128, H):
            raise ValueError(f"kept must be [{(L + 127) // 128}, {H}]")
    _check("attention_fp8_skip", lib().h3_attention_fp8_skip(
        _p(ops["qc"]), _p(ops["kc"]), _p(ops["vc"]), _p(ops["sq"]), _p(ops["sk"]),
        _p(ops["sv"]), _p(o), S, L, H, Dh, scale, skip_eps, _p(kept), _s(stream)))


def swiglu(gate_up, out, L=None, stream=None):
    _need(gate_up, torch.bfloat16, "gate_up")
    _need(out, torch.bfloat16, "out")
    S, F = out.shape
    L = S if L is None else L
    _check("swiglu", lib().h3_swiglu(_p(gate_up), _p(out), S, L, F, _s(stream)))


def linear(x, w, y, L=None, stream=None):
    """y[:L] = x[:L] @ w^T; x [S,K], w [N,K], y [S,N] bf16."""
    for n, t in (("x", x), ("w", w), ("y", y)):
        _need(t, torch.bfloat16, n)
    S, K = x.shape
    N = w.shape[0]
    L = S if L is None else L
    _check("linear", lib().h3_linear(_p(x), _p(w), _p(y), S, L, N, K, _s(stream)))


def linear_swiglu(x, w_gu, out, L=None, stream=None):
    """out[:L] = SiLU(x w_g^T) * (x w_u^T); w_gu [2F,K] rows [gate | up]."""
    for n, t in (("x", x), ("w_gu", w_gu), ("out", out)):
        _need(t, torch.bfloat16, n)
    S, K = x.shape
    F = out.shape[1]
    L = S if L is None else L
    _check("linear_swiglu", lib().h3_linear_swiglu(_p(x), _p(w_gu), _p(out), S, L, F, K,
                                                    _s(stream)))


def rope_table(pos, axis_dims, table, L=None, theta=1e4, stream=None):
    """table[:L] = (cos, sin) of every RoPE angle; pos [S,3] int32, table [S,64,2] f32."""
    _need(pos, torch.int32, "pos")
    _need(table, torch.float32, "table")
    S = pos.shape[0]
    L = S if L is None else L
    ax = (ctypes.c_int * 3)(*axis_dims)
    _check("rope_table", lib().h3_rope_table(_p(pos), ctypes.cast(ax, ctypes.c_void_p), S, L,
                                              theta, _p(table), _s(stream)))


def linear_qk_norm_rope(x, w_qkv, qkv, q_gain, k_gain, table, axis_dims, L=None, eps=1e-6,
                        pairing=0, stream=None):
    """qkv[:L] = x @ w_qkv^T with per-head Q/K RMSNorm + RoPE (table from
    rope_table, sections axis_dims, pairing as qk_norm_rope) in the epilogue;
    x [S,K], w_qkv [3D,K], qkv [S,3D] bf16."""
    for n, t in (("x", x), ("w_qkv", w_qkv), ("qkv", qkv)):
        _need(t, torch.bfloat16, n)
    S, K = x.shape
    H = w_qkv.shape[0] // 3 // 128
    L = S if L is None else L
    ax = ctypes.cast((ctypes.c_int * 3)(*axis_dims), ctypes.c_void_p)
    _check("linear_qk_norm_rope", lib().h3_linear_qk_norm_rope(
        _p(x), _p(w_qkv), _p(qkv), _p(q_gain), _p(k_gain), _p(table), ax, pairing, S, L, H, K,
        eps, _s(stream)))


def linear_residual(x, w, resid, gate, L=None, stream=None):
    """resid[:L] += gate * bf16(x @ w^T) in FP32; x [S,K], w [N,K] bf16, resid [S,N] f32."""
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w")
    _need(resid, torch.float32, "resid")
    S, K = x.shape
    N = w.shape[0]
    L = S if L is None else L
    _check("linear_residual", lib().h3_linear_residual(_p(x), _p(w), _p(resid), _p(gate), S, L,
                                                        N, K, _s(stream)))


def block_config(S, L, D, H, Dh, F, axis_dims, theta=1e4, eps_ln=1e-6, eps_qk=1e-6,
                 rope_pairing=0) -> BlockConfig:
    return BlockConfig(S, L, D, H, Dh, F, (ctypes.c_int * 3)(*axis_dims), theta, eps_ln, eps_qk,
                       rope_pairing)


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def block_forward_noalloc(cfg: BlockConfig, weights, resid, mod, pos, stream=None):
    """h3_block_forward_noalloc: the block forward with the library's own
    fixed scratch array instead of a caller workspace, for callers that cannot
    allocate device memory (blocks up to NOALLOC_SCRATCH_BYTES of workspace)."""
    w = weights if isinstance(weights, BlockWeights) else block_weights(weights)
    _check("block_forward_noalloc", lib().h3_block_forward_noalloc(
        ctypes.byref(cfg), ctypes.byref(w), _p(resid), _p(mod), _p(pos), _s(stream)))


def stack_forward(cfg: BlockConfig, weights_list, resid, mods, pos, workspace, seg=None,
                  stream=None):
    """Blocks applied in order: weights_list[b] (dict or BlockWeights) with
    mods [num_blocks, G, 6, D] f32 (or [num_blocks, 6, D] when seg is None);
    seg [S] int32 picks each row's group."""
    n = len(weights_list)
    arr = (BlockWeights * n)(*(w if isinstance(w, BlockWeights) else block_weights(w)
                               for w in weights_list))
    G = 1 if mods.dim() == 3 else mods.shape[1]
    _need(mods, torch.float32, "mods")
    _check("stack_forward", lib().h3_stack_forward(
        ctypes.byref(cfg), arr, n, _p(resid), _p(mods), G, _p(seg), _p(pos), _p(workspace),
        workspace.numel() * workspace.element_size(), _s(stream)))


def frames_to_u8(frames, out, stream=None):
    """frames [B, C, T, H, W] f32 -> out [B, T, H, W, C] uint8."""
    _need(frames, torch.float32, "frames")
    _need(out, torch.uint8, "out")
    B, C, T, H, W = frames.shape
    _check("frames_to_u8", lib().h3_frames_to_u8(_p(frames), _p(out), B, C, T, H, W,
                                                  _s(stream)))


def quantize_fp8_rows(x, q, scale, stream=None):
    """x [R, K] bf16 -> q [R, K] uint8 (E4M3 codes), scale [R] f32."""
    _need(x, torch.bfloat16, "x")
    _need(q, torch.uint8, "q")
    _need(scale, torch.float32, "scale")
    R, K = x.shape
    _check("quantize_fp8_rows", lib().h3_quantize_fp8_rows(_p(x), _p(q), _p(scale), R, K,
                                                            _s(stream)))


def linear_fp8(qx, sx, qw, sw, y, L=None, stream=None):
    S, K = qx.shape
    N = qw.shape[0]
    L = S if L is None else L
    _check("linear_fp8", lib().h3_linear_fp8(_p(qx), _p(sx), _p(qw), _p(sw), _p(y), S, L, N, K,
                                              _s(stream)))


def linear_swiglu_fp8(qx, sx, qw_gu, sw_gu, out, L=None, stream=None):
    S, K = qx.shape
    F = out.shape[1]
    L = S if L is None else L
    _check("linear_swiglu_fp8", lib().h3_linear_swiglu_fp8(
        _p(qx), _p(sx), _p(qw_gu), _p(sw_gu), _p(out), S, L, F, K, _s(stream)))


def quantize_block_weights_fp8(weights: dict, stream=None) -> dict:
    """Load-time FP8 quantisation of a block's four projection weights:
    returns a dict with codes (uint8) and per-row scales for each, plus the
    Q/K gains, ready for block_forward_fp8."""
    out = {"q_gain": weights["q_gain"], "k_gain": weights["k_gain"]}
    for k in ("w_qkv", "w_o", "w_gu", "w_down"):
        w = weights[k]
        q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
        sc = torch.empty(w.shape[0], dtype=torch.float32, device=w.device)
        quantize_fp8_rows(w, q, sc, stream)
        out[k] = q
        out["s_" + k[2:]] = sc
    return out


def block_weights_fp8(w: dict) -> BlockWeightsFp8:
    return BlockWeightsFp8(*(w[k].data_ptr() for k in (
        "w_qkv", "s_qkv", "w_o", "s_o", "w_gu", "s_gu", "w_down", "s_down", "q_gain", "k_gain")))


def block_workspace_bytes_fp8(cfg: BlockConfig) -> int:
    n = lib().h3_block_workspace_bytes_fp8(ctypes.byref(cfg))
    if n == 0:
        raise H3Error("block_workspace_bytes_fp8", 1, last_error())
    return n


def block_forward_fp8(cfg: BlockConfig, weights_fp8, resid, mod, pos, workspace, stream=None,
                      fp8_attention=False):
    w = weights_fp8 if isinstance(weights_fp8, BlockWeightsFp8) else block_weights_fp8(weights_fp8)
    _check("block_forward_fp8", lib().h3_block_forward_fp8(
        ctypes.byref(cfg), ctypes.byref(w), _p(resid), _p(mod), _p(pos), int(fp8_attention),
        _p(workspace), workspace.numel() * workspace.element_size(), _s(stream)))


def block_workspace_bytes(cfg: BlockConfig) -> int:
    n = lib().h3_block_workspace_bytes(ctypes.byref(cfg))
    if n == 0:
        raise H3Error("block_workspace_bytes", 1, last_error())
    return n


BLOCK_STAGES = 7
STAGE_NAMES = ("mod_norm", "qkv_proj_qk_norm_rope", "attention", "out_proj",
               "residual_mod_norm", "gate_up_swiglu", "down_proj_residual")
# kernels one block launches: one per stage
BLOCK_LAUNCHES = BLOCK_STAGES


def block_weights(weights: dict) -> BlockWeights:
    return BlockWeights(*(weights[k].data_ptr() for k in
                          ("w_qkv", "w_o", "w_gu", "w_down", "q_gain", "k_gain")))


def block_forward(cfg: BlockConfig, weights, resid, mod, pos, workspace, stream=None,
                  events=None):
    """One block forward, in place on resid [S,D] f32. weights: dict with
    w_qkv, w_o, w_gu, w_down (bf16) and q_gain, k_gain (f32), or a prepared
    BlockWeights; workspace: uint8 device tensor. events: optional list of
    BLOCK_STAGES + 1 recorded-once torch.cuda.Event, marked before each stage."""
    w = weights if isinstance(weights, BlockWeights) else block_weights(weights)
    nbytes = workspace.numel() * workspace.element_size()
    if events is None:
        _check("block_forward", lib().h3_block_forward(
            ctypes.byref(cfg), ctypes.byref(w), _p(resid), _p(mod), _p(pos), _p(workspace),
            nbytes, _s(stream)))
        return
    arr = (_P * len(events))(*(e.cuda_event for e in events))
    _check("block_forward_events", lib().h3_block_forward_events(
        ctypes.byref(cfg), ctypes.byref(w), _p(resid), _p(mod), _p(pos), _p(workspace), nbytes,
        _s(stream), arr, len(events)))
