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
                ("theta", ctypes.c_float), ("eps_ln", ctypes.c_float), ("eps_qk", ctypes.c_float)]


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
    "h3_linear": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "h3_linear_swiglu": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "h3_block_workspace_bytes": (_SZ, [ctypes.POINTER(BlockConfig)]),
    "h3_block_forward": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights), _P, _P,
                              _P, _P, _SZ, _P]),
    "h3_block_forward_events": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights),
                                     _P, _P, _P, _P, _SZ, _P, ctypes.POINTER(_P), _I]),
    "h3_block_forward_noalloc": (_I, [ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights),
                                      _P, _P, _P, _P]),
    "h3_debug_wait_timeout": (_I, [_U64, _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libh3block.so (built by dit_transformer_block_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m "
                               "dit_transformer_block_gb300.build` or __graft_entry__.build()")
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


def qk_norm_rope(q, k, q_gain, k_gain, pos, axis_dims, L=None, theta=1e4, eps=1e-6, stream=None):
    """In-place per-head RMSNorm + RoPE of q, k [S,H,Dh] bf16."""
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(pos, torch.int32, "pos")
    S, H, Dh = q.shape
    L = S if L is None else L
    ax = (ctypes.c_int * 3)(*axis_dims)
    _check("qk_norm_rope", lib().h3_qk_norm_rope(
        _p(q), _p(k), _p(q_gain), _p(k_gain), _p(pos), ctypes.cast(ax, ctypes.c_void_p), S, L, H,
        Dh, theta, eps, _s(stream)))


def attention_varlen(q, k, v, o, L=None, scale=None, stream=None):
    """o[:L] = softmax(q k^T * scale) v over keys < L; all [S,H,Dh] bf16."""
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need(t, torch.bfloat16, n)
    S, H, Dh = q.shape
    L = S if L is None else L
    scale = Dh ** -0.5 if scale is None else scale
    _check("attention_varlen", lib().h3_attention_varlen(
        _p(q), _p(k), _p(v), _p(o), S, L, H, Dh, scale, _s(stream)))


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


def block_config(S, L, D, H, Dh, F, axis_dims, theta=1e4, eps_ln=1e-6, eps_qk=1e-6) -> BlockConfig:
    return BlockConfig(S, L, D, H, Dh, F, (ctypes.c_int * 3)(*axis_dims), theta, eps_ln, eps_qk)


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def block_forward_noalloc(cfg: BlockConfig, weights, resid, mod, pos, stream=None):
    """h3_block_forward_noalloc: the block forward with the library's own
    fixed scratch array instead of a caller workspace, for callers that cannot
    allocate device memory (blocks up to NOALLOC_SCRATCH_BYTES of workspace)."""
    w = weights if isinstance(weights, BlockWeights) else block_weights(weights)
    _check("block_forward_noalloc", lib().h3_block_forward_noalloc(
        ctypes.byref(cfg), ctypes.byref(w), _p(resid), _p(mod), _p(pos), _s(stream)))


def block_workspace_bytes(cfg: BlockConfig) -> int:
    n = lib().h3_block_workspace_bytes(ctypes.byref(cfg))
    if n == 0:
        raise H3Error("block_workspace_bytes", 1, last_error())
    return n


BLOCK_STAGES = 9
STAGE_NAMES = ("mod_norm", "qkv_proj", "qk_norm_rope", "attention", "out_proj",
               "residual_mod_norm", "gate_up_swiglu", "down_proj", "residual")


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
