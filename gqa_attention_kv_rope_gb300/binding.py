"""Thin Python binding over libminf.so: argument marshalling only.

Every function has the C ABI's name and argument order (include/minf.h), takes
torch CUDA tensors in place of device pointers, and raises MinfError on a
non-zero status.  All arithmetic runs in the library's kernels; there is no
CPU path.  If the library is missing, the first call raises -- nothing falls
back to another implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

MINF_OK = 0
MINF_ERR_ARG = 1
MINF_ERR_GEOMETRY = 2
MINF_ERR_UNSUPPORTED = 3
MINF_ERR_WORKSPACE = 5
MINF_ERR_CUDA = 6
ERRBIT_STORE_POS = 0x1
ERRBIT_ROPE_POS = 0x2
ERRBIT_ATTN_POS = 0x4
ERRBIT_TIMEOUT = 0x8
ERRBIT_BLOCK = 0x10
ERRBIT_WORKSPACE = 0x20

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_I64 = ctypes.c_int64

_SIGS = {
    "minf_status_string": ([_I], ctypes.c_char_p),
    "minf_version": ([], _I),
    "minf_rope_freqs": ([_P, _I, _F, _F], _I),
    "minf_rms_norm": ([_P, _P, _P, _I, _I, _F, _P], _I),
    "minf_rope": ([_P, _P, _I, _I, _I, _F, _F, _I, _P, _P], _I),
    "minf_kv_append": ([_P, _P, _I, _I, _P, _P, _P, _I, _P, _P], _I),
    "minf_rope_kv_append": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _I, _P, _P], _I),
    "minf_attn_decode_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "minf_attn_prefill_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "minf_gqa_attn_decode": ([_P, _P, _P, _P, _P, _P, _I, _I64, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P], _I),
    "minf_gqa_attn_decode_static_ws": ([_P, _P, _P, _P, _P, _P, _I, _I64, _P, _I, _I, _I, _I, _I, _F, _P, _P], _I),
    "minf_gqa_attn_prefill": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                              _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    # the same step with early start (the launch before writes neither pos nor cached rows)
    "minf_layer_attn_step_chained": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                      _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_chained_f16": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                          _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_chained_q8": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                         _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_batched": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I64,
                                      _I, _I, _I, _I, _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_silu_mul": ([_P, _P, _P, _I64, _P], _I),
    # binary16 regions (torch.float16 tensors): the same arguments as the fp32 entry points
    "minf_kv_append_f16": ([_P, _P, _I, _I, _P, _P, _P, _I, _P, _P], _I),
    "minf_rope_kv_append_f16": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _I, _P, _P], _I),
    "minf_gqa_attn_decode_f16": ([_P, _P, _P, _P, _P, _P, _I, _I64, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P,
                                  _P], _I),
    "minf_gqa_attn_prefill_f16": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_f16": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                  _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_batched_f16": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I64,
                                          _I, _I, _I, _I, _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    # Q8_0 regions (torch.uint8 tensors of rows of minf_q8_row_bytes(W) bytes)
    "minf_q8_row_bytes": ([_I], _SZ),
    "minf_kv_append_q8": ([_P, _P, _I, _I, _P, _P, _P, _I, _P, _P], _I),
    "minf_rope_kv_append_q8": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _I, _P, _P], _I),
    "minf_gqa_attn_decode_q8": ([_P, _P, _P, _P, _P, _P, _I, _I64, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P],
                                _I),
    "minf_gqa_attn_prefill_q8": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_q8": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                 _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_batched_q8": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I64,
                                         _I, _I, _I, _I, _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_kv_append_paged_q8": ([_P, _P, _I64, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P], _I),
    "minf_gqa_attn_decode_paged_q8": ([_P, _P, _P, _P, _I64, _P, _I, _I, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P,
                                       _P], _I),
    "minf_layer_attn_step_paged_q8": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I64, _P, _I, _I, _I, _I,
                                       _I, _I, _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    # the fused QKV decode op
    "minf_fused_qkv": ([_P, _P, _P, _F, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _I, _P,
                        _P], _I),
    "minf_layer_attn_step_qkv": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F,
                                  _I, _P, _P, _SZ, _P, _P], _I),
    # paged regions: a pool of blocks and a block table per sequence
    "minf_kv_append_paged": ([_P, _P, _I64, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P], _I),
    "minf_kv_append_paged_f16": ([_P, _P, _I64, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P], _I),
    "minf_gqa_attn_decode_paged": ([_P, _P, _P, _P, _I64, _P, _I, _I, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P],
                                   _I),
    "minf_gqa_attn_decode_paged_f16": ([_P, _P, _P, _P, _I64, _P, _I, _I, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P,
                                        _P], _I),
    "minf_layer_attn_step_paged": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I64, _P, _I, _I, _I, _I, _I,
                                    _I, _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
    "minf_layer_attn_step_paged_f16": ([_P, _P, _P, _F, _I, _P, _P, _P, _P, _I, _P, _P, _I64, _P, _I, _I, _I, _I,
                                        _I, _I, _F, _F, _I, _P, _P, _SZ, _P, _P], _I),
}


class MinfError(RuntimeError):
    def __init__(self, status: int, name: str):
        msg = lib().minf_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{name}: status {status} ({msg})")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded library (ctypes).  Raises if libminf.so has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libminf.so is not built ({path}); run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'` first")
            handle = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def _check(status: int, name: str):
    if status != MINF_OK:
        raise MinfError(status, name)


def _dev(t, dtype=torch.float32, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def minf_rope_freqs(hd: int, theta: float, freq_scale: float = 1.0) -> list[float]:
    import array

    buf = (ctypes.c_float * max(hd // 2, 1))()
    _check(lib().minf_rope_freqs(ctypes.cast(buf, _P), hd, theta, freq_scale), "minf_rope_freqs")
    return array.array("f", buf[: hd // 2])


def minf_rms_norm(y, x, w, eps: float, stream=None):
    rows, n = x.shape
    _check(lib().minf_rms_norm(_dev(y, name="y"), _dev(x, name="x"), _dev(w, name="w"), rows, n, eps,
                               _stream(stream)), "minf_rms_norm")


def minf_rope(x, pos, n_head: int, hd: int, theta: float, freq_scale: float, style: int, err,
              stream=None):
    nt = pos.numel()
    _check(lib().minf_rope(_dev(x, name="x"), _dev(pos, torch.int32, "pos"), nt, n_head, hd, theta,
                           freq_scale, style, _dev(err, torch.int32, "err"), _stream(stream)),
           "minf_rope")


def minf_kv_append(k_reg, v_reg, k_rows, v_rows, pos, err, stream=None):
    cap, W = k_reg.shape
    _check(lib().minf_kv_append(_dev(k_reg, name="k_reg"), _dev(v_reg, name="v_reg"), cap, W,
                                _dev(k_rows, name="k_rows"), _dev(v_rows, name="v_rows"),
                                _dev(pos, torch.int32, "pos"), pos.numel(),
                                _dev(err, torch.int32, "err"), _stream(stream)), "minf_kv_append")


def minf_rope_kv_append(q, k, v, pos, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, k_reg,
                        v_reg, err, stream=None):
    cap = k_reg.shape[0]
    _check(lib().minf_rope_kv_append(_dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"),
                                     _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head,
                                     hd, hd_kv, theta, freq_scale, style, _dev(k_reg, name="k_reg"),
                                     _dev(v_reg, name="v_reg"), cap, _dev(err, torch.int32, "err"),
                                     _stream(stream)), "minf_rope_kv_append")


def minf_attn_decode_workspace_bytes(n_seq, n_head, n_kv_head, hd_kv, max_cap) -> int:
    return int(lib().minf_attn_decode_workspace_bytes(n_seq, n_head, n_kv_head, hd_kv, max_cap))


def minf_attn_prefill_workspace_bytes(nt, n_head, n_kv_head, hd_kv, cap) -> int:
    return int(lib().minf_attn_prefill_workspace_bytes(nt, n_head, n_kv_head, hd_kv, cap))


def minf_gqa_attn_decode(out, q, k_reg, v_reg, seq_row_off, seq_cap, max_cap, pos, n_head, n_kv_head,
                         hd, hd_kv, scale, ws, err, stream=None):
    """k_reg/v_reg: the [rows, W] arena (or one sequence's [cap, W] regions)."""
    _check(lib().minf_gqa_attn_decode(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_reg, name="k_reg"), _dev(v_reg, name="v_reg"),
        _dev(seq_row_off, torch.int64, "seq_row_off"), _dev(seq_cap, torch.int32, "seq_cap"), max_cap,
        k_reg.shape[0], _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv, scale,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_gqa_attn_decode")


def minf_gqa_attn_decode_static_ws(out, q, k_reg, v_reg, seq_row_off, seq_cap, max_cap, pos, n_head,
                                   n_kv_head, hd, hd_kv, scale, err, stream=None):
    """minf_gqa_attn_decode for callers that cannot allocate: the library's own fixed device
    scratch replaces the workspace argument (see include/minf.h for its limits)."""
    _check(lib().minf_gqa_attn_decode_static_ws(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_reg, name="k_reg"), _dev(v_reg, name="v_reg"),
        _dev(seq_row_off, torch.int64, "seq_row_off"), _dev(seq_cap, torch.int32, "seq_cap"), max_cap,
        k_reg.shape[0], _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv, scale,
        _dev(err, torch.int32, "err"), _stream(stream)), "minf_gqa_attn_decode_static_ws")


def minf_gqa_attn_prefill(out, q, k_reg, v_reg, pos, n_head, n_kv_head, hd, hd_kv, scale, ws, err,
                          stream=None):
    cap = k_reg.shape[0]
    _check(lib().minf_gqa_attn_prefill(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_reg, name="k_reg"), _dev(v_reg, name="v_reg"),
        cap, _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv, scale,
        _dev(ws, torch.uint8, "ws"), _nbytes(ws), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_gqa_attn_prefill")


def _layer_step(name, reg_dtype, xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv,
                theta, freq_scale, style, out, ws, err, stream):
    nt, n_embd = h.shape
    cap = k_reg.shape[0]
    _check(getattr(lib(), name)(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd,
        _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), _dev(pos, torch.int32, "pos"), nt,
        _dev(k_reg, reg_dtype, "k_reg"), _dev(v_reg, reg_dtype, "v_reg"), cap, n_head, n_kv_head, hd, hd_kv,
        theta, freq_scale, style, _dev(out, name="out"), _dev(ws, torch.uint8, "ws"), _nbytes(ws),
        _dev(err, torch.int32, "err"), _stream(stream)), name)


def minf_layer_attn_step(xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv,
                         theta, freq_scale, style, out, ws, err, stream=None):
    _layer_step("minf_layer_attn_step", torch.float32, xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head,
                n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream)


def minf_layer_attn_step_chained(xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv,
                                 theta, freq_scale, style, out, ws, err, stream=None):
    _layer_step("minf_layer_attn_step_chained", torch.float32, xn, h, gain, eps, q, k, v, pos, k_reg, v_reg,
                n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream)


def minf_layer_attn_step_chained_f16(xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv,
                                     theta, freq_scale, style, out, ws, err, stream=None):
    _layer_step("minf_layer_attn_step_chained_f16", torch.float16, xn, h, gain, eps, q, k, v, pos, k_reg, v_reg,
                n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream)


def minf_layer_attn_step_chained_q8(xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv,
                                    theta, freq_scale, style, out, ws, err, stream=None):
    _layer_step("minf_layer_attn_step_chained_q8", torch.uint8, xn, h, gain, eps, q, k, v, pos, k_reg, v_reg,
                n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream)


def minf_layer_attn_step_batched(xn, h, gain, eps, q, k, v, pos, k_arena, v_arena, seq_row_off, seq_cap,
                                 max_cap, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out,
                                 ws, err, stream=None):
    n_seq, n_embd = h.shape
    _check(lib().minf_layer_attn_step_batched(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd,
        _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), _dev(pos, torch.int32, "pos"), n_seq,
        _dev(k_arena, name="k_arena"), _dev(v_arena, name="v_arena"),
        _dev(seq_row_off, torch.int64, "seq_row_off"), _dev(seq_cap, torch.int32, "seq_cap"), max_cap,
        k_arena.shape[0], n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, _dev(out, name="out"),
        _dev(ws, torch.uint8, "ws"), ws.numel(), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_layer_attn_step_batched")


def minf_silu_mul(y, gate, up, stream=None):
    _check(lib().minf_silu_mul(_dev(y, name="y"), _dev(gate, name="gate"), _dev(up, name="up"),
                               gate.numel(), _stream(stream)), "minf_silu_mul")


# ----------------------------------------------------------------------------- binary16 regions
# The regions (or arena) are torch.float16 tensors; everything else is as for fp32 regions.
_H = torch.float16


def minf_kv_append_f16(k_reg, v_reg, k_rows, v_rows, pos, err, stream=None):
    cap, W = k_reg.shape
    _check(lib().minf_kv_append_f16(_dev(k_reg, _H, "k_reg"), _dev(v_reg, _H, "v_reg"), cap, W,
                                    _dev(k_rows, name="k_rows"), _dev(v_rows, name="v_rows"),
                                    _dev(pos, torch.int32, "pos"), pos.numel(),
                                    _dev(err, torch.int32, "err"), _stream(stream)), "minf_kv_append_f16")


def minf_rope_kv_append_f16(q, k, v, pos, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, k_reg,
                            v_reg, err, stream=None):
    cap = k_reg.shape[0]
    _check(lib().minf_rope_kv_append_f16(_dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"),
                                         _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head,
                                         hd, hd_kv, theta, freq_scale, style, _dev(k_reg, _H, "k_reg"),
                                         _dev(v_reg, _H, "v_reg"), cap, _dev(err, torch.int32, "err"),
                                         _stream(stream)), "minf_rope_kv_append_f16")


def minf_gqa_attn_decode_f16(out, q, k_reg, v_reg, seq_row_off, seq_cap, max_cap, pos, n_head, n_kv_head,
                             hd, hd_kv, scale, ws, err, stream=None):
    _check(lib().minf_gqa_attn_decode_f16(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_reg, _H, "k_reg"), _dev(v_reg, _H, "v_reg"),
        _dev(seq_row_off, torch.int64, "seq_row_off"), _dev(seq_cap, torch.int32, "seq_cap"), max_cap,
        k_reg.shape[0], _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv, scale,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_gqa_attn_decode_f16")


def minf_gqa_attn_prefill_f16(out, q, k_reg, v_reg, pos, n_head, n_kv_head, hd, hd_kv, scale, ws, err,
                              stream=None):
    cap = k_reg.shape[0]
    _check(lib().minf_gqa_attn_prefill_f16(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_reg, _H, "k_reg"), _dev(v_reg, _H, "v_reg"),
        cap, _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv, scale,
        _dev(ws, torch.uint8, "ws"), _nbytes(ws), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_gqa_attn_prefill_f16")


def minf_layer_attn_step_f16(xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv,
                             theta, freq_scale, style, out, ws, err, stream=None):
    nt, n_embd = h.shape
    cap = k_reg.shape[0]
    _check(lib().minf_layer_attn_step_f16(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd,
        _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), _dev(pos, torch.int32, "pos"), nt,
        _dev(k_reg, _H, "k_reg"), _dev(v_reg, _H, "v_reg"), cap, n_head, n_kv_head, hd, hd_kv,
        theta, freq_scale, style, _dev(out, name="out"), _dev(ws, torch.uint8, "ws"), _nbytes(ws),
        _dev(err, torch.int32, "err"), _stream(stream)), "minf_layer_attn_step_f16")


def minf_layer_attn_step_batched_f16(xn, h, gain, eps, q, k, v, pos, k_arena, v_arena, seq_row_off, seq_cap,
                                     max_cap, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out,
                                     ws, err, stream=None):
    n_seq, n_embd = h.shape
    _check(lib().minf_layer_attn_step_batched_f16(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd,
        _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), _dev(pos, torch.int32, "pos"), n_seq,
        _dev(k_arena, _H, "k_arena"), _dev(v_arena, _H, "v_arena"),
        _dev(seq_row_off, torch.int64, "seq_row_off"), _dev(seq_cap, torch.int32, "seq_cap"), max_cap,
        k_arena.shape[0], n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, _dev(out, name="out"),
        _dev(ws, torch.uint8, "ws"), ws.numel(), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_layer_attn_step_batched_f16")


# ----------------------------------------------------------------------------- paged regions
# k_pool/v_pool: [pool_rows, W] (float32, or float16 for the _f16 forms); block_table: int32
# [n_seq, max_blocks] on the device; block_rows: rows per block.
def _pool_dtype(name):
    return _H if name.endswith("_f16") else (torch.uint8 if name.endswith("_q8") else torch.float32)


def _kv_append_paged(name, k_pool, v_pool, block_table, block_rows, k_rows, v_rows, pos, err, stream):
    dt = _pool_dtype(name)
    n_seq, max_blocks = block_table.shape
    _check(getattr(lib(), name)(
        _dev(k_pool, dt, "k_pool"), _dev(v_pool, dt, "v_pool"), k_pool.shape[0], k_pool.shape[1],
        _dev(block_table, torch.int32, "block_table"), max_blocks, block_rows, _dev(k_rows, name="k_rows"),
        _dev(v_rows, name="v_rows"), _dev(pos, torch.int32, "pos"), n_seq, _dev(err, torch.int32, "err"),
        _stream(stream)), name)


def minf_kv_append_paged(k_pool, v_pool, block_table, block_rows, k_rows, v_rows, pos, err, stream=None):
    _kv_append_paged("minf_kv_append_paged", k_pool, v_pool, block_table, block_rows, k_rows, v_rows, pos, err,
                     stream)


def minf_kv_append_paged_f16(k_pool, v_pool, block_table, block_rows, k_rows, v_rows, pos, err, stream=None):
    _kv_append_paged("minf_kv_append_paged_f16", k_pool, v_pool, block_table, block_rows, k_rows, v_rows, pos, err,
                     stream)


def _decode_paged(name, out, q, k_pool, v_pool, block_table, block_rows, pos, n_head, n_kv_head, hd, hd_kv, scale,
                  ws, err, stream):
    dt = _pool_dtype(name)
    n_seq, max_blocks = block_table.shape
    _check(getattr(lib(), name)(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_pool, dt, "k_pool"), _dev(v_pool, dt, "v_pool"),
        k_pool.shape[0], _dev(block_table, torch.int32, "block_table"), max_blocks, block_rows,
        _dev(pos, torch.int32, "pos"), n_seq, n_head, n_kv_head, hd, hd_kv, scale, _dev(ws, torch.uint8, "ws"),
        ws.numel(), _dev(err, torch.int32, "err"), _stream(stream)), name)


def minf_gqa_attn_decode_paged(out, q, k_pool, v_pool, block_table, block_rows, pos, n_head, n_kv_head, hd, hd_kv,
                               scale, ws, err, stream=None):
    _decode_paged("minf_gqa_attn_decode_paged", out, q, k_pool, v_pool, block_table, block_rows, pos, n_head,
                  n_kv_head, hd, hd_kv, scale, ws, err, stream)


def minf_gqa_attn_decode_paged_f16(out, q, k_pool, v_pool, block_table, block_rows, pos, n_head, n_kv_head, hd,
                                   hd_kv, scale, ws, err, stream=None):
    _decode_paged("minf_gqa_attn_decode_paged_f16", out, q, k_pool, v_pool, block_table, block_rows, pos, n_head,
                  n_kv_head, hd, hd_kv, scale, ws, err, stream)


def _step_paged(name, xn, h, gain, eps, q, k, v, pos, k_pool, v_pool, block_table, block_rows, n_head, n_kv_head,
                hd, hd_kv, theta, freq_scale, style, out, ws, err, stream):
    dt = _pool_dtype(name)
    n_seq, n_embd = h.shape
    max_blocks = block_table.shape[1]
    _check(getattr(lib(), name)(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd,
        _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), _dev(pos, torch.int32, "pos"), n_seq,
        _dev(k_pool, dt, "k_pool"), _dev(v_pool, dt, "v_pool"), k_pool.shape[0],
        _dev(block_table, torch.int32, "block_table"), max_blocks, block_rows, n_head, n_kv_head, hd, hd_kv, theta,
        freq_scale, style, _dev(out, name="out"), _dev(ws, torch.uint8, "ws"), ws.numel(),
        _dev(err, torch.int32, "err"), _stream(stream)), name)


def minf_layer_attn_step_paged(xn, h, gain, eps, q, k, v, pos, k_pool, v_pool, block_table, block_rows, n_head,
                               n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream=None):
    _step_paged("minf_layer_attn_step_paged", xn, h, gain, eps, q, k, v, pos, k_pool, v_pool, block_table,
                block_rows, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream)


def minf_layer_attn_step_paged_f16(xn, h, gain, eps, q, k, v, pos, k_pool, v_pool, block_table, block_rows, n_head,
                                   n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream=None):
    _step_paged("minf_layer_attn_step_paged_f16", xn, h, gain, eps, q, k, v, pos, k_pool, v_pool, block_table,
                block_rows, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream)


def minf_kv_append_paged_q8(k_pool, v_pool, block_table, block_rows, k_rows, v_rows, pos, err, stream=None):
    """Pools [pool_rows, minf_q8_row_bytes(W)] uint8; W is taken from k_rows."""
    n_seq, max_blocks = block_table.shape
    _check(lib().minf_kv_append_paged_q8(
        _dev(k_pool, torch.uint8, "k_pool"), _dev(v_pool, torch.uint8, "v_pool"), k_pool.shape[0], k_rows.shape[-1],
        _dev(block_table, torch.int32, "block_table"), max_blocks, block_rows, _dev(k_rows, name="k_rows"),
        _dev(v_rows, name="v_rows"), _dev(pos, torch.int32, "pos"), n_seq, _dev(err, torch.int32, "err"),
        _stream(stream)), "minf_kv_append_paged_q8")


def minf_gqa_attn_decode_paged_q8(out, q, k_pool, v_pool, block_table, block_rows, pos, n_head, n_kv_head, hd, hd_kv,
                                  scale, ws, err, stream=None):
    _decode_paged("minf_gqa_attn_decode_paged_q8", out, q, k_pool, v_pool, block_table, block_rows, pos, n_head,
                  n_kv_head, hd, hd_kv, scale, ws, err, stream)


def minf_layer_attn_step_paged_q8(xn, h, gain, eps, q, k, v, pos, k_pool, v_pool, block_table, block_rows, n_head,
                                  n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream=None):
    _step_paged("minf_layer_attn_step_paged_q8", xn, h, gain, eps, q, k, v, pos, k_pool, v_pool, block_table,
                block_rows, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err, stream)


# ----------------------------------------------------------------------------- Q8_0 regions
# The regions (or arena) are torch.uint8 tensors [rows, minf_q8_row_bytes(W)]; the row width W
# (values) comes from the fp32 rows or the head geometry.
_U8 = torch.uint8


def minf_q8_row_bytes(row_width: int) -> int:
    return int(lib().minf_q8_row_bytes(row_width))


def minf_kv_append_q8(k_reg, v_reg, k_rows, v_rows, pos, err, stream=None):
    _check(lib().minf_kv_append_q8(_dev(k_reg, _U8, "k_reg"), _dev(v_reg, _U8, "v_reg"), k_reg.shape[0],
                                   k_rows.shape[-1], _dev(k_rows, name="k_rows"), _dev(v_rows, name="v_rows"),
                                   _dev(pos, torch.int32, "pos"), pos.numel(), _dev(err, torch.int32, "err"),
                                   _stream(stream)), "minf_kv_append_q8")


def minf_rope_kv_append_q8(q, k, v, pos, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, k_reg, v_reg, err,
                           stream=None):
    _check(lib().minf_rope_kv_append_q8(_dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"),
                                        _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv,
                                        theta, freq_scale, style, _dev(k_reg, _U8, "k_reg"), _dev(v_reg, _U8, "v_reg"),
                                        k_reg.shape[0], _dev(err, torch.int32, "err"), _stream(stream)),
           "minf_rope_kv_append_q8")


def minf_gqa_attn_decode_q8(out, q, k_reg, v_reg, seq_row_off, seq_cap, max_cap, pos, n_head, n_kv_head, hd, hd_kv,
                            scale, ws, err, stream=None):
    _check(lib().minf_gqa_attn_decode_q8(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_reg, _U8, "k_reg"), _dev(v_reg, _U8, "v_reg"),
        _dev(seq_row_off, torch.int64, "seq_row_off"), _dev(seq_cap, torch.int32, "seq_cap"), max_cap,
        k_reg.shape[0], _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv, scale,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_gqa_attn_decode_q8")


def minf_gqa_attn_prefill_q8(out, q, k_reg, v_reg, pos, n_head, n_kv_head, hd, hd_kv, scale, ws, err, stream=None):
    _check(lib().minf_gqa_attn_prefill_q8(
        _dev(out, name="out"), _dev(q, name="q"), _dev(k_reg, _U8, "k_reg"), _dev(v_reg, _U8, "v_reg"),
        k_reg.shape[0], _dev(pos, torch.int32, "pos"), pos.numel(), n_head, n_kv_head, hd, hd_kv, scale,
        _dev(ws, torch.uint8, "ws"), _nbytes(ws), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_gqa_attn_prefill_q8")


def minf_layer_attn_step_q8(xn, h, gain, eps, q, k, v, pos, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv, theta,
                            freq_scale, style, out, ws, err, stream=None):
    nt, n_embd = h.shape
    _check(lib().minf_layer_attn_step_q8(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd,
        _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), _dev(pos, torch.int32, "pos"), nt,
        _dev(k_reg, _U8, "k_reg"), _dev(v_reg, _U8, "v_reg"), k_reg.shape[0], n_head, n_kv_head, hd, hd_kv,
        theta, freq_scale, style, _dev(out, name="out"), _dev(ws, torch.uint8, "ws"), _nbytes(ws),
        _dev(err, torch.int32, "err"), _stream(stream)), "minf_layer_attn_step_q8")


def minf_layer_attn_step_batched_q8(xn, h, gain, eps, q, k, v, pos, k_arena, v_arena, seq_row_off, seq_cap, max_cap,
                                    n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, err,
                                    stream=None):
    n_seq, n_embd = h.shape
    _check(lib().minf_layer_attn_step_batched_q8(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd,
        _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), _dev(pos, torch.int32, "pos"), n_seq,
        _dev(k_arena, _U8, "k_arena"), _dev(v_arena, _U8, "v_arena"),
        _dev(seq_row_off, torch.int64, "seq_row_off"), _dev(seq_cap, torch.int32, "seq_cap"), max_cap,
        k_arena.shape[0], n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, _dev(out, name="out"),
        _dev(ws, torch.uint8, "ws"), ws.numel(), _dev(err, torch.int32, "err"), _stream(stream)),
        "minf_layer_attn_step_batched_q8")


# ----------------------------------------------------------------------------- fused QKV op
def minf_fused_qkv(xn, h, gain, eps, w_qkv, b_qkv, pos, q, k, v, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv, theta,
                   freq_scale, style, err, stream=None):
    nt, n_embd = h.shape
    _check(lib().minf_fused_qkv(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd, _dev(w_qkv, name="w_qkv"),
        _dev(b_qkv, name="b_qkv"), _dev(pos, torch.int32, "pos"), nt, _dev(q, name="q"), _dev(k, name="k"),
        _dev(v, name="v"), _dev(k_reg, name="k_reg"), _dev(v_reg, name="v_reg"), k_reg.shape[0], n_head, n_kv_head,
        hd, hd_kv, theta, freq_scale, style, _dev(err, torch.int32, "err"), _stream(stream)), "minf_fused_qkv")


def minf_layer_attn_step_qkv(xn, h, gain, eps, w_qkv, b_qkv, pos, q, k, v, k_reg, v_reg, n_head, n_kv_head, hd, hd_kv,
                             theta, freq_scale, style, out, ws, err, stream=None):
    n_embd = h.shape[-1]
    _check(lib().minf_layer_attn_step_qkv(
        _dev(xn, name="xn"), _dev(h, name="h"), _dev(gain, name="gain"), eps, n_embd, _dev(w_qkv, name="w_qkv"),
        _dev(b_qkv, name="b_qkv"), _dev(pos, torch.int32, "pos"), _dev(q, name="q"), _dev(k, name="k"),
        _dev(v, name="v"), _dev(k_reg, name="k_reg"), _dev(v_reg, name="v_reg"), k_reg.shape[0], n_head, n_kv_head,
        hd, hd_kv, theta, freq_scale, style, _dev(out, name="out"), _dev(ws, torch.uint8, "ws"), ws.numel(),
        _dev(err, torch.int32, "err"), _stream(stream)), "minf_layer_attn_step_qkv")
