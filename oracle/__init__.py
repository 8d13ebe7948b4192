"""CPU oracle for the attention stage -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its Python
binding) never imports it and shares no code with it.

The arithmetic lives in ``minf_oracle.c`` (plain C, built here with gcc and
``-ffp-contract=off``); this module only builds it and marshals numpy arrays.
Every function cites the page and section it restates, in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "minf_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

OK = 0
ERR_ARG = 1
ERR_GEOMETRY = 2
ERR_POS = 4

_lock = threading.Lock()
_lib = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.orc_rope_freqs.argtypes = [_f32p, ctypes.c_int, ctypes.c_float, ctypes.c_float]
        lib.orc_rope_freqs.restype = None
        lib.orc_rms_norm.argtypes = [_f32p, _f32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_float]
        lib.orc_rms_norm.restype = None
        lib.orc_rope.argtypes = [_f32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_float, ctypes.c_float, ctypes.c_int]
        lib.orc_rope.restype = ctypes.c_int
        lib.orc_kv_append.argtypes = [_f32p, _f32p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, _i32p,
                                      ctypes.c_int]
        lib.orc_kv_append.restype = ctypes.c_int
        lib.orc_gqa_attn.argtypes = [_f32p, _f32p, _f32p, _f32p, ctypes.c_int, _i32p, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_float, ctypes.c_int]
        lib.orc_gqa_attn.restype = ctypes.c_int
        lib.orc_attn_bruteforce_f64.argtypes = [_f64p, _f32p, _f32p, _f32p, ctypes.c_int, _i32p,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_double]
        lib.orc_attn_bruteforce_f64.restype = ctypes.c_int
        lib.orc_silu_mul.argtypes = [_f32p, _f32p, _f32p, ctypes.c_long]
        lib.orc_silu_mul.restype = None
        lib.orc_layer_attn_step.argtypes = [
            _f32p, _f32p, _f32p, ctypes.c_float, ctypes.c_int,
            _f32p, _f32p, _f32p, _i32p, ctypes.c_int,
            _f32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_float, ctypes.c_float, ctypes.c_int, _f32p, ctypes.c_int]
        lib.orc_layer_attn_step.restype = ctypes.c_int
        _u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.orc_f32_to_f16_array.argtypes = [_u16p, _f32p, ctypes.c_long]
        lib.orc_f32_to_f16_array.restype = None
        lib.orc_f16_to_f32_array.argtypes = [_f32p, _u16p, ctypes.c_long]
        lib.orc_f16_to_f32_array.restype = None
        lib.orc_kv_append_f16.argtypes = [_u16p, _u16p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, _i32p,
                                          ctypes.c_int]
        lib.orc_kv_append_f16.restype = ctypes.c_int
        lib.orc_layer_attn_step_f16.argtypes = [
            _f32p, _f32p, _f32p, ctypes.c_float, ctypes.c_int,
            _f32p, _f32p, _f32p, _i32p, ctypes.c_int,
            _u16p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_float, ctypes.c_float, ctypes.c_int, _f32p, ctypes.c_int]
        lib.orc_layer_attn_step_f16.restype = ctypes.c_int
        lib.orc_kv_append_paged.argtypes = [_f32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p,
                                            ctypes.c_int, _f32p, _f32p, _i32p, ctypes.c_int]
        lib.orc_kv_append_paged.restype = ctypes.c_int
        lib.orc_gqa_attn_paged.argtypes = [_f32p, _f32p, _f32p, _f32p, ctypes.c_int, ctypes.c_int, _i32p,
                                           ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_float]
        lib.orc_gqa_attn_paged.restype = ctypes.c_int
        _u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.orc_q8_row_bytes.argtypes = [ctypes.c_int]
        lib.orc_q8_row_bytes.restype = ctypes.c_long
        lib.orc_q8_quantize_rows.argtypes = [_u8p, _f32p, ctypes.c_long, ctypes.c_int]
        lib.orc_q8_quantize_rows.restype = None
        lib.orc_q8_dequant_rows.argtypes = [_f32p, _u8p, ctypes.c_long, ctypes.c_int]
        lib.orc_q8_dequant_rows.restype = None
        lib.orc_kv_append_q8.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, _i32p, ctypes.c_int]
        lib.orc_kv_append_q8.restype = ctypes.c_int
        lib.orc_fused_qkv.argtypes = [_f32p, _f32p, _f32p, _f32p, _f32p, _f32p, ctypes.c_float, ctypes.c_int,
                                      _f32p, _f32p, _i32p, ctypes.c_int, _f32p, _f32p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int]
        lib.orc_fused_qkv.restype = ctypes.c_int
        _lib = lib
        return lib


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: oracle status {status}")
        self.status = status


def _f32(a, writable=False):
    a = np.asarray(a)
    if a.dtype != np.float32 or not a.flags.c_contiguous:
        if writable:
            raise TypeError("in-place argument must be a C-contiguous float32 array")
        a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _i32(a):
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _p(a, t):
    return a.ctypes.data_as(t)


def rope_freqs(hd: int, theta: float, freq_scale: float = 1.0) -> np.ndarray:
    out = np.zeros(hd // 2, dtype=np.float32)
    _load().orc_rope_freqs(_p(out, _f32p), hd, theta, freq_scale)
    return out


def rms_norm(x, w=None, eps: float = 1e-6, out=None) -> np.ndarray:
    """x: [rows, n] float32.  Returns y (or writes ``out``, which may be ``x``)."""
    x = _f32(x)
    rows, n = x.shape
    y = np.empty_like(x) if out is None else _f32(out, writable=True)
    wkeep = _f32(w) if w is not None else None
    wp = _p(wkeep, _f32p) if wkeep is not None else None
    _load().orc_rms_norm(_p(y, _f32p), _p(x, _f32p), wp, rows, n, eps)
    return y


def rope(x, pos, n_head: int, hd: int, theta: float, freq_scale: float = 1.0, style: int = 0):
    """In place on a float32 array laid out [nt, n_head, hd]; returns it."""
    x = _f32(x, writable=True)
    pos = _i32(pos)
    nt = pos.shape[0]
    assert x.size == nt * n_head * hd
    st = _load().orc_rope(_p(x, _f32p), _p(pos, _i32p), nt, n_head, hd, theta, freq_scale, style)
    if st != OK:
        raise OracleError(st, "rope")
    return x


def kv_append(k_reg, v_reg, k_rows, v_rows, pos, check=True) -> int:
    """Regions [cap, W] (modified in place), rows [nt, W]."""
    k_reg = _f32(k_reg, writable=True)
    v_reg = _f32(v_reg, writable=True)
    cap, W = k_reg.shape
    k_rows = _f32(k_rows).reshape(-1, W)
    v_rows = _f32(v_rows).reshape(-1, W)
    pos = _i32(pos)
    st = _load().orc_kv_append(_p(k_reg, _f32p), _p(v_reg, _f32p), cap, W, _p(k_rows, _f32p),
                               _p(v_rows, _f32p), _p(pos, _i32p), pos.shape[0])
    if check and st != OK:
        raise OracleError(st, "kv_append")
    return st


def gqa_attn(q, k_reg, v_reg, pos, n_head: int, n_kv_head: int, hd: int, hd_kv: int,
             scale: float | None = None, n_threads: int = 1, cap: int | None = None) -> np.ndarray:
    """q [nt, n_head, hd]; regions [cap, n_kv_head*hd_kv]; returns out [nt, n_head*hd_kv]."""
    q = _f32(q)
    k_reg = _f32(k_reg)
    v_reg = _f32(v_reg)
    pos = _i32(pos)
    nt = pos.shape[0]
    if cap is None:
        cap = k_reg.shape[0]
    if scale is None:
        scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    out = np.zeros((nt, n_head * hd_kv), dtype=np.float32)
    st = _load().orc_gqa_attn(_p(out, _f32p), _p(q, _f32p), _p(k_reg, _f32p), _p(v_reg, _f32p), cap,
                              _p(pos, _i32p), nt, n_head, n_kv_head, hd, hd_kv, scale, n_threads)
    if st != OK:
        raise OracleError(st, "gqa_attn")
    return out


def attn_bruteforce_f64(q, k_reg, v_reg, pos, n_head: int, n_kv_head: int, hd: int, hd_kv: int,
                        scale: float, cap: int | None = None) -> np.ndarray:
    q = _f32(q)
    k_reg = _f32(k_reg)
    v_reg = _f32(v_reg)
    pos = _i32(pos)
    nt = pos.shape[0]
    if cap is None:
        cap = k_reg.shape[0]
    out = np.zeros((nt, n_head * hd_kv), dtype=np.float64)
    st = _load().orc_attn_bruteforce_f64(_p(out, _f64p), _p(q, _f32p), _p(k_reg, _f32p),
                                         _p(v_reg, _f32p), cap, _p(pos, _i32p), nt, n_head,
                                         n_kv_head, hd, hd_kv, scale)
    if st != OK:
        raise OracleError(st, "attn_bruteforce_f64")
    return out


def silu_mul(gate, up) -> np.ndarray:
    gate = _f32(gate)
    up = _f32(up)
    y = np.empty_like(gate)
    _load().orc_silu_mul(_p(y, _f32p), _p(gate, _f32p), _p(up, _f32p), gate.size)
    return y


def layer_attn_step(h, gain, q, k, v, pos, k_reg, v_reg, *, n_head: int, n_kv_head: int, hd: int,
                    hd_kv: int, eps: float = 1e-6, theta: float = 1e6, freq_scale: float = 1.0,
                    style: int = 0, n_threads: int = 1):
    """One layer's attention stage.  q and k are rotated in place, the regions are
    appended in place; returns (xn, out)."""
    h = _f32(h)
    gain = _f32(gain)
    q = _f32(q, writable=True)
    k = _f32(k, writable=True)
    v = _f32(v)
    pos = _i32(pos)
    k_reg = _f32(k_reg, writable=True)
    v_reg = _f32(v_reg, writable=True)
    nt = pos.shape[0]
    n_embd = h.size // max(nt, 1)
    xn = np.empty_like(h)
    out = np.zeros((nt, n_head * hd_kv), dtype=np.float32)
    st = _load().orc_layer_attn_step(
        _p(xn, _f32p), _p(h, _f32p), _p(gain, _f32p), eps, n_embd,
        _p(q, _f32p), _p(k, _f32p), _p(v, _f32p), _p(pos, _i32p), nt,
        _p(k_reg, _f32p), _p(v_reg, _f32p), k_reg.shape[0], n_head, n_kv_head, hd, hd_kv,
        theta, freq_scale, style, _p(out, _f32p), n_threads)
    if st != OK:
        raise OracleError(st, "layer_attn_step")
    return xn, out


# ----------------------------------------------------------------------------- f16 cache
def _u16(a, writable=False):
    a = np.asarray(a)
    if a.dtype != np.uint16 or not a.flags.c_contiguous:
        if writable:
            raise TypeError("in-place argument must be a C-contiguous uint16 array")
        a = np.ascontiguousarray(a, dtype=np.uint16)
    return a


def f32_to_f16(x) -> np.ndarray:
    """binary16 bit patterns (uint16) of float32 values, round to nearest even."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_f32_to_f16_array(_p(out, _u16p), _p(x, _f32p), x.size)
    return out


def f16_to_f32(h) -> np.ndarray:
    """float32 values of binary16 bit patterns (exact)."""
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float32)
    _load().orc_f16_to_f32_array(_p(out, _f32p), _p(h, _u16p), h.size)
    return out


def kv_append_f16(k_reg, v_reg, k_rows, v_rows, pos, check=True) -> int:
    """f16 regions [cap, W] as uint16 bit patterns (modified in place), fp32 rows [nt, W]."""
    k_reg = _u16(k_reg, writable=True)
    v_reg = _u16(v_reg, writable=True)
    cap, W = k_reg.shape
    k_rows = _f32(k_rows).reshape(-1, W)
    v_rows = _f32(v_rows).reshape(-1, W)
    pos = _i32(pos)
    st = _load().orc_kv_append_f16(_p(k_reg, _u16p), _p(v_reg, _u16p), cap, W, _p(k_rows, _f32p),
                                   _p(v_rows, _f32p), _p(pos, _i32p), pos.shape[0])
    if check and st != OK:
        raise OracleError(st, "kv_append_f16")
    return st


def layer_attn_step_f16(h, gain, q, k, v, pos, k_reg, v_reg, *, n_head: int, n_kv_head: int, hd: int,
                        hd_kv: int, eps: float = 1e-6, theta: float = 1e6, freq_scale: float = 1.0,
                        style: int = 0, n_threads: int = 1):
    """layer_attn_step over f16 regions (uint16 bit patterns, appended in place)."""
    h = _f32(h)
    gain = _f32(gain)
    q = _f32(q, writable=True)
    k = _f32(k, writable=True)
    v = _f32(v)
    pos = _i32(pos)
    k_reg = _u16(k_reg, writable=True)
    v_reg = _u16(v_reg, writable=True)
    nt = pos.shape[0]
    n_embd = h.size // max(nt, 1)
    xn = np.empty_like(h)
    out = np.zeros((nt, n_head * hd_kv), dtype=np.float32)
    st = _load().orc_layer_attn_step_f16(
        _p(xn, _f32p), _p(h, _f32p), _p(gain, _f32p), eps, n_embd,
        _p(q, _f32p), _p(k, _f32p), _p(v, _f32p), _p(pos, _i32p), nt,
        _p(k_reg, _u16p), _p(v_reg, _u16p), k_reg.shape[0], n_head, n_kv_head, hd, hd_kv,
        theta, freq_scale, style, _p(out, _f32p), n_threads)
    if st != OK:
        raise OracleError(st, "layer_attn_step_f16")
    return xn, out


# ----------------------------------------------------------------------------- paged regions
def kv_append_paged(k_pool, v_pool, table, block_rows: int, k_rows, v_rows, pos, check=True) -> int:
    """Pools [pool_blocks*block_rows, W] (modified in place); table int32 [n_seq, max_blocks];
    one row per sequence, rows [n_seq, W], at pos[s]."""
    k_pool = _f32(k_pool, writable=True)
    v_pool = _f32(v_pool, writable=True)
    rows, W = k_pool.shape
    table = _i32(table)
    n_seq, max_blocks = table.shape
    k_rows = _f32(k_rows).reshape(-1, W)
    v_rows = _f32(v_rows).reshape(-1, W)
    pos = _i32(pos)
    st = _load().orc_kv_append_paged(_p(k_pool, _f32p), _p(v_pool, _f32p), rows // block_rows, block_rows, W,
                                     _p(table, _i32p), max_blocks, _p(k_rows, _f32p), _p(v_rows, _f32p),
                                     _p(pos, _i32p), n_seq)
    if check and st != OK:
        raise OracleError(st, "kv_append_paged")
    return st


def gqa_attn_paged(q, k_pool, v_pool, table, block_rows: int, pos, n_head: int, n_kv_head: int, hd: int,
                   hd_kv: int, scale: float | None = None) -> np.ndarray:
    """Decode attention through a block table; q [n_seq, n_head, hd] -> out [n_seq, n_head*hd_kv]."""
    q = _f32(q)
    k_pool = _f32(k_pool)
    v_pool = _f32(v_pool)
    table = _i32(table)
    n_seq, max_blocks = table.shape
    pos = _i32(pos)
    if scale is None:
        scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    out = np.zeros((n_seq, n_head * hd_kv), dtype=np.float32)
    st = _load().orc_gqa_attn_paged(_p(out, _f32p), _p(q, _f32p), _p(k_pool, _f32p), _p(v_pool, _f32p),
                                    k_pool.shape[0] // block_rows, block_rows, _p(table, _i32p), max_blocks,
                                    _p(pos, _i32p), n_seq, n_head, n_kv_head, hd, hd_kv, scale)
    if st != OK:
        raise OracleError(st, "gqa_attn_paged")
    return out


# ----------------------------------------------------------------------------- Q8_0 cache
def q8_row_bytes(W: int) -> int:
    """Bytes of one Q8_0 row of W values: W quants, W/32 binary16 scales, padding to 16 bytes."""
    return int(_load().orc_q8_row_bytes(W))


def q8_quantize(x) -> np.ndarray:
    """[rows, W] float32 -> [rows, q8_row_bytes(W)] uint8."""
    x = _f32(x)
    rows, W = x.shape
    out = np.empty((rows, q8_row_bytes(W)), dtype=np.uint8)
    _load().orc_q8_quantize_rows(_p(out, _u8p), _p(x, _f32p), rows, W)
    return out


def q8_dequant(q, W: int) -> np.ndarray:
    """[rows, q8_row_bytes(W)] uint8 -> [rows, W] float32 (the values the rows hold)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows = q.shape[0]
    out = np.empty((rows, W), dtype=np.float32)
    _load().orc_q8_dequant_rows(_p(out, _f32p), _p(q, _u8p), rows, W)
    return out


def kv_append_q8(k_reg, v_reg, W: int, k_rows, v_rows, pos, check=True) -> int:
    """Q8_0 regions [cap, q8_row_bytes(W)] uint8 (modified in place), fp32 rows [nt, W]."""
    for r in (k_reg, v_reg):
        if r.dtype != np.uint8 or not r.flags.c_contiguous:
            raise TypeError("regions must be C-contiguous uint8 arrays")
    cap = k_reg.shape[0]
    k_rows = _f32(k_rows).reshape(-1, W)
    v_rows = _f32(v_rows).reshape(-1, W)
    pos = _i32(pos)
    st = _load().orc_kv_append_q8(_p(k_reg, _u8p), _p(v_reg, _u8p), cap, W, _p(k_rows, _f32p), _p(v_rows, _f32p),
                                  _p(pos, _i32p), pos.shape[0])
    if check and st != OK:
        raise OracleError(st, "kv_append_q8")
    return st


# ----------------------------------------------------------------------------- fused QKV op
def fused_qkv(h, gain, w, b, pos, k_reg, v_reg, *, n_head: int, n_kv_head: int, hd: int, hd_kv: int,
              eps: float = 1e-6, theta: float = 1e6, freq_scale: float = 1.0, style: int = 0):
    """RMSNorm, the q/k/v projections (w [n_out, n_embd], b [n_out] or None), RoPE on q and k,
    and the K/V store at pos (regions modified in place).  Returns (xn, q, k, v)."""
    h = _f32(h)
    nt, n_embd = h.shape
    gain = _f32(gain)
    w = _f32(w)
    bb = _f32(b) if b is not None else None
    pos = _i32(pos)
    k_reg = _f32(k_reg, writable=True)
    v_reg = _f32(v_reg, writable=True)
    W = n_kv_head * hd_kv
    xn = np.empty_like(h)
    q = np.empty((nt, n_head * hd), np.float32)
    k = np.empty((nt, W), np.float32)
    v = np.empty((nt, W), np.float32)
    st = _load().orc_fused_qkv(_p(xn, _f32p), _p(q, _f32p), _p(k, _f32p), _p(v, _f32p), _p(h, _f32p),
                               _p(gain, _f32p), eps, n_embd, _p(w, _f32p), _p(bb, _f32p) if bb is not None else None,
                               _p(pos, _i32p), nt, _p(k_reg, _f32p), _p(v_reg, _f32p), k_reg.shape[0], n_head,
                               n_kv_head, hd, hd_kv, theta, freq_scale, style)
    if st != OK:
        raise OracleError(st, "fused_qkv")
    return xn, q, k, v
