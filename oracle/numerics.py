"""ctypes wrappers around oracle/liboracle.so (built from kvc_oracle.c).

Test infrastructure only; see oracle/__init__.py.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))

F16, Q4_0, Q8_0 = 1, 2, 8


def _load():
    path = _build.build()
    L = C.CDLL(path)
    p, i64, i32, f64 = C.c_void_p, C.c_int64, C.c_int, C.c_double
    L.orc_f16_to_f64.restype = f64
    L.orc_f16_to_f64.argtypes = [C.c_uint16]
    L.orc_f64_to_f16.restype = C.c_uint16
    L.orc_f64_to_f16.argtypes = [f64]
    L.orc_f32_to_f16.restype = C.c_uint16
    L.orc_f32_to_f16.argtypes = [C.c_float]
    L.orc_f32_to_f16_array.argtypes = [p, p, i64]
    L.orc_f16_to_f64_array.argtypes = [p, p, i64]
    L.orc_q8_0_quantize_block.argtypes = [p, p, p]
    L.orc_q8_0_quantize_row.argtypes = [p, i64, p, p]
    L.orc_q8_0_value.restype = f64
    L.orc_q8_0_value.argtypes = [C.c_int8, C.c_uint16]
    L.orc_q8_0_dequantize_row.argtypes = [p, p, i64, p]
    L.orc_q4_0_quantize_block.argtypes = [p, p, p]
    L.orc_q4_0_quantize_row.argtypes = [p, i64, p, p]
    L.orc_q4_0_dequantize_row.argtypes = [p, p, i64, p]
    L.orc_attn.restype = i32
    L.orc_attn.argtypes = [p, i32, i32, i32, i64, i32, p, p, i32, p, p, f64, i32, i32, p]
    L.orc_attn_bruteforce.restype = i32
    L.orc_attn_bruteforce.argtypes = [p, i32, i32, i32, i64, i32, p, p, i32, p, p, f64, p]
    L.orc_rope_rotate.argtypes = [p, i32, i32, f64, i64]
    L.orc_rope_shift_q8_0.restype = i32
    L.orc_rope_shift_q8_0.argtypes = [p, p, i64, i32, i32, f64, i64]
    L.orc_rope_shift_f16.restype = i32
    L.orc_rope_shift_f16.argtypes = [p, i64, i32, i32, f64, i64]
    L.orc_keydiff_scores.restype = i32
    L.orc_keydiff_scores.argtypes = [i32, p, p, i64, i32, i32, p]
    L.orc_min_window.restype = i64
    L.orc_min_window.argtypes = [p, i64, i64, i64, i64]
    return L


lib = _load()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def f16_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib.orc_f16_to_f64_array(_ptr(h), _ptr(out), h.size)
    return out


def f32_to_f16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.orc_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def q8_0_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """x fp32 [..., D] (D % 32 == 0) -> (codes int8 [..., D], scales u16 [..., D/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    D = x.shape[-1]
    assert D % 32 == 0
    codes = np.empty(x.shape, dtype=np.int8)
    scales = np.empty(x.shape[:-1] + (D // 32,), dtype=np.uint16)
    lib.orc_q8_0_quantize_row(_ptr(x), x.size, _ptr(codes), _ptr(scales))
    return codes, scales


def q8_0_dequantize(codes, scales) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    assert codes.shape[:-1] == scales.shape[:-1] and codes.shape[-1] == 32 * scales.shape[-1]
    out = np.empty(codes.shape, dtype=np.float64)
    # rows are contiguous, so the flat call sees blocks in order
    lib.orc_q8_0_dequantize_row(_ptr(codes), _ptr(scales), codes.size, _ptr(out))
    return out


def q4_0_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """x fp32 [..., D] (D % 32 == 0) -> (packed u8 [..., D/2], scales u16 [..., D/32]).
    Byte j of a block holds code j (low four bits) and code j + 16 (high)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    D = x.shape[-1]
    assert D % 32 == 0
    packed = np.empty(x.shape[:-1] + (D // 2,), dtype=np.uint8)
    scales = np.empty(x.shape[:-1] + (D // 32,), dtype=np.uint16)
    lib.orc_q4_0_quantize_row(_ptr(x), x.size, _ptr(packed), _ptr(scales))
    return packed, scales


def q4_0_dequantize(packed, scales) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    assert packed.shape[:-1] == scales.shape[:-1] and packed.shape[-1] == 16 * scales.shape[-1]
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.float64)
    lib.orc_q4_0_dequantize_row(_ptr(packed), _ptr(scales), out.size, _ptr(out))
    return out


def _kv_args(type_, data, scales):
    dt = {Q8_0: np.int8, Q4_0: np.uint8}.get(type_, np.uint16)
    data = np.ascontiguousarray(data, dtype=dt)
    scales = None if type_ == F16 else np.ascontiguousarray(scales, dtype=np.uint16)
    return data, scales


def attn(q, type_k, k, ks, type_v, v, vs, kq_scale, heads=None) -> np.ndarray:
    """Single-query attention for one sequence.

    q fp32 [H][D]; k/v: q8_0 codes int8 [n][Hk][D] + scales u16 [n][Hk][D/32],
    q4_0 packed u8 [n][Hk][D/2] + scales u16 [n][Hk][D/32] (V only), or f16
    bits u16 [n][Hk][D] (scales None).  Returns fp64 [H][D]; rows
    outside `heads` (a (h0, h1) range) are left zero."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    H, D = q.shape
    k, ks = _kv_args(type_k, k, ks)
    v, vs = _kv_args(type_v, v, vs)
    n, Hk = k.shape[0], k.shape[1]
    out = np.zeros((H, D), dtype=np.float64)
    h0, h1 = heads if heads is not None else (0, H)
    rc = lib.orc_attn(_ptr(q), H, Hk, D, n, type_k, _ptr(k), _ptr(ks), type_v, _ptr(v), _ptr(vs),
                      float(kq_scale), h0, h1, _ptr(out))
    if rc:
        raise ValueError("orc_attn failed: %d" % rc)
    return out


def attn_bruteforce(q, type_k, k, ks, type_v, v, vs, kq_scale) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    H, D = q.shape
    k, ks = _kv_args(type_k, k, ks)
    v, vs = _kv_args(type_v, v, vs)
    n, Hk = k.shape[0], k.shape[1]
    out = np.zeros((H, D), dtype=np.float64)
    rc = lib.orc_attn_bruteforce(_ptr(q), H, Hk, D, n, type_k, _ptr(k), _ptr(ks), type_v, _ptr(v),
                                 _ptr(vs), float(kq_scale), _ptr(out))
    if rc:
        raise ValueError("orc_attn_bruteforce failed: %d" % rc)
    return out


def rope_rotate(x, mode: int, base: float, delta: int) -> np.ndarray:
    """Rotate a copy of fp64 rows x [..., D] by delta positions."""
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    D = x.shape[-1]
    rows = x.reshape(-1, D)
    for r in range(rows.shape[0]):
        row = np.ascontiguousarray(rows[r])
        lib.orc_rope_rotate(_ptr(row), D, mode, float(base), int(delta))
        rows[r] = row
    return rows.reshape(x.shape)


def rope_shift_q8_0(codes, scales, mode: int, base: float, delta: int):
    """Shift q8_0 head-rows (codes [..., D], scales [..., D/32]); returns new copies."""
    codes = np.array(codes, dtype=np.int8, copy=True, order="C")
    scales = np.array(scales, dtype=np.uint16, copy=True, order="C")
    D = codes.shape[-1]
    n = codes.size // D
    rc = lib.orc_rope_shift_q8_0(_ptr(codes), _ptr(scales), n, D, mode, float(base), int(delta))
    if rc:
        raise ValueError("orc_rope_shift_q8_0 failed")
    return codes, scales


def rope_shift_f16(h, mode: int, base: float, delta: int) -> np.ndarray:
    h = np.array(h, dtype=np.uint16, copy=True, order="C")
    D = h.shape[-1]
    rc = lib.orc_rope_shift_f16(_ptr(h), h.size // D, D, mode, float(base), int(delta))
    if rc:
        raise ValueError("orc_rope_shift_f16 failed")
    return h


def keydiff_scores(type_k, k, ks) -> np.ndarray:
    """KeyDiff score of every row of one layer's K ([n][Hk][D] stored form),
    in row order: mean over KV heads of 1 - cos(key, that head's mean key)."""
    k, ks = _kv_args(type_k, k, ks)
    n, Hk, D = k.shape
    out = np.zeros(n, dtype=np.float64)
    if lib.orc_keydiff_scores(type_k, _ptr(k), _ptr(ks), n, Hk, D, _ptr(out)):
        raise ValueError("orc_keydiff_scores failed")
    return out


def min_window(score, lo: int, hi: int, w: int) -> int:
    """Start of the width-w window inside [lo, hi) with the smallest score sum
    (first on ties); -1 when none fits."""
    score = np.ascontiguousarray(score, dtype=np.float64)
    return int(lib.orc_min_window(_ptr(score), score.size, lo, hi, w))
