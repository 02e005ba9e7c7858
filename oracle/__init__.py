"""ctypes wrapper of the scalar C oracle (``gguf_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library and never imports it.

Every function takes and returns numpy arrays.  Packed weight / q8_1 buffers
are ``uint8`` arrays of shape ``[rows, row_bytes]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gguf_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgguf_oracle.so")

F32, F16, Q4_0, Q8_0, Q8_1, Q4_K, Q5_K, Q6_K, BF16 = 0, 1, 2, 8, 9, 12, 13, 14, 30
MXFP4 = 39
Q4_1, Q5_0, Q5_1 = 3, 6, 7


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no FMA contraction, no fast math)."""
    src_m = os.path.getmtime(_SRC)
    hdr_m = os.path.getmtime(os.path.join(_HERE, "gguf_oracle.h"))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(src_m, hdr_m):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        sig = {
            "orc_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_block_elems": (i64, [i32]),
            "orc_block_bytes": (i64, [i32]),
            "orc_row_size": (i64, [i32, i64]),
            "orc_sub_elems": (i64, [i32]),
            "orc_quantize_q8_1": (i32, [p, i64, i64, i64, p]),
            "orc_quantize_weights": (i32, [i32, p, i64, i64, p]),
            "orc_dequantize_row": (i32, [i32, p, i64, p]),
            "orc_dequantize_row_f64": (i32, [i32, p, i64, p]),
            "orc_dequantize": (i32, [i32, p, i64, i64, p, i32]),
            "orc_moe_plain": (i32, [i32, p, i64, i64, i64, i64, p, p, i64, i64, p]),
            "orc_get_rows": (i32, [i32, p, i64, i64, p, i64, p, i32]),
            "orc_block_dots": (i32, [i32, p, i64, i64, p, i64, p]),
            "orc_mul_mat": (i32, [i32, p, i64, i64, p, i64, p]),
            "orc_mul_mat_rows": (i32, [i32, p, i64, i64, p, i64, p, i64, i64, i32]),
            "orc_mul_mat_dequant_f64": (i32, [i32, p, i64, i64, p, i64, p]),
            "orc_moe_gate_up": (i32, [i32, p, i64, i64, i64, i64, p, p, i64, i64, p, p, i64, i64, i32]),
            "orc_moe_down": (i32, [i32, p, i64, i64, i64, i64, p, p, p, i64, i64, p, i64, i64, i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _ok(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def row_size(t: int, k: int) -> int:
    rs = lib().orc_row_size(t, k)
    if rs < 0:
        raise ValueError(f"k={k} is not a multiple of the block of type {t}")
    return rs


def block_elems(t: int) -> int:
    return lib().orc_block_elems(t)


def block_bytes(t: int) -> int:
    return lib().orc_block_bytes(t)


def sub_elems(t: int) -> int:
    return lib().orc_sub_elems(t)


def f16_bits(x: float) -> int:
    return lib().orc_f32_to_f16(x)


def f16_value(bits: int) -> float:
    return lib().orc_f16_to_f32(bits)


def bf16_bits(x: float) -> int:
    return lib().orc_f32_to_bf16(x)


def bf16_bits_f64(x: float) -> int:
    """fp64 -> bf16 bits, rounded once (no fp32 step)."""
    return lib().orc_f64_to_bf16(x)


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_to_f32(bits)


def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """fp32 [m, k] -> q8_1 bytes [m, k/32*36]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    m, k = x.shape
    out = np.zeros((m, row_size(Q8_1, k)), dtype=np.uint8)
    _ok(lib().orc_quantize_q8_1(_ptr(x), m, k, k, _ptr(out)), "quantize_q8_1")
    return out


def quantize_weights(t: int, w: np.ndarray) -> np.ndarray:
    """fp32 [n, k] -> packed weight bytes [n, row_size]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    out = np.zeros((n, row_size(t, k)), dtype=np.uint8)
    _ok(lib().orc_quantize_weights(t, _ptr(w), n, k, _ptr(out)), "quantize_weights")
    return out


def dequantize_f32(t: int, w: np.ndarray, k: int) -> np.ndarray:
    """packed [rows, row_size] -> fp32 [rows, k] (fixed fp32 operation order)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    rows = w.shape[0]
    out = np.zeros((rows, k), dtype=np.float32)
    _ok(lib().orc_dequantize(t, _ptr(w), rows, k, _ptr(out), F32), "dequantize")
    return out


def dequantize(t: int, w: np.ndarray, k: int, ot: int = F32) -> np.ndarray:
    """packed -> out dtype; fp16/bf16 outputs are returned as uint16 bit patterns."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    rows = w.shape[0]
    out = np.zeros((rows, k), dtype=np.float32 if ot == F32 else np.uint16)
    _ok(lib().orc_dequantize(t, _ptr(w), rows, k, _ptr(out), ot), "dequantize")
    return out


def dequantize_f64(t: int, w: np.ndarray, k: int) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint8)
    rows = w.shape[0]
    out = np.zeros((rows, k), dtype=np.float64)
    for r in range(rows):
        _ok(lib().orc_dequantize_row_f64(t, _ptr(w[r]), k, out[r].ctypes.data), "dequantize_f64")
    return out


def get_rows(t: int, table: np.ndarray, k: int, ids: np.ndarray, ot: int = F32) -> np.ndarray:
    table = np.ascontiguousarray(table, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.zeros((ids.size, k), dtype=np.float32 if ot == F32 else np.uint16)
    _ok(lib().orc_get_rows(t, _ptr(table), table.shape[0], k, _ptr(ids), ids.size, _ptr(out), ot), "get_rows")
    return out


def block_dots(t: int, w: np.ndarray, k: int, xq: np.ndarray) -> np.ndarray:
    """int32 [m, n, k/sub] per-sub-block dot products."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    n, m = w.shape[0], xq.shape[0]
    out = np.zeros((m, n, k // sub_elems(t)), dtype=np.int32)
    _ok(lib().orc_block_dots(t, _ptr(w), n, k, _ptr(xq), m, _ptr(out)), "block_dots")
    return out


def mul_mat(t: int, w: np.ndarray, k: int, xq: np.ndarray, rows: tuple[int, int] | None = None,
            nthreads: int = 1) -> np.ndarray:
    """fp64 y[m, n] by the blockwise formula.  ``rows`` restricts the weight rows
    computed (others stay 0)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    n, m = w.shape[0], xq.shape[0]
    y = np.zeros((m, n), dtype=np.float64)
    n0, n1 = rows if rows is not None else (0, n)
    _ok(lib().orc_mul_mat_rows(t, _ptr(w), n, k, _ptr(xq), m, _ptr(y), n0, n1, nthreads), "mul_mat")
    return y


def mul_mat_dequant_f64(t: int, w: np.ndarray, k: int, xq: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    n, m = w.shape[0], xq.shape[0]
    y = np.zeros((m, n), dtype=np.float64)
    _ok(lib().orc_mul_mat_dequant_f64(t, _ptr(w), n, k, _ptr(xq), m, _ptr(y)), "mul_mat_dequant_f64")
    return y


def moe_gate_up(wt: int, bank: np.ndarray, n_experts: int, stride: int, two_i: int, h: int, xq: np.ndarray,
                ids: np.ndarray, routes: tuple[int, int] | None = None, nthreads: int = 1):
    """Returns (h_f32 [R, I] (bf16 values as fp32), h_q8_1 [R, I/32*36]) for all
    routes R = T * top_k; rows outside ``routes`` stay zero."""
    bank = np.ascontiguousarray(bank, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n_tokens, top_k = ids.shape
    i_dim = two_i // 2
    hbuf = np.zeros((n_tokens * top_k, i_dim), dtype=np.float32)
    hq = np.zeros((n_tokens * top_k, row_size(Q8_1, i_dim)), dtype=np.uint8)
    r0, r1 = routes if routes is not None else (0, n_tokens * top_k)
    _ok(lib().orc_moe_gate_up(wt, _ptr(bank), n_experts, stride, two_i, h, _ptr(xq), _ptr(ids), n_tokens, top_k,
                              _ptr(hbuf), _ptr(hq), r0, r1, nthreads), "moe_gate_up")
    return hbuf, hq


def moe_down(wt: int, bank: np.ndarray, n_experts: int, stride: int, n_out: int, i_dim: int, hq: np.ndarray,
             ids: np.ndarray, route_w: np.ndarray | None, tokens: tuple[int, int] | None = None,
             nthreads: int = 1) -> np.ndarray:
    """fp64 y[T, n_out] = sum_k w[t,k] * (W_down[e] . hq[route]); tokens outside
    ``tokens`` stay zero."""
    bank = np.ascontiguousarray(bank, dtype=np.uint8)
    hq = np.ascontiguousarray(hq, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n_tokens, top_k = ids.shape
    rw = None if route_w is None else np.ascontiguousarray(route_w, dtype=np.float32)
    y = np.zeros((n_tokens, n_out), dtype=np.float64)
    t0, t1 = tokens if tokens is not None else (0, n_tokens)
    _ok(lib().orc_moe_down(wt, _ptr(bank), n_experts, stride, n_out, i_dim, _ptr(hq), _ptr(ids), _ptr(rw),
                           n_tokens, top_k, _ptr(y), t0, t1, nthreads), "moe_down")
    return y


def moe_plain(wt: int, bank: np.ndarray, n_experts: int, stride: int, n: int, k: int, xq: np.ndarray,
              ids: np.ndarray) -> np.ndarray:
    """fp64 y[T * top_k, n]: route r = t * top_k + j gives W[ids[t, j]] . xq[t]
    (zero row for an inactive route)."""
    bank = np.ascontiguousarray(bank, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n_tokens, top_k = ids.shape
    y = np.zeros((n_tokens * top_k, n), dtype=np.float64)
    _ok(lib().orc_moe_plain(wt, _ptr(bank), n_experts, stride, n, k, _ptr(xq), _ptr(ids), n_tokens, top_k, _ptr(y)),
        "moe_plain")
    return y


def q8_1_fields(xq: np.ndarray):
    """Split q8_1 bytes [m, nb*36] into (d fp16 bits [m, nb], s fp16 bits [m, nb], q int8 [m, nb, 32])."""
    m = xq.shape[0]
    b = xq.reshape(m, -1, 36)
    d = b[:, :, 0].astype(np.uint16) | (b[:, :, 1].astype(np.uint16) << 8)
    s = b[:, :, 2].astype(np.uint16) | (b[:, :, 3].astype(np.uint16) << 8)
    q = b[:, :, 4:].view(np.int8)
    return d, s, q
