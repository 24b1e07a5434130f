"""CPU oracle for paged multi-token attention, the paged KV append and block swap.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The product path never imports this
package, and this package imports nothing from the product package.

``oracle.c`` holds the definition (fp64, plain loops, one output row at a
time); this module compiles it with gcc, loads it with ctypes and wraps it for
numpy arrays.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(brute force, closed forms, permutation invariance, library routines).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP when available)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_paged_attn_rows.argtypes = [P, P, P, I, I, I, I, I, P, I, P, P, P, I, D, P, P, I, P, P]
            lib.oracle_paged_attn.argtypes = [P, P, P, I, I, I, I, I, P, I, P, P, P, I, I, D, P, P]
            lib.oracle_append.argtypes = [P, P, I, I, I, I, P, I, P, P, I, I, P, P]
            lib.oracle_swap_out.argtypes = [P, P, I, I, I, I, P, I, P]
            lib.oracle_swap_in.argtypes = [P, P, I, I, I, I, P, I, P]
            lib.oracle_paged_attn_rows_fp8.argtypes = [P, P, P, D, D, I, I, I, I, I, P, I, P, P, P, I, D, P, P, I,
                                                       P, P]
            lib.oracle_append_fp8.argtypes = [P, P, ctypes.c_float, ctypes.c_float, I, I, I, I, P, I, P, P, I, I,
                                              P, P]
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = D
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            for f in (lib.oracle_paged_attn_rows, lib.oracle_paged_attn, lib.oracle_append,
                      lib.oracle_swap_out, lib.oracle_swap_in, lib.oracle_paged_attn_rows_fp8,
                      lib.oracle_append_fp8):
                f.restype = I
            lib.oracle_num_threads.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paged_attn(q, k_pool, v_pool, block_tables, ctx_lens, cu_q_lens, q_positions, scale,
               num_kv_heads=None):
    """Full oracle attention.  q [T,Hq,D], pools [NB,Hkv,B,D] (bf16 bits, uint16).

    Returns (O [T,Hq,D] fp64, LSE [T,Hq] fp64).  Raises ValueError on a
    precondition violation (position >= ctx, bad block id, Hq % Hkv != 0).
    """
    lib = _load()
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    bt = _c(block_tables, np.int32)
    ctx = _c(ctx_lens, np.int32)
    cu = _c(cu_q_lens, np.int32)
    pos = _c(q_positions, np.int32)
    T, Hq, D = q.shape
    NB, Hkv, B, D2 = k_pool.shape
    assert D == D2
    out = np.zeros((T, Hq, D), np.float64)
    lse = np.zeros((T, Hq), np.float64)
    rc = lib.oracle_paged_attn(_p(q), _p(k_pool), _p(v_pool), NB, Hkv, B, D, Hq, _p(bt),
                               bt.shape[1], _p(ctx), _p(cu), _p(pos), ctx.shape[0], T,
                               float(scale), _p(out), _p(lse))
    if rc:
        raise ValueError("oracle_paged_attn: precondition violated")
    return out, lse


def paged_attn_rows(q, k_pool, v_pool, block_tables, ctx_lens, cu_q_lens, q_positions, scale,
                    rows_t, rows_h):
    """Oracle attention for selected (token, query head) rows; returns (O [n,D], LSE [n])."""
    lib = _load()
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    bt = _c(block_tables, np.int32)
    ctx = _c(ctx_lens, np.int32)
    cu = _c(cu_q_lens, np.int32)
    pos = _c(q_positions, np.int32)
    rt = _c(rows_t, np.int32)
    rh = _c(rows_h, np.int32)
    T, Hq, D = q.shape
    NB, Hkv, B, _ = k_pool.shape
    n = rt.shape[0]
    out = np.zeros((n, D), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = lib.oracle_paged_attn_rows(_p(q), _p(k_pool), _p(v_pool), NB, Hkv, B, D, Hq, _p(bt),
                                    bt.shape[1], _p(ctx), _p(cu), _p(pos), ctx.shape[0],
                                    float(scale), _p(rt), _p(rh), n, _p(out), _p(lse))
    if rc:
        raise ValueError("oracle_paged_attn_rows: precondition violated")
    return out, lse


# ----------------------------------------------------------------------------- FP8 (E4M3) KV cache

def e4m3_decode(codes) -> np.ndarray:
    """Values (fp64) of E4M3 codes (uint8 array), from the format's definition."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_decode(c) for c in range(256)], np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, finite values saturating) of float32 values."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).ravel()
    out = np.fromiter((lib.oracle_e4m3_encode(float(v)) for v in flat), dtype=np.uint8, count=flat.size)
    return out.reshape(np.shape(x))


def paged_attn_rows_fp8(q, k_pool, v_pool, k_scale, v_scale, block_tables, ctx_lens, cu_q_lens, q_positions,
                        scale, rows_t, rows_h):
    """Oracle attention over FP8 pools (uint8 E4M3 codes [NB,Hkv,B,D]) for selected rows."""
    lib = _load()
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint8)
    v_pool = _c(v_pool, np.uint8)
    bt = _c(block_tables, np.int32)
    ctx = _c(ctx_lens, np.int32)
    cu = _c(cu_q_lens, np.int32)
    pos = _c(q_positions, np.int32)
    rt = _c(rows_t, np.int32)
    rh = _c(rows_h, np.int32)
    T, Hq, D = q.shape
    NB, Hkv, B, _ = k_pool.shape
    n = rt.shape[0]
    out = np.zeros((n, D), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = lib.oracle_paged_attn_rows_fp8(_p(q), _p(k_pool), _p(v_pool), float(np.float32(k_scale)),
                                        float(np.float32(v_scale)), NB, Hkv, B, D, Hq, _p(bt), bt.shape[1],
                                        _p(ctx), _p(cu), _p(pos), ctx.shape[0], float(scale), _p(rt), _p(rh), n,
                                        _p(out), _p(lse))
    if rc:
        raise ValueError("oracle_paged_attn_rows_fp8: precondition violated")
    return out, lse


def paged_attn_fp8(q, k_pool, v_pool, k_scale, v_scale, block_tables, ctx_lens, cu_q_lens, q_positions, scale):
    """Full oracle attention over FP8 pools; returns (O [T,Hq,D], LSE [T,Hq]) in fp64."""
    T, Hq, D = np.shape(q)
    rt = np.repeat(np.arange(T, dtype=np.int32), Hq)
    rh = np.tile(np.arange(Hq, dtype=np.int32), T)
    o, l = paged_attn_rows_fp8(q, k_pool, v_pool, k_scale, v_scale, block_tables, ctx_lens, cu_q_lens,
                               q_positions, scale, rt, rh)
    return o.reshape(T, Hq, D), l.reshape(T, Hq)


def append_fp8(k_pool, v_pool, k_scale, v_scale, block_tables, cu_q_lens, positions, k_new, v_new):
    """In-place FP8 append: new bf16 rows (uint16 bits) quantised into uint8 code pools."""
    lib = _load()
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == np.uint8 and v_pool.dtype == np.uint8
    bt = _c(block_tables, np.int32)
    cu = _c(cu_q_lens, np.int32)
    pos = _c(positions, np.int32)
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    NB, Hkv, B, D = k_pool.shape
    rc = lib.oracle_append_fp8(_p(k_pool), _p(v_pool), float(k_scale), float(v_scale), NB, Hkv, B, D, _p(bt),
                               bt.shape[1], _p(cu), _p(pos), cu.shape[0] - 1, pos.shape[0], _p(kn), _p(vn))
    if rc:
        raise ValueError("oracle_append_fp8: slot out of range")


def append(k_pool, v_pool, block_tables, cu_q_lens, positions, k_new, v_new):
    """In-place oracle append into numpy pools (uint16 bf16 bits)."""
    lib = _load()
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == np.uint16 and v_pool.dtype == np.uint16
    bt = _c(block_tables, np.int32)
    cu = _c(cu_q_lens, np.int32)
    pos = _c(positions, np.int32)
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    NB, Hkv, B, D = k_pool.shape
    rc = lib.oracle_append(_p(k_pool), _p(v_pool), NB, Hkv, B, D, _p(bt), bt.shape[1], _p(cu),
                           _p(pos), cu.shape[0] - 1, pos.shape[0], _p(kn), _p(vn))
    if rc:
        raise ValueError("oracle_append: slot out of range")


def swap_out(k_pool, v_pool, ids):
    """Return host buffer [n,2,Hkv,B,D] holding blocks ``ids`` (K then V)."""
    lib = _load()
    ids = _c(ids, np.int32)
    NB, Hkv, B, D = k_pool.shape
    host = np.zeros((ids.shape[0], 2, Hkv, B, D), np.uint16)
    rc = lib.oracle_swap_out(_p(_c(k_pool, np.uint16)), _p(_c(v_pool, np.uint16)), NB, Hkv, B, D,
                             _p(ids), ids.shape[0], _p(host))
    if rc:
        raise ValueError("oracle_swap_out: block id out of range")
    return host


def swap_in(k_pool, v_pool, ids, host):
    """In-place: write host [n,2,Hkv,B,D] into blocks ``ids`` of the pools."""
    lib = _load()
    ids = _c(ids, np.int32)
    host = _c(host, np.uint16)
    NB, Hkv, B, D = k_pool.shape
    rc = lib.oracle_swap_in(_p(k_pool), _p(v_pool), NB, Hkv, B, D, _p(ids), ids.shape[0], _p(host))
    if rc:
        raise ValueError("oracle_swap_in: block id out of range")

