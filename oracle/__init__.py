"""CPU oracle for the FP8 (E4M3FN) per-token/per-head KV cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` arms of
``bench.py`` may import this package.  The product path (``fp8_kv_cache_ftkv_gb300``) never imports
it, and it never imports the product: the two share only the seeded input generators in
``fp8_kv_cache_ftkv_gb300.inputs``, which hold none of the method's arithmetic.

The arithmetic lives in ``ftkv_oracle.c`` (plain C, FP64 attention, one function per step, each citing
the page passage it follows).  This module compiles it with gcc on first use (or through
``build()``) and exposes numpy-level wrappers.  BF16 tensors are passed as ``uint16`` bit patterns.

Pins (what ties the oracle to something other than itself) live in ``tests/test_oracle_*.py``:
the codec against torch's ``float8_e4m3fn`` cast and the format's landmarks, the byte accounting
against the integers printed in FreeToken PR #853 ("Validation", "Follow-up model/workload
search"), and attention against torch's FP64 ``scaled_dot_product_attention`` plus closed-form
special cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ftkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libftkv_oracle.so")
_lib = None
_lock = threading.Lock()

E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (IEEE arithmetic, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.ftkv_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.ftkv_oracle_e4m3_decode.restype = f64
        lib.ftkv_oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.ftkv_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.ftkv_oracle_e4m3_encode_array.argtypes = [P, P, i64]
        lib.ftkv_oracle_e4m3_decode_array.argtypes = [P, P, i64]
        lib.ftkv_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.ftkv_oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.ftkv_oracle_store_quant.argtypes = [P, P, P, i64, i32, i32, P, P, P, P, i64]
        lib.ftkv_oracle_store_quant.restype = i32
        lib.ftkv_oracle_reconstruct.argtypes = [P, P, P, P, i64, i32, i32, P, i64, P, P]
        lib.ftkv_oracle_reconstruct.restype = i32
        lib.ftkv_oracle_decode_attn.argtypes = [P, P, P, P, i64, i32, i32, i32, P, P, i64, P, P, i32,
                                                f64, i64, i32, P]
        lib.ftkv_oracle_decode_attn.restype = i32
        lib.ftkv_oracle_decode_attn_bf16.argtypes = [P, P, i64, i32, i32, i32, P, P, i64, P, P, i32, f64, i64, i32, P]
        lib.ftkv_oracle_decode_attn_bf16.restype = i32
        lib.ftkv_oracle_prefill_attn.argtypes = [i32, i32, i32, P, P, P, i64, P, P, i64, f64, P, i64, i32, P]
        lib.ftkv_oracle_prefill_attn.restype = i32
        lib.ftkv_oracle_pool_bytes.argtypes = [i64, i64, i64, i64, P, P, P]
        lib.ftkv_oracle_set_threads.argtypes = [i32]
        lib.ftkv_oracle_get_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    _load().ftkv_oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().ftkv_oracle_get_threads())


# --------------------------------------------------------------------------------------------
# codec
# --------------------------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """E4M3FN byte codes -> float64 values (NaN for 0x7F/0xFF)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().ftkv_oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    """FP32 values -> E4M3FN codes (nearest, ties to even, saturating at +-448, NaN -> 0x7F)."""
    a = _c(x, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().ftkv_oracle_e4m3_encode_array(_ptr(a), _ptr(out), a.size)
    return out


def f32_to_bf16_bits(x: float) -> int:
    return int(_load().ftkv_oracle_f32_to_bf16(float(x)))


# --------------------------------------------------------------------------------------------
# pool
# --------------------------------------------------------------------------------------------
class Pool:
    """Host FP8 pool for one layer: codes uint8 [rows, Hkv, D], scales float32 [rows, Hkv]."""

    def __init__(self, num_rows: int, num_kv_heads: int, head_dim: int):
        self.num_rows, self.Hkv, self.D = int(num_rows), int(num_kv_heads), int(head_dim)
        self.k_codes = np.zeros((num_rows, num_kv_heads, head_dim), np.uint8)
        self.v_codes = np.zeros((num_rows, num_kv_heads, head_dim), np.uint8)
        self.k_scales = np.zeros((num_rows, num_kv_heads), np.float32)
        self.v_scales = np.zeros((num_rows, num_kv_heads), np.float32)


def store_quant(pool: Pool, k_bits, v_bits, slots) -> None:
    """Quantize-on-write of T tokens (BF16 bit patterns [T, Hkv, D]) into pool rows ``slots``."""
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    s = _c(slots, np.int32)
    T = s.shape[0]
    assert k.shape == (T, pool.Hkv, pool.D) and v.shape == k.shape
    rc = _load().ftkv_oracle_store_quant(_ptr(k), _ptr(v), _ptr(s), T, pool.Hkv, pool.D,
                                         _ptr(pool.k_codes), _ptr(pool.v_codes),
                                         _ptr(pool.k_scales), _ptr(pool.v_scales), pool.num_rows)
    if rc != 0:
        raise ValueError("slot out of range")


def reconstruct(pool: Pool, slots):
    """Rebuild rows ``slots`` (logical order) into BF16 workspaces; returns (ws_k, ws_v) uint16."""
    s = _c(slots, np.int32)
    P = s.shape[0]
    ws_k = np.empty((P, pool.Hkv, pool.D), np.uint16)
    ws_v = np.empty((P, pool.Hkv, pool.D), np.uint16)
    rc = _load().ftkv_oracle_reconstruct(_ptr(pool.k_codes), _ptr(pool.v_codes), _ptr(pool.k_scales),
                                         _ptr(pool.v_scales), pool.num_rows, pool.Hkv, pool.D,
                                         _ptr(s), P, _ptr(ws_k), _ptr(ws_v))
    if rc != 0:
        raise ValueError("slot out of range")
    return ws_k, ws_v


def _decode_args(q_bits, req_to_slot, seq_lens, q_row_offsets, num_q_heads, D):
    q = _c(q_bits, np.uint16)
    r2s = _c(req_to_slot, np.int32)
    if r2s.ndim == 1:
        r2s = r2s.reshape(1, -1)
    sl = _c(seq_lens, np.int32)
    qo = _c(q_row_offsets, np.int32)
    B = sl.shape[0]
    total = int(qo[B])
    assert q.shape == (total, num_q_heads, D)
    return q, r2s, sl, qo, B, np.empty((total, num_q_heads, D), np.float64)


def decode_attn(pool: Pool, q_bits, req_to_slot, seq_lens, q_row_offsets, sm_scale: float,
                num_q_heads: int, abs_v: bool = False, window: int = 0) -> np.ndarray:
    """FP64 decode attention over the FP8 pool; returns float64 [total_rows, Hq, D].

    ``window`` > 0: sliding window of the last ``window`` visible keys.  ``abs_v=True`` returns
    sum_j p_j |v_j| / sum_j p_j instead (a test helper that sizes rounding bounds)."""
    q, r2s, sl, qo, B, out = _decode_args(q_bits, req_to_slot, seq_lens, q_row_offsets, num_q_heads, pool.D)
    rc = _load().ftkv_oracle_decode_attn(_ptr(pool.k_codes), _ptr(pool.v_codes), _ptr(pool.k_scales),
                                         _ptr(pool.v_scales), pool.num_rows, num_q_heads, pool.Hkv,
                                         pool.D, _ptr(q), _ptr(r2s), r2s.shape[1], _ptr(sl), _ptr(qo), B,
                                         float(sm_scale), int(window), int(abs_v), _ptr(out))
    if rc != 0:
        raise ValueError("invalid decode arguments")
    return out


def decode_attn_bf16(k_bits, v_bits, q_bits, req_to_slot, seq_lens, q_row_offsets, sm_scale: float,
                     num_q_heads: int, abs_v: bool = False, window: int = 0) -> np.ndarray:
    """FP64 decode attention over a BF16 pool (k, v: BF16 bit patterns [rows, Hkv, D])."""
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    assert k.shape == v.shape and k.ndim == 3
    q, r2s, sl, qo, B, out = _decode_args(q_bits, req_to_slot, seq_lens, q_row_offsets, num_q_heads, k.shape[2])
    rc = _load().ftkv_oracle_decode_attn_bf16(_ptr(k), _ptr(v), k.shape[0], num_q_heads, k.shape[1], k.shape[2],
                                              _ptr(q), _ptr(r2s), r2s.shape[1], _ptr(sl), _ptr(qo), B,
                                              float(sm_scale), int(window), int(abs_v), _ptr(out))
    if rc != 0:
        raise ValueError("invalid decode arguments")
    return out


def prefill_attn(q_bits, k_chunk_bits, v_chunk_bits, ws_k_bits, ws_v_bits, sm_scale: float,
                 rows=None, abs_v: bool = False) -> np.ndarray:
    """FP64 causal prefill attention of chunk queries over prefix (+) chunk.

    Returns float64 [len(rows), Hq, D] (all C rows when ``rows`` is None)."""
    q = _c(q_bits, np.uint16)
    kc = _c(k_chunk_bits, np.uint16)
    vc = _c(v_chunk_bits, np.uint16)
    wk = _c(ws_k_bits, np.uint16)
    wv = _c(ws_v_bits, np.uint16)
    C, Hq, D = q.shape
    Hkv = kc.shape[1]
    P = wk.shape[0]
    if rows is None:
        r = None
        n = C
    else:
        r = _c(rows, np.int64)
        n = r.shape[0]
    out = np.empty((n, Hq, D), np.float64)
    rc = _load().ftkv_oracle_prefill_attn(Hq, Hkv, D, _ptr(q), _ptr(kc), _ptr(vc), C,
                                          _ptr(wk) if P else None, _ptr(wv) if P else None, P,
                                          float(sm_scale), _ptr(r) if r is not None else None, n,
                                          int(abs_v), _ptr(out))
    if rc != 0:
        raise ValueError("invalid prefill arguments")
    return out


def pool_bytes(rows: int, layers: int, num_kv_heads: int, head_dim: int) -> dict:
    """Byte accounting: persistent BF16 KV, persistent FP8 codes+scales, one-layer BF16 workspace."""
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _load().ftkv_oracle_pool_bytes(rows, layers, num_kv_heads, head_dim, ctypes.byref(a),
                                   ctypes.byref(b), ctypes.byref(c))
    return {"bf16": a.value, "fp8": b.value, "workspace": c.value}
