"""ctypes loader for libftkv.so: the C ABI declared in include/ftkv.h, nothing else.

The library is built in-tree by ``fp8_kv_cache_ftkv_gb300.build`` (``__graft_entry__.build()`` does it).
Loading fails loudly -- there is no CPU fallback anywhere in the product path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libftkv.so")

FTKV_OK = 0
FTKV_ERR_INVALID = -1
FTKV_ERR_UNSUPPORTED = -2
FTKV_ERR_ALIGN = -3
FTKV_ERR_WORKSPACE = -4
FTKV_ERR_CUDA = -6
FTKV_MAX_SPLITS = 256
FTKV_MAX_Q_ROWS = 8
FTKV_MAX_BATCH = 65535
FTKV_DECODE_STABLE_HISTORY = 0x1
FTKV_DEVERR_BAD_SLOT = 0x1
FTKV_DEVERR_SEQ_LEN = 0x2
FTKV_DEVERR_Q_ROWS = 0x4
FTKV_DEVERR_TIMEOUT = 0x8
FTKV_NOALLOC_SCRATCH_BYTES = 16 << 20

# Every symbol include/ftkv.h declares.
EXPORTS = (
    "ftkv_store_quant", "ftkv_reconstruct_bf16", "ftkv_decode_workspace_bytes", "ftkv_decode_auto_splits",
    "ftkv_decode_attn", "ftkv_prefill_attn", "ftkv_prefill_attn_ws", "ftkv_prefill_workspace_bytes",
    "ftkv_e4m3_encode_f32", "ftkv_e4m3_decode_f32", "ftkv_pool_bytes", "ftkv_device_errors", "ftkv_status_str",
    "ftkv_last_cuda_error", "ftkv_abi_version", "ftkv_decode_attn_noalloc", "ftkv_decode_attn_store",
    "ftkv_decode_attn_bf16", "ftkv_gather_bf16",
)


class FtkvPool(ctypes.Structure):
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("num_rows", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
    ]


class FtkvBf16Pool(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("num_rows", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
    ]


class FtkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} {last_cuda_error()}".strip())


_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libftkv.so is not built ({LIB_PATH}); run fp8_kv_cache_ftkv_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F32, SZ, U32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t,
                                     ctypes.c_uint32)
        PP = ctypes.POINTER(FtkvPool)
        PB = ctypes.POINTER(FtkvBf16Pool)
        sig = {
            "ftkv_store_quant": (ctypes.c_int, [PP, P, P, P, I64, P]),
            "ftkv_reconstruct_bf16": (ctypes.c_int, [PP, P, I64, P, P, P]),
            "ftkv_decode_workspace_bytes": (SZ, [I32, I32, I32, I32, I64, I32]),
            "ftkv_decode_auto_splits": (I32, [I32, I32, I64, I32]),
            "ftkv_decode_attn": (ctypes.c_int, [PP, I32, P, P, I64, P, P, I32, I64, I32, I64, F32, I64, I32, U32, P,
                                                SZ, P, P]),
            "ftkv_decode_attn_store": (ctypes.c_int, [PP, I32, P, P, P, P, I64, P, P, I32, I64, I32, I64, F32, I64,
                                                      I32, U32, P, SZ, P, P]),
            "ftkv_decode_attn_bf16": (ctypes.c_int, [PB, I32, P, P, P, P, I64, P, P, I32, I64, I32, I64, F32, I64,
                                                     I32, U32, P, SZ, P, P]),
            "ftkv_gather_bf16": (ctypes.c_int, [PB, P, I64, P, P, P]),
            "ftkv_decode_attn_noalloc": (ctypes.c_int, [PP, I32, P, P, I64, P, P, I32, I64, I32, I64, F32, I32, P,
                                                        P]),
            "ftkv_prefill_attn": (ctypes.c_int, [I32, I32, I32, P, P, P, I64, P, P, I64, F32, P, P]),
            "ftkv_prefill_attn_ws": (ctypes.c_int, [I32, I32, I32, P, P, P, I64, P, P, I64, F32, I32, P, I64, P, P]),
            "ftkv_prefill_workspace_bytes": (I64, [I32]),
            "ftkv_e4m3_encode_f32": (ctypes.c_int, [P, P, I64, P]),
            "ftkv_e4m3_decode_f32": (ctypes.c_int, [P, P, I64, P]),
            "ftkv_pool_bytes": (ctypes.c_int, [I64, I32, I32, I32, P, P, P]),
            "ftkv_device_errors": (ctypes.c_int, [ctypes.POINTER(I32)]),
            "ftkv_status_str": (ctypes.c_char_p, [ctypes.c_int]),
            "ftkv_last_cuda_error": (ctypes.c_char_p, []),
            "ftkv_abi_version": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_str(status: int) -> str:
    return load().ftkv_status_str(int(status)).decode()


def last_cuda_error() -> str:
    return load().ftkv_last_cuda_error().decode()


def check(status: int, what: str) -> None:
    if status != FTKV_OK:
        raise FtkvError(status, what)
