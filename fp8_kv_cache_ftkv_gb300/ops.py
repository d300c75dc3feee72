"""Torch-tensor front end of libftkv.so: argument marshalling only.

Every function checks device/dtype/shape/contiguity, passes raw device pointers and the current CUDA
stream to the C ABI and returns.  All arithmetic happens in the CUDA kernels behind the ABI; there is no
CPU or PyTorch fallback.  BF16 tensors are ``torch.bfloat16`` (passed as their 16-bit patterns).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import FtkvBf16Pool, FtkvPool, check

HEAD_DIM = 128


def _stream_ptr(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _req(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


@dataclass
class KVPool:
    """One layer's FP8 pool on the GPU: codes uint8 [rows, Hkv, 128], scales float32 [rows, Hkv]."""
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_scales: torch.Tensor
    v_scales: torch.Tensor

    @staticmethod
    def empty(num_rows: int, num_kv_heads: int, device="cuda", head_dim: int = HEAD_DIM) -> "KVPool":
        z = dict(device=device)
        return KVPool(torch.zeros(num_rows, num_kv_heads, head_dim, dtype=torch.uint8, **z),
                      torch.zeros(num_rows, num_kv_heads, head_dim, dtype=torch.uint8, **z),
                      torch.zeros(num_rows, num_kv_heads, dtype=torch.float32, **z),
                      torch.zeros(num_rows, num_kv_heads, dtype=torch.float32, **z))

    @property
    def num_rows(self) -> int:
        return self.k_codes.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.k_codes.shape[1]

    @property
    def head_dim(self) -> int:
        return self.k_codes.shape[2]

    def c_struct(self) -> FtkvPool:
        for n in ("k_codes", "v_codes"):
            _req(getattr(self, n), torch.uint8, n, 3)
        for n in ("k_scales", "v_scales"):
            _req(getattr(self, n), torch.float32, n, 2)
        return FtkvPool(self.k_codes.data_ptr(), self.v_codes.data_ptr(), self.k_scales.data_ptr(),
                        self.v_scales.data_ptr(), self.k_codes.shape[0], self.k_codes.shape[1],
                        self.k_codes.shape[2])


@dataclass
class BF16Pool:
    """One layer's unquantized pool on the GPU (the comparison point): K and V bfloat16 [rows, Hkv, 128]."""
    k: torch.Tensor
    v: torch.Tensor

    @staticmethod
    def empty(num_rows: int, num_kv_heads: int, device="cuda", head_dim: int = HEAD_DIM) -> "BF16Pool":
        return BF16Pool(torch.zeros(num_rows, num_kv_heads, head_dim, dtype=torch.bfloat16, device=device),
                        torch.zeros(num_rows, num_kv_heads, head_dim, dtype=torch.bfloat16, device=device))

    @property
    def num_rows(self) -> int:
        return self.k.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.k.shape[1]

    def c_struct(self) -> FtkvBf16Pool:
        _req(self.k, torch.bfloat16, "k", 3)
        _req(self.v, torch.bfloat16, "v", 3)
        if self.v.shape != self.k.shape:
            raise ValueError("k and v pools disagree")
        return FtkvBf16Pool(self.k.data_ptr(), self.v.data_ptr(), self.k.shape[0], self.k.shape[1], self.k.shape[2])


def store_quant(pool: KVPool, k: torch.Tensor, v: torch.Tensor, slots: torch.Tensor, stream=None) -> None:
    """Quantize-on-write of BF16 K/V [T, Hkv, D] into pool rows ``slots`` (int32 [T]); D = the pool's head_dim."""
    _req(k, torch.bfloat16, "k", 3)
    _req(v, torch.bfloat16, "v", 3)
    _req(slots, torch.int32, "slots", 1)
    if k.shape != v.shape or k.shape[0] != slots.shape[0]:
        raise ValueError("k, v, slots disagree")
    if k.shape[1:] != (pool.num_kv_heads, pool.head_dim):
        raise ValueError(f"k/v rows must be [{pool.num_kv_heads}, {pool.head_dim}]")
    ps = pool.c_struct()
    check(_lib.load().ftkv_store_quant(ctypes.byref(ps), _ptr(k), _ptr(v), _ptr(slots), k.shape[0],
                                       _stream_ptr(stream)), "ftkv_store_quant")


def reconstruct_bf16(pool: KVPool, slots: torch.Tensor, ws_k: torch.Tensor = None, ws_v: torch.Tensor = None,
                     stream=None):
    """Rebuild rows ``slots`` (logical order) into BF16 workspaces [P, Hkv, 128]; returns (ws_k, ws_v)."""
    _req(slots, torch.int32, "slots", 1)
    P = slots.shape[0]
    shape = (P, pool.num_kv_heads, HEAD_DIM)
    if ws_k is None:
        ws_k = torch.empty(shape, dtype=torch.bfloat16, device=slots.device)
    if ws_v is None:
        ws_v = torch.empty(shape, dtype=torch.bfloat16, device=slots.device)
    _req(ws_k, torch.bfloat16, "ws_k", 3)
    _req(ws_v, torch.bfloat16, "ws_v", 3)
    if ws_k.shape[0] < P or ws_v.shape[0] < P:
        raise ValueError("workspace too small")
    ps = pool.c_struct()
    check(_lib.load().ftkv_reconstruct_bf16(ctypes.byref(ps), _ptr(slots), P, _ptr(ws_k), _ptr(ws_v),
                                            _stream_ptr(stream)), "ftkv_reconstruct_bf16")
    return ws_k, ws_v


def decode_workspace_bytes(num_q_heads: int, num_kv_heads: int, batch: int, total_q_rows: int,
                           num_splits: int, head_dim: int = HEAD_DIM) -> int:
    return int(_lib.load().ftkv_decode_workspace_bytes(num_q_heads, num_kv_heads, head_dim, batch, total_q_rows,
                                                       num_splits))


def decode_auto_splits(batch: int, num_kv_heads: int, max_seq_len: int, max_q_rows: int = 1) -> int:
    return int(_lib.load().ftkv_decode_auto_splits(batch, num_kv_heads, max_seq_len, max_q_rows))


class DecodePlan:
    """Host-side decode geometry + the zero-filled workspace it needs (allocated once, reused by every call
    on one stream; the kernels leave its arrival counters at zero)."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, batch: int, total_q_rows: int, max_q_rows: int,
                 max_seq_len: int, num_splits: int = 0, device="cuda", window: int = 0, head_dim: int = HEAD_DIM):
        self.num_q_heads, self.num_kv_heads = num_q_heads, num_kv_heads
        self.batch, self.total_q_rows, self.max_q_rows = batch, total_q_rows, max_q_rows
        self.max_seq_len, self.window = max_seq_len, window
        # keys one request attends to at most: with a sliding window, the union of its rows' windows
        span = min(max_seq_len, window + max_q_rows - 1) if window > 0 else max_seq_len
        self.num_splits = num_splits or decode_auto_splits(batch, num_kv_heads, span, max_q_rows)
        nbytes = decode_workspace_bytes(num_q_heads, num_kv_heads, batch, total_q_rows, self.num_splits, head_dim)
        self.workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def decode_attn(pool: KVPool, q: torch.Tensor, req_to_slot: torch.Tensor, seq_lens: torch.Tensor,
                q_row_offsets: torch.Tensor = None, *, max_seq_len: int, max_q_rows: int = 1,
                sm_scale: float = None, window: int = 0, num_splits: int = 0,
                plan: DecodePlan = None, out: torch.Tensor = None, k_new: torch.Tensor = None,
                v_new: torch.Tensor = None, stable_history: bool = False, stream=None) -> torch.Tensor:
    """Split-K decode attention over the FP8 pool.  q/out: BF16 [total_q_rows, Hq, D] (D = the pool's head_dim,
    128 or 256; 256 with one row per request).  ``sm_scale`` defaults to D^-1/2.
    ``window`` > 0: sliding window -- a row that sees keys 0 .. v-1 attends to keys max(0, v - window) .. v-1.
    ``k_new``/``v_new`` (BF16 [total_q_rows, Hkv, 128], the new tokens' rows, one per query row): quantize them
    into the pool at their positions' slots first, in the same launch (``ftkv_decode_attn_store``).
    ``stable_history``: pass FTKV_DECODE_STABLE_HISTORY -- the caller guarantees that no work still pending on the
    stream writes the slot table, the sequence lengths or the history rows, so the kernel may start loading them
    before the preceding kernel has finished."""
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        _req(k_new, torch.bfloat16, "k_new", 3)
        _req(v_new, torch.bfloat16, "v_new", 3)
    _req(q, torch.bfloat16, "q", 3)
    if req_to_slot.dim() == 1:
        req_to_slot = req_to_slot.view(1, -1)
    _req(req_to_slot, torch.int32, "req_to_slot", 2)
    _req(seq_lens, torch.int32, "seq_lens", 1)
    if q_row_offsets is not None:
        _req(q_row_offsets, torch.int32, "q_row_offsets", 1)
    batch = seq_lens.shape[0]
    total, hq, D = q.shape
    if D != pool.head_dim:
        raise ValueError(f"q has head_dim {D}, the pool {pool.head_dim}")
    if sm_scale is None:
        sm_scale = D ** -0.5
    if plan is None:
        plan = DecodePlan(hq, pool.num_kv_heads, batch, total, max_q_rows, max_seq_len, num_splits, q.device,
                          window, D)
    if out is None:
        out = torch.empty_like(q)
    _req(out, torch.bfloat16, "out", 3)
    flags = _lib.FTKV_DECODE_STABLE_HISTORY if stable_history else 0
    ps = pool.c_struct()
    if k_new is not None:
        if k_new.shape != (total, pool.num_kv_heads, D) or v_new.shape != k_new.shape:
            raise ValueError(f"k_new/v_new must be [{total}, {pool.num_kv_heads}, {D}]")
        check(_lib.load().ftkv_decode_attn_store(
            ctypes.byref(ps), hq, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(req_to_slot), req_to_slot.shape[1],
            _ptr(seq_lens), _ptr(q_row_offsets), batch, total, max_q_rows, max_seq_len, float(sm_scale),
            int(window), plan.num_splits, flags, _ptr(plan.workspace), plan.workspace.numel(), _ptr(out),
            _stream_ptr(stream)),
            "ftkv_decode_attn_store")
        return out
    check(_lib.load().ftkv_decode_attn(
        ctypes.byref(ps), hq, _ptr(q), _ptr(req_to_slot), req_to_slot.shape[1], _ptr(seq_lens),
        _ptr(q_row_offsets), batch, total, max_q_rows, max_seq_len, float(sm_scale), int(window), plan.num_splits,
        flags,
        _ptr(plan.workspace), plan.workspace.numel(), _ptr(out), _stream_ptr(stream)), "ftkv_decode_attn")
    return out


def decode_attn_bf16(pool: BF16Pool, q: torch.Tensor, req_to_slot: torch.Tensor, seq_lens: torch.Tensor,
                     q_row_offsets: torch.Tensor = None, *, max_seq_len: int, max_q_rows: int = 1,
                     sm_scale: float = HEAD_DIM ** -0.5, window: int = 0, num_splits: int = 0,
                     plan: DecodePlan = None, out: torch.Tensor = None, k_new: torch.Tensor = None,
                     v_new: torch.Tensor = None, stable_history: bool = False, stream=None) -> torch.Tensor:
    """Split-K decode attention over a BF16 pool (``ftkv_decode_attn_bf16``); the arguments of ``decode_attn``.
    ``k_new``/``v_new``: the new tokens' rows are copied into the pool and attended from these tensors."""
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    _req(q, torch.bfloat16, "q", 3)
    if req_to_slot.dim() == 1:
        req_to_slot = req_to_slot.view(1, -1)
    _req(req_to_slot, torch.int32, "req_to_slot", 2)
    _req(seq_lens, torch.int32, "seq_lens", 1)
    if q_row_offsets is not None:
        _req(q_row_offsets, torch.int32, "q_row_offsets", 1)
    batch = seq_lens.shape[0]
    total, hq, _ = q.shape
    if k_new is not None:
        _req(k_new, torch.bfloat16, "k_new", 3)
        _req(v_new, torch.bfloat16, "v_new", 3)
        if k_new.shape != (total, pool.num_kv_heads, HEAD_DIM) or v_new.shape != k_new.shape:
            raise ValueError(f"k_new/v_new must be [{total}, {pool.num_kv_heads}, {HEAD_DIM}]")
    if plan is None:
        plan = DecodePlan(hq, pool.num_kv_heads, batch, total, max_q_rows, max_seq_len, num_splits, q.device,
                          window)
    if out is None:
        out = torch.empty_like(q)
    _req(out, torch.bfloat16, "out", 3)
    flags = _lib.FTKV_DECODE_STABLE_HISTORY if stable_history else 0
    ps = pool.c_struct()
    check(_lib.load().ftkv_decode_attn_bf16(
        ctypes.byref(ps), hq, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(req_to_slot), req_to_slot.shape[1],
        _ptr(seq_lens), _ptr(q_row_offsets), batch, total, max_q_rows, max_seq_len, float(sm_scale), int(window),
        plan.num_splits, flags, _ptr(plan.workspace), plan.workspace.numel(), _ptr(out), _stream_ptr(stream)),
        "ftkv_decode_attn_bf16")
    return out


def gather_bf16(pool: BF16Pool, slots: torch.Tensor, ws_k: torch.Tensor = None, ws_v: torch.Tensor = None,
                stream=None):
    """Gather BF16 pool rows ``slots`` (logical order) into workspaces [P, Hkv, 128]; returns (ws_k, ws_v)."""
    _req(slots, torch.int32, "slots", 1)
    P = slots.shape[0]
    shape = (P, pool.num_kv_heads, HEAD_DIM)
    if ws_k is None:
        ws_k = torch.empty(shape, dtype=torch.bfloat16, device=slots.device)
    if ws_v is None:
        ws_v = torch.empty(shape, dtype=torch.bfloat16, device=slots.device)
    _req(ws_k, torch.bfloat16, "ws_k", 3)
    _req(ws_v, torch.bfloat16, "ws_v", 3)
    if ws_k.shape[0] < P or ws_v.shape[0] < P:
        raise ValueError("workspace too small")
    ps = pool.c_struct()
    check(_lib.load().ftkv_gather_bf16(ctypes.byref(ps), _ptr(slots), P, _ptr(ws_k), _ptr(ws_v),
                                       _stream_ptr(stream)), "ftkv_gather_bf16")
    return ws_k, ws_v


def prefill_workspace_bytes(max_ctas: int = 0) -> int:
    n = int(_lib.load().ftkv_prefill_workspace_bytes(max_ctas))
    if n < 0:
        raise RuntimeError("ftkv_prefill_workspace_bytes: the current device could not be queried")
    return n


class PrefillPlan:
    """Zero-filled stream-K workspace for ``prefill_attn`` (allocated once; calls that share it must be
    ordered on one stream; the kernel leaves its tickets at zero)."""

    def __init__(self, max_ctas: int = 0, device="cuda"):
        self.max_ctas = max_ctas
        self.workspace = torch.zeros(prefill_workspace_bytes(max_ctas), dtype=torch.uint8, device=device)


def prefill_attn(q: torch.Tensor, k_chunk: torch.Tensor, v_chunk: torch.Tensor, ws_k: torch.Tensor = None,
                 ws_v: torch.Tensor = None, *, sm_scale: float = HEAD_DIM ** -0.5, out: torch.Tensor = None,
                 plan: PrefillPlan = None, stream=None) -> torch.Tensor:
    """Causal prefill of the chunk over prefix (+) chunk on the tcgen05 kernel.  With ``plan`` the launch is
    scheduled stream-K over the plan's workspace (``ftkv_prefill_attn_ws``)."""
    _req(q, torch.bfloat16, "q", 3)
    _req(k_chunk, torch.bfloat16, "k_chunk", 3)
    _req(v_chunk, torch.bfloat16, "v_chunk", 3)
    C, hq, _ = q.shape
    hkv = k_chunk.shape[1]
    P = 0 if ws_k is None else ws_k.shape[0]
    if P:
        _req(ws_k, torch.bfloat16, "ws_k", 3)
        _req(ws_v, torch.bfloat16, "ws_v", 3)
    if out is None:
        out = torch.empty_like(q)
    _req(out, torch.bfloat16, "out", 3)
    args = (hq, hkv, HEAD_DIM, _ptr(q), _ptr(k_chunk), _ptr(v_chunk), C, _ptr(ws_k) if P else None,
            _ptr(ws_v) if P else None, P, float(sm_scale))
    if plan is not None:
        check(_lib.load().ftkv_prefill_attn_ws(*args, plan.max_ctas, _ptr(plan.workspace), plan.workspace.numel(),
                                                _ptr(out), _stream_ptr(stream)), "ftkv_prefill_attn_ws")
        return out
    check(_lib.load().ftkv_prefill_attn(*args, _ptr(out), _stream_ptr(stream)), "ftkv_prefill_attn")
    return out


def e4m3_encode(x: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    _req(x, torch.float32, "x")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    check(_lib.load().ftkv_e4m3_encode_f32(_ptr(x), _ptr(out), x.numel(), _stream_ptr(stream)), "e4m3_encode")
    return out


def e4m3_decode(c: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    _req(c, torch.uint8, "codes")
    if out is None:
        out = torch.empty(c.shape, dtype=torch.float32, device=c.device)
    check(_lib.load().ftkv_e4m3_decode_f32(_ptr(c), _ptr(out), c.numel(), _stream_ptr(stream)), "e4m3_decode")
    return out


def pool_bytes(rows: int, layers: int, num_kv_heads: int, head_dim: int = HEAD_DIM) -> dict:
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    check(_lib.load().ftkv_pool_bytes(rows, layers, num_kv_heads, head_dim, ctypes.byref(a), ctypes.byref(b),
                                      ctypes.byref(c)), "ftkv_pool_bytes")
    return {"bf16": a.value, "fp8": b.value, "workspace": c.value}


def device_errors() -> int:
    v = ctypes.c_int32()
    check(_lib.load().ftkv_device_errors(ctypes.byref(v)), "ftkv_device_errors")
    return v.value
