"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module draws random numbers and nothing else: it holds none of the method's arithmetic (no
quantization, no attention).  Every tensor is drawn with numpy's PCG64 in FP32 and rounded to BF16
(round-to-nearest-even, by torch's dtype cast); BF16 tensors are returned as ``uint16`` bit patterns
so that the oracle and the GPU path receive the identical bits.

Workloads (shapes and value distributions of the FP8 KV-cache workloads; seeds are 1000 + id):

* ``decode_small``    -- one layer, batch 1, Hq=32, Hkv=4, D=128, 512-token context in a 1,024-row pool,
  slots = first 512 entries of a permutation of the pool rows.  K/V = N(0,1) x per-token LogN(0,1).
* ``store``           -- quantize-on-write of 8,192 tokens per layer into a 33,059-row pool; K/V =
  N(0,1) x per-token LogN(0,2), 1 % of tokens x1e3, 0.1 % all-zero (chosen independently for K and V).
  The same 8,192 slots serve every layer.
* ``decode_long``     -- batch 1 at 32,768 keys in a 33,059-row pool (or 40,000 in 40,290), one pool
  per layer, distributions as ``decode_small``; the slot permutation is shared by all layers.
* ``prefill``         -- 8,192 historical rows (33,059-row pool) then 8,192 new tokens in chunks of
  2,048; distributions as ``decode_small``.
* ``decode_batched``  -- 64 requests, context ~ U[1,024, 40,000], 1..8 query rows each, 2,000,000-row
  pool, one permutation cut into consecutive blocks; magnitudes as ``store``.

The per-token magnitude is one draw per (token, tensor) shared by all KV heads of the token.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HQ, HKV, D = 32, 4, 128
SM_SCALE = float(np.float32(1.0 / np.sqrt(128.0)))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 array -> BF16 bit patterns (uint16), round-to-nearest-even (torch dtype cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> FP32 values (exact widening)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


def kv_tokens(rng: np.random.Generator, T: int, sigma: float, big_frac: float = 0.0,
              zero_frac: float = 0.0, Hkv: int = HKV, head_dim: int = D):
    """K and V for T tokens: N(0,1) times one LogN(0, sigma) magnitude per (token, tensor).

    ``big_frac`` of the tokens are scaled x1e3 and ``zero_frac`` are all-zero, chosen independently
    for K and V.  Returns (k_bits, v_bits), uint16 [T, Hkv, head_dim]."""
    out = []
    for _ in range(2):
        x = rng.standard_normal((T, Hkv, head_dim), dtype=np.float32)
        mag = rng.lognormal(0.0, sigma, size=T).astype(np.float32)
        if big_frac > 0:
            mag[rng.random(T) < big_frac] *= np.float32(1e3)
        if zero_frac > 0:
            mag[rng.random(T) < zero_frac] = 0.0
        x *= mag[:, None, None]
        out.append(to_bf16_bits(x))
    return out[0], out[1]


def queries(rng: np.random.Generator, rows: int, Hq: int = HQ, head_dim: int = D) -> np.ndarray:
    """BF16 queries N(0,1), uint16 [rows, Hq, head_dim]."""
    return to_bf16_bits(rng.standard_normal((rows, Hq, head_dim), dtype=np.float32))


# --------------------------------------------------------------------------------------------
@dataclass
class DecodeLayer:
    """One layer of a decode workload before quantization (the pool is built by a store call)."""
    k: np.ndarray          # uint16 [n_tokens, Hkv, D]   every context token, in logical order per request
    v: np.ndarray
    slots: np.ndarray      # int32 [n_tokens]            pool row of each token above
    q: np.ndarray          # uint16 [total_q_rows, Hq, D]


@dataclass
class DecodeWorkload:
    name: str
    num_rows: int
    req_to_slot: np.ndarray      # int32 [B, stride]
    seq_lens: np.ndarray         # int32 [B]
    q_row_offsets: np.ndarray    # int32 [B+1]
    layers: int
    sigma: float
    big_frac: float = 0.0
    zero_frac: float = 0.0
    seed: int = 0
    Hq: int = HQ
    Hkv: int = HKV
    head_dim: int = D
    sm_scale: float = SM_SCALE
    meta: dict = field(default_factory=dict)

    @property
    def token_slots(self) -> np.ndarray:
        """Pool rows of all context tokens, request by request, in logical order."""
        return np.concatenate([self.req_to_slot[b, :self.seq_lens[b]] for b in range(len(self.seq_lens))])

    def layer(self, l: int) -> DecodeLayer:
        rng = _rng(self.seed, 1, l)
        slots = self.token_slots.astype(np.int32)
        k, v = kv_tokens(rng, slots.shape[0], self.sigma, self.big_frac, self.zero_frac, self.Hkv,
                         self.head_dim)
        q = queries(_rng(self.seed, 2, l), int(self.q_row_offsets[-1]), self.Hq, self.head_dim)
        return DecodeLayer(k=k, v=v, slots=slots, q=q)


def decode_small(seed: int = 1000) -> DecodeWorkload:
    """One decode step, one layer, batch 1, 512-token context, 1,024-row pool."""
    R, n = 1024, 512
    perm = _rng(seed, 0).permutation(R).astype(np.int32)
    return DecodeWorkload("decode_small", R, perm[:n].reshape(1, n).copy(), np.array([n], np.int32),
                          np.array([0, 1], np.int32), layers=1, sigma=1.0, seed=seed)


def decode_long(n: int = 32768, num_rows: int = 33059, layers: int = 48, seed: int = 1002) -> DecodeWorkload:
    """Batch-1 decode at n keys, one pool of ``num_rows`` rows per layer (shared slot table)."""
    perm = _rng(seed, 0, n).permutation(num_rows).astype(np.int32)
    return DecodeWorkload(f"decode_long_{n}", num_rows, perm[:n].reshape(1, n).copy(),
                          np.array([n], np.int32), np.array([0, 1], np.int32), layers=layers, sigma=1.0,
                          seed=seed)


def decode_batched(B: int = 64, num_rows: int = 2_000_000, lo: int = 1024, hi: int = 40000,
                   max_rows: int = 8, seed: int = 1004) -> DecodeWorkload:
    """Batched multi-row decode: context ~ U[lo, hi], 1..max_rows query rows per request."""
    rng = _rng(seed, 0)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    rows = rng.integers(1, max_rows + 1, size=B).astype(np.int32)
    assert int(lens.sum()) <= num_rows
    perm = rng.permutation(num_rows).astype(np.int32)
    stride = int(lens.max())
    table = np.zeros((B, stride), np.int32)
    pos = 0
    for b in range(B):
        table[b, :lens[b]] = perm[pos:pos + lens[b]]
        pos += int(lens[b])
    offs = np.zeros(B + 1, np.int32)
    offs[1:] = np.cumsum(rows)
    return DecodeWorkload("decode_batched", num_rows, table, lens, offs, layers=1, sigma=2.0,
                          big_frac=0.01, zero_frac=0.001, seed=seed)


def decode_custom(seq_lens, q_rows, num_rows: int, sigma: float = 1.0, big_frac: float = 0.0,
                  zero_frac: float = 0.0, seed: int = 7, Hq: int = HQ, Hkv: int = HKV,
                  head_dim: int = D) -> DecodeWorkload:
    """Small ad-hoc decode workloads for edge cases (ragged lengths, GQA variants, empty rows)."""
    lens = np.asarray(seq_lens, np.int32)
    rows = np.asarray(q_rows, np.int32)
    B = lens.shape[0]
    assert int(lens.sum()) <= num_rows
    rng = _rng(seed, 0)
    perm = rng.permutation(num_rows).astype(np.int32)
    stride = max(int(lens.max()) if B else 1, 1)
    table = np.zeros((B, stride), np.int32)
    pos = 0
    for b in range(B):
        table[b, :lens[b]] = perm[pos:pos + lens[b]]
        pos += int(lens[b])
    offs = np.zeros(B + 1, np.int32)
    offs[1:] = np.cumsum(rows)
    return DecodeWorkload("decode_custom", num_rows, table, lens, offs, layers=1, sigma=sigma,
                          big_frac=big_frac, zero_frac=zero_frac, seed=seed, Hq=Hq, Hkv=Hkv,
                          head_dim=head_dim)


# --------------------------------------------------------------------------------------------
@dataclass
class StoreWorkload:
    num_rows: int
    slots: np.ndarray     # int32 [T] -- the same slots for every layer
    layers: int
    seed: int

    def layer(self, l: int):
        rng = _rng(self.seed, 1, l)
        return kv_tokens(rng, self.slots.shape[0], 2.0, 0.01, 0.001)


def store(T: int = 8192, num_rows: int = 33059, layers: int = 48, seed: int = 1001) -> StoreWorkload:
    perm = _rng(seed, 0).permutation(num_rows).astype(np.int32)
    return StoreWorkload(num_rows, perm[:T].copy(), layers, seed)


# --------------------------------------------------------------------------------------------
@dataclass
class PrefillWorkload:
    num_rows: int
    hist_slots: np.ndarray     # int32 [H]
    new_slots: np.ndarray      # int32 [N]
    hist_k: np.ndarray         # uint16 [H, Hkv, D]
    hist_v: np.ndarray
    q: np.ndarray              # uint16 [N, Hq, D]
    k: np.ndarray              # uint16 [N, Hkv, D]
    v: np.ndarray
    chunk: int
    sm_scale: float = SM_SCALE

    @property
    def num_chunks(self) -> int:
        return (self.q.shape[0] + self.chunk - 1) // self.chunk


def prefill(hist: int = 8192, new: int = 8192, chunk: int = 2048, num_rows: int = 33059,
            seed: int = 1003, Hq: int = HQ, Hkv: int = HKV, head_dim: int = D) -> PrefillWorkload:
    perm = _rng(seed, 0).permutation(num_rows).astype(np.int32)
    hk, hv = kv_tokens(_rng(seed, 1), hist, 1.0, Hkv=Hkv, head_dim=head_dim)
    k, v = kv_tokens(_rng(seed, 2), new, 1.0, Hkv=Hkv, head_dim=head_dim)
    q = queries(_rng(seed, 3), new, Hq, head_dim)
    return PrefillWorkload(num_rows, perm[:hist].copy(), perm[hist:hist + new].copy(), hk, hv, q, k, v,
                           chunk)
