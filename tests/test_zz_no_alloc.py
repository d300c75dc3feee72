"""GPU test of the decode entry point that allocates nothing (ftkv_decode_attn_noalloc).

Callers that cannot allocate device memory -- a runtime that forbids out-of-band device allocations, a
plug-in that only receives buffers from its host -- use ftkv_decode_attn_noalloc, whose split partials
and counters live in a static device array inside the library.  Through the C ABI (ctypes, no torch
wrapper), two calls in a row with different shapes (so the second meets the first one's leftovers in
the shared array), then the first shape again, must match the regular ftkv_decode_attn and the FP64
oracle within the attention tolerance used by the other tests; a call too large for the array, or with a
bad argument, must be refused without touching the array.
This file is collected last and needs nothing from the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_ftkv_gb300 import _lib, inputs, ops
from parity import bits_to_cuda_bf16, check_attention

pytestmark = pytest.mark.gpu


def _setup(wl):
    L = wl.layer(0)
    pool = ops.KVPool.empty(wl.num_rows, wl.Hkv)
    ops.store_quant(pool, bits_to_cuda_bf16(L.k), bits_to_cuda_bf16(L.v), torch.from_numpy(L.slots).cuda())
    dev = dict(q=bits_to_cuda_bf16(L.q), r2s=torch.from_numpy(wl.req_to_slot).cuda(),
               lens=torch.from_numpy(wl.seq_lens).cuda(), offs=torch.from_numpy(wl.q_row_offsets).cuda())
    return pool, dev


def _noalloc(wl, pool, dev, max_q_rows):
    lib = _lib.load()
    out = torch.empty_like(dev["q"])
    ps = pool.c_struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.ftkv_decode_attn_noalloc(ctypes.byref(ps), wl.Hq, p(dev["q"]), p(dev["r2s"]), wl.req_to_slot.shape[1],
                                      p(dev["lens"]), p(dev["offs"]), len(wl.seq_lens), dev["q"].shape[0],
                                      max_q_rows, int(wl.req_to_slot.shape[1]), wl.sm_scale, 0, p(out), stream)
    assert st == _lib.FTKV_OK, _lib.status_str(st)
    torch.cuda.synchronize()
    return out


def _regular(wl, pool, dev, max_q_rows):
    return ops.decode_attn(pool, dev["q"], dev["r2s"], dev["lens"], dev["offs"], max_seq_len=int(wl.req_to_slot.shape[1]),
                           max_q_rows=max_q_rows, sm_scale=wl.sm_scale)


def test_noalloc_decode_matches_regular_entry_point():
    cases = [(inputs.decode_small(), 1),
             (inputs.decode_custom([300, 1000, 77], [3, 1, 8], 3000, sigma=2.0, big_frac=0.01, seed=11), 8)]
    runs = [cases[0], cases[1], cases[0]]   # two calls in a row with different shapes, then the first again
    for wl, mq in runs:
        pool, dev = _setup(wl)
        got = _noalloc(wl, pool, dev, mq)
        ref = _regular(wl, pool, dev, mq)
        check_attention(got, ref.float().cpu().numpy().astype(np.float64), f"noalloc vs ftkv_decode_attn {wl.name}")
        L = wl.layer(0)
        op = oracle.Pool(wl.num_rows, wl.Hkv, 128)
        oracle.store_quant(op, L.k, L.v, L.slots)
        exact = oracle.decode_attn(op, L.q, wl.req_to_slot, wl.seq_lens, wl.q_row_offsets, wl.sm_scale, wl.Hq)
        check_attention(got, exact, f"noalloc vs oracle {wl.name}")
    assert ops.device_errors() == 0


def test_noalloc_refuses_requests_beyond_its_scratch():
    wl = inputs.decode_small()
    pool, dev = _setup(wl)
    lib = _lib.load()
    big_rows = 4096                     # 4096 rows x 32 heads x 64 slices of partials: far beyond 16 MiB
    ps = pool.c_struct()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.ftkv_decode_attn_noalloc(ctypes.byref(ps), 32, p(dev["q"]), p(dev["r2s"]), wl.req_to_slot.shape[1],
                                      p(dev["lens"]), None, big_rows, big_rows, 1, 512, wl.sm_scale, 64,
                                      p(dev["q"]), None)
    assert st == _lib.FTKV_ERR_WORKSPACE
    # a refused call enqueues nothing: a bad argument after a good call leaves the good call's output intact
    good = _noalloc(wl, pool, dev, 1)
    bad_out = torch.full_like(dev["q"], 7.0)
    st = lib.ftkv_decode_attn_noalloc(ctypes.byref(ps), 32, ctypes.c_void_p(dev["q"].data_ptr() + 2), p(dev["r2s"]),
                                      wl.req_to_slot.shape[1], p(dev["lens"]), None, 1, 1, 1, 512, wl.sm_scale, 0,
                                      p(bad_out), None)
    assert st == _lib.FTKV_ERR_ALIGN
    torch.cuda.synchronize()
    assert (bad_out.float() == 7.0).all()
    again = _noalloc(wl, pool, dev, 1)
    assert torch.equal(good, again)
