"""GPU parity: prefill attention over the reconstructed prefix plus the BF16 chunk.

The chunked workload runs exactly as the benchmark does (8,192 historical rows, 8,192 new tokens in
4 chunks of 2,048: reconstruct -> prefill -> quantize-on-write of the chunk) on both sides; every 16th
query row of each chunk is compared (all heads, all d).  Small cases cover an empty prefix, ragged
chunk and prefix lengths and GQA group sizes, one CTA per work item ("tc") and stream-K ("tc_sk").

Tolerance.  Prefill is BF16 attention over the BF16 workspace (FreeToken PR #853, "What changes": the
historical rows are rebuilt into BF16 for the existing BF16 attention): the probabilities P enter the
tensor-core PV product as BF16 (8 significant bits; A and B of one kind::f16 MMA share one type, and V is
BF16).  Each term p_j v_j then carries a relative error up to 2^-9, so an output element that is small
next to the terms it sums is off by ~2^-9 of those terms, not of itself: measured max-abs 0.06-0.19 for
|ref| up to ~80 (max-abs / max|ref| 2e-3 - 5e-3), relative L2 1.1e-3 - 1.8e-3, and the elementwise
|o - ref| <= 1e-2 + 1e-2 |ref| fails for a handful of elements per case.  These checks therefore use the
"terms" bound of parity.py (absolute part scaled by the attention-weighted term magnitude, per output
vector) plus relative L2 <= 1e-2.  Decode uses FP32 probabilities into its FP16 PV product and meets the
elementwise bound.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_ftkv_gb300 import inputs, ops
from parity import bits_to_cuda_bf16, check_attention

pytestmark = pytest.mark.gpu

IMPLS = ["tc", "tc_sk"]
BOUND = "terms"  # see the module docstring
_PLANS = {}


def _prefill(impl, q, kc, vc, wk, wv, ctas=5):
    """impl "tc_sk": the tcgen05 kernel scheduled stream-K over `ctas` persistent CTAs (0: the SM count;
    a small count on small inputs makes every CTA run several items and cuts items between CTAs).  The
    plans are shared by all tests, so each test also checks that the previous calls left the tickets at
    zero."""
    if impl == "tc_sk":
        if ctas not in _PLANS:
            _PLANS[ctas] = ops.PrefillPlan(ctas)
        return ops.prefill_attn(q, kc, vc, wk, wv, plan=_PLANS[ctas])
    return ops.prefill_attn(q, kc, vc, wk, wv)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("P,C", [(0, 1), (0, 77), (37, 29), (128, 128), (1000, 300), (257, 513)])
def test_prefill_small(impl, P, C):
    rng = np.random.default_rng(P * 1000 + C)
    wk, wv = inputs.kv_tokens(rng, P, 1.0)
    kc, vc = inputs.kv_tokens(rng, C, 1.0)
    q = inputs.queries(rng, C)
    ref = oracle.prefill_attn(q, kc, vc, wk, wv, inputs.SM_SCALE)
    mag = oracle.prefill_attn(q, kc, vc, wk, wv, inputs.SM_SCALE, abs_v=True)
    out = _prefill(impl, bits_to_cuda_bf16(q), bits_to_cuda_bf16(kc), bits_to_cuda_bf16(vc),
                   bits_to_cuda_bf16(wk) if P else None, bits_to_cuda_bf16(wv) if P else None)
    check_attention(out, ref, f"{impl} P={P} C={C}", mag, bound=BOUND)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("Hq,Hkv", [(16, 4), (8, 8), (64, 8), (8, 4)])
def test_prefill_gqa(impl, Hq, Hkv):
    rng = np.random.default_rng(Hq)
    P, C = 200, 150
    wk, wv = inputs.kv_tokens(rng, P, 1.0, Hkv=Hkv)
    kc, vc = inputs.kv_tokens(rng, C, 1.0, Hkv=Hkv)
    q = inputs.queries(rng, C, Hq)
    ref = oracle.prefill_attn(q, kc, vc, wk, wv, inputs.SM_SCALE)
    mag = oracle.prefill_attn(q, kc, vc, wk, wv, inputs.SM_SCALE, abs_v=True)
    out = _prefill(impl, bits_to_cuda_bf16(q), bits_to_cuda_bf16(kc), bits_to_cuda_bf16(vc),
                   bits_to_cuda_bf16(wk), bits_to_cuda_bf16(wv))
    check_attention(out, ref, f"{impl} Hq={Hq} Hkv={Hkv}", mag, bound=BOUND)


@pytest.mark.parametrize("impl", IMPLS)
def test_chunked_prefill_full_workload(impl):
    wl = inputs.prefill()
    R = wl.num_rows
    gp = ops.KVPool.empty(R, 4)
    op = oracle.Pool(R, 4, 128)
    hist = torch.from_numpy(wl.hist_slots).cuda()
    ops.store_quant(gp, bits_to_cuda_bf16(wl.hist_k), bits_to_cuda_bf16(wl.hist_v), hist)
    oracle.store_quant(op, wl.hist_k, wl.hist_v, wl.hist_slots)
    slots_all = np.concatenate([wl.hist_slots, wl.new_slots])
    q_d, k_d, v_d = bits_to_cuda_bf16(wl.q), bits_to_cuda_bf16(wl.k), bits_to_cuda_bf16(wl.v)
    slots_d = torch.from_numpy(slots_all).cuda()
    H = wl.hist_slots.shape[0]
    for c in range(wl.num_chunks):
        c0, c1 = c * wl.chunk, min((c + 1) * wl.chunk, wl.q.shape[0])
        P = H + c0
        wk, wv = ops.reconstruct_bf16(gp, slots_d[:P])
        out = _prefill(impl, q_d[c0:c1], k_d[c0:c1], v_d[c0:c1], wk, wv, ctas=0)
        ops.store_quant(gp, k_d[c0:c1], v_d[c0:c1], slots_d[P:P + c1 - c0])
        # oracle: the same pipeline
        owk, owv = oracle.reconstruct(op, slots_all[:P])
        rows = np.arange(0, c1 - c0, 16, dtype=np.int64)
        ref = oracle.prefill_attn(wl.q[c0:c1], wl.k[c0:c1], wl.v[c0:c1], owk, owv, wl.sm_scale, rows)
        mag = oracle.prefill_attn(wl.q[c0:c1], wl.k[c0:c1], wl.v[c0:c1], owk, owv, wl.sm_scale, rows, abs_v=True)
        oracle.store_quant(op, wl.k[c0:c1], wl.v[c0:c1], slots_all[P:P + c1 - c0])
        check_attention(out[torch.from_numpy(rows).cuda()], ref, f"{impl} chunk {c}", mag, bound=BOUND)
    assert ops.device_errors() == 0


@pytest.mark.parametrize("ctas", [2, 3, 7, 19])
def test_prefill_stream_k_cuts(ctas):
    """Stream-K with CTA counts that cut items at many different tiles (prefix and chunk tiles, first
    and last query tiles): same attention as the oracle, bit-identical on a repeated call (the tickets
    were reset), and within FP32 summation order of the one-CTA-per-item launch."""
    rng = np.random.default_rng(100 + ctas)
    P, C = 700, 390  # 6 prefix tiles (the last one ragged), 4 query tiles (the last one ragged)
    wk, wv = inputs.kv_tokens(rng, P, 1.0)
    kc, vc = inputs.kv_tokens(rng, C, 1.0)
    q = inputs.queries(rng, C)
    ref = oracle.prefill_attn(q, kc, vc, wk, wv, inputs.SM_SCALE)
    mag = oracle.prefill_attn(q, kc, vc, wk, wv, inputs.SM_SCALE, abs_v=True)
    args = [bits_to_cuda_bf16(x) for x in (q, kc, vc, wk, wv)]
    plan = ops.PrefillPlan(ctas)
    out1 = ops.prefill_attn(*args, plan=plan)
    out2 = ops.prefill_attn(*args, plan=plan)
    whole = ops.prefill_attn(*args)
    check_attention(out1, ref, f"stream-K ctas={ctas}", mag, bound=BOUND)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    tickets = ((ctas + 1) * 16 + 255) // 256 * 256
    assert torch.count_nonzero(plan.workspace[:tickets]).item() == 0  # every ticket back at zero
    d = (out1.float() - whole.float()).abs().max().item()
    assert d <= 2.0 ** -6 * max(1.0, whole.float().abs().max().item()), d
    assert ops.device_errors() == 0
