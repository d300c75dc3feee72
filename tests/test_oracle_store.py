"""Pins for the oracle's quantize-on-write, reconstruct and byte accounting (CPU only).

* Byte accounting: the integers printed in FreeToken PR #853 ("Validation": 3,249,831,936 B BF16 KV,
  1,675,694,592 B FP8 codes+scales and a 67,704,832 B workspace at 33,059 rows, 46.35 % saved;
  "Follow-up model/workload search": 98,304 vs 50,688 bytes per token), read from
  tests/golden/byte_accounting.txt.
* Store: the scale against numpy's FP32 division of the row absmax by 448, the codes against torch's
  float8_e4m3fn cast of numpy's FP32 quotient, and the E4M3 error bound on the dequantized values.
* Reconstruct: power-of-two scales (exact products) and torch's FP32 product + BF16 cast.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_ftkv_gb300 import inputs


# ---------------------------------------------------------------------------------------------
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "byte_accounting.txt")


def _golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            cases.append({k: float(v) if "." in v else int(v) for k, v in (f.split("=") for f in line.split())})
    return cases


def test_golden_byte_accounting_fixture_is_complete():
    cases = _golden_cases()
    assert len(cases) == 2
    assert {"bf16", "fp8", "workspace", "saved_with_workspace_pct"} <= set(cases[0])
    assert {"bf16", "fp8", "saved_pct"} <= set(cases[1])


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: f"rows{c['rows']}")
def test_byte_accounting_matches_printed_integers(case):
    b = oracle.pool_bytes(case["rows"], case["layers"], case["kv_heads"], case["head_dim"])
    assert b["bf16"] == case["bf16"]
    assert b["fp8"] == case["fp8"]
    if "workspace" in case:
        assert b["workspace"] == case["workspace"]
        saved = 1.0 - (b["fp8"] + b["workspace"]) / b["bf16"]
        assert round(100 * saved, 2) == case["saved_with_workspace_pct"]
    if "saved_pct" in case:
        assert round(100 * (1 - b["fp8"] / b["bf16"]), 1) == case["saved_pct"]


# ---------------------------------------------------------------------------------------------
def _independent_quantize(x_bits: np.ndarray):
    """Row quantization restated with numpy FP32 arithmetic and torch's E4M3FN cast."""
    x = inputs.bf16_bits_to_f32(x_bits)                       # [..., D]
    amax = np.max(np.abs(np.nan_to_num(x, nan=0.0)), axis=-1)  # NaN-ignoring absmax
    s = (amax / np.float32(448.0)).astype(np.float32)
    div = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    qv = (x / div[..., None]).astype(np.float32)
    codes = torch.from_numpy(np.clip(qv, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    codes = np.where(np.isnan(qv), np.uint8(0x7F), codes)
    return codes, s


def test_store_matches_independent_restatement():
    rng = np.random.default_rng(11)
    T, R = 300, 777
    k, v = inputs.kv_tokens(rng, T, 2.0, big_frac=0.05, zero_frac=0.05)
    slots = rng.permutation(R)[:T].astype(np.int32)
    pool = oracle.Pool(R, 4, 128)
    oracle.store_quant(pool, k, v, slots)
    for src, codes, scales in ((k, pool.k_codes, pool.k_scales), (v, pool.v_codes, pool.v_scales)):
        want_c, want_s = _independent_quantize(src)
        assert np.array_equal(codes[slots], want_c)
        assert np.array_equal(scales[slots].view(np.uint32), want_s.view(np.uint32))
    # rows not written stay untouched (zero)
    untouched = np.setdiff1d(np.arange(R), slots)
    assert not pool.k_codes[untouched].any() and not pool.k_scales[untouched].any()


def test_store_256d_matches_independent_restatement():
    """The 256-d row (FTKV_HEAD_DIM_256) is quantized by the same definition over all 256 elements."""
    rng = np.random.default_rng(12)
    T, R = 120, 300
    k, v = inputs.kv_tokens(rng, T, 2.0, big_frac=0.05, zero_frac=0.05, head_dim=256)
    slots = rng.permutation(R)[:T].astype(np.int32)
    pool = oracle.Pool(R, 4, 256)
    oracle.store_quant(pool, k, v, slots)
    for src, codes, scales in ((k, pool.k_codes, pool.k_scales), (v, pool.v_codes, pool.v_scales)):
        want_c, want_s = _independent_quantize(src)
        assert np.array_equal(codes[slots], want_c)
        assert np.array_equal(scales[slots].view(np.uint32), want_s.view(np.uint32))


def test_store_error_bound_and_landmarks():
    rng = np.random.default_rng(12)
    T = 200
    k, v = inputs.kv_tokens(rng, T, 2.0, big_frac=0.02)
    slots = np.arange(T, dtype=np.int32)
    pool = oracle.Pool(T, 4, 128)
    oracle.store_quant(pool, k, v, slots)
    x = inputs.bf16_bits_to_f32(k).astype(np.float64)
    s = pool.k_scales.astype(np.float64)[..., None]
    deq = oracle.e4m3_decode(pool.k_codes) * s
    # E4M3 RNE: relative error <= 2^-4 in the normal range, absolute <= 2^-10 * s below 2^-6 * s
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)
    assert (err <= bound).all()
    # the row's absmax element maps to +-448 exactly
    idx = np.argmax(np.abs(x), axis=-1)
    top = np.take_along_axis(pool.k_codes, idx[..., None], axis=-1)[..., 0]
    assert np.isin(top, [0x7E, 0xFE]).all()


def test_store_degenerate_rows():
    z = np.zeros((3, 4, 128), np.uint16)
    z[1, :, ::2] = 0x8000                       # -0.0 in half the lanes
    pool = oracle.Pool(3, 4, 128)
    oracle.store_quant(pool, z, z, np.array([0, 1, 2], np.int32))
    assert (pool.k_scales == 0).all()
    assert (pool.k_codes[0] == 0).all()
    assert (pool.k_codes[1, :, ::2] == 0x80).all() and (pool.k_codes[1, :, 1::2] == 0).all()
    # a NaN element is ignored by absmax and encodes to 0x7F; an Inf row gives scale Inf
    x = np.zeros((1, 4, 128), np.float32)
    x[0, 0, :] = np.linspace(-3, 3, 128)
    x[0, 0, 5] = np.nan
    x[0, 1, :] = 1.0
    x[0, 1, 7] = np.inf
    bits = inputs.to_bf16_bits(x)
    pool = oracle.Pool(1, 4, 128)
    oracle.store_quant(pool, bits, bits, np.array([0], np.int32))
    assert pool.k_scales[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert pool.k_codes[0, 0, 5] == 0x7F
    assert np.isinf(pool.k_scales[0, 1])
    assert pool.k_codes[0, 1, 7] == 0x7F                 # Inf / Inf
    assert (np.delete(pool.k_codes[0, 1], 7) == 0).all()  # finite / Inf = +0


# ---------------------------------------------------------------------------------------------
def test_reconstruct_power_of_two_scales_exact():
    rng = np.random.default_rng(13)
    R, P = 64, 40
    pool = oracle.Pool(R, 4, 128)
    codes = rng.integers(0, 256, size=(R, 4, 128), dtype=np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    pool.k_codes[:] = codes
    pool.v_codes[:] = codes[::-1]
    pool.k_scales[:] = np.exp2(rng.integers(-20, 20, size=(R, 4))).astype(np.float32)
    pool.v_scales[:] = np.exp2(rng.integers(-20, 20, size=(R, 4))).astype(np.float32)
    slots = rng.permutation(R)[:P].astype(np.int32)
    ws_k, ws_v = oracle.reconstruct(pool, slots)
    want_k = oracle.e4m3_decode(pool.k_codes[slots]) * pool.k_scales[slots][..., None].astype(np.float64)
    assert np.array_equal(inputs.bf16_bits_to_f32(ws_k).astype(np.float64), want_k)
    want_v = oracle.e4m3_decode(pool.v_codes[slots]) * pool.v_scales[slots][..., None].astype(np.float64)
    assert np.array_equal(inputs.bf16_bits_to_f32(ws_v).astype(np.float64), want_v)


def test_reconstruct_matches_torch_product_and_cast():
    rng = np.random.default_rng(14)
    T, R = 256, 512
    k, v = inputs.kv_tokens(rng, T, 2.0, big_frac=0.05, zero_frac=0.02)
    slots = rng.permutation(R)[:T].astype(np.int32)
    pool = oracle.Pool(R, 4, 128)
    oracle.store_quant(pool, k, v, slots)
    ws_k, ws_v = oracle.reconstruct(pool, slots)
    for ws, codes, scales in ((ws_k, pool.k_codes, pool.k_scales), (ws_v, pool.v_codes, pool.v_scales)):
        dec = torch.from_numpy(codes[slots]).view(torch.float8_e4m3fn).to(torch.float32)
        prod = dec * torch.from_numpy(scales[slots])[..., None]
        want = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(ws, want)


def test_bf16_rounding_helper():
    # nearest-even at the BF16 boundary, overflow to Inf, NaN quiet
    assert oracle.f32_to_bf16_bits(1.0) == 0x3F80
    assert oracle.f32_to_bf16_bits(float(np.float32(1.0 + 2 ** -8))) == 0x3F80        # tie -> even
    assert oracle.f32_to_bf16_bits(float(np.float32(1.0 + 3 * 2 ** -8))) == 0x3F82    # tie -> even (up)
    assert oracle.f32_to_bf16_bits(3.4e38) == 0x7F80
    assert oracle.f32_to_bf16_bits(float("nan")) == 0x7FC0
