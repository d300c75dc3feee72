"""Pins for the oracle's E4M3FN codec (CPU only).

The codec is tied to three things outside the oracle:
* the format's landmarks (1.0, 448, the smallest normal and subnormal, signed zero, NaN);
* torch's ``float8_e4m3fn`` dtype (an independent library implementation of the same format), for
  decode of all 256 codes and for encode of every FP32 bit pattern (finite inputs clamped to +-448,
  since torch's cast is not saturating);
* an arithmetic restatement of round-to-nearest-even at 3 mantissa bits (numpy's ``rint`` rounds half
  to even), independent of the oracle's table search.
FreeToken PR #897 ("Regression and CUDA isolation") requires every finite E4M3FN value, signed zero
included, to survive bit-for-bit: the round-trip test below.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _torch_decode_all():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_landmarks():
    d = oracle.e4m3_decode(np.array([0x38, 0x7E, 0x08, 0x01, 0x00, 0x80, 0xB8, 0xFE, 0x07, 0x77], np.uint8))
    assert d[0] == 1.0
    assert d[1] == 448.0
    assert d[2] == 2.0 ** -6          # smallest normal
    assert d[3] == 2.0 ** -9          # smallest subnormal
    assert d[4] == 0.0 and not math.copysign(1.0, d[4]) < 0
    assert d[5] == 0.0 and math.copysign(1.0, d[5]) < 0   # -0
    assert d[6] == -1.0
    assert d[7] == -448.0
    assert d[8] == 7 * 2.0 ** -9       # largest subnormal
    assert d[9] == 240.0               # 2^7 * 1.875
    nan = oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))
    assert np.isnan(nan).all()


def test_decode_matches_torch_all_codes():
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _torch_decode_all()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero bit-for-bit
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    # exactly two NaN codes
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]


def test_round_trip_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    finite = ~np.isnan(vals)
    assert np.array_equal(back[finite], codes[finite])
    assert (back[~finite] == 0x7F).all()
    assert back[0x80] == 0x80  # -0 keeps its sign


def test_special_values():
    x = np.array([np.nan, -np.nan, np.inf, -np.inf, 448.0, 449.0, 463.99, 464.0, 480.0, 1e30, -1e30,
                  0.0, -0.0, 1e-45, -1e-45], np.float32)
    c = oracle.e4m3_encode(x)
    assert c[0] == 0x7F and c[1] == 0x7F                     # NaN -> canonical 0x7F
    assert c[2] == 0x7E and c[3] == 0xFE                     # +-Inf saturate
    assert (c[4:9] == 0x7E).all()                            # everything at or past 448 -> 448
    assert c[9] == 0x7E and c[10] == 0xFE
    assert c[11] == 0x00 and c[12] == 0x80                   # signed zero
    assert c[13] == 0x00 and c[14] == 0x80                   # FP32 subnormals round to +-0


def test_ties_go_to_even_mantissa():
    codes = np.arange(0, 126, dtype=np.uint8)
    lo = oracle.e4m3_decode(codes)
    hi = oracle.e4m3_decode(codes + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # midpoints are exact in FP32
    got = oracle.e4m3_encode(mid)
    want = np.where(codes % 2 == 0, codes, codes + 1)
    assert np.array_equal(got, want)
    # just below / above the midpoint
    below = np.nextafter(mid, np.float32(-np.inf))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(oracle.e4m3_encode(below), codes)
    assert np.array_equal(oracle.e4m3_encode(above), codes + 1)


def _rne_restated(x: np.ndarray) -> np.ndarray:
    """Round |x| <= 448 to E4M3 by arithmetic: 3 fractional mantissa bits, subnormal spacing 2^-9."""
    a = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                      # below 2^-6 the spacing is fixed at 2^-9
    step = np.exp2(e - 3.0)
    r = np.rint(a / step) * step                 # rint: round half to even
    return np.copysign(r, x.astype(np.float64))


def test_encode_matches_arithmetic_restatement():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(40),
        (rng.random(200000) * 448).astype(np.float32),
        (rng.random(100000) * 2.0 ** -5).astype(np.float32),
    ])
    x = np.clip(x, -448, 448)
    want = _rne_restated(x)
    got = oracle.e4m3_decode(oracle.e4m3_encode(x))
    assert np.array_equal(got, want)


def test_encode_matches_torch_all_fp32_bit_patterns():
    """Every one of the 2^32 FP32 bit patterns: oracle == torch cast of the input clamped to +-448."""
    chunk = 1 << 26
    base = np.arange(chunk, dtype=np.uint32)
    bits = np.empty(chunk, np.uint32)
    for start in range(0, 1 << 32, chunk):
        np.add(base, np.uint32(start), out=bits)
        x = torch.from_numpy(bits.view(np.float32))
        ref = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = oracle.e4m3_encode(x.numpy())
        nan = torch.isnan(x).numpy()
        # NaN inputs: torch keeps the sign bit of the NaN, the oracle emits the canonical 0x7F
        assert (got[nan] == 0x7F).all()
        assert np.array_equal(ref[nan] & 0x7F, np.full(int(nan.sum()), 0x7F, np.uint8))
        ok = np.array_equal(got[~nan], ref[~nan])
        if not ok:
            bad = np.flatnonzero(got[~nan] != ref[~nan])[:5]
            pytest.fail(f"mismatch at chunk {start:#x}: inputs {x.numpy()[~nan][bad]}, "
                        f"oracle {got[~nan][bad]}, torch {ref[~nan][bad]}")
