"""GPU parity: E4M3 codec, quantize-on-write and reconstruct -- bit-exact against the oracle.

Quantize-on-write runs the full 8,192-token x 48-layer workload into a 33,059-row pool (the
configuration the benchmark times); reconstruct runs the chunked-prefill prefix sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_ftkv_gb300 import inputs, ops
from parity import bits_to_cuda_bf16, cuda_bf16_to_bits, pool_to_host

pytestmark = pytest.mark.gpu


def test_decode_all_codes_exact():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).cuda()
    got = ops.e4m3_decode(codes).cpu().numpy().astype(np.float64)
    want = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all()
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_encode_every_fp32_bit_pattern():
    """The store kernel's encoder (same device function) on all 2^32 FP32 inputs."""
    chunk = 1 << 28
    base = torch.arange(chunk, dtype=torch.int64, device="cuda")
    for start in range(0, 1 << 32, chunk):
        bits = (base + start)
        bits = torch.where(bits >= (1 << 31), bits - (1 << 32), bits).to(torch.int32)
        x = bits.view(torch.float32)
        got = ops.e4m3_encode(x).cpu().numpy()
        want = oracle.e4m3_encode(x.cpu().numpy())
        if not np.array_equal(got, want):
            bad = np.flatnonzero(got != want)[:8]
            xs = x.cpu().numpy()[bad]
            pytest.fail(f"chunk {start:#x}: x={xs} gpu={got[bad]} oracle={want[bad]}")


def _store_both(T, R, sigma=2.0, big=0.01, zero=0.001, seed=5, slots=None):
    rng = np.random.default_rng(seed)
    k, v = inputs.kv_tokens(rng, T, sigma, big, zero)
    if slots is None:
        slots = rng.permutation(R)[:T].astype(np.int32)
    gp = ops.KVPool.empty(R, 4)
    ops.store_quant(gp, bits_to_cuda_bf16(k), bits_to_cuda_bf16(v), torch.from_numpy(slots).cuda())
    op = oracle.Pool(R, 4, 128)
    oracle.store_quant(op, k, v, slots)
    return gp, op, slots


def _assert_pool_equal(gp, op, slots):
    kc, vc, ks, vs = pool_to_host(gp)
    assert np.array_equal(kc[slots], op.k_codes[slots])
    assert np.array_equal(vc[slots], op.v_codes[slots])
    assert np.array_equal(ks[slots].view(np.uint32), op.k_scales[slots].view(np.uint32))
    assert np.array_equal(vs[slots].view(np.uint32), op.v_scales[slots].view(np.uint32))


def test_store_full_workload_48_layers_bit_exact():
    wl = inputs.store()
    slots_d = torch.from_numpy(wl.slots).cuda()
    gp = ops.KVPool.empty(wl.num_rows, 4)
    for l in range(wl.layers):
        k, v = wl.layer(l)
        ops.store_quant(gp, bits_to_cuda_bf16(k), bits_to_cuda_bf16(v), slots_d)
        op = oracle.Pool(wl.num_rows, 4, 128)
        oracle.store_quant(op, k, v, wl.slots)
        _assert_pool_equal(gp, op, wl.slots)
    assert ops.device_errors() == 0


@pytest.mark.parametrize("T", [1, 7, 33, 1000])
def test_store_ragged_sizes(T):
    gp, op, slots = _store_both(T, 2048, seed=T)
    _assert_pool_equal(gp, op, slots)


def test_store_degenerate_rows():
    x = np.zeros((4, 4, 128), np.float32)
    x[1, :, ::2] = -0.0
    x[2, 0, :] = np.linspace(-3, 3, 128)
    x[2, 0, 5] = np.nan
    x[2, 1, :] = 1.0
    x[2, 1, 7] = np.inf
    x[3] = 1e-40  # BF16 subnormals
    x[3, 2, 3] = -3e-39
    bits = inputs.to_bf16_bits(x)
    slots = np.array([3, 0, 2, 1], np.int32)
    gp = ops.KVPool.empty(4, 4)
    ops.store_quant(gp, bits_to_cuda_bf16(bits), bits_to_cuda_bf16(bits), torch.from_numpy(slots).cuda())
    op = oracle.Pool(4, 4, 128)
    oracle.store_quant(op, bits, bits, slots)
    _assert_pool_equal(gp, op, slots)


def test_store_empty_is_noop_and_bad_slot_is_flagged():
    gp = ops.KVPool.empty(16, 4)
    empty = torch.empty(0, 4, 128, dtype=torch.bfloat16, device="cuda")
    ops.store_quant(gp, empty, empty, torch.empty(0, dtype=torch.int32, device="cuda"))
    assert ops.device_errors() == 0
    k = torch.ones(2, 4, 128, dtype=torch.bfloat16, device="cuda")
    ops.store_quant(gp, k, k, torch.tensor([3, 99], dtype=torch.int32, device="cuda"))
    assert ops.device_errors() & 0x1
    assert ops.device_errors() == 0  # cleared
    assert (gp.k_codes[3] == 0x7E).all()  # the valid row was written (1.0 / (1/448) = 448)


@pytest.mark.parametrize("P", [1, 5, 8192, 14336])
def test_reconstruct_bit_exact(P):
    R = 33059
    gp, op, slots = _store_both(P, R, sigma=1.0, big=0.0, zero=0.0, seed=100 + P)
    wk, wv = ops.reconstruct_bf16(gp, torch.from_numpy(slots).cuda())
    ok, ov = oracle.reconstruct(op, slots)
    assert np.array_equal(cuda_bf16_to_bits(wk), ok)
    assert np.array_equal(cuda_bf16_to_bits(wv), ov)


def test_reconstruct_wide_magnitudes_bit_exact():
    gp, op, slots = _store_both(3000, 5000, sigma=2.0, big=0.05, zero=0.01, seed=9)
    wk, wv = ops.reconstruct_bf16(gp, torch.from_numpy(slots).cuda())
    ok, ov = oracle.reconstruct(op, slots)
    assert np.array_equal(cuda_bf16_to_bits(wk), ok)
    assert np.array_equal(cuda_bf16_to_bits(wv), ov)


def test_store_random_bit_patterns_bit_exact():
    """Rows of random finite BF16 bit patterns over the whole exponent range (and rows confined to a
    few binades at random offsets): codes and scales bit-exact, which checks the per-element division."""
    rng = np.random.default_rng(77)
    T, R = 20000, 40000
    bits = rng.integers(0, 1 << 16, size=(T, 4, 128), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] &= 0xBF7F          # no Inf/NaN
    narrow = rng.random(T) < 0.5                        # half the tokens: exponents within 3 binades
    e = rng.integers(1, 250, size=(T, 1, 1)).astype(np.uint16)
    mant = rng.integers(0, 1 << 7, size=(T, 4, 128)).astype(np.uint16)
    sign = rng.integers(0, 2, size=(T, 4, 128)).astype(np.uint16) << 15
    ex = np.clip(e + rng.integers(0, 3, size=(T, 4, 128)).astype(np.uint16), 1, 254)
    bits[narrow] = (sign | (ex << 7) | mant)[narrow]
    v = bits[::-1].copy()
    slots = rng.permutation(R)[:T].astype(np.int32)
    gp = ops.KVPool.empty(R, 4)
    ops.store_quant(gp, bits_to_cuda_bf16(bits), bits_to_cuda_bf16(v), torch.from_numpy(slots).cuda())
    op = oracle.Pool(R, 4, 128)
    oracle.store_quant(op, bits, v, slots)
    _assert_pool_equal(gp, op, slots)


def _mantissa_pair_rows(exps, rng):
    """Rows that hold, for every BF16 mantissa m_a of the row's absmax (element 0) and every row exponent b in
    `exps`, every BF16 mantissa m_x at every exponent b - k, k = 0..21, below the absmax (random signs, 127
    elements a row, the last row of a group padded with zeros)."""
    rows = []
    mx = np.arange(128)
    for b in exps:
        for ma in range(128):
            amax = np.float32((1 + ma / 128) * 2.0 ** b)
            xs = [(1 + mx / 128) * 2.0 ** (b - k) for k in range(22)]
            xs = np.concatenate(xs)
            xs = xs[xs <= amax].astype(np.float32)
            xs *= np.where(rng.random(xs.size) < 0.5, -1.0, 1.0).astype(np.float32)
            pad = (-xs.size) % 127
            xs = np.concatenate([xs, np.zeros(pad, np.float32)]).reshape(-1, 127)
            rows.append(np.concatenate([np.full((xs.shape[0], 1), amax, np.float32), xs], axis=1))
    return np.concatenate(rows)


def test_store_every_bf16_mantissa_pair_bit_exact():
    """The store's quotient x / scale, scale = RN(absmax / 448), depends on the BF16 mantissas of x and of the
    absmax and on their exponent gap only (away from FP32 subnormals): these rows hold every such combination
    whose quotient is in or below the E4M3 range (over row exponents from FP32-subnormal scales to 2^126): the
    code of every quotient a BF16 row can produce, 7,592 of them exact ties at E4M3 rounding midpoints.  Codes
    and scales bit-exact against the oracle."""
    rng = np.random.default_rng(2024)
    x = _mantissa_pair_rows([-120, -100, -37, 0, 11, 60, 126], rng)
    T = (x.shape[0] + 3) // 4
    x = np.concatenate([x, np.zeros((4 * T - x.shape[0], 128), np.float32)]).reshape(T, 4, 128)
    bits = inputs.to_bf16_bits(x)
    v = bits[rng.permutation(T)].copy()
    R = T + 100
    slots = rng.permutation(R)[:T].astype(np.int32)
    gp = ops.KVPool.empty(R, 4)
    ops.store_quant(gp, bits_to_cuda_bf16(bits), bits_to_cuda_bf16(v), torch.from_numpy(slots).cuda())
    op = oracle.Pool(R, 4, 128)
    oracle.store_quant(op, bits, v, slots)
    _assert_pool_equal(gp, op, slots)
    assert ops.device_errors() == 0


def test_store_quotients_at_e4m3_midpoints_bit_exact():
    """Rows whose quotients x / scale land on or within a few ulps of E4M3 rounding midpoints, over scales
    from 2^-40 to 2^40: any shortcut for the per-element IEEE division shows up here as a changed code.
    Element 0 of every row is its absmax, so the scale is known."""
    rng = np.random.default_rng(123)
    T, R = 8192, 9000
    amax = (2.0 ** rng.uniform(-40, 40, size=(T, 4, 1))).astype(np.float32)
    amax = inputs.to_bf16_bits(amax).astype(np.uint32) << 16
    amax = amax.view(np.float32)
    codes = rng.integers(0, 126, size=(T, 4, 128))
    mids = (oracle.e4m3_decode(codes.astype(np.uint8)) + oracle.e4m3_decode((codes + 1).astype(np.uint8))) / 2
    wiggle = 1.0 + rng.integers(-4, 5, size=(T, 4, 128)) * 2.0 ** -8  # a few BF16 ulps around the midpoint
    sign = np.where(rng.random((T, 4, 128)) < 0.5, -1.0, 1.0)
    x = (sign * mids * wiggle * amax.astype(np.float64) / 448.0).astype(np.float32)
    x = np.clip(x, -amax, amax)
    x[:, :, 0] = amax[:, :, 0]
    bits = inputs.to_bf16_bits(x)
    slots = rng.permutation(R)[:T].astype(np.int32)
    gp = ops.KVPool.empty(R, 4)
    ops.store_quant(gp, bits_to_cuda_bf16(bits), bits_to_cuda_bf16(bits[::-1].copy()), torch.from_numpy(slots).cuda())
    op = oracle.Pool(R, 4, 128)
    oracle.store_quant(op, bits, bits[::-1].copy(), slots)
    _assert_pool_equal(gp, op, slots)
