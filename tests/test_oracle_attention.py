"""Pins for the oracle's FP64 attention (CPU only).

* Library special case: torch's FP64 ``scaled_dot_product_attention`` on tiny inputs, with the K/V
  dequantized by torch's float8_e4m3fn dtype (decode) and the GQA groups expanded explicitly.
* Closed forms: one key -> that key's value; identical keys -> mean of the values; q = 0 -> uniform mean.
* Invariants: query heads of one GQA group with equal queries agree; multi-row decode's last row is the
  single-row decode over all keys, and row r is the single-row decode over the first n-R+r+1 keys;
  permuting pool rows (with the slot table) changes nothing; prefill with an empty prefix is plain
  causal attention.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from fp8_kv_cache_ftkv_gb300 import inputs

SM = inputs.SM_SCALE


def _pool_from(rng, R, n, Hkv=4, D=128, sigma=1.0):
    k, v = inputs.kv_tokens(rng, n, sigma, Hkv=Hkv, head_dim=D)
    slots = rng.permutation(R)[:n].astype(np.int32)
    pool = oracle.Pool(R, Hkv, D)
    oracle.store_quant(pool, k, v, slots)
    return pool, slots


def _torch_deq(codes, scales):
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)
    return c * torch.from_numpy(scales).to(torch.float64)[..., None]


def _sdpa(q, k, v, mask=None):
    """q [Hq, Lq, D], k/v [Hkv, Lk, D] (FP64) -> [Hq, Lq, D]; GQA by repeating KV heads."""
    G = q.shape[0] // k.shape[0]
    k = k.repeat_interleave(G, dim=0)
    v = v.repeat_interleave(G, dim=0)
    return F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=SM)


@pytest.mark.parametrize("Hq,Hkv", [(32, 4), (16, 4), (8, 8)])
def test_decode_matches_torch_sdpa(Hq, Hkv):
    rng = np.random.default_rng(21)
    R, n = 97, 61
    pool, slots = _pool_from(rng, R, n, Hkv=Hkv)
    q = inputs.queries(rng, 1, Hq)
    got = oracle.decode_attn(pool, q, slots[None], [n], [0, 1], SM, Hq)[0]
    kd = _torch_deq(pool.k_codes[slots], pool.k_scales[slots]).permute(1, 0, 2)   # [Hkv, n, D]
    vd = _torch_deq(pool.v_codes[slots], pool.v_scales[slots]).permute(1, 0, 2)
    qd = torch.from_numpy(inputs.bf16_bits_to_f32(q[0])).to(torch.float64)[:, None, :]
    want = _sdpa(qd, kd, vd)[:, 0, :].numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv", [(32, 4), (16, 2)])
def test_decode_256d_matches_torch_sdpa(Hq, Hkv):
    """256-d heads (the Qwen3.6 full-attention case of PR #897): the same definition, scale 1/16."""
    rng = np.random.default_rng(23)
    R, n = 90, 57
    pool, slots = _pool_from(rng, R, n, Hkv=Hkv, D=256)
    q = inputs.queries(rng, 1, Hq, 256)
    got = oracle.decode_attn(pool, q, slots[None], [n], [0, 1], 1.0 / 16.0, Hq)[0]
    kd = _torch_deq(pool.k_codes[slots], pool.k_scales[slots]).permute(1, 0, 2)
    vd = _torch_deq(pool.v_codes[slots], pool.v_scales[slots]).permute(1, 0, 2)
    qd = torch.from_numpy(inputs.bf16_bits_to_f32(q[0])).to(torch.float64)[:, None, :]
    G = Hq // Hkv
    want = F.scaled_dot_product_attention(qd, kd.repeat_interleave(G, 0), vd.repeat_interleave(G, 0),
                                          scale=1.0 / 16.0)[:, 0, :].numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_decode_multirow_matches_torch_sdpa_with_causal_mask():
    rng = np.random.default_rng(22)
    R, n, rows = 128, 50, 5
    pool, slots = _pool_from(rng, R, n)
    q = inputs.queries(rng, rows)
    got = oracle.decode_attn(pool, q, slots[None], [n], [0, rows], SM, 32)
    kd = _torch_deq(pool.k_codes[slots], pool.k_scales[slots]).permute(1, 0, 2)
    vd = _torch_deq(pool.v_codes[slots], pool.v_scales[slots]).permute(1, 0, 2)
    qd = torch.from_numpy(inputs.bf16_bits_to_f32(q)).to(torch.float64).permute(1, 0, 2)  # [Hq, rows, D]
    r = torch.arange(rows)[:, None]
    j = torch.arange(n)[None, :]
    mask = j <= (n - rows + r)
    want = _sdpa(qd, kd, vd, mask).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_decode_closed_forms():
    rng = np.random.default_rng(23)
    R = 40
    pool, slots = _pool_from(rng, R, 20)
    q = inputs.queries(rng, 1)
    # one key -> its dequantized value
    one = oracle.decode_attn(pool, q, slots[None, :1], [1], [0, 1], SM, 32)[0]
    v0 = oracle.e4m3_decode(pool.v_codes[slots[0]]) * pool.v_scales[slots[0]][:, None]
    np.testing.assert_array_equal(one, np.repeat(v0, 8, axis=0))
    # identical keys -> arithmetic mean of the values
    pool.k_codes[slots[1:6]] = pool.k_codes[slots[0]]
    pool.k_scales[slots[1:6]] = pool.k_scales[slots[0]]
    out = oracle.decode_attn(pool, q, slots[None, :6], [6], [0, 1], SM, 32)[0]
    vals = np.stack([oracle.e4m3_decode(pool.v_codes[s]) * pool.v_scales[s][:, None] for s in slots[:6]])
    np.testing.assert_allclose(out, np.repeat(vals.mean(axis=0), 8, axis=0), rtol=1e-13, atol=1e-13)
    # q = 0 -> uniform mean over all keys
    qz = np.zeros_like(q)
    out = oracle.decode_attn(pool, qz, slots[None], [20], [0, 1], SM, 32)[0]
    vals = np.stack([oracle.e4m3_decode(pool.v_codes[s]) * pool.v_scales[s][:, None] for s in slots])
    np.testing.assert_allclose(out, np.repeat(vals.mean(axis=0), 8, axis=0), rtol=1e-13, atol=1e-13)


def test_decode_invariants():
    rng = np.random.default_rng(24)
    R, n, rows = 300, 120, 4
    pool, slots = _pool_from(rng, R, n)
    q = inputs.queries(rng, rows)
    q[:, 9] = q[:, 8]          # heads 8 and 9 share KV head 1 and now the same query
    multi = oracle.decode_attn(pool, q, slots[None], [n], [0, rows], SM, 32)
    np.testing.assert_array_equal(multi[:, 8], multi[:, 9])
    for r in range(rows):
        single = oracle.decode_attn(pool, q[r:r + 1], slots[None], [n - rows + r + 1], [0, 1], SM, 32)
        np.testing.assert_array_equal(multi[r], single[0])
    # permuting the pool rows together with the slot table changes nothing
    perm = rng.permutation(R)
    inv = np.argsort(perm)
    pool2 = oracle.Pool(R, 4, 128)
    pool2.k_codes[:] = pool.k_codes[perm]
    pool2.v_codes[:] = pool.v_codes[perm]
    pool2.k_scales[:] = pool.k_scales[perm]
    pool2.v_scales[:] = pool.v_scales[perm]
    slots2 = inv[slots].astype(np.int32)
    again = oracle.decode_attn(pool2, q, slots2[None], [n], [0, rows], SM, 32)
    np.testing.assert_array_equal(multi, again)


def test_decode_batch_and_empty_rows():
    rng = np.random.default_rng(25)
    R = 200
    wl = inputs.decode_custom([30, 1, 45], [2, 1, 3], R, seed=3)
    layer = wl.layer(0)
    pool = oracle.Pool(R, 4, 128)
    oracle.store_quant(pool, layer.k, layer.v, layer.slots)
    out = oracle.decode_attn(pool, layer.q, wl.req_to_slot, wl.seq_lens, wl.q_row_offsets, SM, 32)
    # request 1 has one key and one row -> that value
    s = wl.req_to_slot[1, 0]
    v = oracle.e4m3_decode(pool.v_codes[s]) * pool.v_scales[s][:, None]
    np.testing.assert_array_equal(out[2], np.repeat(v, 8, axis=0))
    # each request on its own gives the same rows
    for b in range(3):
        o0, o1 = wl.q_row_offsets[b], wl.q_row_offsets[b + 1]
        alone = oracle.decode_attn(pool, layer.q[o0:o1], wl.req_to_slot[b:b + 1], wl.seq_lens[b:b + 1],
                                   [0, o1 - o0], SM, 32)
        np.testing.assert_array_equal(out[o0:o1], alone)
    # a row that sees no key (seq_len < rows) outputs zeros
    z = oracle.decode_attn(pool, layer.q[:3], wl.req_to_slot[:1], [1], [0, 3], SM, 32)
    assert (z[0] == 0).all() and (z[1] == 0).all() and (z[2] != 0).any()


def test_prefill_matches_torch_sdpa():
    rng = np.random.default_rng(26)
    P, C = 37, 29
    wk, wv = inputs.kv_tokens(rng, P, 1.0)
    kc, vc = inputs.kv_tokens(rng, C, 1.0)
    q = inputs.queries(rng, C)
    got = oracle.prefill_attn(q, kc, vc, wk, wv, SM)
    t = lambda b: torch.from_numpy(inputs.bf16_bits_to_f32(b)).to(torch.float64).permute(1, 0, 2)
    K = torch.cat([t(wk), t(kc)], dim=1)
    V = torch.cat([t(wv), t(vc)], dim=1)
    i = torch.arange(C)[:, None]
    j = torch.arange(P + C)[None, :]
    mask = j <= P + i
    want = _sdpa(t(q), K, V, mask).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # sampled rows equal the full evaluation
    rows = np.array([0, 5, 28], np.int64)
    np.testing.assert_array_equal(oracle.prefill_attn(q, kc, vc, wk, wv, SM, rows), got[rows])


def test_prefill_empty_prefix_is_causal_attention():
    rng = np.random.default_rng(27)
    C = 33
    kc, vc = inputs.kv_tokens(rng, C, 1.0)
    q = inputs.queries(rng, C)
    empty = np.zeros((0, 4, 128), np.uint16)
    got = oracle.prefill_attn(q, kc, vc, empty, empty, SM)
    t = lambda b: torch.from_numpy(inputs.bf16_bits_to_f32(b)).to(torch.float64).permute(1, 0, 2)
    G = 8
    want = F.scaled_dot_product_attention(t(q), t(kc).repeat_interleave(G, 0), t(vc).repeat_interleave(G, 0),
                                          is_causal=True, scale=SM).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # first chunk row sees only itself
    np.testing.assert_array_equal(got[0], np.repeat(inputs.bf16_bits_to_f32(vc[0]).astype(np.float64), 8, 0))


def test_abs_mode_is_attention_over_absolute_values():
    """The test helper mode (sum p |v| / sum p) equals torch SDPA with |v| as values."""
    rng = np.random.default_rng(28)
    R, n = 80, 50
    pool, slots = _pool_from(rng, R, n)
    q = inputs.queries(rng, 1)
    got = oracle.decode_attn(pool, q, slots[None], [n], [0, 1], SM, 32, abs_v=True)[0]
    kd = _torch_deq(pool.k_codes[slots], pool.k_scales[slots]).permute(1, 0, 2)
    vd = _torch_deq(pool.v_codes[slots], pool.v_scales[slots]).permute(1, 0, 2).abs()
    qd = torch.from_numpy(inputs.bf16_bits_to_f32(q[0])).to(torch.float64)[:, None, :]
    np.testing.assert_allclose(got, _sdpa(qd, kd, vd)[:, 0, :].numpy(), rtol=1e-12, atol=1e-12)
    P, C = 20, 15
    wk, wv = inputs.kv_tokens(rng, P, 1.0)
    kc, vc = inputs.kv_tokens(rng, C, 1.0)
    q = inputs.queries(rng, C)
    absd = lambda b: inputs.to_bf16_bits(np.abs(inputs.bf16_bits_to_f32(b)))
    np.testing.assert_array_equal(oracle.prefill_attn(q, kc, vc, wk, wv, SM, abs_v=True),
                                  oracle.prefill_attn(q, kc, absd(vc), wk, absd(wv), SM))


# ---- decode over a BF16 pool, and the sliding window ----

def _bf16_pool(rng, R, n, Hkv=4, D=128, sigma=1.0):
    k, v = inputs.kv_tokens(rng, n, sigma, Hkv=Hkv, head_dim=D)
    slots = rng.permutation(R)[:n].astype(np.int32)
    kp = np.zeros((R, Hkv, D), np.uint16)
    vp = np.zeros_like(kp)
    kp[slots], vp[slots] = k, v
    return kp, vp, slots


def _bf16_t(bits):
    return torch.from_numpy(inputs.bf16_bits_to_f32(bits)).to(torch.float64)


@pytest.mark.parametrize("Hq,Hkv,rows", [(32, 4, 1), (16, 4, 3), (8, 8, 1)])
def test_decode_bf16_pool_matches_torch_sdpa(Hq, Hkv, rows):
    rng = np.random.default_rng(61)
    R, n = 90, 57
    kp, vp, slots = _bf16_pool(rng, R, n, Hkv=Hkv)
    q = inputs.queries(rng, rows, Hq)
    got = oracle.decode_attn_bf16(kp, vp, q, slots[None], [n], [0, rows], SM, Hq)
    kd = _bf16_t(kp[slots]).permute(1, 0, 2)
    vd = _bf16_t(vp[slots]).permute(1, 0, 2)
    qd = _bf16_t(q).permute(1, 0, 2)
    mask = torch.arange(n)[None, :] <= (n - rows + torch.arange(rows)[:, None])
    want = _sdpa(qd, kd, vd, mask).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_decode_bf16_pool_equals_fp8_pool_on_identical_values():
    """With power-of-two scales every dequantized FP8 value is a BF16 value: both pool kinds then hold the
    same numbers, and the two decodes must agree exactly (a dropped scale or a wrong row would show)."""
    rng = np.random.default_rng(62)
    R, n, Hkv = 64, 40, 4
    pool = oracle.Pool(R, Hkv, 128)
    codes = rng.integers(0, 256, size=(R, Hkv, 128), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38           # no NaN codes
    pool.k_codes[:], pool.v_codes[:] = codes, codes[::-1]
    pool.k_scales[:] = 2.0 ** rng.integers(-6, 6, size=(R, Hkv))
    pool.v_scales[:] = 2.0 ** rng.integers(-6, 6, size=(R, Hkv))
    kval = oracle.e4m3_decode(pool.k_codes) * pool.k_scales[..., None]
    vval = oracle.e4m3_decode(pool.v_codes) * pool.v_scales[..., None]
    kb, vb = inputs.to_bf16_bits(kval.astype(np.float32)), inputs.to_bf16_bits(vval.astype(np.float32))
    assert np.array_equal(inputs.bf16_bits_to_f32(kb).astype(np.float64), kval)   # exact in BF16
    slots = rng.permutation(R)[:n].astype(np.int32)
    q = inputs.queries(rng, 2)
    a = oracle.decode_attn(pool, q, slots[None], [n], [0, 2], SM, 32)
    b = oracle.decode_attn_bf16(kb, vb, q, slots[None], [n], [0, 2], SM, 32)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("window,rows", [(1, 1), (7, 1), (13, 3), (56, 1), (1000, 2)])
def test_decode_sliding_window_matches_torch_sdpa_with_banded_mask(window, rows):
    rng = np.random.default_rng(63 + window)
    R, n = 80, 57
    pool, slots = _pool_from(rng, R, n)
    q = inputs.queries(rng, rows)
    got = oracle.decode_attn(pool, q, slots[None], [n], [0, rows], SM, 32, window=window)
    kd = _torch_deq(pool.k_codes[slots], pool.k_scales[slots]).permute(1, 0, 2)
    vd = _torch_deq(pool.v_codes[slots], pool.v_scales[slots]).permute(1, 0, 2)
    qd = torch.from_numpy(inputs.bf16_bits_to_f32(q)).to(torch.float64).permute(1, 0, 2)
    last = n - rows + torch.arange(rows)[:, None]             # last visible key of each row
    j = torch.arange(n)[None, :]
    mask = (j <= last) & (j > last - window)
    want = _sdpa(qd, kd, vd, mask).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # the same window over the BF16 pool holding the same values
    kb = inputs.to_bf16_bits(kd.permute(1, 0, 2).numpy().astype(np.float32))
    if np.array_equal(inputs.bf16_bits_to_f32(kb).astype(np.float64), kd.permute(1, 0, 2).numpy()):
        vb = inputs.to_bf16_bits(vd.permute(1, 0, 2).numpy().astype(np.float32))
        kp = np.zeros((R, 4, 128), np.uint16)
        vp = np.zeros_like(kp)
        kp[slots], vp[slots] = kb, vb
        got_b = oracle.decode_attn_bf16(kp, vp, q, slots[None], [n], [0, rows], SM, 32, window=window)
        np.testing.assert_allclose(got_b, want, rtol=1e-12, atol=1e-12)


def test_decode_sliding_window_closed_forms():
    rng = np.random.default_rng(64)
    R, n = 50, 30
    pool, slots = _pool_from(rng, R, n)
    q = inputs.queries(rng, 1)
    # window 1: the value of the last key alone
    got = oracle.decode_attn(pool, q, slots[None], [n], [0, 1], SM, 32, window=1)[0]
    vlast = oracle.e4m3_decode(pool.v_codes[slots[n - 1]]) * pool.v_scales[slots[n - 1]][:, None]
    for i in range(32):
        np.testing.assert_allclose(got[i], vlast[i // 8], rtol=1e-12, atol=1e-12)
    # a window of n or more keys is full attention
    full = oracle.decode_attn(pool, q, slots[None], [n], [0, 1], SM, 32)
    np.testing.assert_array_equal(oracle.decode_attn(pool, q, slots[None], [n], [0, 1], SM, 32, window=n), full)
    # window w equals full attention over the last w keys only
    w = 9
    sub = oracle.decode_attn(pool, q, slots[None, n - w:], [w], [0, 1], SM, 32)
    np.testing.assert_allclose(oracle.decode_attn(pool, q, slots[None], [n], [0, 1], SM, 32, window=w), sub,
                               rtol=1e-13, atol=1e-13)
