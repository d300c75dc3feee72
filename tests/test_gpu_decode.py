"""GPU parity: split-K FP8 decode attention against the FP64 oracle.

Covers the 512-token single step, ragged key counts (1, 17, 513, 4099), split counts 1/8/64/152/256 and
automatic, GQA group sizes 8/4/2/1 and 8 KV heads, multi-row decode (1..8 rows, rows that see no key), the
sliding windows (1 key to more than the sequence, single- and multi-row, with the fused store), the
32,768- and 40,000-key batch-1 workloads at full size (sampled layers, every output element), the batched
64-request multi-row workload at full size, negative and zero softmax scales, and chains of decode launches in one stream with and without
FTKV_DECODE_STABLE_HISTORY (history loads issued before the preceding kernel has finished).  Single-row
cases run with the flag off and on ("stable").
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_ftkv_gb300 import inputs, ops
from parity import bits_to_cuda_bf16, check_attention

pytestmark = pytest.mark.gpu
STABLE = [False, True]


def _setup(wl: inputs.DecodeWorkload, layer: int = 0):
    """Store one layer of the workload on both sides; return GPU pool, oracle pool, device tensors."""
    L = wl.layer(layer)
    gp = ops.KVPool.empty(wl.num_rows, wl.Hkv)
    if L.slots.size:
        ops.store_quant(gp, bits_to_cuda_bf16(L.k), bits_to_cuda_bf16(L.v), torch.from_numpy(L.slots).cuda())
    op = oracle.Pool(wl.num_rows, wl.Hkv, 128)
    if L.slots.size:
        oracle.store_quant(op, L.k, L.v, L.slots)
    dev = dict(q=bits_to_cuda_bf16(L.q), r2s=torch.from_numpy(wl.req_to_slot).cuda(),
               lens=torch.from_numpy(wl.seq_lens).cuda(), offs=torch.from_numpy(wl.q_row_offsets).cuda())
    return gp, op, L, dev


def _run(wl, gp, dev, num_splits=0, max_q_rows=None, stable=False, window=0):
    R = np.diff(wl.q_row_offsets)
    mq = int(max(R.max(), 1)) if max_q_rows is None else max_q_rows
    return ops.decode_attn(gp, dev["q"], dev["r2s"], dev["lens"], dev["offs"], max_seq_len=int(wl.req_to_slot.shape[1]),
                           max_q_rows=mq, sm_scale=wl.sm_scale, num_splits=num_splits, stable_history=stable,
                           window=window)


def _ref(wl, op, L, window=0):
    args = (op, L.q, wl.req_to_slot, wl.seq_lens, wl.q_row_offsets, wl.sm_scale, wl.Hq)
    return (oracle.decode_attn(*args, window=window), oracle.decode_attn(*args, abs_v=True, window=window))


def _check(out, refs, what):
    return check_attention(out, refs[0], what, refs[1])


@pytest.mark.parametrize("stable", STABLE)
def test_decode_small_step(stable):
    wl = inputs.decode_small()
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev, stable=stable)
    stats = _check(out, _ref(wl, op, L), "decode_small")
    assert stats["max_abs"] < 0.05
    assert ops.device_errors() == 0


@pytest.mark.parametrize("stable", STABLE)
@pytest.mark.parametrize("n", [1, 17, 513, 4099])
@pytest.mark.parametrize("splits", [0, 1, 8, 64, 152, 256])
def test_decode_ragged_lengths_and_split_caps(n, splits, stable):
    wl = inputs.decode_custom([n], [1], max(2 * n, 64), seed=n)
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev, num_splits=splits, stable=stable)
    _check(out, _ref(wl, op, L), f"n={n} splits={splits} stable={stable}")


@pytest.mark.parametrize("stable", STABLE)
@pytest.mark.parametrize("n,splits", [(9000, 1), (20000, 3), (2049, 2), (131, 1), (131, 2)])
def test_decode_long_slices_cross_slot_windows(n, splits, stable):
    """Slices of thousands of keys (several 1,024-slot windows of the single-row kernel, several 4,096-slot
    windows of the multi-row kernel), a slice ending one key past a window, and slices shorter than one
    16-key block per key group."""
    wl = inputs.decode_custom([n], [1], n + 7, seed=n + splits)
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev, num_splits=splits, stable=stable)
    _check(out, _ref(wl, op, L), f"n={n} splits={splits}")
    assert ops.device_errors() == 0


@pytest.mark.parametrize("stable", STABLE)
@pytest.mark.parametrize("Hq,Hkv", [(32, 4), (16, 4), (8, 4), (4, 4), (64, 8), (16, 2), (8, 1), (12, 6)])
def test_decode_gqa_groups(Hq, Hkv, stable):
    """GQA groups 8/4/2/1 with 4 KV heads per CTA, 8 KV heads (two CTAs per key slice), and 2, 1 and 6 KV heads
    (CTAs of 2 or 1 heads)."""
    wl = inputs.decode_custom([300, 1000], [1, 1], 4000, seed=Hq, Hq=Hq, Hkv=Hkv)
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev, stable=stable)
    _check(out, _ref(wl, op, L), f"Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("rows", [[2], [3, 1, 8], [8, 8], [5, 7, 6, 4]])
def test_decode_multirow(rows):
    lens = [200 + 97 * i for i in range(len(rows))]
    wl = inputs.decode_custom(lens, rows, 5000, sigma=2.0, big_frac=0.01, zero_frac=0.01, seed=len(rows))
    gp, op, L, dev = _setup(wl)
    for splits in (0, 1, 5):
        out = _run(wl, gp, dev, num_splits=splits)
        _check(out, _ref(wl, op, L), f"rows={rows} splits={splits}")


@pytest.mark.parametrize("rows", [[1], [3, 8]])
@pytest.mark.parametrize("scale", [-0.0883883, 0.0, 2.0])
def test_decode_softmax_scale_sign_and_zero(rows, scale):
    """A negative softmax scale (the scores change sign), a zero one (uniform weights over the visible keys) and
    a large one, on the single-row and the multi-row kernels (one and two groups of 32 query rows)."""
    lens = [700 + 301 * i for i in range(len(rows))]
    wl = inputs.decode_custom(lens, rows, 4000, seed=11 + len(rows))
    wl.sm_scale = scale
    gp, op, L, dev = _setup(wl)
    for splits in (0, 3):
        out = _run(wl, gp, dev, num_splits=splits)
        _check(out, _ref(wl, op, L), f"rows={rows} scale={scale} splits={splits}")
    assert ops.device_errors() == 0


def test_decode_rows_that_see_no_key_are_zero():
    wl = inputs.decode_custom([2, 40], [5, 3], 100, seed=3)
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev)
    refs = _ref(wl, op, L)
    assert (refs[0][:3] == 0).all()
    _check(out, refs, "empty rows")
    assert (out[:3].float() == 0).all()


@pytest.mark.parametrize("stable", STABLE)
def test_decode_zero_length_request_and_single_row_path_with_offsets(stable):
    wl = inputs.decode_custom([0, 33, 1], [1, 1, 1], 64, seed=4)
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev, stable=stable)
    _check(out, _ref(wl, op, L), "zero-length request")
    assert (out[0].float() == 0).all()


@pytest.mark.parametrize("stable", STABLE)
@pytest.mark.parametrize("n,R", [(32768, 33059), (40000, 40290)])
def test_decode_long_context_full_size(n, R, stable):
    wl = inputs.decode_long(n, R, layers=48)
    for layer in (0, 47):
        gp, op, L, dev = _setup(wl, layer)
        out = _run(wl, gp, dev, stable=stable)
        stats = _check(out, _ref(wl, op, L), f"n={n} layer={layer} stable={stable}")
        assert stats["rel_l2"] < 2e-3
    assert ops.device_errors() == 0


def test_decode_batched_multirow_full_size():
    wl = inputs.decode_batched()
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev)
    # sampled outputs: every query row of 12 requests (all heads, all d)
    rng = np.random.default_rng(0)
    for b in sorted(rng.choice(len(wl.seq_lens), size=12, replace=False)):
        o0, o1 = int(wl.q_row_offsets[b]), int(wl.q_row_offsets[b + 1])
        args = (op, L.q[o0:o1], wl.req_to_slot[b:b + 1], wl.seq_lens[b:b + 1],
                np.array([0, o1 - o0], np.int32), wl.sm_scale, wl.Hq)
        check_attention(out[o0:o1], oracle.decode_attn(*args), f"request {b}", oracle.decode_attn(*args, abs_v=True))
    assert ops.device_errors() == 0


@pytest.mark.parametrize("rows", [[8], [4], [5, 3]])
def test_decode_multirow_long_request_full_size(rows):
    """One or two long requests with several query rows (8 rows x 8 heads: two groups of 32 query rows per
    KV head; 4 rows: one group repeated over the four TMEM lane quarters) at 32,768 keys: ~38 key slices of
    ~7 tiles each, every output element against the FP64 oracle."""
    lens = [32768] if len(rows) == 1 else [32768, 20001]
    wl = inputs.decode_custom(lens, rows, 60000, sigma=1.0, seed=31 + sum(rows))
    gp, op, L, dev = _setup(wl)
    out = _run(wl, gp, dev)
    _check(out, _ref(wl, op, L), f"long multirow rows={rows}")
    assert ops.device_errors() == 0


@pytest.mark.parametrize("max_q_rows", [1, 2])
@pytest.mark.parametrize("stable", STABLE)
def test_decode_bad_slot_and_seq_len_are_flagged_not_faulted(stable, max_q_rows):
    wl = inputs.decode_custom([50], [1], 128, seed=5)
    gp, op, L, dev = _setup(wl)
    bad = dev["r2s"].clone()
    bad[0, 3] = 10 ** 6
    bad[0, 4] = -7
    ops.decode_attn(gp, dev["q"], bad, dev["lens"], dev["offs"], max_seq_len=50, max_q_rows=max_q_rows,
                    stable_history=stable)
    assert ops.device_errors() & 0x1
    lens = torch.tensor([60], dtype=torch.int32, device="cuda")
    ops.decode_attn(gp, dev["q"], dev["r2s"], lens, dev["offs"], max_seq_len=50, max_q_rows=max_q_rows,
                    stable_history=stable)
    assert ops.device_errors() & 0x2
    assert ops.device_errors() == 0


@pytest.mark.parametrize("max_q_rows,stable", [(1, False), (1, True), (2, False)])
def test_decode_dominant_key_with_small_v_scale(max_q_rows, stable):
    """A key holding almost all the probability has a V scale 1e6 x smaller than a key with tiny
    probability; both terms matter (ratio ~0.1) and the dominant one must keep full precision."""
    rng = np.random.default_rng(31)
    n, R = 48, 64
    k = np.zeros((n, 4, 128), np.float32)
    v = rng.standard_normal((n, 4, 128)).astype(np.float32)
    k[:, :, 0] = rng.standard_normal((n, 4)).astype(np.float32)
    k[7, :, 0] = 181.0          # dominant logit: s = 181 * 0.0884 = 16 above the rest
    v[7] *= 1.0                 # V scale ~ 1/448 * 3
    v[23] *= 1.0e6              # e^-16 * 1e6 ~ 0.1 relative contribution
    q = np.zeros((max_q_rows, 32, 128), np.float32)
    q[:, :, 0] = 1.0
    kb, vb, qb = inputs.to_bf16_bits(k), inputs.to_bf16_bits(v), inputs.to_bf16_bits(q)
    slots = rng.permutation(R)[:n].astype(np.int32)
    gp = ops.KVPool.empty(R, 4)
    ops.store_quant(gp, bits_to_cuda_bf16(kb), bits_to_cuda_bf16(vb), torch.from_numpy(slots).cuda())
    op = oracle.Pool(R, 4, 128)
    oracle.store_quant(op, kb, vb, slots)
    offs = np.array([0, max_q_rows], np.int32)
    lens = np.array([n], np.int32)
    out = ops.decode_attn(gp, bits_to_cuda_bf16(qb), torch.from_numpy(slots[None]).cuda(),
                          torch.from_numpy(lens).cuda(), torch.from_numpy(offs).cuda(), max_seq_len=n,
                          max_q_rows=max_q_rows, stable_history=stable)
    args = (op, qb, slots[None], lens, offs, inputs.SM_SCALE, 32)
    ref, mag = oracle.decode_attn(*args), oracle.decode_attn(*args, abs_v=True)
    stats = check_attention(out, ref, "dominant small-scale key", mag)
    assert stats["rel_l2"] < 2e-3


@pytest.mark.parametrize("stable", STABLE)
def test_decode_one_hot_attention_with_huge_logits(stable):
    """Logits near 1e5 (a x1e3 key aligned with the query) make the attention one-hot: the output must
    be that key's dequantized value to BF16 rounding, which fails if the V scale is applied through an
    addition to the logit (its log would be rounded to the ulp of the logit)."""
    rng = np.random.default_rng(41)
    n, R = 40, 64
    k = rng.standard_normal((n, 4, 128)).astype(np.float32)
    v = rng.standard_normal((n, 4, 128)).astype(np.float32) * np.float32(0.37)
    q = rng.standard_normal((1, 32, 128)).astype(np.float32)
    k[11] = np.repeat(q[0, ::8], 1, axis=0)[:4] * np.float32(3e3)   # kv head h aligned with query head 8h
    kb, vb, qb = inputs.to_bf16_bits(k), inputs.to_bf16_bits(v), inputs.to_bf16_bits(q)
    slots = rng.permutation(R)[:n].astype(np.int32)
    gp = ops.KVPool.empty(R, 4)
    ops.store_quant(gp, bits_to_cuda_bf16(kb), bits_to_cuda_bf16(vb), torch.from_numpy(slots).cuda())
    op = oracle.Pool(R, 4, 128)
    oracle.store_quant(op, kb, vb, slots)
    lens, offs = np.array([n], np.int32), np.array([0, 1], np.int32)
    out = ops.decode_attn(gp, bits_to_cuda_bf16(qb), torch.from_numpy(slots[None]).cuda(),
                          torch.from_numpy(lens).cuda(), torch.from_numpy(offs).cuda(), max_seq_len=n,
                          stable_history=stable)
    args = (op, qb, slots[None], lens, offs, inputs.SM_SCALE, 32)
    ref, mag = oracle.decode_attn(*args), oracle.decode_attn(*args, abs_v=True)
    vhat = oracle.e4m3_decode(op.v_codes[slots[11]]) * op.v_scales[slots[11]][:, None]
    for h in range(4):                                   # the aligned heads are one-hot on key 11
        np.testing.assert_allclose(ref[0, 8 * h], vhat[h], rtol=1e-9, atol=1e-12)
    o = out.float().cpu().numpy().astype(np.float64)
    for h in range(4):
        assert np.abs(o[0, 8 * h] - vhat[h]).max() <= 2.0 ** -8 * np.abs(vhat[h]).max() + 1e-6
    check_attention(out, ref, "one-hot huge logits", mag)


# ---- sliding window ----

@pytest.mark.parametrize("stable", STABLE)
@pytest.mark.parametrize("lens,rows,window,splits", [
    ([4099], [1], 513, 0), ([4099], [1], 513, 8), ([4099], [1], 1, 0), ([4099], [1], 7, 1), ([300], [1], 299, 0),
    ([300], [1], 300, 3), ([300], [1], 5000, 0), ([32768], [1], 4095, 0), ([1000, 17, 2500], [1, 1, 1], 127, 0),
    ([200, 297, 394], [3, 1, 8], 9, 0), ([200, 297, 394], [3, 1, 8], 131, 5), ([900, 2000], [4, 2], 1, 1),
    ([5, 40], [5, 3], 2, 0), ([0, 33, 1], [1, 1, 1], 16, 0),
])
def test_decode_sliding_window(lens, rows, window, splits, stable):
    """Sliding windows of 1 key to more than the sequence, odd sizes, several slices over the window and
    one; multi-row requests, whose rows each end their window at their own causal limit."""
    wl = inputs.decode_custom(lens, rows, max(sum(lens) + 9, 64), seed=window + len(rows))
    gp, op, L, dev = _setup(wl)
    if stable and max(rows) > 1:
        pytest.skip("the stable-history path is the single-row kernel's")
    out = _run(wl, gp, dev, num_splits=splits, stable=stable, window=window)
    _check(out, _ref(wl, op, L, window), f"window={window} lens={lens} rows={rows} splits={splits}")
    assert ops.device_errors() == 0


@pytest.mark.parametrize("lens,rows,window", [([4099], [1], 513), ([200, 297, 394], [3, 1, 8], 33)])
def test_decode_sliding_window_reads_no_key_before_it(lens, rows, window):
    """Slot entries before a request's first window key are set outside the pool: nothing is flagged, so no
    CTA reads them, and the result is unchanged."""
    wl = inputs.decode_custom(lens, rows, sum(lens) + 9, seed=window)
    gp, op, L, dev = _setup(wl)
    R = np.diff(wl.q_row_offsets)
    r2s = dev["r2s"].clone()
    for b, n in enumerate(wl.seq_lens):
        first = max(0, int(n) - int(R[b]) + 1 - window)
        r2s[b, :first] = 10 ** 7
    out = ops.decode_attn(gp, dev["q"], r2s, dev["lens"], dev["offs"], max_seq_len=int(wl.req_to_slot.shape[1]),
                          max_q_rows=int(R.max()), sm_scale=wl.sm_scale, window=window)
    assert ops.device_errors() == 0
    _check(out, _ref(wl, op, L, window), f"window={window} poisoned history")


# ---- fused store + decode (ftkv_decode_attn_store) ----

def _new_tokens(wl, L):
    """K/V rows of each request's new tokens (its last R_b positions, one per query row; zeros for a
    position below 0) and a mask of those tokens among the workload's tokens."""
    R = np.diff(wl.q_row_offsets)
    starts = np.concatenate([[0], np.cumsum(wl.seq_lens)[:-1]]).astype(np.int64)
    total = int(wl.q_row_offsets[-1])
    k_new = np.zeros((total, wl.Hkv, wl.head_dim), np.uint16)
    v_new = np.zeros_like(k_new)
    new = np.zeros(L.slots.shape[0], bool)
    for b in range(len(wl.seq_lens)):
        n = int(wl.seq_lens[b])
        for r in range(int(R[b])):
            pos = n - int(R[b]) + r
            if pos < 0:
                continue
            t = starts[b] + pos
            k_new[wl.q_row_offsets[b] + r] = L.k[t]
            v_new[wl.q_row_offsets[b] + r] = L.v[t]
            new[t] = True
    return k_new, v_new, new


@pytest.mark.parametrize("stable", STABLE)
@pytest.mark.parametrize("lens,rows,splits", [
    ([512], [1], 0), ([33], [1], 1), ([4099], [1], 8), ([9000], [1], 1), ([1], [1], 0), ([32768], [1], 0),
    ([200, 297, 394], [3, 1, 8], 0), ([200, 297, 394], [3, 1, 8], 5), ([2, 40], [5, 3], 0), ([0, 33, 1], [1, 1, 1], 0),
])
@pytest.mark.parametrize("window", [0, 77])
def test_decode_fused_store_equals_store_then_decode(lens, rows, splits, stable, window):
    """The new tokens' rows land in the pool bit-exactly as the store kernel writes them (oracle store),
    and the attention over them matches the oracle; new tokens split across slices and windows, rows
    past the start of the sequence, and an empty request included."""
    wl = inputs.decode_custom(lens, rows, max(2 * sum(lens), 64), sigma=2.0, big_frac=0.01, zero_frac=0.01,
                              seed=sum(lens) + len(rows))
    L = wl.layer(0)
    k_new, v_new, new = _new_tokens(wl, L)
    gp = ops.KVPool.empty(wl.num_rows, wl.Hkv)
    old = ~new
    if old.any():
        ops.store_quant(gp, bits_to_cuda_bf16(L.k[old]), bits_to_cuda_bf16(L.v[old]),
                        torch.from_numpy(L.slots[old]).cuda())
    op = oracle.Pool(wl.num_rows, wl.Hkv, 128)
    if L.slots.size:
        oracle.store_quant(op, L.k, L.v, L.slots)
    R = np.diff(wl.q_row_offsets)
    out = ops.decode_attn(gp, bits_to_cuda_bf16(L.q), torch.from_numpy(wl.req_to_slot).cuda(),
                          torch.from_numpy(wl.seq_lens).cuda(), torch.from_numpy(wl.q_row_offsets).cuda(),
                          max_seq_len=int(wl.req_to_slot.shape[1]), max_q_rows=int(max(R.max(), 1)),
                          sm_scale=wl.sm_scale, num_splits=splits, k_new=bits_to_cuda_bf16(k_new),
                          v_new=bits_to_cuda_bf16(v_new), stable_history=stable, window=window)
    s = L.slots
    assert np.array_equal(gp.k_codes.cpu().numpy()[s], op.k_codes[s])
    assert np.array_equal(gp.v_codes.cpu().numpy()[s], op.v_codes[s])
    assert np.array_equal(gp.k_scales.cpu().numpy()[s].view(np.uint32), op.k_scales[s].view(np.uint32))
    assert np.array_equal(gp.v_scales.cpu().numpy()[s].view(np.uint32), op.v_scales[s].view(np.uint32))
    _check(out, _ref(wl, op, L, window), f"fused lens={lens} rows={rows} splits={splits} stable={stable} W={window}")
    assert ops.device_errors() == 0


def test_decode_fused_store_bad_slot_is_flagged_and_not_written():
    wl = inputs.decode_custom([50], [1], 128, seed=6)
    L = wl.layer(0)
    k_new, v_new, new = _new_tokens(wl, L)
    gp = ops.KVPool.empty(wl.num_rows, wl.Hkv)
    ops.store_quant(gp, bits_to_cuda_bf16(L.k[~new]), bits_to_cuda_bf16(L.v[~new]),
                    torch.from_numpy(L.slots[~new]).cuda())
    before = (gp.k_codes.cpu().clone(), gp.k_scales.cpu().clone())
    bad = torch.from_numpy(wl.req_to_slot).cuda().clone()
    bad[0, 49] = 10 ** 6  # the new token's slot
    ops.decode_attn(gp, bits_to_cuda_bf16(L.q), bad, torch.from_numpy(wl.seq_lens).cuda(), None, max_seq_len=50,
                    k_new=bits_to_cuda_bf16(k_new), v_new=bits_to_cuda_bf16(v_new))
    assert ops.device_errors() & 0x1
    assert torch.equal(gp.k_codes.cpu(), before[0]) and torch.equal(gp.k_scales.cpu(), before[1])
    assert ops.device_errors() == 0


@pytest.mark.parametrize("lens,rows", [([4099], [1]), ([3000, 70, 1], [1, 1, 1]), ([900, 2000], [4, 2])])
def test_decode_shared_merge_state_resets_between_calls(lens, rows):
    """Consecutive calls on one workspace: the arrival tickets left by one call must be clean for the next;
    groups with different slice counts in one batch."""
    wl = inputs.decode_custom(lens, rows, 2 * sum(lens) + 64, seed=len(lens) + 40)
    gp, op, L, dev = _setup(wl)
    R = np.diff(wl.q_row_offsets)
    mq = int(max(R.max(), 1))
    plan = ops.DecodePlan(wl.Hq, wl.Hkv, len(lens), int(wl.q_row_offsets[-1]), mq, int(wl.req_to_slot.shape[1]), 0,
                          "cuda")
    refs = _ref(wl, op, L)
    first = None
    for it in range(4):
        out = ops.decode_attn(gp, dev["q"], dev["r2s"], dev["lens"], dev["offs"],
                              max_seq_len=int(wl.req_to_slot.shape[1]), max_q_rows=mq, sm_scale=wl.sm_scale,
                              plan=plan)
        _check(out, refs, f"call {it}")
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first)
    assert ops.device_errors() == 0


# ---- chains of launches in one stream: history loads before the preceding kernel ends ----

def _chain_layers(n, R, layers, seed):
    """`layers` pools of one request with n keys; the last key of each is the new token (stored by the decode)."""
    wl = inputs.decode_custom([n], [1], R, seed=seed)
    wl.layers = layers
    out = []
    for l in range(layers):
        L = wl.layer(l)
        gp = ops.KVPool.empty(R, wl.Hkv)
        ops.store_quant(gp, bits_to_cuda_bf16(L.k[:n - 1]), bits_to_cuda_bf16(L.v[:n - 1]),
                        torch.from_numpy(L.slots[:n - 1]).cuda())
        op = oracle.Pool(R, wl.Hkv, 128)
        oracle.store_quant(op, L.k, L.v, L.slots)
        out.append((L, gp, op))
    return wl, out


@pytest.mark.parametrize("graph", [False, True])
def test_decode_stable_history_chain_of_layers(graph):
    """A decode step of 12 layers as back-to-back fused store + decode launches with FTKV_DECODE_STABLE_HISTORY
    (eager, and as one CUDA graph replayed twice): every layer's new token lands bit-exact and every output
    matches the oracle."""
    n, R, layers = 6000, 6100, 12
    wl, ls = _chain_layers(n, R, layers, seed=77)
    r2s = torch.from_numpy(wl.req_to_slot).cuda()
    lens = torch.from_numpy(wl.seq_lens).cuda()
    plan = ops.DecodePlan(wl.Hq, wl.Hkv, 1, 1, 1, n, 0, "cuda")
    q = [bits_to_cuda_bf16(L.q) for L, _, _ in ls]
    kn = [bits_to_cuda_bf16(L.k[n - 1:n]) for L, _, _ in ls]
    vn = [bits_to_cuda_bf16(L.v[n - 1:n]) for L, _, _ in ls]
    outs = [torch.empty_like(x) for x in q]
    stream = torch.cuda.Stream()

    def step():
        for l, (L, gp, op) in enumerate(ls):
            ops.decode_attn(gp, q[l], r2s, lens, None, max_seq_len=n, plan=plan, out=outs[l], k_new=kn[l],
                            v_new=vn[l], stable_history=True, stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step()
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            for o in outs:
                o.zero_()
            g.replay()
            g.replay()
    torch.cuda.synchronize()
    s = ls[0][0].slots
    for l, (L, gp, op) in enumerate(ls):
        assert np.array_equal(gp.k_codes.cpu().numpy()[s], op.k_codes[s]), l
        assert np.array_equal(gp.v_scales.cpu().numpy()[s].view(np.uint32), op.v_scales[s].view(np.uint32)), l
        _check(outs[l], _ref(wl, op, L), f"chain layer {l} graph={graph}")
    assert ops.device_errors() == 0


@pytest.mark.parametrize("stable", STABLE)
def test_decode_after_store_kernel_on_the_same_pool(stable):
    """ftkv_store_quant writes the new token's rows, then ftkv_decode_attn reads the same pool, back to back in
    one stream: the decode must see the stored rows.  The new token is not history, so this order is allowed
    with FTKV_DECODE_STABLE_HISTORY as well (its block is loaded only after the store kernel has finished)."""
    n, R = 4000, 4100
    wl, ls = _chain_layers(n, R, 3, seed=78)
    r2s = torch.from_numpy(wl.req_to_slot).cuda()
    lens = torch.from_numpy(wl.seq_lens).cuda()
    new_slot = torch.from_numpy(wl.req_to_slot[0, n - 1:n].copy()).cuda()
    plan = ops.DecodePlan(wl.Hq, wl.Hkv, 1, 1, 1, n, 0, "cuda")
    outs = []
    for L, gp, op in ls:
        ops.store_quant(gp, bits_to_cuda_bf16(L.k[n - 1:n]), bits_to_cuda_bf16(L.v[n - 1:n]), new_slot)
        outs.append(ops.decode_attn(gp, bits_to_cuda_bf16(L.q), r2s, lens, None, max_seq_len=n, plan=plan,
                                    stable_history=stable))
    torch.cuda.synchronize()
    for l, (L, gp, op) in enumerate(ls):
        _check(outs[l], _ref(wl, op, L), f"store then decode layer {l} stable={stable}")
    assert ops.device_errors() == 0
