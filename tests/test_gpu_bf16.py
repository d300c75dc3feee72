"""GPU parity: the BF16-pool comparison point (decode over a BF16 KV pool, prefix gather, prefill over it).

Decode over a BF16 pool is compared element by element with the FP64 oracle's attention over the same BF16
rows (oracle.decode_attn_bf16) under the strict bound |o - ref| <= 1e-2 + 1e-2 |ref| plus rel-L2 <= 1e-2:
the 512-token step, ragged key counts and split caps (1/8/64/152/256), GQA groups, multi-row requests, rows
that see no key, sliding windows, the fused copy of the new tokens into the pool (bit-exact), the stable-
history chain, and the 32,768-key batch-1 workload at full size.  The gather is bit-exact against plain
indexing; the chunked prefill over the BF16 pool runs the gather -> prefill -> copy pipeline on both sides
(prefill bound as in test_gpu_prefill.py).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_ftkv_gb300 import inputs, ops
from parity import bits_to_cuda_bf16, check_attention, cuda_bf16_to_bits

pytestmark = pytest.mark.gpu
STABLE = [False, True]


def _pool(wl, L, skip=None):
    """BF16 pool of one layer on both sides: host bit array [rows, Hkv, D] and the device pool.  Tokens
    flagged in ``skip`` are left out of the device pool (the fused copy writes them)."""
    host_k = np.zeros((wl.num_rows, wl.Hkv, wl.head_dim), np.uint16)
    host_v = np.zeros_like(host_k)
    host_k[L.slots] = L.k
    host_v[L.slots] = L.v
    gp = ops.BF16Pool.empty(wl.num_rows, wl.Hkv)
    keep = np.ones(L.slots.shape[0], bool) if skip is None else ~skip
    if keep.any():
        s = torch.from_numpy(L.slots[keep].astype(np.int64)).cuda()
        gp.k[s] = bits_to_cuda_bf16(L.k[keep])
        gp.v[s] = bits_to_cuda_bf16(L.v[keep])
    return host_k, host_v, gp


def _dev(wl, L):
    return dict(q=bits_to_cuda_bf16(L.q), r2s=torch.from_numpy(wl.req_to_slot).cuda(),
                lens=torch.from_numpy(wl.seq_lens).cuda(), offs=torch.from_numpy(wl.q_row_offsets).cuda())


def _run(wl, gp, dev, num_splits=0, stable=False, window=0, offsets=True, **kw):
    R = np.diff(wl.q_row_offsets)
    return ops.decode_attn_bf16(gp, dev["q"], dev["r2s"], dev["lens"], dev["offs"] if offsets else None,
                                max_seq_len=int(wl.req_to_slot.shape[1]), max_q_rows=int(max(R.max(), 1)),
                                sm_scale=wl.sm_scale, num_splits=num_splits, stable_history=stable,
                                window=window, **kw)


def _ref(wl, hk, hv, L, window=0):
    args = (hk, hv, L.q, wl.req_to_slot, wl.seq_lens, wl.q_row_offsets, wl.sm_scale, wl.Hq)
    return oracle.decode_attn_bf16(*args, window=window), oracle.decode_attn_bf16(*args, abs_v=True, window=window)


def _check(out, refs, what):
    return check_attention(out, refs[0], what, refs[1])


@pytest.mark.parametrize("stable", STABLE)
def test_bf16_decode_small_step(stable):
    wl = inputs.decode_small()
    L = wl.layer(0)
    hk, hv, gp = _pool(wl, L)
    out = _run(wl, gp, _dev(wl, L), stable=stable, offsets=False)
    stats = _check(out, _ref(wl, hk, hv, L), f"bf16 decode_small stable={stable}")
    assert stats["max_abs"] < 0.05  # BF16 rounding of outputs up to |13|
    assert ops.device_errors() == 0


@pytest.mark.parametrize("n", [1, 17, 513, 4099])
@pytest.mark.parametrize("splits", [0, 1, 8, 64, 152, 256])
def test_bf16_decode_ragged_lengths_and_split_caps(n, splits):
    wl = inputs.decode_custom([n], [1], max(2 * n, 64), seed=n + 7)
    L = wl.layer(0)
    hk, hv, gp = _pool(wl, L)
    out = _run(wl, gp, _dev(wl, L), num_splits=splits)
    _check(out, _ref(wl, hk, hv, L), f"bf16 n={n} splits={splits}")


@pytest.mark.parametrize("Hq,Hkv", [(32, 4), (16, 4), (8, 4), (4, 4), (64, 8), (16, 2), (8, 1), (12, 6)])
def test_bf16_decode_gqa_groups(Hq, Hkv):
    wl = inputs.decode_custom([300, 1000], [1, 1], 4000, seed=Hq + 1, Hq=Hq, Hkv=Hkv)
    L = wl.layer(0)
    hk, hv, gp = _pool(wl, L)
    out = _run(wl, gp, _dev(wl, L))
    _check(out, _ref(wl, hk, hv, L), f"bf16 Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("rows", [[2], [3, 1, 8], [8, 8], [5, 7, 6, 4]])
def test_bf16_decode_multirow(rows):
    lens = [200 + 97 * i for i in range(len(rows))]
    wl = inputs.decode_custom(lens, rows, 5000, sigma=2.0, big_frac=0.01, zero_frac=0.01, seed=len(rows) + 20)
    L = wl.layer(0)
    hk, hv, gp = _pool(wl, L)
    dev = _dev(wl, L)
    for splits in (0, 1, 5):
        out = _run(wl, gp, dev, num_splits=splits)
        _check(out, _ref(wl, hk, hv, L), f"bf16 rows={rows} splits={splits}")


def test_bf16_decode_rows_that_see_no_key_are_zero():
    wl = inputs.decode_custom([2, 40, 0], [5, 3, 1], 100, seed=3)
    L = wl.layer(0)
    hk, hv, gp = _pool(wl, L)
    out = _run(wl, gp, _dev(wl, L))
    refs = _ref(wl, hk, hv, L)
    assert (refs[0][:3] == 0).all() and (refs[0][8] == 0).all()
    _check(out, refs, "bf16 empty rows")
    assert (out[:3].float() == 0).all() and (out[8].float() == 0).all()


@pytest.mark.parametrize("lens,rows,window,splits", [
    ([4099], [1], 513, 0), ([4099], [1], 1, 8), ([300], [1], 5000, 0), ([200, 297, 394], [3, 1, 8], 9, 0),
    ([900, 2000], [4, 2], 131, 5),
])
def test_bf16_decode_sliding_window(lens, rows, window, splits):
    wl = inputs.decode_custom(lens, rows, sum(lens) + 9, seed=window + 5)
    L = wl.layer(0)
    hk, hv, gp = _pool(wl, L)
    out = _run(wl, gp, _dev(wl, L), num_splits=splits, window=window)
    _check(out, _ref(wl, hk, hv, L, window), f"bf16 window={window} lens={lens} rows={rows}")


def _new_tokens(wl, L):
    """K/V rows of each request's new tokens (its last R_b positions, one per query row) and their mask."""
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
            k_new[wl.q_row_offsets[b] + r] = L.k[starts[b] + pos]
            v_new[wl.q_row_offsets[b] + r] = L.v[starts[b] + pos]
            new[starts[b] + pos] = True
    return k_new, v_new, new


@pytest.mark.parametrize("stable", STABLE)
@pytest.mark.parametrize("lens,rows,splits,window", [
    ([512], [1], 0, 0), ([4099], [1], 8, 0), ([32768], [1], 0, 0), ([4099], [1], 0, 77),
    ([200, 297, 394], [3, 1, 8], 0, 0), ([2, 40], [5, 3], 0, 0), ([0, 33, 1], [1, 1, 1], 0, 0),
])
def test_bf16_decode_fused_copy(lens, rows, splits, window, stable):
    """The new tokens' rows land in the pool bit for bit, and the attention over them matches the oracle."""
    wl = inputs.decode_custom(lens, rows, max(2 * sum(lens), 64), sigma=2.0, big_frac=0.01, seed=sum(lens) + 3)
    L = wl.layer(0)
    k_new, v_new, new = _new_tokens(wl, L)
    hk, hv, gp = _pool(wl, L, skip=new)
    single = max(rows) == 1
    out = _run(wl, gp, _dev(wl, L), num_splits=splits, stable=stable, window=window, offsets=not single,
               k_new=bits_to_cuda_bf16(k_new), v_new=bits_to_cuda_bf16(v_new))
    s = L.slots
    assert np.array_equal(cuda_bf16_to_bits(gp.k)[s], hk[s])
    assert np.array_equal(cuda_bf16_to_bits(gp.v)[s], hv[s])
    _check(out, _ref(wl, hk, hv, L, window), f"bf16 fused lens={lens} rows={rows} W={window} stable={stable}")
    assert ops.device_errors() == 0


def test_bf16_decode_bad_slot_is_flagged_not_faulted():
    wl = inputs.decode_custom([300], [1], 600, seed=8)
    L = wl.layer(0)
    hk, hv, gp = _pool(wl, L)
    dev = _dev(wl, L)
    dev["r2s"] = dev["r2s"].clone()
    dev["r2s"][0, 5] = 10 ** 7
    _run(wl, gp, dev)
    torch.cuda.synchronize()
    assert ops.device_errors() & 0x1
    assert ops.device_errors() == 0


@pytest.mark.parametrize("graph", [False, True])
def test_bf16_decode_stable_history_chain_of_layers(graph):
    """48 decode launches in one stream with the stable-history flag, each with its own pool, new tokens and
    output; layers 0, 23 and 47 against the oracle."""
    wl = inputs.decode_custom([3000], [1], 3100, seed=31)
    layers = 48
    Ls = [wl.layer(l) for l in range(layers)]
    news = [_new_tokens(wl, L) for L in Ls]
    pools = [_pool(wl, L, skip=nw[2]) for L, nw in zip(Ls, news)]
    q = [bits_to_cuda_bf16(L.q) for L in Ls]
    kn = [bits_to_cuda_bf16(nw[0]) for nw in news]
    vn = [bits_to_cuda_bf16(nw[1]) for nw in news]
    r2s = torch.from_numpy(wl.req_to_slot).cuda()
    lens = torch.from_numpy(wl.seq_lens).cuda()
    n = int(wl.req_to_slot.shape[1])
    plan = ops.DecodePlan(wl.Hq, wl.Hkv, 1, 1, 1, n)
    outs = [torch.empty_like(q[0]) for _ in range(layers)]

    def step():
        for l in range(layers):
            ops.decode_attn_bf16(pools[l][2], q[l], r2s, lens, None, max_seq_len=n, plan=plan, out=outs[l],
                                 k_new=kn[l], v_new=vn[l], stable_history=True)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()  # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
    else:
        step()
    torch.cuda.synchronize()
    for l in (0, 23, 47):
        hk, hv, _ = pools[l]
        _check(outs[l], _ref(wl, hk, hv, Ls[l]), f"bf16 chain layer {l} graph={graph}")
    assert ops.device_errors() == 0


def test_bf16_decode_long_context_full_size():
    wl = inputs.decode_long(32768, 33059, layers=48)
    for layer in (0, 47):
        L = wl.layer(layer)
        hk, hv, gp = _pool(wl, L)
        for stable in STABLE:
            out = _run(wl, gp, _dev(wl, L), stable=stable, offsets=False)
            stats = _check(out, _ref(wl, hk, hv, L), f"bf16 32K layer={layer} stable={stable}")
            assert stats["rel_l2"] < 2e-3
    assert ops.device_errors() == 0


# ---- prefix gather and prefill over the BF16 pool ----

@pytest.mark.parametrize("P", [1, 5, 8192, 14336])
def test_bf16_gather_bit_exact(P):
    rng = np.random.default_rng(P)
    rows, hkv = 33059, 8
    k, v = inputs.kv_tokens(rng, rows, 1.0, Hkv=hkv)
    gp = ops.BF16Pool(bits_to_cuda_bf16(k), bits_to_cuda_bf16(v))
    slots = rng.permutation(rows)[:P].astype(np.int32)
    wk, wv = ops.gather_bf16(gp, torch.from_numpy(slots).cuda())
    assert np.array_equal(cuda_bf16_to_bits(wk), k[slots])
    assert np.array_equal(cuda_bf16_to_bits(wv), v[slots])
    assert ops.device_errors() == 0


def test_bf16_gather_bad_slot_writes_zeros_and_flags():
    rng = np.random.default_rng(9)
    k, v = inputs.kv_tokens(rng, 100, 1.0)
    gp = ops.BF16Pool(bits_to_cuda_bf16(k), bits_to_cuda_bf16(v))
    slots = np.array([3, 200, -1, 7], np.int32)
    wk = bits_to_cuda_bf16(np.full((4, 4, 128), 0x3F80, np.uint16))
    wv = wk.clone()
    ops.gather_bf16(gp, torch.from_numpy(slots).cuda(), wk, wv)
    torch.cuda.synchronize()
    assert ops.device_errors() & 0x1
    got = cuda_bf16_to_bits(wk)
    assert np.array_equal(got[0], k[3]) and np.array_equal(got[3], k[7])
    assert (got[1] == 0).all() and (got[2] == 0).all()
    assert ops.device_errors() == 0


def test_bf16_chunked_prefill_full_workload():
    """8,192 historical rows, 8,192 new tokens in 4 chunks of 2,048: gather -> prefill -> copy of the chunk
    into the pool, on both sides; every 16th query row of each chunk."""
    wl = inputs.prefill()
    R = wl.num_rows
    host_k = np.zeros((R, 4, 128), np.uint16)
    host_v = np.zeros_like(host_k)
    host_k[wl.hist_slots] = wl.hist_k
    host_v[wl.hist_slots] = wl.hist_v
    gp = ops.BF16Pool(bits_to_cuda_bf16(host_k), bits_to_cuda_bf16(host_v))
    slots_all = np.concatenate([wl.hist_slots, wl.new_slots])
    q_d, k_d, v_d = bits_to_cuda_bf16(wl.q), bits_to_cuda_bf16(wl.k), bits_to_cuda_bf16(wl.v)
    slots_d = torch.from_numpy(slots_all).cuda()
    plan = ops.PrefillPlan(0)
    H = wl.hist_slots.shape[0]
    for c in range(wl.num_chunks):
        c0, c1 = c * wl.chunk, min((c + 1) * wl.chunk, wl.q.shape[0])
        P = H + c0
        wk, wv = ops.gather_bf16(gp, slots_d[:P])
        out = ops.prefill_attn(q_d[c0:c1], k_d[c0:c1], v_d[c0:c1], wk, wv, plan=plan)
        dst = slots_d[P:P + c1 - c0].long()
        gp.k[dst] = k_d[c0:c1]
        gp.v[dst] = v_d[c0:c1]
        owk, owv = host_k[slots_all[:P]], host_v[slots_all[:P]]
        rows = np.arange(0, c1 - c0, 16, dtype=np.int64)
        ref = oracle.prefill_attn(wl.q[c0:c1], wl.k[c0:c1], wl.v[c0:c1], owk, owv, wl.sm_scale, rows)
        mag = oracle.prefill_attn(wl.q[c0:c1], wl.k[c0:c1], wl.v[c0:c1], owk, owv, wl.sm_scale, rows, abs_v=True)
        host_k[slots_all[P:P + c1 - c0]] = wl.k[c0:c1]
        host_v[slots_all[P:P + c1 - c0]] = wl.v[c0:c1]
        check_attention(out[torch.from_numpy(rows).cuda()], ref, f"bf16 prefill chunk {c}", mag, bound="terms")
    assert ops.device_errors() == 0
