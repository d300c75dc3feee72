"""GPU parity: 256-d heads (the Qwen3.6 full-attention case of FreeToken PR #897, "Known regression and
uncertainty") -- quantize-on-write of 256-d rows, bit-exact against the oracle, and single-row split-K decode
over a 256-d FP8 pool against the FP64 oracle under the strict bound: ragged key counts and split caps, GQA
groups, the fused store, sliding windows, the stable-history chain and the 32,768-key workload.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_ftkv_gb300 import inputs, ops
from parity import bits_to_cuda_bf16, check_attention

pytestmark = pytest.mark.gpu
D = 256
SM = 1.0 / 16.0


def _setup(wl, layer=0, skip=None):
    L = wl.layer(layer)
    gp = ops.KVPool.empty(wl.num_rows, wl.Hkv, head_dim=D)
    keep = np.ones(L.slots.shape[0], bool) if skip is None else ~skip
    if keep.any():
        ops.store_quant(gp, bits_to_cuda_bf16(L.k[keep]), bits_to_cuda_bf16(L.v[keep]),
                        torch.from_numpy(L.slots[keep]).cuda())
    op = oracle.Pool(wl.num_rows, wl.Hkv, D)
    if L.slots.size:
        oracle.store_quant(op, L.k, L.v, L.slots)
    return gp, op, L


def _wl(lens, num_rows, seed, Hq=32, Hkv=4, sigma=1.0):
    return inputs.decode_custom(lens, [1] * len(lens), num_rows, sigma=sigma, seed=seed, Hq=Hq, Hkv=Hkv,
                                head_dim=D)


def _run(wl, gp, L, splits=0, stable=False, window=0, **kw):
    return ops.decode_attn(gp, bits_to_cuda_bf16(L.q), torch.from_numpy(wl.req_to_slot).cuda(),
                           torch.from_numpy(wl.seq_lens).cuda(), None, max_seq_len=int(wl.req_to_slot.shape[1]),
                           sm_scale=SM, num_splits=splits, stable_history=stable, window=window, **kw)


def _ref(wl, op, L, window=0):
    args = (op, L.q, wl.req_to_slot, wl.seq_lens, wl.q_row_offsets, SM, wl.Hq)
    return oracle.decode_attn(*args, window=window), oracle.decode_attn(*args, abs_v=True, window=window)


def test_store_256d_bit_exact():
    rng = np.random.default_rng(256)
    T, R = 3000, 5000
    k, v = inputs.kv_tokens(rng, T, 2.0, big_frac=0.05, zero_frac=0.05, Hkv=4, head_dim=D)
    slots = rng.permutation(R)[:T].astype(np.int32)
    gp = ops.KVPool.empty(R, 4, head_dim=D)
    ops.store_quant(gp, bits_to_cuda_bf16(k), bits_to_cuda_bf16(v), torch.from_numpy(slots).cuda())
    op = oracle.Pool(R, 4, D)
    oracle.store_quant(op, k, v, slots)
    assert np.array_equal(gp.k_codes.cpu().numpy(), op.k_codes)
    assert np.array_equal(gp.v_codes.cpu().numpy(), op.v_codes)
    assert np.array_equal(gp.k_scales.cpu().numpy().view(np.uint32), op.k_scales.view(np.uint32))
    assert np.array_equal(gp.v_scales.cpu().numpy().view(np.uint32), op.v_scales.view(np.uint32))
    assert ops.device_errors() == 0


@pytest.mark.parametrize("stable", [False, True])
@pytest.mark.parametrize("n", [1, 17, 513, 4099])
@pytest.mark.parametrize("splits", [0, 1, 8, 64])
def test_decode_256d_ragged_lengths_and_split_caps(n, splits, stable):
    wl = _wl([n], max(2 * n, 64), seed=n + 256)
    gp, op, L = _setup(wl)
    out = _run(wl, gp, L, splits=splits, stable=stable)
    ref, mag = _ref(wl, op, L)
    check_attention(out, ref, f"D256 n={n} splits={splits} stable={stable}", mag)
    assert ops.device_errors() == 0


@pytest.mark.parametrize("Hq,Hkv", [(32, 4), (16, 2), (8, 1), (64, 8), (12, 6), (4, 4)])
def test_decode_256d_gqa_groups(Hq, Hkv):
    wl = _wl([300, 1000], 4000, seed=Hq + 257, Hq=Hq, Hkv=Hkv)
    gp, op, L = _setup(wl)
    out = _run(wl, gp, L)
    ref, mag = _ref(wl, op, L)
    check_attention(out, ref, f"D256 Hq={Hq} Hkv={Hkv}", mag)


def _new_tokens(wl, L):
    starts = np.concatenate([[0], np.cumsum(wl.seq_lens)[:-1]]).astype(np.int64)
    k_new = np.zeros((len(wl.seq_lens), wl.Hkv, D), np.uint16)
    v_new = np.zeros_like(k_new)
    new = np.zeros(L.slots.shape[0], bool)
    for b, n in enumerate(wl.seq_lens):
        if n > 0:
            k_new[b] = L.k[starts[b] + n - 1]
            v_new[b] = L.v[starts[b] + n - 1]
            new[starts[b] + n - 1] = True
    return k_new, v_new, new


@pytest.mark.parametrize("stable", [False, True])
@pytest.mark.parametrize("lens,splits,window", [([512], 0, 0), ([4099], 8, 0), ([4099], 0, 77), ([33, 0, 1], 0, 0)])
def test_decode_256d_fused_store(lens, splits, window, stable):
    wl = _wl(lens, max(2 * sum(lens), 64), seed=sum(lens) + 258, sigma=2.0)
    L = wl.layer(0)
    k_new, v_new, new = _new_tokens(wl, L)
    gp, op, L = _setup(wl, skip=new)
    out = _run(wl, gp, L, splits=splits, stable=stable, window=window, k_new=bits_to_cuda_bf16(k_new),
               v_new=bits_to_cuda_bf16(v_new))
    s = L.slots
    assert np.array_equal(gp.k_codes.cpu().numpy()[s], op.k_codes[s])
    assert np.array_equal(gp.v_codes.cpu().numpy()[s], op.v_codes[s])
    assert np.array_equal(gp.k_scales.cpu().numpy()[s].view(np.uint32), op.k_scales[s].view(np.uint32))
    assert np.array_equal(gp.v_scales.cpu().numpy()[s].view(np.uint32), op.v_scales[s].view(np.uint32))
    ref, mag = _ref(wl, op, L, window)
    check_attention(out, ref, f"D256 fused lens={lens} W={window} stable={stable}", mag)
    assert ops.device_errors() == 0


@pytest.mark.parametrize("window,splits", [(1, 0), (513, 8), (5000, 0)])
def test_decode_256d_sliding_window(window, splits):
    wl = _wl([4099, 300], 4500, seed=window + 259)
    gp, op, L = _setup(wl)
    out = _run(wl, gp, L, splits=splits, window=window)
    ref, mag = _ref(wl, op, L, window)
    check_attention(out, ref, f"D256 window={window}", mag)


@pytest.mark.parametrize("graph", [False, True])
def test_decode_256d_stable_history_chain(graph):
    """16 fused-store decode launches in one stream with the stable-history flag; layers 0, 7, 15 checked."""
    wl = _wl([3000], 3100, seed=260)
    layers = 16
    Ls = [wl.layer(l) for l in range(layers)]
    news = [_new_tokens(wl, L) for L in Ls]
    pools = []
    for l in range(layers):
        gp, op, _ = _setup(wl, l, skip=news[l][2])
        pools.append((gp, op))
    q = [bits_to_cuda_bf16(L.q) for L in Ls]
    kn = [bits_to_cuda_bf16(nw[0]) for nw in news]
    vn = [bits_to_cuda_bf16(nw[1]) for nw in news]
    r2s = torch.from_numpy(wl.req_to_slot).cuda()
    lens = torch.from_numpy(wl.seq_lens).cuda()
    n = int(wl.req_to_slot.shape[1])
    plan = ops.DecodePlan(wl.Hq, wl.Hkv, 1, 1, 1, n, head_dim=D)
    outs = [torch.empty_like(q[0]) for _ in range(layers)]

    def step():
        for l in range(layers):
            ops.decode_attn(pools[l][0], q[l], r2s, lens, None, max_seq_len=n, plan=plan, out=outs[l],
                            k_new=kn[l], v_new=vn[l], stable_history=True, sm_scale=SM)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
    else:
        step()
    torch.cuda.synchronize()
    for l in (0, 7, 15):
        ref, mag = _ref(wl, pools[l][1], Ls[l])
        check_attention(outs[l], ref, f"D256 chain layer {l} graph={graph}", mag)
    assert ops.device_errors() == 0


def test_decode_256d_long_context_full_size():
    wl = inputs.decode_long(32768, 33059, layers=2)
    wl.head_dim = D
    wl.sm_scale = SM
    gp, op, L = _setup(wl, 1)
    for stable in (False, True):
        out = _run(wl, gp, L, stable=stable)
        ref, mag = _ref(wl, op, L)
        stats = check_attention(out, ref, f"D256 32K stable={stable}", mag)
        assert stats["rel_l2"] < 2e-3
    assert ops.device_errors() == 0
