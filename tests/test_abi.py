"""C-ABI checks that need no GPU: the library loads, exports every function include/ftkv.h declares, and
rejects bad arguments on the host (nothing is enqueued, no device memory is touched).

Fake device pointers below are never dereferenced: every call returns during host validation.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from fp8_kv_cache_ftkv_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ftkv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ftkv_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ftkv_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    assert lib.ftkv_abi_version() == 2
    for code, name in [(0, "FTKV_OK"), (-1, "FTKV_ERR_INVALID"), (-2, "FTKV_ERR_UNSUPPORTED"), (-3, "FTKV_ERR_ALIGN"),
                       (-4, "FTKV_ERR_WORKSPACE"), (-6, "FTKV_ERR_CUDA"), (-99, "FTKV_ERR_UNKNOWN")]:
        assert _lib.status_str(code) == name


def test_pool_bytes_matches_printed_accounting(lib):
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    assert lib.ftkv_pool_bytes(33059, 48, 4, 128, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == 0
    assert (a.value, b.value, c.value) == (3_249_831_936, 1_675_694_592, 67_704_832)
    assert lib.ftkv_pool_bytes(-1, 48, 4, 128, None, None, None) == _lib.FTKV_ERR_INVALID


def _pool(k=0x10000, v=0x20000, ks=0x30000, vs=0x40000, rows=100, hkv=4, d=128):
    return _lib.FtkvPool(k, v, ks, vs, rows, hkv, d)


def test_store_validation(lib):
    P = ctypes.byref
    assert lib.ftkv_store_quant(None, None, None, None, 1, None) == _lib.FTKV_ERR_INVALID
    assert lib.ftkv_store_quant(P(_pool(d=64)), 0x1000, 0x2000, 0x3000, 1, None) == _lib.FTKV_ERR_UNSUPPORTED
    assert lib.ftkv_store_quant(P(_pool(k=0x10001)), 0x1000, 0x2000, 0x3000, 1, None) == _lib.FTKV_ERR_ALIGN
    assert lib.ftkv_store_quant(P(_pool()), 0x1008, 0x2000, 0x3000, 1, None) == _lib.FTKV_ERR_ALIGN
    assert lib.ftkv_store_quant(P(_pool()), 0x1000, 0x2000, 0x3000, -1, None) == _lib.FTKV_ERR_INVALID
    assert lib.ftkv_store_quant(P(_pool()), None, 0x2000, 0x3000, 1, None) == _lib.FTKV_ERR_INVALID
    assert lib.ftkv_store_quant(P(_pool()), None, None, None, 0, None) == _lib.FTKV_OK  # empty: no-op
    assert lib.ftkv_store_quant(P(_pool(rows=0)), 0x1000, 0x2000, 0x3000, 1, None) == _lib.FTKV_ERR_INVALID


def test_reconstruct_validation(lib):
    P = ctypes.byref
    assert lib.ftkv_reconstruct_bf16(P(_pool(d=256)), 0x3000, 5, 0x5000, 0x6000, None) == _lib.FTKV_ERR_UNSUPPORTED
    assert lib.ftkv_reconstruct_bf16(P(_pool()), 0x3000, 5, 0x5008, 0x6000, None) == _lib.FTKV_ERR_ALIGN
    assert lib.ftkv_reconstruct_bf16(P(_pool()), None, 5, 0x5000, 0x6000, None) == _lib.FTKV_ERR_INVALID
    assert lib.ftkv_reconstruct_bf16(P(_pool()), None, 0, None, None, None) == _lib.FTKV_OK


def test_decode_validation(lib):
    P = ctypes.byref
    ws = lib.ftkv_decode_workspace_bytes(32, 4, 128, 1, 1, 4)
    assert ws > 0 and ws % 256 == 0
    assert lib.ftkv_decode_workspace_bytes(32, 4, 64, 1, 1, 8) == 0
    ws256 = lib.ftkv_decode_workspace_bytes(32, 4, 256, 1, 1, 4)
    assert ws256 > ws and ws256 % 256 == 0                    # 256-d partials: twice the accumulators
    base = dict(q=0x1000, r2s=0x2000, stride=64, lens=0x3000, offs=None, B=1, total=1, mq=1, maxlen=64,
                sm=0.0884, win=0, splits=4, flags=0, ws=0x100000, wsb=ws, out=0x4000)

    def call(pool=None, hq=32, **kw):
        a = dict(base, **kw)
        return lib.ftkv_decode_attn(P(pool or _pool()), hq, a["q"], a["r2s"], a["stride"], a["lens"], a["offs"],
                                    a["B"], a["total"], a["mq"], a["maxlen"], a["sm"], a["win"], a["splits"],
                                    a["flags"], a["ws"], a["wsb"], a["out"], None)

    assert call(hq=24) == _lib.FTKV_ERR_UNSUPPORTED          # group 6
    assert call(hq=30) == _lib.FTKV_ERR_UNSUPPORTED          # not a multiple of Hkv
    assert call(hq=64, pool=_pool(hkv=4)) == _lib.FTKV_ERR_UNSUPPORTED  # group 16
    assert call(mq=9) == _lib.FTKV_ERR_UNSUPPORTED
    assert call(B=65536, total=65536) == _lib.FTKV_ERR_UNSUPPORTED  # above FTKV_MAX_BATCH
    assert call(splits=_lib.FTKV_MAX_SPLITS + 1) == _lib.FTKV_ERR_INVALID
    assert call(flags=2) == _lib.FTKV_ERR_INVALID             # unknown flag bits
    assert call(flags=_lib.FTKV_DECODE_STABLE_HISTORY, q=0x1002) == _lib.FTKV_ERR_ALIGN
    assert call(r2s=0x2002) == _lib.FTKV_ERR_ALIGN             # int32 tables are 4-byte aligned
    assert call(maxlen=65) == _lib.FTKV_ERR_INVALID          # above req_stride
    assert call(total=2) == _lib.FTKV_ERR_INVALID            # no offsets: one row per request
    assert call(q=0x1002) == _lib.FTKV_ERR_ALIGN
    assert call(ws=0x100010) == _lib.FTKV_ERR_ALIGN          # workspace must be 256-B aligned
    assert call(wsb=ws - 1) == _lib.FTKV_ERR_WORKSPACE
    assert call(sm=float("nan")) == _lib.FTKV_ERR_INVALID
    assert call(win=-1) == _lib.FTKV_ERR_INVALID             # sliding window: 0 (off) or >= 1 keys
    assert call(pool=_pool(d=256), mq=2) == _lib.FTKV_ERR_UNSUPPORTED  # 256-d heads: single-row decode only
    assert call(pool=_pool(d=256)) == _lib.FTKV_ERR_WORKSPACE  # 256-d: the 128-d workspace is too small
    assert call(pool=_pool(d=192)) == _lib.FTKV_ERR_UNSUPPORTED
    assert call(win=8, wsb=255) == _lib.FTKV_ERR_WORKSPACE    # the workspace rule holds with a window too
    assert call(B=0, total=0) == _lib.FTKV_OK                # nothing to do

    def call_store(kn=0x7000, vn=0x8000, **kw):
        a = dict(base, **kw)
        return lib.ftkv_decode_attn_store(P(_pool()), 32, a["q"], kn, vn, a["r2s"], a["stride"], a["lens"],
                                          a["offs"], a["B"], a["total"], a["mq"], a["maxlen"], a["sm"], a["win"],
                                          a["splits"], a["flags"], a["ws"], a["wsb"], a["out"], None)

    assert call_store(kn=None) == _lib.FTKV_ERR_INVALID       # the fused store needs the new rows
    assert call_store(vn=None) == _lib.FTKV_ERR_INVALID
    assert call_store(kn=0x7008) == _lib.FTKV_ERR_ALIGN
    assert call_store(vn=0x8004) == _lib.FTKV_ERR_ALIGN
    assert call_store(mq=9) == _lib.FTKV_ERR_UNSUPPORTED       # the decode checks still apply
    assert call_store(win=-2) == _lib.FTKV_ERR_INVALID
    assert call_store(kn=None, vn=None, B=0, total=0) == _lib.FTKV_OK

    def call_noalloc(**kw):
        a = dict(base, **kw)
        return lib.ftkv_decode_attn_noalloc(P(_pool()), 32, a["q"], a["r2s"], a["stride"], a["lens"], a["offs"],
                                            a["B"], a["total"], a["mq"], a["maxlen"], a["sm"], a["splits"], a["out"],
                                            None)

    # every decode check runs before the allocation-free entry point touches its scratch array
    assert call_noalloc(q=0x1002) == _lib.FTKV_ERR_ALIGN
    assert call_noalloc(out=None) == _lib.FTKV_ERR_INVALID
    assert call_noalloc(mq=9) == _lib.FTKV_ERR_UNSUPPORTED
    assert call_noalloc(maxlen=65) == _lib.FTKV_ERR_INVALID
    assert call_noalloc(B=4096, total=4096, offs=0x5000, mq=1, splits=64) == _lib.FTKV_ERR_WORKSPACE
    assert call_noalloc(B=0, total=0) == _lib.FTKV_OK


def test_decode_auto_splits_host_logic(lib):
    """The automatic split count (host only; without a GPU the SM count defaults to 152).  Single-row CTAs
    cover 4 KV heads (two CTAs fit per SM); multi-row CTAs one KV head (one CTA per SM)."""
    if torch.cuda.is_available():
        pytest.skip("the expected values assume the 152-SM default")
    f = lib.ftkv_decode_auto_splits
    assert f(1, 4, 32768, 1) == 152           # one group: one CTA per SM
    assert f(1, 8, 32768, 1) == 76            # 8 KV heads: two groups of 4
    assert f(1, 4, 1000, 1) == 125            # at least ~8 keys per slice (single-row kernel)
    assert f(1, 4, 1000, 2) == 8              # at least ~128 keys per slice (multi-row kernel)
    assert f(4, 4, 32768, 1) == 38            # up to 4 groups: one CTA per SM, 152 // 4
    assert f(8, 4, 32768, 1) == 38            # more: one wave of two CTAs per SM, 304 // 8
    assert f(16, 4, 16384, 1) == 19
    assert f(32, 4, 16384, 1) == 9
    assert f(64, 4, 40000, 1) == 9            # many groups: 2 whole waves for >= ~8 slices, 608 // 64
    assert f(256, 4, 40000, 1) == 8           # 7 waves, 2128 // 256
    assert f(64, 4, 40000, 8) == 5            # multi-row: ~8 waves of one CTA per SM, ceil(8 * 152 / 256)
    assert f(1, 1, 10 ** 9, 1) == 152
    assert f(0, 4, 100, 1) == 1


def test_prefill_validation(lib):
    for fn in (lib.ftkv_prefill_attn,):
        assert fn(32, 4, 64, 0x1000, 0x2000, 0x3000, 16, 0x4000, 0x5000, 16, 0.08, 0x6000, None) == \
            _lib.FTKV_ERR_UNSUPPORTED
        assert fn(32, 5, 128, 0x1000, 0x2000, 0x3000, 16, 0x4000, 0x5000, 16, 0.08, 0x6000, None) == \
            _lib.FTKV_ERR_UNSUPPORTED
        assert fn(32, 4, 128, 0x1000, 0x2000, 0x3000, 16, None, None, 16, 0.08, 0x6000, None) == \
            _lib.FTKV_ERR_INVALID
        assert fn(32, 4, 128, 0x1004, 0x2000, 0x3000, 16, 0x4000, 0x5000, 16, 0.08, 0x6000, None) == \
            _lib.FTKV_ERR_ALIGN
        assert fn(32, 4, 128, None, None, None, 0, None, None, 0, 0.08, None, None) == _lib.FTKV_OK


def test_prefill_stream_k_validation(lib):
    def call(ws=0x7000, nbytes=1 << 30, **kw):
        a = dict(hq=32, hkv=4, d=128, q=0x1000, k=0x2000, v=0x3000, C=16, wk=0x4000, wv=0x5000, P=16, ctas=4)
        a.update(kw)
        return lib.ftkv_prefill_attn_ws(a["hq"], a["hkv"], a["d"], a["q"], a["k"], a["v"], a["C"], a["wk"], a["wv"],
                                        a["P"], 0.08, a["ctas"], ws, nbytes, 0x6000, None)
    assert call(ws=None) == _lib.FTKV_ERR_INVALID          # the workspace is required
    assert call(nbytes=-1) == _lib.FTKV_ERR_INVALID
    assert call(d=64) == _lib.FTKV_ERR_UNSUPPORTED         # the prefill checks still apply
    assert call(q=0x1004) == _lib.FTKV_ERR_ALIGN
    # workspace size: tickets [ctas + 1][4] rounded up to 256 B, then two FP32 pieces per boundary
    piece = (2 * 128 * 128 + 4 * 128) * 4
    for ctas in (1, 5, 152):
        n = ctas + 1
        assert lib.ftkv_prefill_workspace_bytes(ctas) == (n * 16 + 255) // 256 * 256 + n * 2 * piece


def test_codec_validation(lib):
    assert lib.ftkv_e4m3_encode_f32(None, None, 0, None) == _lib.FTKV_OK
    assert lib.ftkv_e4m3_encode_f32(None, 0x1000, 4, None) == _lib.FTKV_ERR_INVALID
    assert lib.ftkv_e4m3_decode_f32(0x1000, 0x2002, 4, None) == _lib.FTKV_ERR_ALIGN


def _bpool(k=0x10000, v=0x20000, rows=100, hkv=4, d=128):
    return _lib.FtkvBf16Pool(k, v, rows, hkv, d)


def test_bf16_pool_validation(lib):
    """The BF16-pool entry points check their pool, then every decode check of ftkv_decode_attn."""
    P = ctypes.byref
    ws = lib.ftkv_decode_workspace_bytes(32, 4, 128, 1, 1, 4)
    base = dict(q=0x1000, kn=None, vn=None, r2s=0x2000, stride=64, lens=0x3000, offs=None, B=1, total=1, mq=1,
                maxlen=64, sm=0.0884, win=0, splits=4, flags=0, ws=0x100000, wsb=ws, out=0x4000)

    def call(pool=None, hq=32, **kw):
        a = dict(base, **kw)
        return lib.ftkv_decode_attn_bf16(P(pool or _bpool()), hq, a["q"], a["kn"], a["vn"], a["r2s"], a["stride"],
                                         a["lens"], a["offs"], a["B"], a["total"], a["mq"], a["maxlen"], a["sm"],
                                         a["win"], a["splits"], a["flags"], a["ws"], a["wsb"], a["out"], None)

    assert call(pool=_bpool(k=0)) == _lib.FTKV_ERR_INVALID          # null pool array
    assert call(pool=_bpool(rows=0)) == _lib.FTKV_ERR_INVALID
    assert call(pool=_bpool(d=256)) == _lib.FTKV_ERR_UNSUPPORTED
    assert call(pool=_bpool(v=0x20008)) == _lib.FTKV_ERR_ALIGN
    assert call(hq=24) == _lib.FTKV_ERR_UNSUPPORTED                  # group 6
    assert call(mq=9) == _lib.FTKV_ERR_UNSUPPORTED
    assert call(win=-1) == _lib.FTKV_ERR_INVALID
    assert call(q=0x1002) == _lib.FTKV_ERR_ALIGN
    assert call(wsb=255) == _lib.FTKV_ERR_WORKSPACE
    assert call(kn=0x7000) == _lib.FTKV_ERR_INVALID                 # k_new without v_new
    assert call(kn=0x7000, vn=0x8008) == _lib.FTKV_ERR_ALIGN
    assert call(B=70000, total=70000, wsb=1 << 40) == _lib.FTKV_ERR_UNSUPPORTED  # one grid row per query row
    assert call(B=0, total=0) == _lib.FTKV_OK

    g = lib.ftkv_gather_bf16
    assert g(P(_bpool()), 0x3000, -1, 0x5000, 0x6000, None) == _lib.FTKV_ERR_INVALID
    assert g(P(_bpool()), None, 5, 0x5000, 0x6000, None) == _lib.FTKV_ERR_INVALID
    assert g(P(_bpool()), 0x3002, 5, 0x5000, 0x6000, None) == _lib.FTKV_ERR_ALIGN
    assert g(P(_bpool()), 0x3000, 5, 0x5008, 0x6000, None) == _lib.FTKV_ERR_ALIGN
    assert g(P(_bpool(d=64)), 0x3000, 5, 0x5000, 0x6000, None) == _lib.FTKV_ERR_UNSUPPORTED
    assert g(P(_bpool()), None, 0, None, None, None) == _lib.FTKV_OK
