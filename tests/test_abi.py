"""The C-ABI library loads and exports what include/fp8kv.h declares, and its
host-side checks reject bad arguments before any CUDA call (no GPU needed)."""
import ctypes
import math
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8kv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "fp8kv_build", os.path.join(ROOT, "fp8_e4m3_kv_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import fp8_e4m3_kv_gb300 as fk
    return fk


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kv_store_e4m3", "paged_attn_fp8_decode", "attn_fp8_varlen_prefill",
              "kv_amax_calibrate", "fp8kv_scale_from_amax", "fp8kv_decode_workspace_size",
              "fp8kv_status_string", "fp8kv_device_error", "fp8kv_cache_bytes",
              "paged_attn_fp8_decode_ex", "kv_band_counts", "fp8kv_set_prefill_max_ctas"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in declared_functions():
        assert n in exported, n
    for n in lib.EXPORTED:
        assert n in exported, n


def test_prefill_cta_cap_is_host_only(lib):
    with pytest.raises(lib.Fp8KVError) as e:
        lib.set_prefill_max_ctas(-1)
    assert e.value.status == 1
    lib.set_prefill_max_ctas(5)
    lib.set_prefill_max_ctas(0)


def test_status_strings(lib):
    assert lib.status_string(0) == "ok"
    assert "scale" in lib.status_string(2)
    assert lib.status_string(99) == "unknown status"


def test_scale_rules_match_oracle(lib, oracle_lib):
    for a in [1272.0, 114.6, 23.1, 11.6, 55.8, 0.37, 1e-3]:
        for rule in (0, 1, 2):
            assert lib.scale_from_amax(a, rule) == oracle_lib.scale_from_amax(a, rule)
    assert lib.scale_from_amax(0.0, 2) == 1.0
    for bad in (0.0, float("nan"), float("inf"), -1.0):
        with pytest.raises(lib.Fp8KVError) as e:
            lib.scale_from_amax(bad, 0)
        assert e.value.status == lib.ERR_SCALE
    with pytest.raises(lib.Fp8KVError) as e:
        lib.scale_from_amax(1.0, 7)
    assert e.value.status == lib.ERR_ARG


def test_cache_bytes(lib):
    # 4 KV heads x 128 dims: 512 bytes per token per K (1,024 with V)
    assert lib.cache_bytes(1, 1, 4, 128) * 2 == 1024
    assert lib.cache_bytes(65536, 16, 4, 128) == 1 << 29
    assert lib.cache_bytes(-1, 16, 4, 128) == 0


def _c(lib):
    return lib._lib


def test_store_rejects_bad_arguments_on_host(lib):
    L = _c(lib)
    cache = lib.CacheStruct(16, 16, 4, 16, 1, 128)  # fake, never dereferenced
    f = L.kv_store_e4m3
    assert f(None, 16, 16, 128, 128, 16, 1, 1.0, 1.0, None) == lib.ERR_ARG
    assert f(ctypes.byref(cache), 16, 16, 128, 128, 16, -1, 1.0, 1.0, None) == lib.ERR_ARG
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert f(ctypes.byref(cache), 16, 16, 128, 128, 16, 1, bad, 1.0, None) == lib.ERR_SCALE
        assert f(ctypes.byref(cache), 16, 16, 128, 128, 16, 1, 1.0, bad, None) == lib.ERR_SCALE
    assert f(ctypes.byref(cache), 16, 16, 128, 128, 16, 0, 1.0, 1.0, None) == lib.OK  # no-op
    assert f(ctypes.byref(cache), None, 16, 128, 128, 16, 1, 1.0, 1.0, None) == lib.ERR_ARG
    assert f(ctypes.byref(cache), 16, 16, 100, 128, 16, 1, 1.0, 1.0, None) == lib.ERR_ARG
    assert f(ctypes.byref(cache), 8, 16, 128, 128, 16, 1, 1.0, 1.0, None) == lib.ERR_ARG
    odd = lib.CacheStruct(16, 16, 4, 16, 1, 100)       # row not a multiple of 16
    assert f(ctypes.byref(odd), 16, 16, 128, 128, 16, 1, 1.0, 1.0, None) == lib.ERR_UNSUPPORTED


def _decode(lib, cache, **kw):
    a = dict(q=16, Hq=8, bt=16, mb=4, lens=16, B=1, qs=1.0, ks=1.0, vs=1.0, sm=0.1, rel=None,
             bstride=0, E=0, window=0, out=16, ws=16, wsb=1 << 20, split=0)
    a.update(kw)
    return _c(lib).paged_attn_fp8_decode_ex(
        ctypes.byref(cache) if cache is not None else None, a["q"], a["Hq"], a["bt"], a["mb"],
        a["lens"], a["B"], a["qs"], a["ks"], a["vs"], a["sm"], a["rel"], a["bstride"], a["E"],
        a["window"], a["out"], a["ws"], a["wsb"], a["split"], None)


def test_decode_rejects_bad_arguments_on_host(lib):
    cache = lib.CacheStruct(16, 16, 4, 16, 2, 128)
    assert _decode(lib, None) == lib.ERR_ARG
    for k in ("qs", "ks", "vs", "sm"):
        assert _decode(lib, cache, **{k: float("nan")}) == lib.ERR_SCALE
        assert _decode(lib, cache, **{k: 0.0}) == lib.ERR_SCALE
    assert _decode(lib, cache, Hq=7) == lib.ERR_ARG                  # not a multiple of Hkv
    assert _decode(lib, cache, Hq=34) == lib.ERR_UNSUPPORTED         # 17 heads per KV head
    assert _decode(lib, lib.CacheStruct(16, 16, 4, 16, 2, 64)) == lib.ERR_UNSUPPORTED
    assert _decode(lib, lib.CacheStruct(16, 16, 4, 24, 2, 128)) == lib.ERR_UNSUPPORTED
    assert _decode(lib, cache, rel=16, E=0) == lib.ERR_ARG
    assert _decode(lib, cache, split=100) == lib.ERR_ARG
    assert _decode(lib, cache, split=64) == lib.ERR_ARG              # not a whole key tile
    assert _decode(lib, cache, window=-1) == lib.ERR_ARG
    assert _decode(lib, cache, B=0) == lib.OK                        # nothing to do
    assert _decode(lib, cache, q=None) == lib.ERR_ARG
    assert _decode(lib, cache, q=8) == lib.ERR_ARG                   # q not 16-byte aligned


def test_workspace_size_is_host_only_with_explicit_splits(lib):
    def per_slot(B, Hq, D):
        return B * Hq * (D + 2) * 4          # fp32 partial o plus (m, l) per query head
    sched = 256                              # the persistent launch's work-item counter
    # 2 seqs x 8 q heads, max 4 blocks of 16 = 64 keys -> one split of 256 keys
    n1 = lib.decode_workspace_size(2, 8, 2, 128, 4, 16, 0, 256) - sched
    assert n1 % per_slot(2, 8, 128) == 0
    slots_per_split = n1 // per_slot(2, 8, 128)
    assert 1 <= slots_per_split <= 4
    # 1024 keys in splits of 256 keys: 4 splits
    n2 = lib.decode_workspace_size(1, 4, 1, 256, 64, 16, 0, 256) - sched
    assert n2 % per_slot(1, 4, 256) == 0 and (n2 // per_slot(1, 4, 256)) % 4 == 0
    assert lib.decode_workspace_size(1, 4, 1, 64, 4, 16, 0, 128) == 0


def test_band_counts_rejects_bad_arguments_on_host(lib):
    f = _c(lib).kv_band_counts
    # (x, stride, slots, tokens, row, scale, counts, stream); the pointers are
    # fakes, and every case below is rejected (or is empty) before any CUDA call
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert f(16, 128, None, 4, 128, bad, 16, None) == lib.ERR_SCALE
    assert f(16, 128, None, -1, 128, 1.0, 16, None) == lib.ERR_ARG
    assert f(16, 128, None, 4, 0, 1.0, 16, None) == lib.ERR_ARG
    assert f(16, 128, None, 4, 100, 1.0, 16, None) == lib.ERR_UNSUPPORTED   # row % 16
    assert f(16, 128, None, 0, 128, 1.0, None, None) == lib.OK               # nothing to do
    assert f(None, 128, None, 4, 128, 1.0, 16, None) == lib.ERR_ARG
    assert f(16, 64, None, 4, 128, 1.0, 16, None) == lib.ERR_ARG             # stride < row
    assert f(8, 128, None, 4, 128, 1.0, 16, None) == lib.ERR_ARG             # x not 16-byte aligned
    assert f(16, 128, None, 4, 128, 1.0, 12, None) == lib.ERR_ARG            # counts not 8-byte aligned
    assert f(16, 128, None, 4, 128, 1.0, None, None) == lib.ERR_ARG


def _prefill(lib, cache, **kw):
    a = dict(q=16, Hq=8, cu=16, lk=16, bt=16, mb=4, B=1, maxq=16, qs=1.0, ks=1.0, vs=1.0, sm=0.1,
             rel=None, bstride=0, E=0, window=0, out=16, ws=None, wsb=0)
    a.update(kw)
    return _c(lib).attn_fp8_varlen_prefill(
        ctypes.byref(cache) if cache is not None else None, a["q"], a["Hq"], a["cu"], a["lk"],
        a["bt"], a["mb"], a["B"], a["maxq"], a["qs"], a["ks"], a["vs"], a["sm"], a["rel"],
        a["bstride"], a["E"], a["window"], a["out"], a["ws"], a["wsb"], None)


def test_prefill_rejects_bad_arguments_on_host(lib):
    cache = lib.CacheStruct(16, 16, 4, 16, 2, 128)   # fake pointers, never dereferenced
    assert _prefill(lib, None) == lib.ERR_ARG
    for k in ("qs", "ks", "vs", "sm"):
        for bad in (float("nan"), 0.0, -1.0, float("inf")):
            assert _prefill(lib, cache, **{k: bad}) == lib.ERR_SCALE
    assert _prefill(lib, cache, B=-1) == lib.ERR_ARG
    assert _prefill(lib, cache, Hq=0) == lib.ERR_ARG
    assert _prefill(lib, cache, Hq=7) == lib.ERR_ARG                 # not a multiple of Hkv
    assert _prefill(lib, cache, mb=0) == lib.ERR_ARG
    assert _prefill(lib, cache, window=-1) == lib.ERR_ARG
    assert _prefill(lib, cache, maxq=-1) == lib.ERR_ARG
    assert _prefill(lib, lib.CacheStruct(16, 16, 4, 16, 2, 64)) == lib.ERR_UNSUPPORTED   # D 64
    assert _prefill(lib, lib.CacheStruct(16, 16, 4, 8, 2, 128)) == lib.ERR_UNSUPPORTED   # bs 8
    assert _prefill(lib, cache, rel=16, E=0) == lib.ERR_ARG
    assert _prefill(lib, cache, rel=16, E=128, bstride=-1) == lib.ERR_ARG
    assert _prefill(lib, cache, B=0) == lib.OK                       # nothing to do
    assert _prefill(lib, cache, maxq=0) == lib.OK
    assert _prefill(lib, cache, q=None) == lib.ERR_ARG
    assert _prefill(lib, cache, cu=None) == lib.ERR_ARG
    assert _prefill(lib, cache, q=8) == lib.ERR_ARG                  # q not 16-byte aligned
    assert _prefill(lib, cache, out=8) == lib.ERR_ARG


def _decode_store(lib, cache, **kw):
    a = dict(q=16, Hq=8, kn=16, vn=16, bt=16, mb=4, lens=16, B=1, qs=1.0, ks=1.0, vs=1.0, sm=0.1,
             rel=None, bstride=0, E=0, window=0, ak=None, av=None, out=16, ws=16, wsb=1 << 20)
    a.update(kw)
    return _c(lib).paged_attn_fp8_decode_store(
        ctypes.byref(cache), a["q"], a["Hq"], a["kn"], a["vn"], a["bt"], a["mb"], a["lens"],
        a["B"], a["qs"], a["ks"], a["vs"], a["sm"], a["rel"], a["bstride"], a["E"], a["window"],
        a["ak"], a["av"], a["out"], a["ws"], a["wsb"], None)


def test_decode_store_rejects_bad_arguments_on_host(lib):
    cache = lib.CacheStruct(16, 16, 4, 16, 2, 128)
    assert _decode_store(lib, cache, kn=None) == lib.ERR_ARG
    assert _decode_store(lib, cache, vn=None) == lib.ERR_ARG
    assert _decode_store(lib, cache, kn=8) == lib.ERR_ARG            # not 16-byte aligned
    assert _decode_store(lib, cache, ak=2) == lib.ERR_ARG            # amax not 4-byte aligned
    assert _decode_store(lib, cache, ks=float("nan")) == lib.ERR_SCALE
    assert _decode_store(lib, cache, B=0, kn=None, vn=None) == lib.OK


def test_per_token_calls_reject_bad_arguments_on_host(lib):
    L = _c(lib)
    cache = lib.CacheStruct(16, 16, 4, 16, 2, 128)                   # row = Hkv * D = 256
    st = L.kv_store_e4m3_per_token   # (cache, k, v, k_stride, v_stride, slots, T, k_sc, v_sc, s)
    assert st(None, 16, 16, 256, 256, 16, 1, 16, 16, None) == lib.ERR_ARG
    assert st(ctypes.byref(cache), 16, 16, 256, 256, 16, -1, 16, 16, None) == lib.ERR_ARG
    d64 = lib.CacheStruct(16, 16, 4, 16, 2, 64)
    assert st(ctypes.byref(d64), 16, 16, 128, 128, 16, 1, 16, 16, None) == lib.ERR_UNSUPPORTED
    assert st(ctypes.byref(cache), 16, 16, 256, 256, 16, 0, 16, 16, None) == lib.OK
    assert st(ctypes.byref(cache), 16, 16, 256, 256, 16, 1, None, 16, None) == lib.ERR_ARG
    assert st(ctypes.byref(cache), 16, 16, 256, 256, None, 1, 16, 16, None) == lib.ERR_ARG
    assert st(ctypes.byref(cache), 16, 16, 256, 256, 16, 1, 18, 16, None) == lib.ERR_ARG  # align 4
    assert st(ctypes.byref(cache), 16, 16, 128, 256, 16, 1, 16, 16, None) == lib.ERR_ARG  # stride
    assert st(ctypes.byref(cache), 8, 16, 256, 256, 16, 1, 16, 16, None) == lib.ERR_ARG   # align 16
    dec = L.paged_attn_fp8_decode_per_token
    # (cache, q, Hq, bt, mb, lens, B, q_scale, softmax_scale, k_sc, v_sc, rel, bstride, E,
    #  window, out, ws, ws_bytes, stream)
    args = [ctypes.byref(cache), 16, 8, 16, 4, 16, 1, 1.0, 0.1, 16, 16, None, 0, 0, 0, 16, 16,
            1 << 20, None]
    for i, bad in ((9, None), (10, None), (9, 18), (7, float("nan")), (8, 0.0)):
        a = list(args)
        a[i] = bad
        assert dec(*a) == (lib.ERR_SCALE if i in (7, 8) else lib.ERR_ARG), (i, bad)
    a = list(args)
    a[6], a[9], a[10] = 0, None, None
    assert dec(*a) == lib.OK                                           # nothing to do


def test_amax_rejects_bad_arguments_on_host(lib):
    f = _c(lib).kv_amax_calibrate   # (k, v, k_stride, v_stride, slots, T, Hkv, D, amax_k, amax_v, s)
    assert f(16, 16, 256, 256, None, -1, 2, 128, 16, 16, None) == lib.ERR_ARG
    assert f(16, 16, 256, 256, None, 1, 0, 128, 16, 16, None) == lib.ERR_ARG
    assert f(16, 16, 256, 256, None, 1, 2, 100, 16, 16, None) == lib.ERR_UNSUPPORTED  # row % 16
    assert f(16, None, 256, 256, None, 1, 2, 128, None, None, None) == lib.ERR_ARG    # no amax_k
    assert f(16, None, 128, 256, None, 1, 2, 128, 16, None, None) == lib.ERR_ARG      # stride < row
    assert f(8, None, 256, 256, None, 1, 2, 128, 16, None, None) == lib.ERR_ARG       # align 16
    assert f(None, None, 256, 256, None, 1, 2, 128, None, None, None) == lib.OK       # nothing to do
    assert f(16, 16, 256, 256, None, 0, 2, 128, 16, 16, None) == lib.OK


def test_decode_bindings_check_table_and_lengths(lib):
    """Every decode binding checks block_table and seq_lens (dtype, device,
    shape, contiguity) before the call: the kernels read them through raw
    device pointers.  The cache here is a host tensor, so a "device" mismatch
    is a meta tensor; nothing reaches CUDA."""
    import torch
    cache = lib.KVCache.empty(4, 16, 1, 128, device="cpu")
    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16)
    bt = torch.zeros(2, 3, dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    calls = {
        "decode": lambda t, n: lib.paged_attn_fp8_decode(cache, q, t, n, 1.0, 1.0, 1.0),
        "noalloc": lambda t, n: lib.paged_attn_fp8_decode_noalloc(cache, q, t, n, 1.0, 1.0, 1.0),
        "store": lambda t, n: lib.paged_attn_fp8_decode_store(
            cache, q, torch.zeros(2, 1, 128, dtype=torch.bfloat16),
            torch.zeros(2, 1, 128, dtype=torch.bfloat16), t, n, 1.0, 1.0, 1.0),
        "per_token": lambda t, n: lib.paged_attn_fp8_decode_per_token(
            cache, q, t, n, 1.0, torch.ones(4, 1, 16), torch.ones(4, 1, 16)),
        "bound_step": lambda t, n: lib.DecodeStep(cache, q, t, n, 1.0, 1.0, 1.0),
    }
    bad = [
        (bt.to(torch.int64), lens, TypeError),                  # int64 table
        (bt, lens.to(torch.int64), TypeError),                  # int64 lengths
        (torch.zeros(1, 3, dtype=torch.int32), lens, ValueError),   # fewer rows than B
        (torch.zeros(2, dtype=torch.int32), lens, ValueError),      # not 2-D
        (torch.zeros(3, 2, dtype=torch.int32).t(), lens, ValueError),   # not contiguous
        (bt, torch.ones(3, dtype=torch.int32), ValueError),     # lengths of another batch
        (torch.zeros(2, 3, dtype=torch.int32, device="meta"), lens, ValueError),  # other device
        (bt, torch.ones(2, dtype=torch.int32, device="meta"), ValueError),
    ]
    for name, call in calls.items():
        for t, n, exc in bad:
            with pytest.raises(exc):
                call(t, n)


def test_per_token_prefill_rejects_bad_arguments_on_host(lib):
    f = _c(lib).attn_fp8_varlen_prefill_per_token
    cache = lib.CacheStruct(16, 16, 4, 16, 2, 128)   # fake pointers, never dereferenced
    # (cache, q, Hq, cu, lens_k, bt, mb, B, maxq, q_scale, softmax_scale, k_sc, v_sc, rel,
    #  bstride, E, window, out, stream)
    args = [ctypes.byref(cache), 16, 8, 16, 16, 16, 4, 1, 16, 1.0, 0.1, 16, 16, None, 0, 0, 0, 16,
            None]
    for i, bad, want in ((11, None, lib.ERR_ARG), (12, None, lib.ERR_ARG), (11, 18, lib.ERR_ARG),
                         (9, float("nan"), lib.ERR_SCALE), (10, 0.0, lib.ERR_SCALE)):
        a = list(args)
        a[i] = bad
        assert f(*a) == want, (i, bad)
    a = list(args)
    a[7], a[11], a[12] = 0, None, None
    assert f(*a) == lib.OK                                             # nothing to do
    d256 = lib.CacheStruct(16, 16, 4, 16, 2, 256)
    a = list(args)
    a[0] = ctypes.byref(d256)
    assert f(*a) == lib.ERR_UNSUPPORTED
