"""The no-allocation decode entry point, called through the C ABI.

paged_attn_fp8_decode_noalloc serves callers that cannot allocate device
memory -- an engine that gave all free HBM to its KV-cache pool, or a decode
loop that must not call cudaMalloc because it can synchronize the device.  It
keeps the split partials in the library's fixed 16 MiB device buffer instead
of a caller workspace.  It runs the same kernels with the same split plan as
the regular entry point, so its output must be bit-identical to the regular
call's (which is stricter than the 2e-2 abs + 2e-2 rel tolerance of the other
tests), on calls in a row: a large call, a smaller one, then one of the large
call's shape on new inputs -- the case where leftovers of an earlier call in
the shared buffer would show.  One case is also checked against the oracle.

This file is named so that pytest collects it last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads
from helpers import to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(fk, seed, lens, Hq, Hkv, E, window):
    spec = workloads.DecodeSpec("noalloc", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, block_size=16,
                                ctx_lo=1, ctx_hi=1, rel_extent=E)
    inp = workloads.make_decode(spec, device="cpu", seed=seed, lens=lens)
    kv = to_device(inp["kv"], DEV)
    cache = fk.KVCache.empty(kv.num_blocks, 16, Hkv, 128, device=DEV, fill=0x7F)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
    q = inp["q"].to(DEV)
    rel = None if inp["rel"] is None else inp["rel"].to(DEV)
    return cache, q, kv, rel


def _noalloc_via_c_abi(fk, cache, q, kv, rel, window, scales):
    lib = fk._lib
    fn = lib.paged_attn_fp8_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(fk.CacheStruct), ctypes.c_void_p, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                   ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p]
    B, Hq, D = q.shape
    out = torch.full_like(q, float("nan"))
    sq, sk, sv = scales
    st = fn(cache.c(), q.data_ptr(), Hq, kv.block_table.data_ptr(), kv.block_table.shape[1],
            kv.seq_lens.data_ptr(), B, sq, sk, sv, 1.0 / math.sqrt(D),
            rel.data_ptr() if rel is not None else None,
            rel.stride(0) if rel is not None else 0, rel.shape[2] if rel is not None else 0,
            window, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, fk.status_string(st)
    return out


def test_noalloc_matches_workspace_decode_on_calls_in_a_row():
    import fp8_e4m3_kv_gb300 as fk
    cases = [
        dict(seed=21, lens=[1, 300, 4000, 9000], Hq=32, Hkv=4, E=1024, window=0),
        dict(seed=22, lens=[700, 15, 2500], Hq=8, Hkv=2, E=128, window=512),
        # the first call's shape again, on new inputs
        dict(seed=23, lens=[1, 300, 4000, 9000], Hq=32, Hkv=4, E=1024, window=0),
    ]
    for c in cases:
        cache, q, kv, rel = _case(fk, c["seed"], c["lens"], c["Hq"], c["Hkv"], c["E"], c["window"])
        scales = (1.0, 1.0, 1.0)
        ref = fk.paged_attn_fp8_decode(cache, q, kv.block_table, kv.seq_lens, *scales,
                                       rel_bias=rel, window=c["window"])
        got = _noalloc_via_c_abi(fk, cache, q, kv, rel, c["window"], scales)
        torch.cuda.synchronize()
        assert fk.device_error() == 0
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got, ref), c


def test_noalloc_matches_the_oracle():
    import fp8_e4m3_kv_gb300 as fk
    from helpers import assert_close, oracle_decode_rows
    lens, Hq, Hkv, E = [5, 777, 3000], 8, 2, 128
    spec = workloads.DecodeSpec("noalloc", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, block_size=16,
                                ctx_lo=1, ctx_hi=1, rel_extent=E)
    inp = workloads.make_decode(spec, device="cpu", seed=24, lens=lens)
    cache, q, kv, rel = _case(fk, 24, lens, Hq, Hkv, E, 0)
    scales = (0.5, 0.5, 1.5)
    cache = fk.KVCache.empty(kv.num_blocks, 16, Hkv, 128, device=DEV, fill=0x7F)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, scales[1], scales[2])
    got = _noalloc_via_c_abi(fk, cache, q, kv, rel, 0, scales)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    rows = [(b, h) for b in range(len(lens)) for h in range(Hq)]
    ref = oracle_decode_rows(inp, rows, *scales, rel=inp["rel"])
    g = got.float().cpu().numpy()
    assert_close(np.stack([g[b, h] for b, h in rows]), ref, "noalloc vs oracle")


def test_noalloc_rejects_sizes_beyond_its_buffer():
    import fp8_e4m3_kv_gb300 as fk
    # 64 sequences x 64 query heads x up to 1M keys needs far more than 16 MiB
    n = fk.decode_workspace_size(64, 64, 4, 256, 65536, 16, 0, 0)
    assert n > 16 << 20
    cache = fk.KVCache.empty(4, 16, 4, 256, device=DEV)
    q = torch.zeros(64, 64, 256, dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros(64, 65536, dtype=torch.int32, device=DEV)
    lens = torch.ones(64, dtype=torch.int32, device=DEV)
    with pytest.raises(fk.Fp8KVError) as e:
        fk.paged_attn_fp8_decode_noalloc(cache, q, bt, lens, 1.0, 1.0, 1.0)
    assert e.value.status == fk.ERR_WORKSPACE
