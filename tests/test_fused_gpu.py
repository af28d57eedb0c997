"""The fused decode step (store of each sequence's new token + amax + decode in
one call) against the separate calls: the cache bytes and the output must be
identical, the amax equal to kv_amax_calibrate's; one case also against the
float64 oracle within 2e-2 abs + 2e-2 rel."""
import numpy as np
import pytest
import torch

import workloads
from helpers import assert_close, oracle_decode_rows, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fk():
    import fp8_e4m3_kv_gb300 as m
    return m


def run_both(fk, lens, Hq, Hkv, D, bs, scales=(1.0, 1.0, 1.0), window=0, E=0, v_dist="normal",
             seed=0):
    spec = workloads.DecodeSpec("case", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                                ctx_lo=1, ctx_hi=1, v_dist=v_dist, rel_extent=E)
    inp = workloads.make_decode(spec, device="cpu", seed=seed, lens=lens)
    kv = inp["kv"]
    kd = to_device(kv, DEV)
    sq, sk, sv = scales
    starts = kv.tok_start.tolist()
    # the step's new token of each sequence is its last one
    last = [starts[b] + L - 1 for b, L in enumerate(lens) if L > 0]
    has = torch.tensor([L > 0 for L in lens])
    k_new = torch.zeros(len(lens), Hkv, D, dtype=torch.bfloat16)
    v_new = torch.zeros(len(lens), Hkv, D, dtype=torch.bfloat16)
    k_new[has] = kv.k[last]
    v_new[has] = kv.v[last]
    k_new, v_new = k_new.to(DEV), v_new.to(DEV)
    before = kd.slot_mapping.clone()
    before[last] = -1
    # the cache before the step: every token but the new ones (stale NaN codes elsewhere)
    a = fk.KVCache.empty(kv.num_blocks, bs, Hkv, D, device=DEV, fill=0x7F)
    fk.kv_store_e4m3(a, kd.k, kd.v, before, sk, sv)
    b = fk.KVCache(a.k.clone(), a.v.clone())
    rel = None if inp["rel"] is None else inp["rel"].to(DEV)
    q = inp["q"].to(DEV)
    # separate calls: amax, store of the new tokens, decode
    am_a = torch.zeros(2, dtype=torch.float32, device=DEV)
    fk.kv_amax_calibrate(k_new, v_new, am_a[0:1], am_a[1:2])
    slot_new = torch.full((len(lens),), -1, dtype=torch.int64, device=DEV)
    slot_new[has.to(DEV)] = kd.slot_mapping[last]
    fk.kv_store_e4m3(a, k_new, v_new, slot_new, sk, sv)
    out_a = fk.paged_attn_fp8_decode(a, q, kd.block_table, kd.seq_lens, sq, sk, sv, rel_bias=rel,
                                     window=window)
    # the fused call
    am_b = torch.zeros(2, dtype=torch.float32, device=DEV)
    out_b = fk.paged_attn_fp8_decode_store(b, q, k_new, v_new, kd.block_table, kd.seq_lens, sq,
                                           sk, sv, rel_bias=rel, window=window,
                                           amax_k=am_b[0:1], amax_v=am_b[1:2])
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    assert torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    assert torch.equal(out_a, out_b)
    assert torch.equal(am_a, am_b)
    return inp, out_b


@pytest.mark.parametrize("bs", [16, 64])
def test_fused_step_equals_separate_calls(fk, bs):
    run_both(fk, [1, 15, 16, 17, 300, 1000, 4097], 32, 4, 128, bs, E=1024, v_dist="v_t3",
             scales=(1.0, 1.0, 3.0))


def test_fused_step_window_and_empty_sequence(fk):
    run_both(fk, [0, 5, 511, 512, 513, 2000], 8, 1, 128, 16, window=512, E=128, seed=3)


def test_fused_step_head_dim_256_nonpow2_scales(fk):
    run_both(fk, [100, 700, 1500], 24, 4, 256, 16, scales=(0.3, 0.05, 0.25), seed=4)


def test_fused_step_against_oracle(fk):
    lens = [3, 130, 900, 2600]
    inp, out = run_both(fk, lens, 16, 2, 128, 16, E=128, seed=5)
    rows = [(b, h) for b in range(len(lens)) for h in range(16)]
    ref = oracle_decode_rows(inp, rows, 1.0, 1.0, 1.0, window=0, rel=inp["rel"])
    got = out.float().cpu().numpy()
    assert_close(np.stack([got[b, h] for b, h in rows]), ref, "fused decode")


@pytest.mark.parametrize("D", [128, 256])
def test_fused_step_through_the_work_counter(fk, D):
    """More splits than the persistent grid has CTAs (the CTAs take them from
    the counter), with an empty and a one-key sequence among them."""
    lens = [40000, 30000, 0, 20000, 9000, 1] if D == 128 else [30000, 20000, 5000, 0]
    run_both(fk, lens, 32 if D == 128 else 24, 4, D, 16, scales=(1.0, 1.0, 3.0), E=1024, seed=7)
