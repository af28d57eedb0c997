"""Paged fp8 decode attention on the GPU against the float64 oracle, element
by element, within 2e-2 abs + 2e-2 rel."""
import math

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


def run_case(fk, lens, Hq, Hkv, D, bs, scales=(1.0, 1.0, 1.0), window=0, E=0, bias_bcast=False,
             v_dist="normal", seed=0, split_tokens=0, fill=0x7F, rows=None, plant=False,
             out_nan=False):
    spec = workloads.DecodeSpec("case", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                                ctx_lo=1, ctx_hi=1, v_dist=v_dist, rel_extent=E, plant_v=plant)
    inp = workloads.make_decode(spec, device="cpu", seed=seed, lens=lens)
    if E and bias_bcast:   # one learned table per head, broadcast over sequences
        inp["rel"] = inp["rel"][:1].expand(len(lens), Hq, E)
    kv = inp["kv"]
    kd = to_device(kv, DEV)
    sq, sk, sv = scales
    # stale NaN codes everywhere the store does not write
    cache = fk.KVCache.empty(kv.num_blocks, bs, Hkv, D, device=DEV, fill=fill)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, sk, sv)
    rel_d = None if inp["rel"] is None else inp["rel"].to(DEV)
    # out_nan: the output starts as NaN, so a row the kernels skip shows up
    out0 = (torch.full((len(lens), Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
            if out_nan else None)
    out = fk.paged_attn_fp8_decode(cache, inp["q"].to(DEV), kd.block_table, kd.seq_lens, sq, sk,
                                   sv, rel_bias=rel_d, window=window, split_tokens=split_tokens,
                                   out=out0)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = out.float().cpu().numpy()
    if rows is None:
        rows = [(b, h) for b in range(len(lens)) for h in range(Hq)]
    rel_h = None if inp["rel"] is None else inp["rel"]
    ref = oracle_decode_rows(inp, rows, sq, sk, sv, window=window, rel=rel_h)
    g = np.stack([got[b, h] for b, h in rows])
    return assert_close(g, ref, "decode"), got


def test_tiny_workload(fk):
    """1 sequence, 4 q heads / 1 KV head, head_dim 128, context 256, block 16."""
    run_case(fk, [256], 4, 1, 128, 16)


@pytest.mark.parametrize("scales", [(1.0, 1.0, 1.0), (0.5, 0.5, 1.5)])
def test_ragged_lengths_gqa8_bias(fk, scales):
    run_case(fk, [1, 2, 15, 16, 17, 127, 128, 129, 255, 300, 1000], 32, 4, 128, 16,
             scales=scales, E=1024)


def test_bias_extent_128_broadcast(fk):
    run_case(fk, [500, 64, 129], 16, 2, 128, 16, E=128, bias_bcast=True, seed=1)


@pytest.mark.parametrize("window", [1, 3, 100, 512])
def test_sliding_window(fk, window):
    run_case(fk, [1, 50, 511, 512, 513, 700, 1500], 8, 1, 128, 16, window=window, E=128, seed=2)


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_block_sizes(fk, bs):
    run_case(fk, [3, 200, 333, 1024], 8, 2, 128, bs, seed=3)


def test_head_dim_256_gqa6(fk):
    run_case(fk, [1, 100, 257, 900], 24, 4, 256, 16, scales=(0.3, 0.05, 0.25), seed=4)


def test_head_dim_256_window(fk):
    run_case(fk, [700, 90], 12, 2, 256, 32, window=512, E=128, seed=5)


@pytest.mark.parametrize("G", [1, 3, 16])
def test_group_sizes(fk, G):
    run_case(fk, [77, 400], 2 * G, 2, 128, 16, seed=6 + G)


@pytest.mark.parametrize("v_scale", [1.0, 3.0])
def test_heavy_tailed_values(fk, v_scale):
    """V = 17.47 t(3) with a planted |V| = 1,272: clipped at v_scale 1, not at 3."""
    run_case(fk, [1024, 2000, 3000], 32, 4, 128, 16, scales=(1.0, 1.0, v_scale), E=1024,
             v_dist="v_t3", plant=True, seed=9)


@pytest.mark.parametrize("split", [256, 512, 1792])
def test_explicit_splits_agree(fk, split):
    lens = [1, 130, 1000, 2500]
    _, auto = run_case(fk, lens, 8, 1, 128, 16, seed=11)
    _, forced = run_case(fk, lens, 8, 1, 128, 16, seed=11, split_tokens=split)
    # Other split boundaries change each split's running max, hence the
    # two-term e4m3 rounding of P (relative error <= 2^-8 per weight) and the
    # fp32 summation order; per row the outputs agree within 2^-8 of the
    # row's largest value plus one bf16 rounding step.
    for b in range(len(lens)):
        for h in range(8):
            a, f = auto[b, h], forced[b, h]
            tol = 2.0 ** -8 * np.abs(a).max() + 2.0 ** -7 * np.abs(a)
            assert (np.abs(f - a) <= tol).all(), (b, h, float(np.abs(f - a).max()))


def test_sixteen_heads_per_kv_head_through_the_work_counter(fk):
    """16 query heads per KV head with more splits than CTAs (the counter
    path), sampled rows against the oracle."""
    rng = np.random.default_rng(3)
    lens = [int(x) for x in rng.integers(5000, 20000, 32)]
    rows = [(b, h) for b in (0, 7, 19, 31) for h in (0, 5, 16, 31)]
    run_case(fk, lens, 32, 2, 128, 16, E=128, seed=21, rows=rows)


@pytest.mark.parametrize("window", [0, 3000])
def test_empty_and_short_sequences_among_long_ones_through_the_work_counter(fk, window):
    """Empty, one-key and short sequences beside long ones, with more items
    than CTAs (the counter path): every row is written (the output starts as
    NaN), empty sequences give zeros, sampled rows match the oracle."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(8000, 20000, 40)]
    for b, n in ((0, 0), (3, 1), (9, 0), (17, 200), (25, 0), (39, 2049)):
        lens[b] = n
    rows = [(b, h) for b in (3, 5, 17, 30, 39) for h in (0, 13, 31)]
    err, got = run_case(fk, lens, 32, 4, 128, 16, E=128, window=window, seed=23, rows=rows,
                        split_tokens=2048, out_nan=True)
    assert not np.isnan(got).any()
    for b in (0, 9, 25):
        assert (got[b] == 0).all()


@pytest.mark.parametrize("D,Hq,Hkv,offset", [(256, 24, 4, 0), (256, 24, 4, 1), (128, 32, 4, 1)])
def test_merge_of_many_rows_and_an_out_not_8_byte_aligned(fk, D, Hq, Hkv, offset):
    """Enough (sequence, head) rows that the merge runs one warp per row (at
    head_dim 256 too), several splits per row, and out at an element offset
    of 0 or 1 (2-byte aligned only): sampled rows match the oracle and the
    padding element before out stays untouched."""
    rng = np.random.default_rng(7 + D + offset)
    B = 16
    lens = [int(x) for x in rng.integers(300, 6000, B)]
    lens[3] = 0
    spec = workloads.DecodeSpec("case", B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=16, ctx_lo=1,
                                ctx_hi=1, rel_extent=128)
    inp = workloads.make_decode(spec, device="cpu", seed=31, lens=lens)
    kd = to_device(inp["kv"], DEV)
    cache = fk.KVCache.empty(kd.num_blocks, 16, Hkv, D, device=DEV)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, 1.0, 1.0)
    flat = torch.full((B * Hq * D + 8,), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = flat[offset:offset + B * Hq * D].view(B, Hq, D)
    fk.paged_attn_fp8_decode(cache, inp["q"].to(DEV), kd.block_table, kd.seq_lens, 1.0, 1.0,
                             1.0, rel_bias=inp["rel"].to(DEV), out=out, split_tokens=1024)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = out.float().cpu().numpy()
    assert not np.isnan(got).any()
    assert (got[3] == 0).all()
    if offset:
        assert torch.isnan(flat[:offset].float()).all()
    rows = [(b, h) for b in (0, 5, 15) for h in (0, Hq // 2, Hq - 1)]
    ref = oracle_decode_rows(inp, rows, 1.0, 1.0, 1.0, rel=inp["rel"])
    assert_close(np.stack([got[b, h] for b, h in rows]), ref, "merge")


def test_empty_and_single_key(fk):
    """len 0 gives zeros; len 1 gives v_scale * v8 of the only key (exact)."""
    err, got = run_case(fk, [0, 1, 5], 4, 1, 128, 16, scales=(1.0, 1.0, 2.0), seed=12,
                        rows=[(1, 0), (1, 3), (2, 2)])
    assert (got[0] == 0).all()


def _full(fk, spec, rows_per_check, seed=0, scales=(1.0, 1.0, 1.0), calibrate=False,
          longest_all_heads=False):
    inp = workloads.make_decode(spec, device=DEV, seed=seed)
    kv = inp["kv"]
    sq, sk, sv = scales
    if calibrate:
        amax = torch.zeros(3, dtype=torch.float32, device=DEV)
        fk.kv_amax_calibrate(kv.k, kv.v, amax[0:1], amax[1:2], kv.slot_mapping)
        fk.kv_amax_calibrate(inp["q"], None, amax[2:3], None)
        ak, av, aq = amax.cpu().tolist()
        sk, sv, sq = fk.scale_from_amax(ak), fk.scale_from_amax(av), fk.scale_from_amax(aq)
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=DEV)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, sk, sv)
    out = fk.paged_attn_fp8_decode(cache, inp["q"], kv.block_table, kv.seq_lens, sq, sk, sv,
                                   rel_bias=inp["rel"], window=spec.window)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    lens = inp["lens"]
    G = spec.Hq // spec.Hkv
    rng = np.random.default_rng(seed)
    order = np.argsort(lens)
    bsel = sorted(set([int(order[0]), int(order[-1])] +
                      [int(x) for x in rng.choice(len(lens), rows_per_check[0], replace=False)]))
    rows = []
    for b in bsel:
        kvh = int(rng.integers(spec.Hkv))
        rows += [(b, kvh * G + g) for g in range(G)][: rows_per_check[1]]
    if longest_all_heads:   # every query head of the longest sequence
        b = int(order[-1])
        rows += [(b, h) for h in range(spec.Hq) if (b, h) not in rows]
    host = dict(inp)
    host["kv"] = kv
    ref = oracle_decode_rows(host, rows, sq, sk, sv, window=spec.window, rel=inp["rel"])
    return assert_close(np.stack([got[b, h] for b, h in rows]), ref, spec.name)


def test_full_decode_64seq_32k(fk):
    _full(fk, workloads.DECODE_32K, (4, 8))


def test_full_decode_64seq_32k_vscale3(fk):
    _full(fk, workloads.DECODE_32K, (2, 8), scales=(1.0, 1.0, 3.0))


def test_full_decode_64seq_32k_vscale3_longest_all_heads(fk):
    """v_scale 3.0 on the full workload: every head of its longest sequence."""
    _full(fk, workloads.DECODE_32K, (0, 0), scales=(1.0, 1.0, 3.0), longest_all_heads=True)


def test_full_decode_64seq_32k_window512(fk):
    """The full workload as a 512-token sliding-window layer."""
    import dataclasses
    _full(fk, dataclasses.replace(workloads.DECODE_32K, window=512), (4, 8))


def test_length_past_block_table_is_flagged(fk):
    """A length past the sequence's block-table row: the keys beyond the row
    read as zeros, FP8KV_DEVERR_BAD_BLOCK is set, and the call completes."""
    spec = workloads.DecodeSpec("case", B=2, Hq=8, Hkv=2, D=128, block_size=16, ctx_lo=1,
                                ctx_hi=1)
    inp = workloads.make_decode(spec, device="cpu", seed=30, lens=[40, 48])
    kv = to_device(inp["kv"], DEV)
    cache = fk.KVCache.empty(kv.num_blocks, 16, 2, 128, device=DEV)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
    assert kv.block_table.shape[1] == 3
    q = inp["q"].to(DEV)
    fk.paged_attn_fp8_decode(cache, q, kv.block_table, kv.seq_lens, 1.0, 1.0, 1.0)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    too_long = torch.tensor([40, 48 + 37], dtype=torch.int32, device=DEV)
    out = fk.paged_attn_fp8_decode(cache, q, kv.block_table, too_long, 1.0, 1.0, 1.0)
    torch.cuda.synchronize()
    assert fk.device_error() & fk.DEVERR_BAD_BLOCK
    assert fk.device_error() == 0          # read with clear: the word is clean again
    assert torch.isfinite(out.float()).all()


def test_full_decode_128k_calibrated_d256(fk):
    _full(fk, workloads.DECODE_128K_CAL, (1, 6), calibrate=True)


def test_full_decode_1m(fk):
    _full(fk, workloads.DECODE_1M, (0, 8))


def test_one_workspace_for_calls_of_different_shapes(fk):
    """The persistent launch's work counter lives in the workspace: calls of
    different sizes in a row on one workspace (the large one through the
    counter, the small one with one CTA per item) give the results of calls on
    fresh workspaces, bit for bit."""
    big = workloads.make_decode(workloads.DecodeSpec("big", B=16, Hq=32, Hkv=4, D=128, block_size=16,
                                                     ctx_lo=1000, ctx_hi=30000, rel_extent=1024),
                                device=DEV, seed=40)
    small = workloads.make_decode(workloads.DecodeSpec("small", B=3, Hq=8, Hkv=1, D=128,
                                                       block_size=16, ctx_lo=10, ctx_hi=3000),
                                  device=DEV, seed=41)
    caches = []
    for inp, spec_h in ((big, (4, 128)), (small, (1, 128))):
        kv = inp["kv"]
        c = fk.KVCache.empty(kv.num_blocks, 16, spec_h[0], spec_h[1], device=DEV)
        fk.kv_store_e4m3(c, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
        caches.append(c)

    def call(i, ws=None):
        inp = (big, small)[i]
        kv = inp["kv"]
        return fk.paged_attn_fp8_decode(caches[i], inp["q"], kv.block_table, kv.seq_lens, 1.0, 1.0,
                                        1.0, rel_bias=inp["rel"], workspace=ws).clone()
    ref_big, ref_small = call(0), call(1)
    kvb = big["kv"]
    n = fk.decode_workspace_size(16, 32, 4, 128, kvb.max_blocks, 16, 0, 0)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    a1 = call(0, ws)
    s1 = call(1, ws)
    a2 = call(0, ws)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    assert torch.equal(a1, ref_big) and torch.equal(a2, ref_big) and torch.equal(s1, ref_small)


def test_bound_decode_step_matches_the_calls(fk):
    """DecodeStep.run() over buffers updated in place gives the one-shot calls'
    results bit for bit, for decode and for the fused store + decode."""
    spec = workloads.DecodeSpec("bound", B=12, Hq=32, Hkv=4, D=128, block_size=16,
                                ctx_lo=500, ctx_hi=9000, rel_extent=1024)
    inp = workloads.make_decode(spec, device=DEV, seed=50)
    kv = inp["kv"]
    cache = fk.KVCache.empty(kv.num_blocks, 16, 4, 128, device=DEV)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
    q = inp["q"].clone()
    step = fk.DecodeStep(cache, q, kv.block_table, kv.seq_lens, 1.0, 1.0, 1.0,
                         rel_bias=inp["rel"])
    for seed in (1, 2):   # new contents of q between runs
        q.copy_(torch.randn(q.shape, generator=torch.Generator(DEV).manual_seed(seed),
                            device=DEV).to(torch.bfloat16))
        got = step.run().clone()
        ref = fk.paged_attn_fp8_decode(cache, q, kv.block_table, kv.seq_lens, 1.0, 1.0, 1.0,
                                       rel_bias=inp["rel"])
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    # fused: the same new token stored by both (the cache bytes are identical)
    k_new = torch.randn(12, 4, 128, device=DEV).to(torch.bfloat16)
    v_new = torch.randn(12, 4, 128, device=DEV).to(torch.bfloat16)
    fused = fk.DecodeStep(cache, q, kv.block_table, kv.seq_lens, 1.0, 1.0, 1.0,
                          rel_bias=inp["rel"], k_new=k_new, v_new=v_new)
    got = fused.run().clone()
    ref = fk.paged_attn_fp8_decode_store(cache, q, k_new, v_new, kv.block_table, kv.seq_lens, 1.0,
                                         1.0, 1.0, rel_bias=inp["rel"])
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    assert torch.equal(got, ref)


def test_decode_step_cuda_graph_replays_the_step(fk):
    """DecodeStep.cuda_graph: a graph of (copy of q, k_new, v_new from pinned
    host memory, the fused store + decode, copy of out to pinned host memory),
    replayed after new inputs are written to the host buffers, gives the
    one-shot fused call's output bit for bit; sampled rows match the oracle."""
    spec = workloads.DecodeSpec("graph", B=40, Hq=32, Hkv=4, D=128, block_size=16,
                                ctx_lo=300, ctx_hi=12000, rel_extent=1024)
    inp = workloads.make_decode(spec, device="cpu", seed=51)
    kv = inp["kv"]
    kd = to_device(kv, DEV)
    cache = fk.KVCache.empty(kv.num_blocks, 16, 4, 128, device=DEV)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, 1.0, 1.0)
    rel = inp["rel"].to(DEV)
    B, Hq, Hkv, D = 40, 32, 4, 128
    q_h = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    kn_h = torch.empty((B, Hkv, D), dtype=torch.bfloat16).pin_memory()
    vn_h = torch.empty_like(kn_h).pin_memory()
    out_h = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    q, k_new, v_new = q_h.to(DEV), kn_h.to(DEV), vn_h.to(DEV)
    step = fk.DecodeStep(cache, q, kd.block_table, kd.seq_lens, 1.0, 1.0, 1.0, rel_bias=rel,
                         k_new=k_new, v_new=v_new)

    def copy_in():
        q.copy_(q_h, non_blocking=True)
        k_new.copy_(kn_h, non_blocking=True)
        v_new.copy_(vn_h, non_blocking=True)

    def copy_out():
        out_h.copy_(step.out, non_blocking=True)
    graph = step.cuda_graph(pre=copy_in, post=copy_out)
    for seed in (1, 2):   # new host inputs before each replay
        g = torch.Generator().manual_seed(seed)
        q_h.copy_(torch.randn((B, Hq, D), generator=g).to(torch.bfloat16))
        kn_h.copy_(torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16))
        vn_h.copy_(torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16))
        graph.replay()
        torch.cuda.current_stream().synchronize()
        assert fk.device_error() == 0
        got = out_h.clone()
        ref = fk.paged_attn_fp8_decode_store(cache, q_h.to(DEV), kn_h.to(DEV), vn_h.to(DEV),
                                             kd.block_table, kd.seq_lens, 1.0, 1.0, 1.0,
                                             rel_bias=rel)
        torch.cuda.synchronize()
        assert torch.equal(got, ref.cpu())
    # the last replay's step against the oracle: the cache holds the new
    # tokens at each sequence's last position
    kv_last = workloads.PagedKV(k=kv.k.clone(), v=kv.v.clone(), seq_lens=kv.seq_lens,
                                tok_start=kv.tok_start, block_table=kv.block_table,
                                slot_mapping=kv.slot_mapping, num_blocks=kv.num_blocks,
                                block_size=kv.block_size)
    for b in range(B):
        last = int(kv.tok_start[b]) + int(kv.seq_lens[b]) - 1
        kv_last.k[last] = kn_h[b]
        kv_last.v[last] = vn_h[b]
    host = dict(inp)
    host["kv"] = kv_last
    host["q"] = q_h.clone()
    rows = [(b, h) for b in (0, 17, 39) for h in (0, 9, 31)]
    ref_rows = oracle_decode_rows(host, rows, 1.0, 1.0, 1.0, rel=inp["rel"])
    assert_close(np.stack([got[b, h].float().numpy() for b, h in rows]), ref_rows, "graph")


def test_bounded_wait_runs_out_and_the_next_call_is_clean(fk):
    """The failure path of a bounded wait, made to happen: the test hook makes
    the decode producer skip its first tile's copy (nothing else changes), so
    the MMA warp's wait for it runs out.  The call returns, the error word
    says FP8KV_DEVERR_WAIT_TIMEOUT, and the next call in the same process is
    clean and matches the oracle."""
    import time
    lens, Hq, Hkv = [100], 4, 1            # one key tile, one CTA
    spec = workloads.DecodeSpec("case", B=1, Hq=Hq, Hkv=Hkv, D=128, block_size=16, ctx_lo=1,
                                ctx_hi=1)
    inp = workloads.make_decode(spec, device="cpu", seed=40, lens=lens)
    kd = to_device(inp["kv"], DEV)
    cache = fk.KVCache.empty(kd.num_blocks, 16, Hkv, 128, device=DEV)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, 1.0, 1.0)
    q = inp["q"].to(DEV)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    fk.test_drop_first_copy(True)
    t0 = time.time()
    fk.paged_attn_fp8_decode(cache, q, kd.block_table, kd.seq_lens, 1.0, 1.0, 1.0)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert fk.device_error() & fk.DEVERR_WAIT_TIMEOUT
    assert 1.5 < waited < 30.0, waited     # the 2 s limit, then the teardown
    out = fk.paged_attn_fp8_decode(cache, q, kd.block_table, kd.seq_lens, 1.0, 1.0, 1.0)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    rows = [(0, h) for h in range(Hq)]
    ref = oracle_decode_rows(inp, rows, 1.0, 1.0, 1.0)
    assert_close(out.float().cpu().numpy()[0], ref, "decode after a timed-out call")
