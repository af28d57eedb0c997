"""Varlen fp8 prefill attention (tcgen05) on the GPU against the float64
oracle, element by element, within 2e-2 abs + 2e-2 rel."""
import numpy as np
import pytest
import torch

import workloads
from helpers import assert_close, oracle_prefill_rows, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fk():
    import fp8_e4m3_kv_gb300 as m
    return m


def run_case(fk, q_lens, k_lens=None, Hq=8, Hkv=2, D=128, bs=16, scales=(1.0, 1.0, 1.0),
             window=0, E=0, seed=0, rows=None, bias_std=0.5, rel_override=None):
    spec = workloads.PrefillSpec("case", q_lens=q_lens, q_lo=0, q_hi=0, n_seqs=len(q_lens),
                                 Hq=Hq, Hkv=Hkv, D=D, block_size=bs, rel_extent=E,
                                 bias_std=bias_std)
    inp = workloads.make_prefill(spec, device="cpu", seed=seed, q_lens=q_lens, k_lens=k_lens)
    if rel_override is not None:
        inp["rel"] = rel_override(inp)
    kv = inp["kv"]
    kd = to_device(kv, DEV)
    sq, sk, sv = scales
    cache = fk.KVCache.empty(kv.num_blocks, bs, Hkv, D, device=DEV, fill=0x7F)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, sk, sv)
    rel_d = None if inp["rel"] is None else inp["rel"].to(DEV)
    out = fk.attn_fp8_varlen_prefill(cache, inp["q"].to(DEV), inp["cu_seqlens_q"].to(DEV),
                                     kd.seq_lens, kd.block_table, max(q_lens), sq, sk, sv,
                                     rel_bias=rel_d, window=window)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = out.float().cpu().numpy()
    if rows is None:
        rows = [(t, h) for t in range(sum(q_lens)) for h in range(Hq)]
    ref = oracle_prefill_rows(inp, rows, sq, sk, sv, window=window, rel=inp["rel"])
    return assert_close(np.stack([got[t, h] for t, h in rows]), ref, "prefill"), got


def test_single_tile(fk):
    run_case(fk, [100])


@pytest.mark.parametrize("scales", [(1.0, 1.0, 1.0), (0.5, 0.5, 1.5)])
def test_ragged_fresh_chunks(fk, scales):
    run_case(fk, [1, 127, 128, 129, 300], scales=scales, E=128, seed=1)


def test_chunk_over_cached_prefix(fk):
    """queries are the last q_len of k_len keys (bottom-right causal)"""
    run_case(fk, [1, 64, 128, 200], k_lens=[1, 500, 129, 777], E=1024, seed=2)


@pytest.mark.parametrize("window", [1, 100, 512])
def test_sliding_window(fk, window):
    run_case(fk, [700, 50, 513], k_lens=[900, 50, 1300], window=window, E=128, seed=3)


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_block_sizes(fk, bs):
    run_case(fk, [130, 257], bs=bs, seed=4)


def test_head_dim_256(fk):
    run_case(fk, [90, 300], k_lens=[90, 450], Hq=6, Hkv=1, D=256, scales=(0.5, 0.25, 1.5),
             E=128, seed=5)


def test_gqa_16(fk):
    run_case(fk, [200], Hq=16, Hkv=1, seed=6)


def test_large_bias_row_max_jumps(fk):
    """A bias that grows towards the diagonal makes the row maximum jump at
    every key tile: the lazy rescale must keep P below 448 (threshold 0.75 <
    log2(448) - 8); at the 4.0 threshold P would clip."""
    def ramp(inp):
        T, H, E = inp["rel"].shape
        d = torch.arange(E, dtype=torch.float32)
        r = (6.0 * (1.0 - d / E)).expand(T, H, E)
        return r.to(torch.bfloat16).contiguous()
    run_case(fk, [600, 260], k_lens=[600, 900], E=1024, seed=7, rel_override=ramp)


@pytest.mark.parametrize("window", [0, 100])
def test_bias_with_extreme_scales(fk, window):
    """q and k scales of 2^-30: the kernel adds the bias unfolded (its factor
    log2(e) / score scale would be 2^63.5; a kernel instantiation of its
    own); every code saturates.  With and without a window."""
    run_case(fk, [200, 70], k_lens=[260, 70], scales=(2.0 ** -30, 2.0 ** -30, 1.0), E=128,
             seed=9, window=window)


def test_bias_broadcast_over_tokens(fk):
    """One bias table per head for every query token (token stride 0), the
    form a learned per-head relative-position table takes; every row against
    the oracle."""
    q_lens, k_lens, Hq, Hkv, E = [300, 129], [300, 400], 8, 2, 128
    spec = workloads.PrefillSpec("case", q_lens=q_lens, q_lo=0, q_hi=0, n_seqs=2, Hq=Hq, Hkv=Hkv,
                                 D=128, block_size=16, rel_extent=E)
    inp = workloads.make_prefill(spec, device="cpu", seed=13, q_lens=q_lens, k_lens=k_lens)
    T = sum(q_lens)
    table = inp["rel"][:1]
    inp["rel"] = table.expand(T, Hq, E)
    kv = inp["kv"]
    kd = to_device(kv, DEV)
    cache = fk.KVCache.empty(kv.num_blocks, 16, Hkv, 128, device=DEV, fill=0x7F)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, 1.0, 1.0)
    rel_d = table.to(DEV).expand(T, Hq, E)
    assert rel_d.stride(0) == 0
    out = fk.attn_fp8_varlen_prefill(cache, inp["q"].to(DEV), inp["cu_seqlens_q"].to(DEV),
                                     kd.seq_lens, kd.block_table, max(q_lens), 1.0, 1.0, 1.0,
                                     rel_bias=rel_d)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    rows = [(t, h) for t in range(T) for h in range(Hq)]
    ref = oracle_prefill_rows(inp, rows, 1.0, 1.0, 1.0, rel=inp["rel"])
    got = out.float().cpu().numpy()
    assert_close(np.stack([got[t, h] for t, h in rows]), ref, "broadcast bias")


def test_heavy_bias(fk):
    run_case(fk, [400], E=512, bias_std=3.0, seed=8)


def _prefill_at_caps(fk, q_lens, k_lens, caps, window=0, E=128, Hq=8, Hkv=2, seed=0, bs=16,
                     scales=(1.0, 1.0, 1.0)):
    """The same prefill once per CTA cap (0: one CTA per SM)."""
    spec = workloads.PrefillSpec("case", q_lens=q_lens, q_lo=0, q_hi=0, n_seqs=len(q_lens),
                                 Hq=Hq, Hkv=Hkv, D=128, block_size=bs, rel_extent=E)
    inp = workloads.make_prefill(spec, device="cpu", seed=seed, q_lens=q_lens, k_lens=k_lens)
    kv = inp["kv"]
    kd = to_device(kv, DEV)
    sq, sk, sv = scales
    cache = fk.KVCache.empty(kv.num_blocks, bs, Hkv, 128, device=DEV, fill=0x7F)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, sk, sv)
    q, cu = inp["q"].to(DEV), inp["cu_seqlens_q"].to(DEV)
    rel = None if inp["rel"] is None else inp["rel"].to(DEV)
    outs = []
    try:
        for cap in caps:
            fk.set_prefill_max_ctas(cap)
            outs.append(fk.attn_fp8_varlen_prefill(cache, q, cu, kd.seq_lens, kd.block_table,
                                                   max(q_lens), sq, sk, sv, rel_bias=rel,
                                                   window=window))
            torch.cuda.synchronize()
            assert fk.device_error() == 0
    finally:
        fk.set_prefill_max_ctas(0)
    return inp, outs


@pytest.mark.parametrize("window", [0, 200])
def test_persistent_schedule_does_not_change_results(fk, window):
    """With one, two or seven CTAs each CTA works through dozens of items
    (query tile pairs of different sequences and heads, second tiles past a
    sequence's queries, cached prefixes, windows) back to back: the output
    must be bit-identical to one CTA per SM's, and match the oracle."""
    q_lens = [1, 129, 256, 300, 700, 1000]
    k_lens = [1, 193, 256, 600, 700, 1001]   # cached prefixes of 0 .. 300 keys
    inp, outs = _prefill_at_caps(fk, q_lens, k_lens, [0, 1, 2, 7], window=window, seed=11)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    rng = np.random.default_rng(window)
    cu = inp["cu_seqlens_q"].tolist()
    rows = []
    for b, n in enumerate(q_lens):
        picks = {0, n - 1, 127, 128, 255, 256} | set(int(x) for x in rng.integers(0, n, 10))
        rows += [(cu[b] + i, int(rng.integers(8))) for i in sorted(picks) if 0 <= i < n]
    ref = oracle_prefill_rows(inp, rows, 1.0, 1.0, 1.0, window=window, rel=inp["rel"])
    got = outs[0].float().cpu().numpy()
    assert_close(np.stack([got[t, h] for t, h in rows]), ref, "persistent prefill")


@pytest.mark.parametrize("seed", range(8))
def test_random_batches_at_several_grids(fk, seed):
    """Random small batches (empty query runs, cached prefixes, windows, GQA
    ratios, block sizes, bias extents, non-power-of-two scales): output
    bit-identical at 0 (one CTA per SM), 1 and 3 CTAs, sampled rows against
    the oracle."""
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 7))
    q_lens = [int(x) for x in rng.choice([0, 1, 5, 127, 128, 129, 200, 256, 300, 513], B)]
    if max(q_lens) == 0:
        q_lens[0] = 70
    k_lens = [q + int(rng.choice([0, 0, 1, 64, 250])) for q in q_lens]
    Hkv = int(rng.choice([1, 2]))
    Hq = Hkv * int(rng.choice([1, 3, 8]))
    bs = int(rng.choice([16, 32, 64]))
    window = int(rng.choice([0, 0, 100, 512]))
    E = int(rng.choice([0, 128, 1024]))
    scales = (float(rng.choice([1.0, 0.75])), float(rng.choice([1.0, 0.3])),
              float(rng.choice([1.0, 2.5])))
    inp, outs = _prefill_at_caps(fk, q_lens, k_lens, [0, 1, 3], window=window, E=E, Hq=Hq,
                                 Hkv=Hkv, seed=seed, bs=bs, scales=scales)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    cu = inp["cu_seqlens_q"].tolist()
    rows = []
    for b, n in enumerate(q_lens):
        if n == 0:
            continue
        picks = {0, n - 1, 127, 128} | set(int(x) for x in rng.integers(0, n, 4))
        rows += [(cu[b] + i, int(rng.integers(Hq))) for i in sorted(picks) if 0 <= i < n]
    ref = oracle_prefill_rows(inp, rows, *scales, window=window, rel=inp["rel"])
    got = outs[0].float().cpu().numpy()
    assert_close(np.stack([got[t, h] for t, h in rows]), ref, "random prefill %d" % seed)


def test_many_sequences_one_cta_per_item(fk):
    """More sequences than the persistent schedule sorts (64): one CTA per two
    query tiles, on sampled rows."""
    rng = np.random.default_rng(12)
    q_lens = [int(x) for x in rng.integers(1, 300, 100)]
    k_lens = [q + int(p) for q, p in zip(q_lens, rng.integers(0, 100, 100))]
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    rows = [(int(cu[b] + rng.integers(q_lens[b])), int(rng.integers(4))) for b in range(0, 100, 3)]
    run_case(fk, q_lens, k_lens=k_lens, Hq=4, Hkv=1, E=128, seed=12, rows=rows)


def _full_group(fk, which, scales=(1.0, 1.0, 1.0)):
    spec = workloads.PREFILL_16K
    inp = workloads.make_prefill(spec, device=DEV, seed=0)
    kv = inp["kv"]
    sq, sk, sv = scales
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=DEV)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, sk, sv)
    half = spec.n_seqs // 2
    lo, hi = (0, half) if which == 0 else (half, spec.n_seqs)
    window = spec.windows[which]
    cu = inp["cu_seqlens_q"].tolist()
    cu_g = torch.tensor([c - cu[lo] for c in cu[lo:hi + 1]], dtype=torch.int32, device=DEV)
    q_g = inp["q"][cu[lo]:cu[hi]]
    rel_g = inp["rel"][cu[lo]:cu[hi]]
    out = fk.attn_fp8_varlen_prefill(cache, q_g, cu_g, kv.seq_lens[lo:hi].contiguous(),
                                     kv.block_table[lo:hi].contiguous(), max(inp["q_lens"][lo:hi]),
                                     sq, sk, sv, rel_bias=rel_g, window=window)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    # a third of the SMs: each CTA takes about three times the items
    try:
        fk.set_prefill_max_ctas(50)
        out2 = fk.attn_fp8_varlen_prefill(cache, q_g, cu_g, kv.seq_lens[lo:hi].contiguous(),
                                          kv.block_table[lo:hi].contiguous(),
                                          max(inp["q_lens"][lo:hi]), sq, sk, sv,
                                          rel_bias=rel_g, window=window)
        torch.cuda.synchronize()
    finally:
        fk.set_prefill_max_ctas(0)
    assert fk.device_error() == 0
    assert torch.equal(out, out2)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(which)
    rows = []
    for b in range(lo, hi):
        s, n = cu[b] - cu[lo], inp["q_lens"][b]
        picks = {0, 1, 127, 128, 129, n - 1, n - 2} | set(int(x) for x in rng.integers(0, n, 12))
        rows += [(s + i, int(rng.integers(spec.Hq))) for i in sorted(picks) if 0 <= i < n]
    g_inp = dict(inp)
    g_inp["q"] = q_g
    g_inp["rel"] = rel_g
    g_inp["cu_seqlens_q"] = cu_g
    g_inp["q_lens"] = inp["q_lens"][lo:hi]
    g_inp["k_lens"] = inp["k_lens"][lo:hi]
    sub = workloads.PagedKV(k=kv.k[int(kv.tok_start[lo]):int(kv.tok_start[hi])],
                            v=kv.v[int(kv.tok_start[lo]):int(kv.tok_start[hi])],
                            seq_lens=kv.seq_lens[lo:hi], tok_start=kv.tok_start[lo:hi + 1] -
                            kv.tok_start[lo], block_table=kv.block_table[lo:hi],
                            slot_mapping=kv.slot_mapping, num_blocks=kv.num_blocks,
                            block_size=kv.block_size)
    g_inp["kv"] = sub
    ref = oracle_prefill_rows(g_inp, rows, sq, sk, sv, window=window, rel=rel_g)
    return assert_close(np.stack([got[t, h] for t, h in rows]), ref, spec.name)


# unit scales, and q / k scales that are not powers of two (the divided
# quantization) with a V scale of 3
FULL_SCALES = [(1.0, 1.0, 1.0), (0.7, 0.45, 3.0)]


@pytest.mark.parametrize("scales", FULL_SCALES)
def test_full_prefill_causal_group(fk, scales):
    _full_group(fk, 0, scales)


@pytest.mark.parametrize("scales", FULL_SCALES)
def test_full_prefill_window_group(fk, scales):
    _full_group(fk, 1, scales)


@pytest.mark.parametrize("scales", FULL_SCALES)
def test_full_chunk_over_64k_prefix(fk, scales):
    """One 4,096-query chunk over 65,536 keys (a 61,440-key cached prefix), the
    bench's chunked-prefill workload, on sampled rows."""
    spec = workloads.PREFILL_CHUNK_64K
    inp = workloads.make_prefill(spec, device=DEV, seed=0)
    kv = inp["kv"]
    sq, sk, sv = scales
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=DEV)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, sk, sv)
    out = fk.attn_fp8_varlen_prefill(cache, inp["q"], inp["cu_seqlens_q"], kv.seq_lens,
                                     kv.block_table, max(inp["q_lens"]), sq, sk, sv,
                                     rel_bias=inp["rel"], window=0)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(2)
    n = inp["q_lens"][0]
    picks = sorted({0, 1, 127, 128, n - 1} | set(int(x) for x in rng.integers(0, n, 10)))
    rows = [(i, int(rng.integers(spec.Hq))) for i in picks]
    host = dict(inp)
    host["kv"] = workloads.PagedKV(k=kv.k.cpu(), v=kv.v.cpu(), seq_lens=kv.seq_lens.cpu(),
                                   tok_start=kv.tok_start.cpu(), block_table=kv.block_table.cpu(),
                                   slot_mapping=kv.slot_mapping.cpu(), num_blocks=kv.num_blocks,
                                   block_size=kv.block_size)
    host["q"] = inp["q"].cpu()
    host["rel"] = inp["rel"].cpu()
    ref = oracle_prefill_rows(host, rows, sq, sk, sv, window=0, rel=host["rel"])
    assert_close(np.stack([got[t, h] for t, h in rows]), ref, spec.name)


def test_length_past_block_table_is_flagged(fk):
    """seq_lens_k past the block-table row: the keys beyond it read as zeros,
    FP8KV_DEVERR_BAD_BLOCK is set, and the call completes."""
    spec = workloads.PrefillSpec("case", q_lens=[100], q_lo=0, q_hi=0, n_seqs=1, Hq=4, Hkv=1,
                                 D=128, block_size=16)
    inp = workloads.make_prefill(spec, device="cpu", seed=31, q_lens=[100], k_lens=[100])
    kv = to_device(inp["kv"], DEV)
    cache = fk.KVCache.empty(kv.num_blocks, 16, 1, 128, device=DEV)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
    assert kv.block_table.shape[1] == 7          # 112 keys of room
    too_long = torch.tensor([100 + 60], dtype=torch.int32, device=DEV)
    out = fk.attn_fp8_varlen_prefill(cache, inp["q"].to(DEV), inp["cu_seqlens_q"].to(DEV),
                                     too_long, kv.block_table, 100, 1.0, 1.0, 1.0)
    torch.cuda.synchronize()
    assert fk.device_error() & fk.DEVERR_BAD_BLOCK
    assert fk.device_error() == 0
    assert torch.isfinite(out.float()).all()
