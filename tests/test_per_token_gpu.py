"""Per-token scales on the GPU against the oracle: the store's codes and
scales bit-exact, decode within 2e-2 abs + 2e-2 rel of the float64 oracle
attending over keys dequantized with their own scales."""
import math

import numpy as np
import pytest
import torch

import workloads
from helpers import assert_close, bits, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fk():
    import fp8_e4m3_kv_gb300 as m
    return m


def store(fk, kv, Hkv, D, bs):
    kd = to_device(kv, DEV)
    cache = fk.KVCache.empty(kv.num_blocks, bs, Hkv, D, device=DEV, fill=0x7F)
    ks = torch.full((kv.num_blocks, Hkv, bs), float("nan"), dtype=torch.float32, device=DEV)
    vs = torch.full_like(ks, float("nan"))
    fk.kv_store_e4m3_per_token(cache, kd.k, kd.v, kd.slot_mapping, ks, vs)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    return cache, ks, vs, kd


def check_store(fk, oracle_lib, kv, Hkv, D, bs):
    cache, ks, vs, _ = store(fk, kv, Hkv, D, bs)
    slots = kv.slot_mapping.cpu().numpy()
    for name, x, c, sc in (("k", kv.k, cache.k, ks), ("v", kv.v, cache.v, vs)):
        codes, scales = oracle_lib.quantize_per_token(bits(x.cpu()), D)
        codes = codes.reshape(-1, Hkv, D)
        scales = scales.reshape(-1, Hkv)
        cc = c.cpu().numpy()
        ss = sc.cpu().numpy()
        keep = slots >= 0
        blk, row = slots[keep] // bs, slots[keep] % bs
        got_c = cc[blk, :, row, :]
        got_s = ss[blk, :, row]
        assert np.array_equal(got_c, codes[keep]), name
        assert np.array_equal(got_s.view(np.uint32), scales[keep].view(np.uint32)), name
    return cache, ks, vs


@pytest.mark.parametrize("D,bs", [(128, 16), (256, 32)])
def test_store_codes_and_scales_bit_exact(fk, oracle_lib, D, bs):
    g = torch.Generator().manual_seed(41)
    lens = [1, 17, 300]
    kv = workloads.make_paged_kv(lens, 4, D, bs, g=g, device="cpu", v_dist="v_t3")
    # rows of special values: all zero, +-Inf, NaN, tiny, one huge outlier
    kv.k[0, 0] = 0.0
    kv.k[1, 1, :3] = torch.tensor([float("inf"), -float("inf"), float("nan")])
    kv.k[2, 2] = 1e-38
    kv.v[3, 3, 5] = 3.0e38
    kv.slot_mapping[4] = -1                      # an unstored token
    check_store(fk, oracle_lib, kv, 4, D, bs)


def oracle_rows_pt(oracle_lib, inp, rows, q_scale, window=0):
    kv, q = inp["kv"], inp["q"]
    B, Hq, D = q.shape
    Hkv = kv.k.shape[1]
    G = Hq // Hkv
    starts = kv.tok_start.cpu().tolist()
    lens = kv.seq_lens.cpu().tolist()
    rel = inp["rel"]
    memo = {}
    out = []
    for b, h in rows:
        kvh = h // G
        if (b, kvh) not in memo:
            s, L = starts[b], lens[b]
            k8, sk = oracle_lib.quantize_per_token(bits(kv.k[s:s + L, kvh].cpu()), D)
            v8, sv = oracle_lib.quantize_per_token(bits(kv.v[s:s + L, kvh].cpu()), D)
            memo[(b, kvh)] = (k8, sk, v8, sv)
        k8, sk, v8, sv = memo[(b, kvh)]
        q8 = oracle_lib.quantize(bits(q[b, h].cpu()), q_scale)
        bias = None if rel is None else bits(rel[b, h].cpu())
        out.append(oracle_lib.attend_row_pt(q8, k8, v8, sk, sv, lens[b] - 1, 1 / math.sqrt(D),
                                            q_scale, bias=bias, window=window))
    return np.stack(out)


def run_decode(fk, oracle_lib, lens, Hq, Hkv, D, bs, window=0, E=0, v_dist="normal", seed=0,
               q_scale=1.0):
    spec = workloads.DecodeSpec("case", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                                ctx_lo=1, ctx_hi=1, v_dist=v_dist, rel_extent=E, plant_v=True)
    inp = workloads.make_decode(spec, device="cpu", seed=seed, lens=lens)
    kv = inp["kv"]
    cache, ks, vs, kd = store(fk, kv, Hkv, D, bs)
    rel = None if inp["rel"] is None else inp["rel"].to(DEV)
    out = fk.paged_attn_fp8_decode_per_token(cache, inp["q"].to(DEV), kd.block_table, kd.seq_lens,
                                             q_scale, ks, vs, rel_bias=rel, window=window)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(seed)
    rows = [(b, int(h)) for b in range(len(lens)) if lens[b] > 0
            for h in rng.choice(Hq, min(Hq, 6), replace=False)]
    ref = oracle_rows_pt(oracle_lib, inp, rows, q_scale, window=window)
    assert_close(np.stack([got[b, h] for b, h in rows]), ref, "per-token decode")
    if 0 in lens:
        assert (got[lens.index(0)] == 0).all()


def test_decode_heavy_tailed_v_with_bias(fk, oracle_lib):
    """V = 17.47 t(3) with a planted 1,272: it would clip at a unity per-tensor
    scale, not with its own scale."""
    run_decode(fk, oracle_lib, [1, 2, 127, 128, 129, 1000, 3000], 32, 4, 128, 16, E=1024,
               v_dist="v_t3", seed=1)


def test_decode_window_and_empty(fk, oracle_lib):
    run_decode(fk, oracle_lib, [0, 50, 511, 513, 1500], 8, 1, 128, 16, window=512, E=128, seed=2,
               q_scale=0.5)


def test_decode_head_dim_256_block_32(fk, oracle_lib):
    run_decode(fk, oracle_lib, [90, 700], 24, 4, 256, 32, seed=3)


def test_decode_sixteen_heads_per_kv_head(fk, oracle_lib):
    run_decode(fk, oracle_lib, [77, 400], 32, 2, 128, 16, seed=4)


def run_prefill(fk, oracle_lib, q_lens, k_lens, Hq, Hkv, window=0, E=0, v_dist="normal", seed=0,
                q_scale=1.0, rows_per_seq=None, caps=(0,)):
    """Per-token prefill (chunks over cached prefixes) against the oracle's
    per-token attention: all rows, or rows_per_seq sampled rows per sequence;
    the output must not depend on the CTA cap."""
    g = torch.Generator().manual_seed(seed)
    kv = workloads.make_paged_kv(k_lens, Hkv, 128, 16, g=g, device="cpu", v_dist=v_dist)
    Tq = sum(q_lens)
    q = workloads.draw_values((Tq, Hq, 128), "normal", g, "cpu")
    rel = None
    if E:
        rel = (0.5 * torch.randn((Tq, Hq, E), generator=g)).to(torch.bfloat16)
    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + n)
    cache, ks, vs, kd = store(fk, kv, Hkv, 128, 16)
    outs = []
    try:
        for cap in caps:
            fk.set_prefill_max_ctas(cap)
            outs.append(fk.attn_fp8_varlen_prefill_per_token(
                cache, q.to(DEV), torch.tensor(cu, dtype=torch.int32, device=DEV), kd.seq_lens,
                kd.block_table, max(q_lens), q_scale, ks, vs,
                rel_bias=None if rel is None else rel.to(DEV), window=window))
            torch.cuda.synchronize()
            assert fk.device_error() == 0
    finally:
        fk.set_prefill_max_ctas(0)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    got = outs[0].float().cpu().numpy()
    assert np.isfinite(got).all()
    G = Hq // Hkv
    starts = kv.tok_start.tolist()
    rng = np.random.default_rng(seed)
    rows, refs = [], []
    memo = {}
    for b, n in enumerate(q_lens):
        picks = range(n) if rows_per_seq is None else sorted(
            {0, n - 1} | set(int(x) for x in rng.integers(0, n, rows_per_seq)))
        for i in picks:
            h = int(rng.integers(Hq))
            kvh = h // G
            if (b, kvh) not in memo:
                s, L = starts[b], k_lens[b]
                k8, sk = oracle_lib.quantize_per_token(bits(kv.k[s:s + L, kvh]), 128)
                v8, sv = oracle_lib.quantize_per_token(bits(kv.v[s:s + L, kvh]), 128)
                memo[(b, kvh)] = (k8, sk, v8, sv)
            k8, sk, v8, sv = memo[(b, kvh)]
            t = cu[b] + i
            q8 = oracle_lib.quantize(bits(q[t, h]), q_scale)
            bias = None if rel is None else bits(rel[t, h])
            refs.append(oracle_lib.attend_row_pt(q8, k8, v8, sk, sv, k_lens[b] - n + i,
                                                 1 / math.sqrt(128), q_scale, bias=bias,
                                                 window=window))
            rows.append((t, h))
    assert_close(np.stack([got[t, h] for t, h in rows]), np.stack(refs), "per-token prefill")


def test_prefill_ragged_fresh_chunks(fk, oracle_lib):
    """Fresh chunks (queries = keys), ragged tiles, heavy-tailed V with a planted
    1,272, every row."""
    run_prefill(fk, oracle_lib, [1, 127, 129, 300], [1, 127, 129, 300], 8, 2, E=128,
                v_dist="v_t3", seed=5, caps=(0, 1, 3))


def test_prefill_chunks_over_cached_prefixes(fk, oracle_lib):
    run_prefill(fk, oracle_lib, [64, 200, 5], [500, 777, 40], 8, 2, E=1024, seed=6, q_scale=0.5)


def test_prefill_sliding_window(fk, oracle_lib):
    run_prefill(fk, oracle_lib, [700, 50], [900, 50], 8, 1, window=512, E=128, seed=7,
                rows_per_seq=40)


def test_prefill_long_chunk_sampled(fk, oracle_lib):
    """A 2,048-query chunk over 4,000 keys, sampled rows."""
    run_prefill(fk, oracle_lib, [2048], [4000], 32, 4, E=128, seed=8, rows_per_seq=48)


def test_prefill_per_token_rejects_head_dim_256(fk):
    cache = fk.KVCache.empty(4, 16, 1, 256, device=DEV)
    ks = torch.ones((4, 1, 16), dtype=torch.float32, device=DEV)
    q = torch.zeros(4, 2, 256, dtype=torch.bfloat16, device=DEV)
    cu = torch.tensor([0, 4], dtype=torch.int32, device=DEV)
    lens = torch.tensor([4], dtype=torch.int32, device=DEV)
    bt = torch.zeros(1, 4, dtype=torch.int32, device=DEV)
    with pytest.raises(fk.Fp8KVError) as e:
        fk.attn_fp8_varlen_prefill_per_token(cache, q, cu, lens, bt, 4, 1.0, ks, ks)
    assert e.value.status == fk.ERR_UNSUPPORTED


def test_decode_dominant_keys_with_tiny_v(fk, oracle_lib):
    """Keys whose V rows are tiny (scale ~1e-33 / 448) but whose scores
    dominate: the V scale folded into the exponent must not drop them from
    the row sum (the output is then close to zero, as the oracle's)."""
    spec = workloads.DecodeSpec("case", B=2, Hq=8, Hkv=2, D=128, block_size=16, ctx_lo=1, ctx_hi=1)
    inp = workloads.make_decode(spec, device="cpu", seed=9, lens=[300, 77])
    kv = inp["kv"]
    q = inp["q"]
    starts = kv.tok_start.tolist()
    for b, j in ((0, 5), (0, 299), (1, 40)):
        t = starts[b] + j
        kv.v[t] = (kv.v[t].float() * 1e-33).to(torch.bfloat16)
        # align the key with every query head of its KV head: a dominant score
        kv.k[t, 0] = (q[b, :4].float().mean(0) * 6.0).to(torch.bfloat16)
        kv.k[t, 1] = (q[b, 4:].float().mean(0) * 6.0).to(torch.bfloat16)
    cache, ks, vs, kd = store(fk, kv, 2, 128, 16)
    out = fk.paged_attn_fp8_decode_per_token(cache, q.to(DEV), kd.block_table, kd.seq_lens, 1.0,
                                             ks, vs)
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    rows = [(b, h) for b in range(2) for h in range(8)]
    ref = oracle_rows_pt(oracle_lib, inp, rows, 1.0)
    assert_close(np.stack([got[b, h] for b, h in rows]), ref, "tiny V scales")


def test_decode_long_sequences_through_the_work_counter(fk, oracle_lib):
    """Enough splits (more work items than the persistent grid has CTAs) that
    the CTAs take them from the counter; empty and one-key sequences among
    them."""
    run_decode(fk, oracle_lib, [40000, 33000, 0, 20000, 5000, 1, 12345, 38000], 32, 4, 128, 16,
               E=1024, v_dist="v_t3", seed=5)
