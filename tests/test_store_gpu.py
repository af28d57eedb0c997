"""Quant-on-store and amax on the GPU against the oracle: cache bytes must be
bit-identical, amax exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import bits, oracle_store, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fk():
    import fp8_e4m3_kv_gb300 as m
    return m


DEV = "cuda"


def _store_case(fk, lens, Hkv, D, bs, k_scale, v_scale, v_dist="normal", seed=0, plant=False):
    g = torch.Generator().manual_seed(seed)
    kv = workloads.make_paged_kv(lens, Hkv, D, bs, g=g, device="cpu", v_dist=v_dist,
                                 plant_v=plant)
    kd = to_device(kv, DEV)
    cache = fk.KVCache.empty(kv.num_blocks, bs, Hkv, D, device=DEV, fill=0xA5)
    fk.kv_store_e4m3(cache, kd.k, kd.v, kd.slot_mapping, k_scale, v_scale)
    torch.cuda.synchronize()
    ck, cv = oracle_store(kv, k_scale, v_scale, fill=0xA5)
    assert np.array_equal(cache.k.cpu().numpy(), ck)
    assert np.array_equal(cache.v.cpu().numpy(), cv)
    assert fk.device_error() == 0


@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.5, 1.5), (1.0, 3.0), (0.0371, 2.84)])
def test_store_bit_exact_ragged(fk, scales):
    _store_case(fk, [1, 15, 16, 17, 33, 129, 300], 4, 128, 16, *scales, v_dist="v_t3",
                plant=True)


@pytest.mark.parametrize("bs,D,Hkv", [(32, 256, 2), (64, 128, 1), (128, 128, 3)])
def test_store_bit_exact_layouts(fk, bs, D, Hkv):
    _store_case(fk, [5, 200, 64], Hkv, D, bs, 0.75, 1.25, seed=3)


@pytest.mark.parametrize("scale", [1.0, 3.0, 0.5, 1272.0 / 448.0, 0.0371])
def test_store_every_bf16_pattern(fk, scale):
    """All 65,536 bf16 bit patterns (NaN, +-Inf, -0, subnormals, ties) as K
    and, reversed, as V: 512 tokens of one 128-wide head."""
    pat = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    k = pat.reshape(512, 1, 128).contiguous()
    v = pat.flip(0).reshape(512, 1, 128).contiguous()
    slots = torch.randperm(512, generator=torch.Generator().manual_seed(1)).to(torch.int64)
    cache = fk.KVCache.empty(32, 16, 1, 128, device=DEV, fill=0xA5)
    fk.kv_store_e4m3(cache, k.to(DEV), v.to(DEV), slots.to(DEV), scale, scale)
    torch.cuda.synchronize()
    ck = np.full((32, 1, 16, 128), 0xA5, dtype=np.uint8)
    cv = ck.copy()
    oracle.kv_store(ck, cv, bits(k), bits(v), slots.numpy(), scale, scale, 16)
    assert np.array_equal(cache.k.cpu().numpy(), ck)
    assert np.array_equal(cache.v.cpu().numpy(), cv)


def test_store_skips_negative_and_flags_out_of_range_slots(fk):
    g = torch.Generator().manual_seed(4)
    k = workloads.draw_values((6, 2, 128), "normal", g, "cpu")
    v = workloads.draw_values((6, 2, 128), "normal", g, "cpu")
    slots = torch.tensor([3, -1, 0, 64, 17, -5], dtype=torch.int64)   # 64 is past 4 blocks x 16
    cache = fk.KVCache.empty(4, 16, 2, 128, device=DEV, fill=0xA5)
    fk.device_error()
    fk.kv_store_e4m3(cache, k.to(DEV), v.to(DEV), slots.to(DEV), 1.0, 1.0)
    err = fk.device_error()
    assert err == fk.DEVERR_BAD_SLOT
    ck = np.full((4, 2, 16, 128), 0xA5, dtype=np.uint8)
    cv = ck.copy()
    keep = slots.clone()
    keep[3] = -1
    oracle.kv_store(ck, cv, bits(k), bits(v), keep.numpy(), 1.0, 1.0, 16)
    assert np.array_equal(cache.k.cpu().numpy(), ck)
    assert np.array_equal(cache.v.cpu().numpy(), cv)


def test_store_strided_rows(fk):
    """k and v as views into a wider [T][3][Hkv*D] buffer (qkv-style)."""
    g = torch.Generator().manual_seed(5)
    qkv = workloads.draw_values((40, 3, 2 * 128), "normal", g, "cpu")
    k, v = qkv[:, 1], qkv[:, 2]
    slots = torch.arange(40, dtype=torch.int64)
    cache = fk.KVCache.empty(3, 16, 2, 128, device=DEV, fill=0)
    qkv_d = qkv.to(DEV)
    fk.kv_store_e4m3(cache, qkv_d[:, 1], qkv_d[:, 2], slots.to(DEV), 1.0, 0.5)
    torch.cuda.synchronize()
    ck = np.zeros((3, 2, 16, 128), dtype=np.uint8)
    cv = ck.copy()
    oracle.kv_store(ck, cv, bits(k.reshape(40, 2, 128)), bits(v.reshape(40, 2, 128)),
                    slots.numpy(), 1.0, 0.5, 16)
    assert np.array_equal(cache.k.cpu().numpy(), ck) and np.array_equal(cache.v.cpu().numpy(), cv)


def test_amax_exact_with_skips_nan_and_running_max(fk):
    g = torch.Generator().manual_seed(6)
    k = workloads.draw_values((300, 4, 128), "v_t3", g, "cpu")
    v = workloads.draw_values((300, 4, 128), "normal", g, "cpu")
    k[7, 1, 3] = float("nan")
    k[9, 0, 0] = 5000.0                      # on a skipped token
    slots = torch.arange(300, dtype=torch.int64)
    slots[9] = -1
    amax = torch.tensor([0.0, 2.5], device=DEV)
    fk.kv_amax_calibrate(k.to(DEV), v.to(DEV), amax[0:1], amax[1:2], slots.to(DEV))
    got = amax.cpu().tolist()
    assert got[0] == oracle.amax(bits(k), slots.numpy(), 0.0)
    assert got[1] == oracle.amax(bits(v), slots.numpy(), 2.5)
    # running: a second call with a larger value raises it, a smaller one does not
    big = k[:1] * 0 + 7777.0                  # bf16: 7776
    fk.kv_amax_calibrate(big.to(DEV), None, amax[0:1], None)
    assert amax[0].item() == float(big.float().max())
    fk.kv_amax_calibrate(big.to(DEV) * 0 + 1.0, None, amax[0:1], None)
    assert amax[0].item() == float(big.float().max())


def test_store_at_decode_pool_size(fk):
    """The cache fill of the 64-sequence decode workload (~1.05M tokens, the
    store launch the bench makes before timing), sampled tokens checked."""
    spec = workloads.DECODE_32K
    inp = workloads.make_decode(spec, device=DEV, seed=0)
    kv = inp["kv"]
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=DEV)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 3.0)
    torch.cuda.synchronize()
    T = kv.k.shape[0]
    idx = torch.randint(0, T, (3000,), generator=torch.Generator().manual_seed(0))
    slots = kv.slot_mapping[idx.to(DEV)]
    blk, row = slots // kv.block_size, slots % kv.block_size
    gk = cache.k[blk, :, row].cpu().numpy()      # [block][head][row][d] -> [n][head][d]
    gv = cache.v[blk, :, row].cpu().numpy()
    hk = kv.k[idx.to(DEV)].cpu()
    hv = kv.v[idx.to(DEV)].cpu()
    assert np.array_equal(gk, oracle.quantize(bits(hk), 1.0))
    assert np.array_equal(gv, oracle.quantize(bits(hv), 3.0))
    assert fk.device_error() == 0
