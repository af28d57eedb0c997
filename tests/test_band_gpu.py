"""Band counters (clip, flush-to-zero, round-trip error) on the GPU against
the oracle: the four counts exactly, the error sum within 1e-6 relative (the
GPU adds it in parallel in fp32/fp64, the oracle in float64 in order)."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fk():
    import fp8_e4m3_kv_gb300 as m
    return m


def check(fk, oracle_lib, x, scale, slots=None):
    counts = fk.kv_band_counts(x.to(DEV), scale,
                               slot_mapping=None if slots is None else slots.to(DEV))
    torch.cuda.synchronize()
    assert fk.device_error() == 0
    got = fk.band_counts_dict(counts)
    want = oracle_lib.band_counts(workloads.bf16_bits(x.reshape(x.shape[0], -1)), scale,
                                  slot_mapping=None if slots is None else slots.numpy())
    for k in ("count", "nonzero", "clipped", "flushed"):
        assert got[k] == want[k], (k, got[k], want[k], scale)
    assert abs(got["rt_err_sum"] - want["rt_err_sum"]) <= 1e-6 * max(1.0, want["rt_err_sum"])
    return got


@pytest.mark.parametrize("scale", [1.0, 3.0, 0.5, 0.37, 114.6 / 448])
def test_every_bf16_pattern(fk, oracle_lib, scale):
    x = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(512, 128)
    got = check(fk, oracle_lib, x, scale)
    assert got["count"] == 65536 - 256          # all but the 254 NaN and 2 Inf patterns


@pytest.mark.parametrize("dist,scale", [("v_t3", 1.0), ("v_t3", 3.0), ("normal", 1.0),
                                        ("normal", 0.0512)])
def test_workload_values_with_unstored_tokens(fk, oracle_lib, dist, scale):
    g = torch.Generator().manual_seed(21)
    x = workloads.draw_values((3000, 4, 128), dist, g, "cpu")
    slots = torch.arange(3000, dtype=torch.int64)
    slots[::7] = -1
    got = check(fk, oracle_lib, x, scale, slots)
    assert got["count"] == int((slots >= 0).sum()) * 512


def test_counts_accumulate_over_calls(fk, oracle_lib):
    g = torch.Generator().manual_seed(22)
    a = workloads.draw_values((100, 256), "v_t3", g, "cpu")
    b = workloads.draw_values((50, 256), "v_t3", g, "cpu")
    counts = fk.kv_band_counts(a.to(DEV), 1.0)
    fk.kv_band_counts(b.to(DEV), 1.0, counts=counts)
    torch.cuda.synchronize()
    got = fk.band_counts_dict(counts)
    want = oracle_lib.band_counts(workloads.bf16_bits(torch.cat([a, b])), 1.0)
    assert (got["count"], got["clipped"], got["flushed"]) == (want["count"], want["clipped"],
                                                              want["flushed"])
