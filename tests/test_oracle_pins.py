"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks an oracle function against a value the pages print, a code
table written from the format definition, a library routine (torch's
float8_e4m3fn cast, scipy's softmax), a closed form, or a hand-enumerated
case, chosen so that a plausible slip (a dropped term, a wrong sign or index,
truncation instead of rounding, a transposed operand) fails one of them.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from conftest import pages_values, read_table


def bf16_bits_of(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return workloads.bf16_bits(t)


# ----------------------------------------------------------------- codec
def test_landmark_codes_match_format_table(oracle_lib):
    for code, value, *_ in read_table("e4m3_codes.txt"):
        got = oracle_lib.e4m3_decode(int(code, 16))
        if value == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(value), code
            assert math.copysign(1.0, got) == math.copysign(1.0, float(value)), code


def test_all_finite_codes_round_trip(oracle_lib):
    for c in range(256):
        v = oracle_lib.e4m3_decode(c)
        if math.isnan(v):
            assert c in (0x7F, 0xFF)
            continue
        assert oracle_lib.e4m3_encode(v) == c, hex(c)


def test_code_values_increase_with_code(oracle_lib):
    vals = [oracle_lib.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))
    assert vals[-1] == pages_values()["e4m3_max"]


def _torch_quantize(bits_u16, scale):
    """Library cross-check: fp32 x/s, clamp to +-448 (NaN kept), torch's
    float8_e4m3fn cast (round to nearest even)."""
    x = torch.from_numpy(bits_u16.view(np.int16).copy()).view(torch.bfloat16).float()
    q = x / torch.tensor(scale, dtype=torch.float32)
    q = torch.where(q > 448.0, torch.tensor(448.0), torch.where(q < -448.0, torch.tensor(-448.0), q))
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("scale", [1.0, 3.0, 0.5, 1272.0 / 448.0, 73.5 / 448.0, 0.0371])
def test_exhaustive_bf16_matches_torch_cast(oracle_lib, scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_lib.quantize(bits, np.float32(scale))
    ref = _torch_quantize(bits, np.float32(scale))
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN keeps its sign and maps to the NaN code (reading: saturating cvt)
    assert set(ours[nan & (np.signbit(x))]) == {0xFF}
    assert set(ours[nan & (~np.signbit(x))]) == {0x7F}


def test_infinity_saturates(oracle_lib):
    assert oracle_lib.e4m3_encode(float("inf")) == 0x7E
    assert oracle_lib.e4m3_encode(float("-inf")) == 0xFE
    assert oracle_lib.e4m3_encode(1e30) == 0x7E


def test_rounding_is_nearest_even_not_truncation(oracle_lib):
    # 1.0625 is halfway between 1.0 (0x38) and 1.125 (0x39): ties go to even
    assert oracle_lib.e4m3_encode(1.0625) == 0x38
    assert oracle_lib.e4m3_encode(1.1875) == 0x3A        # halfway 1.125/1.25 -> even
    assert oracle_lib.e4m3_encode(1.07) == 0x39           # above the midpoint
    assert oracle_lib.e4m3_encode(2.0 ** -10) == 0x00      # halfway 0 / 2^-9 -> 0
    assert oracle_lib.e4m3_encode(1.5 * 2.0 ** -9) == 0x02  # halfway 1/2 subnormal -> even
    assert oracle_lib.e4m3_encode(-1e-6) == 0x80


# ----------------------------------------------------------------- pages' values
def test_v_outlier_clips_at_unity_but_not_at_scale_three(oracle_lib):
    pv = pages_values()
    vmax = bf16_bits_of([pv["v_max_abs"], -pv["v_max_abs"]])
    at1 = oracle_lib.quantize(vmax, pv["v_clips_at_scale"])
    at3 = oracle_lib.quantize(vmax, pv["v_no_clip_at_scale"])
    assert list(at1) == [0x7E, 0xFE]                   # saturated to +-448
    assert oracle_lib.e4m3_decode(int(at1[0])) == pv["e4m3_max"]
    # 1272/3 = 424 rounds to 416, strictly inside the range: not clipped
    assert list(at3) == [0x7D, 0xFD]
    assert oracle_lib.e4m3_decode(int(at3[0])) < pv["e4m3_max"]


def test_safety_rule_scale_of_the_1272_outlier(oracle_lib):
    pv = pages_values()
    s = oracle_lib.scale_from_amax(pv["v_max_abs"], rule=2)
    assert abs(s - pv["rule_safety_scale_of_1272"]) < 0.005
    # the rule never goes below 1 (K, whose amax is far below 448/1.3)
    assert oracle_lib.scale_from_amax(73.5, rule=2) == 1.0


def test_amax_over_448_maps_amax_onto_448(oracle_lib):
    rng = np.random.default_rng(7)
    for a in list(rng.uniform(0.01, 3000.0, 200)) + [11.6, 23.1, 14.9, 114.6, 1272.0]:
        a_bits = bf16_bits_of([a])
        a_val = float(torch.from_numpy(a_bits.view(np.int16).copy()).view(torch.bfloat16).float())
        s = oracle_lib.scale_from_amax(a_val, rule=0)
        assert oracle_lib.quantize(a_bits, s)[0] == 0x7E


def test_ceil_to_bf16_rule_is_smallest_bf16_not_below(oracle_lib):
    for a in [1272.0, 114.6, 23.1, 11.6, 0.37, 55.8]:
        s = oracle_lib.scale_from_amax(a, rule=1)
        plain = np.float32(np.float32(a) / np.float32(448.0))
        bits = np.array([s], dtype=np.float32).view(np.uint32)[0]
        assert bits & 0xFFFF == 0                          # a bf16 value
        assert s >= plain
        below = np.array([bits - 0x10000], dtype=np.uint32).view(np.float32)[0]
        assert below < plain


def test_invalid_scales_rejected(oracle_lib):
    for a in [0.0, float("nan"), float("inf"), -1.0]:
        with pytest.raises(ValueError):
            oracle_lib.scale_from_amax(a, rule=0)


def test_round_trip_error_matches_tier2_statistic(oracle_lib):
    """Mean relative round-trip error of e4m3 at unity scale on heavy-tailed
    V is 2.3-2.6% on the pages' activations; a 3-bit-mantissa nearest
    rounding gives ~2.2-2.4% on these synthetic stand-ins, truncation ~4.5%."""
    pv = pages_values()
    g = torch.Generator().manual_seed(3)
    for dist in ("v_t3", "normal"):
        x = workloads.draw_values((400_000,), dist, g, "cpu")
        q = oracle_lib.quantize(workloads.bf16_bits(x), 1.0)
        xd = x.double().numpy()
        dq = oracle_lib.decode_array(q)
        nz = (xd != 0) & (np.abs(xd) <= 448)
        err = float(np.mean(np.abs(dq[nz] - xd[nz]) / np.abs(xd[nz])))
        assert pv["rt_err_lo"] - 0.003 <= err <= pv["rt_err_hi"] + 0.002, (dist, err)


# ----------------------------------------------------------------- band counters
def test_band_counts_hand_cases(oracle_lib):
    """Every band by hand at unity scale: 1000 and 450 clip (to 448), 2^-11 and
    2^-10 flush (the latter a tie to the even code 0), 2^-9 is the smallest
    subnormal, 1.0625 is a tie between 1 and 1.125 going to the even code 1.0;
    zeros are counted but have no error term; Inf and NaN are not counted."""
    vals = [1000.0, -1000.0, 448.0, 450.0, 2.0 ** -11, 2.0 ** -10, 2.0 ** -9, 1.0625, 0.0,
            -0.0, 3.0, float("inf"), float("nan")]
    got = oracle_lib.band_counts(bf16_bits_of(vals).reshape(1, -1), 1.0)
    assert (got["count"], got["nonzero"], got["clipped"], got["flushed"]) == (11, 9, 3, 2)
    want_err = 2 * (1000 - 448) / 1000 + 2 / 450 + 2 * 1.0 + 0.0625 / 1.0625
    assert abs(got["rt_err_sum"] - want_err) < 1e-12
    # at scale 3 nothing clips (1000/3, 450/3 < 448) and 2^-9/3 < 2^-10 flushes too
    got3 = oracle_lib.band_counts(bf16_bits_of(vals).reshape(1, -1), 3.0)
    assert (got3["clipped"], got3["flushed"]) == (0, 3)


def test_band_counts_skip_unstored_tokens(oracle_lib):
    g = torch.Generator().manual_seed(11)
    x = workloads.bf16_bits(workloads.draw_values((50, 64), "v_t3", g, "cpu"))
    slots = np.where(np.arange(50) % 3 == 0, -1, np.arange(50)).astype(np.int64)
    a = oracle_lib.band_counts(x, 1.0, slot_mapping=slots)
    b = oracle_lib.band_counts(x[slots >= 0], 1.0)
    assert a == b
    assert a["count"] == int((slots >= 0).sum()) * 64


def test_band_counts_flush_band_grows_with_the_scale(oracle_lib):
    """Values flush when |x|/s <= 2^-10, so for N(0,1) the flushed fraction is
    ~2*phi(0)*2^-10*s, and the band at s = 3 is ~3x the band at s = 1 (the
    pages report ~3x on real activations)."""
    pv = pages_values()
    g = torch.Generator().manual_seed(5)
    x = workloads.bf16_bits(workloads.draw_values((4_000_000,), "normal", g, "cpu"))
    f1 = oracle_lib.band_counts(x.reshape(1, -1), 1.0)["flushed"]
    f3 = oracle_lib.band_counts(x.reshape(1, -1), 3.0)["flushed"]
    expect1 = 4_000_000 * 2 * (1 / math.sqrt(2 * math.pi)) * 2.0 ** -10
    assert abs(f1 - expect1) < 0.1 * expect1, (f1, expect1)
    assert abs(f3 / f1 - pv["flush_growth_s3"]) < 0.3, f3 / f1


def test_band_counts_clip_rate_matches_the_t3_tail(oracle_lib):
    """The synthetic global-layer V is 17.47*t(3) (clamped to +-1272): at unity
    scale it clips where |t| > 448/17.47, the two-sided t(3) tail, which is
    of the order the pages measure (1.3e-4 pooled); at scale 3 nothing clips."""
    stats = pytest.importorskip("scipy.stats")
    pv = pages_values()
    g = torch.Generator().manual_seed(9)
    n = 4_000_000
    x = workloads.bf16_bits(workloads.draw_values((n,), "v_t3", g, "cpu")).reshape(1, -1)
    c1 = oracle_lib.band_counts(x, 1.0)
    tail = 2 * stats.t.sf(448.0 / workloads.V_T3_SCALE, 3)
    assert abs(c1["clipped"] / n - tail) < 0.15 * tail, (c1["clipped"] / n, tail)
    assert pv["v_clip_rate_s1_global"] / 2.5 < c1["clipped"] / n < pv["v_clip_rate_s1_global"] * 2.5
    c3 = oracle_lib.band_counts(x, pv["v_no_clip_at_scale"])
    assert c3["clipped"] == 0
    rt = c1["rt_err_sum"] / c1["nonzero"]
    assert pv["rt_err_lo"] - 0.003 <= rt <= pv["rt_err_hi"] + 0.003, rt


def test_rescale_bound_constant():
    pv = pages_values()
    assert abs((math.log2(pv["e4m3_max"]) - 8) - pv["rescale_slack_bound"]) < 5e-4
    assert pv["rescale_threshold_fp8"] < pv["rescale_slack_bound"]
    assert 2.0 ** (8 + pv["rescale_threshold_fp8"]) < pv["e4m3_max"]


def test_cache_byte_figures():
    pv = pages_values()
    heads_per_rank = pv["kv_heads_total"] / pv["tp"]
    per_layer_bf16 = 2 * heads_per_rank * pv["head_dim"] * 2      # K and V, 2 bytes
    assert pv["full_layers"] * per_layer_bf16 == pv["bytes_per_token_rank_bf16"]
    assert pv["full_layers"] * per_layer_bf16 / 2 == pv["bytes_per_token_rank_fp8"]


# ----------------------------------------------------------------- store / amax
def test_paged_store_round_trips_through_block_table(oracle_lib):
    g = torch.Generator().manual_seed(11)
    lens = [37, 16, 1, 70]
    kv = workloads.make_paged_kv(lens, 2, 128, 16, g=g, device="cpu", v_dist="v_t3")
    nb = kv.num_blocks
    ck = np.full((nb, 2, 16, 128), 0xA5, dtype=np.uint8)      # canary, [block][head][row][d]
    cv = np.full((nb, 2, 16, 128), 0xA5, dtype=np.uint8)
    sm = kv.slot_mapping.numpy().copy()
    sm[5] = -1                                                # one skipped token
    oracle_lib.kv_store(ck, cv, workloads.bf16_bits(kv.k), workloads.bf16_bits(kv.v), sm,
                        1.0, 3.0, 16)
    bt = kv.block_table.numpy()
    kq = oracle_lib.quantize(workloads.bf16_bits(kv.k), 1.0)
    vq = oracle_lib.quantize(workloads.bf16_bits(kv.v), 3.0)
    touched = np.zeros((nb, 2, 16), dtype=bool)
    t = 0
    for b, L in enumerate(lens):
        for p in range(L):
            blk, off = bt[b, p // 16], p % 16
            if t == 5:
                assert (ck[blk, :, off] == 0xA5).all()
            else:
                assert np.array_equal(ck[blk, :, off], kq[t]) and np.array_equal(cv[blk, :, off], vq[t])
                touched[blk, :, off] = True
            t += 1
    assert (ck[~touched] == 0xA5).all() and (cv[~touched] == 0xA5).all()


def test_amax_counts_only_stored_tokens(oracle_lib):
    x = bf16_bits_of([[1.0, -5.0], [100.0, 2.0], [-7.5, 0.0]])
    assert oracle_lib.amax(x) == 100.0
    assert oracle_lib.amax(x, slot_mapping=np.array([0, -1, 3])) == 7.5
    assert oracle_lib.amax(x, slot_mapping=np.array([-1, -1, -1]), amax_in=2.5) == 2.5
    assert oracle_lib.amax(x, amax_in=200.0) == 200.0


# ----------------------------------------------------------------- attention
def _rand_e4m3(rng, shape, lo=-4.0, hi=4.0):
    vals = rng.uniform(lo, hi, shape).astype(np.float32)
    return oracle_lib_encode(vals)


def oracle_lib_encode(vals):
    import oracle
    return oracle.encode_f32(vals).reshape(np.shape(vals))


def test_single_key_returns_scaled_value_exactly(oracle_lib):
    rng = np.random.default_rng(0)
    q8 = _rand_e4m3(rng, (128,))
    k8 = _rand_e4m3(rng, (1, 128))
    v8 = _rand_e4m3(rng, (1, 128))
    out = oracle_lib.attend_row(q8, k8, v8, 0, 0.088, 0.5, 0.5, 1.5,
                                bias=bf16_bits_of([3.0] * 16))
    assert np.array_equal(out, 1.5 * oracle_lib.decode_array(v8[0]))


def test_visible_sets_match_hand_enumeration(oracle_lib):
    """Constant keys and zero bias make the weights uniform over the visible
    keys; one-hot values then read the visible set straight off the output."""
    q8 = np.full(64, 0x38, dtype=np.uint8)                # q = 1
    for len_k, pos, window, vis in read_table("mask_visible.txt"):
        len_k, pos, window = int(len_k), int(pos), int(window)
        expect = sorted(int(j) for j in vis.split(","))
        k8 = np.full((len_k, 64), 0x38, dtype=np.uint8)
        v8 = np.zeros((len_k, 64), dtype=np.uint8)
        for j in range(len_k):
            v8[j, j] = 0x38                               # one-hot value of key j
        out = oracle_lib.attend_row(q8, k8, v8, pos, 0.1, 1.0, 1.0, 1.0, window=window)
        got = [j for j in range(64) if out[j] > 0]
        assert got == expect, (len_k, pos, window)
        assert np.allclose(out[got], 1.0 / len(expect), rtol=1e-14)


def test_bias_indexed_by_distance_back_from_the_query(oracle_lib):
    """A large bias at one distance d puts all weight on key pos_q - d."""
    len_k, pos = 30, 25
    q8 = np.full(64, 0x38, dtype=np.uint8)
    k8 = np.full((len_k, 64), 0x38, dtype=np.uint8)
    rng = np.random.default_rng(5)
    v8 = _rand_e4m3(rng, (len_k, 64))
    for d in (0, 1, 7, 19):
        bias = np.zeros(20, dtype=np.float32)
        bias[d] = 80.0
        out = oracle_lib.attend_row(q8, k8, v8, pos, 0.1, 1.0, 1.0, 2.0,
                                    bias=bf16_bits_of(bias))
        assert np.allclose(out, 2.0 * oracle_lib.decode_array(v8[pos - d]), rtol=1e-12, atol=1e-30)


def test_bias_is_zero_beyond_the_extent(oracle_lib):
    """Bias +80 on every distance < E: the weight sits on the last E keys,
    uniformly (constant keys); keys at distance >= E get bias 0."""
    len_k, pos, E = 50, 49, 8
    q8 = np.full(64, 0x38, dtype=np.uint8)
    k8 = np.full((len_k, 64), 0x38, dtype=np.uint8)
    rng = np.random.default_rng(6)
    v8 = _rand_e4m3(rng, (len_k, 64))
    out = oracle_lib.attend_row(q8, k8, v8, pos, 0.1, 1.0, 1.0, 1.0,
                                bias=bf16_bits_of([80.0] * E))
    expect = oracle_lib.decode_array(v8[pos - E + 1:pos + 1]).mean(axis=0)
    assert np.allclose(out, expect, rtol=1e-12, atol=1e-30)


def test_zero_bias_full_window_is_textbook_softmax_attention(oracle_lib):
    from scipy.special import softmax
    rng = np.random.default_rng(8)
    D, L = 128, 300
    sq, sk, sv, sigma = 0.5, 0.75, 1.5, 1 / math.sqrt(128)
    q8 = _rand_e4m3(rng, (D,))
    k8 = _rand_e4m3(rng, (L, D))
    v8 = _rand_e4m3(rng, (L, D))
    Q = sq * oracle_lib.decode_array(q8)
    K = sk * oracle_lib.decode_array(k8)
    V = sv * oracle_lib.decode_array(v8)
    ref = softmax(sigma * (K @ Q)) @ V
    out = oracle_lib.attend_row(q8, k8, v8, L - 1, sigma, sq, sk, sv)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    # the query's position limits the keys (causal): pos 99 sees keys 0..99
    ref99 = softmax(sigma * (K[:100] @ Q)) @ V[:100]
    out99 = oracle_lib.attend_row(q8, k8, v8, 99, sigma, sq, sk, sv)
    assert np.allclose(out99, ref99, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------- per-token scales
def test_per_token_scale_maps_each_row_max_onto_448(oracle_lib):
    """With s = max|x|/448 per row, every row's largest element encodes to
    +-448 (0x7E / 0xFE), the scale is the fp32 quotient, a zero row gets 1 and
    non-finite elements do not enter the max."""
    g = torch.Generator().manual_seed(31)
    x = workloads.draw_values((64, 128), "v_t3", g, "cpu")
    x[5] = 0.0
    x[7, 3] = float("inf")
    x[9, 0] = float("nan")
    bits = workloads.bf16_bits(x)
    codes, scales = oracle_lib.quantize_per_token(bits, 128)
    xf = x.float().numpy()
    for r in range(64):
        fin = np.isfinite(xf[r])
        amax = float(np.abs(xf[r][fin]).max())
        if amax == 0.0:
            assert scales[r] == 1.0 and (codes[r] & 0x7F == 0).all()
            continue
        assert scales[r] == np.float32(np.float32(amax) / np.float32(448.0))
        i = int(np.argmax(np.where(fin, np.abs(xf[r]), -1.0)))
        assert codes[r, i] & 0x7F == 0x7E, r
    assert codes[7, 3] == 0x7E          # +inf saturates at its row's scale


def test_per_token_attention_with_equal_scales_is_the_per_tensor_oracle(oracle_lib):
    rng = np.random.default_rng(32)
    D, L = 128, 200
    q8, k8, v8 = _rand_e4m3(rng, (D,)), _rand_e4m3(rng, (L, D)), _rand_e4m3(rng, (L, D))
    sk = np.full(L, 0.75, dtype=np.float32)
    sv = np.full(L, 1.5, dtype=np.float32)
    bias = bf16_bits_of(list(rng.normal(0, 0.5, 64)))
    for pos, w in ((L - 1, 0), (150, 40)):
        a = oracle_lib.attend_row_pt(q8, k8, v8, sk, sv, pos, 0.09, 0.5, bias=bias, window=w)
        b = oracle_lib.attend_row(q8, k8, v8, pos, 0.09, 0.5, 0.75, 1.5, bias=bias, window=w,
                                  form=5)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_per_token_attention_is_textbook_attention_on_dequantized_keys(oracle_lib):
    from scipy.special import softmax
    rng = np.random.default_rng(33)
    D, L = 128, 90
    q8, k8, v8 = _rand_e4m3(rng, (D,)), _rand_e4m3(rng, (L, D)), _rand_e4m3(rng, (L, D))
    sk = rng.uniform(0.01, 5.0, L).astype(np.float32)
    sv = rng.uniform(0.01, 5.0, L).astype(np.float32)
    Q = 0.5 * oracle_lib.decode_array(q8)
    K = sk.astype(np.float64)[:, None] * oracle_lib.decode_array(k8)
    V = sv.astype(np.float64)[:, None] * oracle_lib.decode_array(v8)
    ref = softmax(0.1 * (K @ Q)) @ V
    out = oracle_lib.attend_row_pt(q8, k8, v8, sk, sv, L - 1, 0.1, 0.5)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_descale_fold_equals_dequantize_then_attend(oracle_lib):
    rng = np.random.default_rng(9)
    D, L = 128, 97
    q8 = _rand_e4m3(rng, (D,), -400, 400)
    k8 = _rand_e4m3(rng, (L, D), -400, 400)
    v8 = _rand_e4m3(rng, (L, D), -400, 400)
    bias = bf16_bits_of(rng.normal(0, 0.5, 64))
    for (sq, sk, sv) in [(1.0, 1.0, 1.0), (0.5, 0.5, 1.5), (0.0371, 0.05, 3.0)]:
        a = oracle_lib.attend_row(q8, k8, v8, 80, 1 / math.sqrt(D), sq, sk, sv, bias=bias,
                                  window=50, form=4)
        b = oracle_lib.attend_row(q8, k8, v8, 80, 1 / math.sqrt(D), sq, sk, sv, bias=bias,
                                  window=50, form=5)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12 * np.abs(b).max())


def test_window_at_least_context_equals_full(oracle_lib):
    rng = np.random.default_rng(10)
    q8 = _rand_e4m3(rng, (128,))
    k8 = _rand_e4m3(rng, (40, 128))
    v8 = _rand_e4m3(rng, (40, 128))
    full = oracle_lib.attend_row(q8, k8, v8, 39, 0.1, 1, 1, 1, window=0)
    for w in (40, 41, 512):
        assert np.array_equal(full, oracle_lib.attend_row(q8, k8, v8, 39, 0.1, 1, 1, 1, window=w))
    assert not np.array_equal(full, oracle_lib.attend_row(q8, k8, v8, 39, 0.1, 1, 1, 1, window=39))


def test_no_visible_key_gives_zeros(oracle_lib):
    q8 = np.full(128, 0x38, dtype=np.uint8)
    k8 = np.zeros((0, 128), dtype=np.uint8)
    out = oracle_lib.attend_row(q8, k8, k8, 0, 0.1, 1, 1, 1)
    assert np.array_equal(out, np.zeros(128))


def test_rows_batch_equals_single_rows(oracle_lib):
    rng = np.random.default_rng(12)
    D, L, H = 128, 33, 3
    k8 = _rand_e4m3(rng, (L, H, D))
    v8 = _rand_e4m3(rng, (L, H, D))
    q8 = _rand_e4m3(rng, (2, H, D))
    rows = [(0, 0, 32), (1, 2, 10), (0, 1, 0)]
    out = oracle_lib.attend_rows(D, q8, [i * H * D + h * D for i, h, _ in rows], k8, v8,
                                 [h * D for _, h, _ in rows], H * D, [L] * 3,
                                 [p for *_, p in rows], 0.1, 1, 1, 1)
    for r, (i, h, p) in enumerate(rows):
        ref = oracle_lib.attend_row(q8[i, h], k8[:, h], v8[:, h], p, 0.1, 1, 1, 1)
        assert np.array_equal(out[r], ref)
