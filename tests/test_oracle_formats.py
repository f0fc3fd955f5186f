"""Pins for the oracle's number formats (CPU only).

Each test checks the oracle against something other than itself: the OCP
bit-field definitions, torch's float8_e4m3fn conversions, hand-worked golden
groups, brute-force nearest-point searches and exhaustive sweeps.
"""
import os

import numpy as np
import pytest
import torch

from oracle import csa2_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_has_16_code_points_matching_bitfields():
    codes = np.arange(16)
    vals = O.e2m1_decode(codes)
    # OCP E2M1 from its bit fields: s e1 e0 m, bias 1, e == 0 subnormal
    ref = []
    for c in codes:
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        ref.append(-mag if s else mag)
    assert np.array_equal(vals, np.array(ref))
    assert len(codes) == 16
    assert set(np.abs(vals)) == {0, 0.5, 1, 1.5, 2, 3, 4, 6}
    assert len(set(vals.tolist())) == 15  # +0 and -0 compare equal
    assert np.signbit(vals[8]) and not np.signbit(vals[0])


def test_e4m3_decode_all_bytes_matches_torch():
    b = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_decode(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(1)
    vals = O.e4m3_decode(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2  # every tie point
    x = np.concatenate([
        rng.normal(0, 30, 200000), rng.uniform(-448, 448, 100000),
        rng.normal(0, 1e-3, 50000), mids, -mids, vals, -vals,
        np.nextafter(mids, 0), np.nextafter(mids, 1e9)])
    x = x[np.abs(x) <= 448].astype(np.float32)
    ours = O.e4m3_encode(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, (x[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_golden_and_saturation():
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for v, byte in rows:
        got = int(O.e4m3_encode(float(v)))
        assert got == int(byte, 16), (v, hex(got), byte)


def _golden_groups():
    out = []
    with open(os.path.join(GOLDEN, "fp4_groups.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            xs, sb, cs = line.split("|")
            x = np.array([float(t) for t in xs.split()])
            assert x.size == 16
            out.append((x, int(sb, 16), np.array([int(t, 16) for t in cs.split()])))
    return out


@pytest.mark.parametrize("case", range(9))
def test_fp4_golden_groups(case):
    groups = _golden_groups()
    assert len(groups) == 9
    x, sbyte, codes = groups[case]
    got_codes, got_scale = O.quantize_fp4(x[None, :])
    assert int(got_scale[0, 0]) == sbyte
    assert np.array_equal(got_codes[0], codes), (got_codes[0], codes)


def test_fp4_nearest_point_brute_force():
    """For groups whose scale does not saturate, every element's code is a
    nearest of the 16 E2M1 points times s (brute force), ties to the even
    code, and s is the nearest E4M3 value to amax/6 (brute force)."""
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, (4000, 16)) * np.exp(rng.uniform(-8, 8, (4000, 1)))
    codes, scales = O.quantize_fp4(x)
    s = O.e4m3_decode(scales)[:, 0]
    allv = O.e4m3_decode(np.arange(0x7F))
    amax = np.abs(x).max(axis=1)
    for i in range(x.shape[0]):
        d = np.abs(allv - amax[i] / 6)
        best = np.nonzero(d == d.min())[0]
        want = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
        assert scales[i, 0] == want
        if s[i] == 0:
            assert np.all(codes[i] == 0)
            continue
        pts = O.e2m1_decode(np.arange(16)) * s[i]
        for j in range(16):
            if abs(x[i, j]) / s[i] > 6:
                assert codes[i, j] & 7 == 7
                continue
            dist = np.abs(pts - x[i, j])
            got = dist[codes[i, j]]
            assert got == dist.min()


def test_fp4_ties_go_to_even_code():
    s = 0.75  # an E4M3 value (0x34)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    x = np.zeros((7, 16))
    x[:, 0] = 6 * s   # amax sets s exactly
    x[:, 1] = mids * s
    codes, scales = O.quantize_fp4(x)
    assert O.e4m3_decode(scales[0, 0]) == s
    assert list(codes[:, 1]) == [0, 2, 2, 4, 4, 6, 6]


def test_scale_quotient_fp32_equals_fp64_for_all_bf16():
    """Every positive finite bf16 amax gives the same E4M3 scale whether
    amax/6 is formed in fp32 (correctly rounded) or fp64: the device's fp32
    quotient cannot land on an E4M3 tie it should not."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16
    a = bits.view(np.float32)
    q32 = (a / np.float32(6)).astype(np.float64)
    q64 = a.astype(np.float64) / 6.0
    assert np.array_equal(O.e4m3_encode(q32), O.e4m3_encode(q64))


def test_pack_low_nibble_is_even_channel():
    codes = np.array([[1, 2, 15, 8]])
    packed = O.pack_codes(codes)
    assert packed.tolist() == [[0x21, 0x8F]]
    assert np.array_equal(O.unpack_codes(packed), codes)


def test_dequantize_roundtrip_is_exact_on_representable_values():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, (100, 64))
    scales = rng.integers(0x01, 0x7F, (100, 4)).astype(np.uint8)
    v = O.dequantize_fp4(codes, scales)
    # re-quantizing exactly representable data (with amax in the group mapping
    # back to the same scale) returns the same values
    c2, s2 = O.quantize_fp4(v)
    v2 = O.dequantize_fp4(c2, s2)
    same_scale = (s2 == scales)
    g = np.repeat(same_scale, 16, axis=1)
    assert np.array_equal(v[g], v2[g])


def test_dequantize_fp4_hand_values_one_scale_per_16_channels():
    """Hand-computed products: channel c takes code c's E2M1 value times the
    E4M3 scale of group c // 16.  The groups carry different scales (0.5 and
    6.0; 448 and the subnormal 3 * 2^-9), so a scale applied to the wrong
    channels, a dropped sign or a mis-decoded scale changes the values."""
    codes = np.array([
        list(range(16)) + [7, 6, 5, 4, 3, 2, 1, 0, 15, 14, 13, 12, 11, 10, 9, 8],
        [7, 7, 7, 1] + [7] * 12 + [7, 9] + [0] * 14,
    ])
    scales = np.array([[0x30, 0x4C], [0x7E, 0x03]], dtype=np.uint8)  # 0.5, 6.0; 448, 3/512
    expect = np.array([
        [0, 0.25, 0.5, 0.75, 1, 1.5, 2, 3, -0.0, -0.25, -0.5, -0.75, -1, -1.5, -2, -3,
         36, 24, 18, 12, 9, 6, 3, 0, -36, -24, -18, -12, -9, -6, -3, -0.0],
        [2688, 2688, 2688, 224] + [2688] * 12 + [0.03515625, -0.0029296875] + [0] * 14,
    ])
    got = O.dequantize_fp4(codes, scales)
    assert np.array_equal(got, expect)
    assert np.array_equal(np.signbit(got), np.signbit(expect))  # code 8 is -0


def test_strict_selection_check_catches_ties_broken_upward():
    """The strict set check used on tie-heavy GPU inputs is not vacuous: a
    selection that breaks ties toward the higher index passes the tolerant
    check (the differing members score exactly the K-th value) but fails the
    strict one."""
    from tests.helpers import check_selection, kth_value
    vals = np.array([5.0, 3.0, 3.0, 3.0, 1.0, 3.0])
    good = O.select_top(vals, 3)                    # 0, 1, 2
    order = np.lexsort((-np.arange(vals.size), -vals))  # ties toward the higher index
    upward = np.sort(order[:3])                     # 0, 3, 5
    assert good.tolist() == [0, 1, 2] and upward.tolist() == [0, 3, 5]
    kth = kth_value(vals, 3)
    check_selection(upward, good, lambda p: vals[p], kth, "tolerant")
    with pytest.raises(AssertionError):
        check_selection(upward, good, lambda p: vals[p], kth, "strict", strict=True)
    check_selection(good, good, lambda p: vals[p], kth, "strict", strict=True)
