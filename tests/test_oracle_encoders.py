"""Pins of the oracle's number formats and its per-128-channel FP8 quantisation.

E4M3 (OCP FP8, "fn" variant: bias 7, max 448, no infinities) is checked
against an independent formulation: decode the 127 non-negative finite codes,
then pick the nearest one (ties to the even code), saturating at 448. BF16 is
checked against PyTorch's float32 -> bfloat16 cast (round to nearest even).
Quantisation follows the DeepEP V1 guide, section 5.2(6) (FP8 data plus float
scales of shape [tokens, hidden/128]); the reading s = amax/448 is checked by
its consequences: each block's largest magnitude maps to the code for 448,
and every element is within half an E4M3 step of x/s.
"""
import numpy as np
import pytest
import torch

import epinputs as ei
import oracle

CODES = np.arange(256, dtype=np.uint8)


def _decode_table():
    """E4M3 code -> value, from the bit fields (independent of the oracle)."""
    v = np.empty(256)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        f, m = (c >> 3) & 15, c & 7
        if f == 15 and m == 7:
            v[c] = np.nan
        elif f == 0:
            v[c] = s * m * 2.0 ** -9
        else:
            v[c] = s * (1 + m / 8) * 2.0 ** (f - 7)
    return v


DEC = _decode_table()
POS = DEC[:127]  # codes 0x00..0x7E: 0 .. 448, strictly increasing


def nearest_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code by search, ties to the even code, saturating."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(POS, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo, dhi = a - POS[lo], POS[hi] - a
    pick = np.where(dhi < dlo, hi, lo)
    tie = (dhi == dlo) & (hi != lo)
    pick = np.where(tie, np.where(hi % 2 == 0, hi, lo), pick)
    pick = np.where(a == POS[hi], hi, pick)
    return (pick | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def test_decode_matches_oracle_decoder():
    got = oracle.e4m3_to_f64(CODES)
    same = (got == DEC) | (np.isnan(got) & np.isnan(DEC))
    assert same.all()
    assert DEC[0x7E] == 448.0 and DEC[0x01] == 2.0 ** -9 and DEC[0x08] == 2.0 ** -6


def test_all_codes_round_trip():
    vals = DEC.astype(np.float32)
    enc = oracle.e4m3_from_f32(vals)
    nan = np.isnan(DEC)
    assert np.array_equal(enc[~nan], CODES[~nan])
    assert np.all(enc[nan] == 0x7F)


def test_midpoints_and_neighbours():
    lo, hi = POS[:-1], POS[1:]
    mid = (lo + hi) / 2  # exact in float32: codes have at most 4 significant bits
    m32 = mid.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mid)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(0))
    xs = np.concatenate([m32, up, dn, -m32, -up, -dn])
    assert np.array_equal(oracle.e4m3_from_f32(xs), nearest_e4m3(xs))
    # ties go to the even code, explicitly
    codes = oracle.e4m3_from_f32(m32)
    assert np.all(codes % 2 == 0)


def test_special_values():
    f = np.array([0.0, -0.0, 448.0, 449.0, 463.99, 464.0, 1e30, np.inf, -np.inf,
                  2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -11, -1e-30, np.nan], np.float32)
    got = oracle.e4m3_from_f32(f).tolist()
    assert got == [0x00, 0x80, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE,
                   0x01, 0x00, 0x02, 0x00, 0x80, 0x7F]


def test_random_against_nearest_search():
    rng_key = ei.stream_key(7, 99)
    u = ei.splitmix64(rng_key, 1 << 21)
    # random sign, exponent in [-16, 10], random mantissa bits
    e = (u % np.uint64(27)).astype(np.int64) - 16
    m = ((u >> np.uint64(8)) & np.uint64(0x7FFFFF)).astype(np.uint32)
    s = ((u >> np.uint64(40)) & np.uint64(1)).astype(np.uint32)
    bits = (s << np.uint32(31)) | ((e + 127).astype(np.uint32) << np.uint32(23)) | m
    f = bits.view(np.float32)
    assert np.array_equal(oracle.e4m3_from_f32(f), nearest_e4m3(f))


def test_bf16_against_torch_cast():
    upper = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    bits = (upper[:, None] | lows[None, :]).reshape(-1)
    u = ei.splitmix64(ei.stream_key(1, 77), 1 << 20).astype(np.uint32)
    bits = np.concatenate([bits, u])
    f = bits.view(np.float32)
    got = oracle.bf16_from_f32(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    # NaN stays NaN (quiet), sign kept
    g = got[nan]
    assert np.all((g & 0x7F80) == 0x7F80) and np.all(g & 0x0040)


def test_quantize_rows_bounds():
    x = ei.make_x(64, 1024, seed=11)
    q, s = oracle.quantize_rows(x)
    xf = oracle.f32_from_bf16(x).astype(np.float64).reshape(64, 8, 128)
    dq = DEC[q].reshape(64, 8, 128)
    s64 = s.astype(np.float64)[:, :, None]
    amax = np.abs(xf).max(axis=2)
    assert np.all(amax > 0)
    # s = amax/448 rounded once to fp32
    assert np.all(np.abs(s.astype(np.float64) * 448.0 - amax) <= amax * 2.0 ** -23)
    # the largest magnitude of each block encodes to +-448
    assert np.all(np.abs(dq).max(axis=2) == 448.0)
    # every element: |dequant - x/s| <= half an E4M3 step at x/s (+ the fp32 division rounding)
    v = xf / s64
    step = 2.0 ** (np.maximum(np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -10))), -6) - 3)
    assert np.all(np.abs(dq - v) <= 0.5 * step + np.abs(v) * 2.0 ** -23)
    # equality with the element-wise encoder on x / s in fp32
    v32 = (oracle.f32_from_bf16(x).reshape(64, 8, 128) / s[:, :, None]).astype(np.float32)
    assert np.array_equal(q.reshape(64, 8, 128), nearest_e4m3(v32))


def test_quantize_zero_block_keeps_signed_zeros():
    x = np.zeros((1, 256), np.uint16)
    x[0, 3] = 0x8000  # -0.0 in block 0; block 1 stays all +0
    x[0, 200] = 0x3F80  # 1.0 in block 1
    q, s = oracle.quantize_rows(x)
    assert s[0, 0] == 0.0
    assert q[0, 3] == 0x80 and np.all(np.delete(q[0, :128], 3) == 0)
    assert s[0, 1] == np.float32(1.0) / np.float32(448.0)
    assert q[0, 200] == 0x7E


def test_round_scale_is_the_smallest_power_of_two_not_below_amax_over_448():
    # "DeepEP V1 guide" 6.3: round_scale rounds the scales to powers of two.
    x = ei.make_x(64, 1024, seed=12)
    q, s = oracle.quantize_rows(x, round_scale=True)
    xf = oracle.f32_from_bf16(x).astype(np.float64).reshape(64, 8, 128)
    amax = np.abs(xf).max(axis=2)
    s64 = s.astype(np.float64)
    m, e = np.frexp(s64)
    assert np.all(m == 0.5)                       # powers of two
    raw = (amax.astype(np.float32) / np.float32(448.0)).astype(np.float64)
    assert np.all(s64 >= raw) and np.all(s64 / 2 < raw)
    # nothing saturates: |x / s| <= 448, and the block max lands in the top binade
    dq = DEC[q].reshape(64, 8, 128)
    assert np.all(np.abs(dq).max(axis=2) <= 448.0) and np.all(np.abs(dq).max(axis=2) > 224.0 - 1e-9)
    v32 = (oracle.f32_from_bf16(x).reshape(64, 8, 128) / s[:, :, None]).astype(np.float32)
    assert np.array_equal(q.reshape(64, 8, 128), nearest_e4m3(v32))


def test_ue8m0_bytes_decode_to_the_scale_and_clamp_tiny_blocks():
    x = ei.make_x(16, 512, seed=13)
    q, s = oracle.quantize_rows(x, ue8m0=True)
    b = oracle.ue8m0_from_scales(s)
    assert np.array_equal(np.ldexp(1.0, b.astype(np.int64) - 127), s.astype(np.float64))
    q2, s2 = oracle.quantize_rows(x, round_scale=True)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)   # normal blocks: same as round_scale
    # a block whose amax is a BF16 subnormal: the power-of-two scale is below
    # 2^-127, so UE8M0 clamps it to 2^-127 (byte 0)
    tiny = np.zeros((1, 128), np.uint16)
    tiny[0, 5] = 0x0001                      # 2^-133
    q, s = oracle.quantize_rows(tiny, ue8m0=True)
    assert s[0, 0] == np.float32(2.0 ** -127) and oracle.ue8m0_from_scales(s)[0, 0] == 0
    assert q[0, 5] == 0x08 and np.all(np.delete(q[0], 5) == 0)   # 2^-133 / 2^-127 = 2^-6
    q, s = oracle.quantize_rows(tiny, round_scale=True)
    assert s[0, 0] < 2.0 ** -127
    assert oracle.ue8m0_from_scales(np.zeros(3, np.float32)).tolist() == [0, 0, 0]


def test_quantisation_divides_by_the_scale():
    # The reading q = e4m3(x / s) with one IEEE fp32 division ("DeepEP V1
    # guide" 5.2(6) gives only the scale's shape). For these BF16 (x, amax)
    # pairs, found by a numpy search, multiplying by fl(1/s) or by
    # fl(448/amax) instead lands on a neighbouring code, so this pins the
    # division itself.
    for x_bits, amax_bits in [(0x3C2F, 0x3CC4), (0x3C1C, 0x3D50), (0x3C3A, 0x3DF8)]:
        row = np.zeros((1, 128), np.uint16)
        row[0, 0], row[0, 1] = amax_bits, x_bits
        q, s = oracle.quantize_rows(row)
        x = np.array([x_bits << 16], np.uint32).view(np.float32)[0]
        amax = np.array([amax_bits << 16], np.uint32).view(np.float32)[0]
        s32 = np.float32(amax) / np.float32(448.0)
        assert s[0, 0] == s32
        by_div = nearest_e4m3(np.array([x / s32], np.float32))[0]
        by_rcp = nearest_e4m3(np.array([x * (np.float32(1.0) / s32)], np.float32))[0]
        by_448 = nearest_e4m3(np.array([x * (np.float32(448.0) / amax)], np.float32))[0]
        assert by_div != by_rcp and by_div != by_448
        assert q[0, 1] == by_div and q[0, 0] == 0x7E
