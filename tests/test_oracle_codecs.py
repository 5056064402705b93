"""Pins for the oracle's number-format codecs (bf16, FP8 E4M3, FP4 E2M1).

Each codec is checked against things fixed outside the oracle: the formats' published value
tables and bit layouts, exhaustive round trips over every code, brute-force nearest-value search
with ties to even, saturation, and PyTorch's own bf16 / float8_e4m3fn casts (a library routine).
"""
import numpy as np
import pytest
import torch

import oracle

E4M3_FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)


def _nearest_even(x: np.ndarray, codes: np.ndarray, values: np.ndarray) -> np.ndarray:
    """Brute force: for each x the code of the closest value; on a tie the code whose last
    fraction bit (bit 0 of the code) is 0. Signed zeros: +0 for x >= 0, -0 for x < 0."""
    out = np.empty(x.shape, np.int64)
    for i, xi in enumerate(x):
        d = np.abs(values - xi)
        best = np.flatnonzero(d == d.min())
        same_sign = [c for c in codes[best] if (np.signbit(values[codes == c][0]) == np.signbit(xi))]
        cand = same_sign if same_sign else list(codes[best])
        even = [c for c in cand if c % 2 == 0]
        out[i] = (even or cand)[0]
    return out


# ---------------------------------------------------------------- FP8 E4M3 (OCP 8-bit FP)
def test_e4m3_named_values():
    # sign | 4-bit exponent (bias 7) | 3-bit fraction; S.1111.111 is NaN, no infinities
    v = oracle.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x7E, 0x80, 0xFE, 0x7F],
                                    np.uint8))
    assert v[0] == 0.0 and v[1] == 2.0 ** -9 and v[2] == 7 * 2.0 ** -9
    assert v[3] == 2.0 ** -6 and v[4] == 1.0 and v[5] == 1.5 and v[6] == 448.0
    assert v[7] == 0.0 and np.signbit(v[7]) and v[8] == -448.0 and np.isnan(v[9])


def test_e4m3_round_trip_all_codes():
    v = oracle.e4m3_decode(E4M3_FINITE)
    assert np.array_equal(oracle.e4m3_encode(v), E4M3_FINITE)


def test_e4m3_midpoints_round_to_even():
    pos = np.arange(0x00, 0x7F, dtype=np.uint8)  # 0 .. 448, increasing
    v = oracle.e4m3_decode(pos)
    mid = (v[:-1] + v[1:]) / 2
    got = oracle.e4m3_encode(mid)
    want = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mid, np.inf)), pos[1:])
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mid, -np.inf)), pos[:-1])
    assert np.array_equal(oracle.e4m3_encode(-mid), want | 0x80)


def test_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, np.inf])
    assert np.all(oracle.e4m3_encode(x) == 0x7E)
    assert np.all(oracle.e4m3_encode(-x) == 0xFE)


def test_e4m3_brute_force_nearest():
    rng = np.random.default_rng(1)
    x = np.sign(rng.standard_normal(3000)) * np.exp2(rng.uniform(-12, 8.8, 3000))
    x = np.clip(x, -448, 448)
    vals = oracle.e4m3_decode(E4M3_FINITE)
    want = _nearest_even(x, E4M3_FINITE.astype(np.int64), vals)
    assert np.array_equal(oracle.e4m3_encode(x).astype(np.int64), want)


def test_e4m3_matches_torch_after_clamp():
    g = torch.Generator().manual_seed(2)
    mag = torch.exp2(torch.empty(200000).uniform_(-14, 9.5, generator=g))
    x = (mag * torch.randn(200000, generator=g).sign()).clamp(-448, 448).to(torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.double().numpy())
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- FP4 E2M1 (OCP MX)
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_value_table():
    v = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert list(v[:8]) == E2M1_TABLE
    assert list(-v[8:]) == E2M1_TABLE and np.signbit(v[8])


def test_e2m1_round_trip_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.e2m1_encode(oracle.e2m1_decode(codes)), codes)


@pytest.mark.parametrize("x,value", [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0),
                                     (2.5, 2.0), (3.5, 4.0), (5.0, 4.0), (0.26, 0.5),
                                     (5.01, 6.0), (7.0, 6.0), (1e9, 6.0)])
def test_e2m1_ties_and_saturation(x, value):
    for s in (1.0, -1.0):
        code = oracle.e2m1_encode(np.array([s * x]))
        assert oracle.e2m1_decode(code)[0] == s * value


def test_e2m1_brute_force_nearest():
    rng = np.random.default_rng(3)
    x = rng.uniform(-6, 6, 4000)
    mids = (np.array(E2M1_TABLE[:-1]) + np.array(E2M1_TABLE[1:])) / 2
    x[:14] = np.concatenate([mids, -mids])
    codes = np.arange(16, dtype=np.int64)
    want = _nearest_even(x, codes, oracle.e2m1_decode(codes.astype(np.uint8)))
    assert np.array_equal(oracle.e2m1_encode(x).astype(np.int64), want)


# ---------------------------------------------------------------- bfloat16
def test_bf16_round_trip_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite_or_inf = ((codes >> 7) & 0xFF) != 0xFF
    finite_or_inf |= (codes & 0x7F) == 0
    codes = codes[finite_or_inf]
    assert np.array_equal(oracle.bf16_encode(oracle.bf16_decode(codes)), codes)


def test_bf16_decode_is_top_half_of_binary32():
    codes = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    codes = codes[((codes >> 7) & 0xFF) != 0xFF]
    as_f32 = (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(oracle.bf16_decode(codes), as_f32)


def test_bf16_matches_torch():
    g = torch.Generator().manual_seed(4)
    x = (torch.randn(300000, generator=g) * torch.exp2(torch.randint(-30, 30, (300000,),
                                                                       generator=g).float()))
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_encode(x.double().numpy()), ref)


def test_bf16_ties_to_even_and_overflow():
    one = np.float64(1.0)
    x = np.array([one + 2.0 ** -8, one + 3 * 2.0 ** -8, 3.4e38, -3.4e38, 2.0 ** -134, 2.0 ** -133])
    v = oracle.bf16_decode(oracle.bf16_encode(x))
    assert v[0] == 1.0 and v[1] == 1.0 + 2.0 ** -6
    assert v[2] == np.inf and v[3] == -np.inf
    assert v[4] == 0.0 and v[5] == 2.0 ** -133
