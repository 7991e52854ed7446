"""Pins of the oracle's FP8 (e4m3) cache: the code values the format defines, round to
nearest with ties to even checked by brute force over every representable value,
saturation, the per-row power-of-two scale, a hand-worked decode and the FP8 append.
CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from mla_latent_kv_13_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _finite_values():
    """(value, code) of every finite non-negative e4m3 code, ascending."""
    vals = [(oracle.e4m3_to_f64(c), c) for c in range(0x80) if c != 0x7F]
    return sorted(vals)


def test_e4m3_landmark_codes():
    # facts of the e4m3 format: largest finite 448 = 1.75 * 2^8, smallest normal 2^-6,
    # smallest subnormal 2^-9, 1.0 = exponent field 7, the all-ones codes are NaN
    assert oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_f64(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0x39) == 1.125
    assert oracle.e4m3_to_f64(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_to_f64(0x7F)) and math.isnan(oracle.e4m3_to_f64(0xFF))
    assert oracle.e4m3_to_f64(0x80) == 0.0 and math.copysign(1, oracle.e4m3_to_f64(0x80)) < 0
    vals = [v for v, _ in _finite_values()]
    assert len(vals) == 127 and len(set(vals)) == 127  # 0 plus 126 distinct magnitudes
    assert all(a < b for a, b in zip(vals, vals[1:]))


def test_e4m3_every_value_round_trips():
    for v, c in _finite_values():
        assert oracle.f64_to_e4m3(v) == c
        if c:
            assert oracle.f64_to_e4m3(-v) == c | 0x80


def test_e4m3_rounding_matches_brute_force_nearest():
    fin = _finite_values()
    vals = np.array([v for v, _ in fin])
    codes = np.array([c for _, c in fin])

    def nearest(x):
        a = abs(x)
        if a >= 448.0:
            c = 0x7E
        else:
            d = np.abs(vals - a)
            best = np.flatnonzero(d == d.min())
            c = int(codes[best[0]]) if len(best) == 1 else int(next(
                codes[i] for i in best if codes[i] % 2 == 0))  # tie: the even mantissa
        return c | (0x80 if math.copysign(1, x) < 0 else 0)

    # every midpoint between neighbours (a tie) and points just beside it
    for (a, ca), (b, cb) in zip(fin, fin[1:]):
        mid = 0.5 * (a + b)
        assert oracle.f64_to_e4m3(mid) == nearest(mid), (a, b)
        assert oracle.f64_to_e4m3(np.nextafter(mid, -1)) == ca
        assert oracle.f64_to_e4m3(np.nextafter(mid, 1e9)) == cb
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(-500, 500, 3000), rng.normal(0, 1, 3000),
                         rng.normal(0, 1e-2, 2000), [2 ** -10, 2 ** -11, 463.9, 464.0, 1e30]])
    for x in xs:
        assert oracle.f64_to_e4m3(float(x)) == nearest(float(x)), x


def test_e4m3_saturation_and_ties_to_even_examples():
    assert oracle.f64_to_e4m3(1e9) == 0x7E and oracle.f64_to_e4m3(-1e9) == 0xFE
    assert oracle.f64_to_e4m3(460.0) == 0x7E      # beyond 448: saturate
    assert oracle.f64_to_e4m3(2 ** -10) == 0x00   # halfway 0 .. 2^-9: the even code 0
    assert oracle.f64_to_e4m3(3 * 2 ** -10) == 0x02  # halfway 2^-9 .. 2^-8: even m = 2
    assert oracle.f64_to_e4m3(1.0625) == 0x38     # halfway 1 .. 1.125: even m = 0
    assert oracle.f64_to_e4m3(1.1875) == 0x3A     # halfway 1.125 .. 1.25: even m = 2


def test_row_scale_is_the_smallest_power_of_two():
    rng = np.random.default_rng(1)
    rows = rng.normal(0, 1, (200, 576)) * np.exp(rng.uniform(-12, 12, (200, 1)))
    rows[7] = 0.0
    rows[8, :] = 0.0
    rows[8, 5] = 448.0 * 2.0 ** -3   # max exactly 448 * 2^e
    codes, exps = oracle.quantize_rows_fp8(rows)
    for r in range(200):
        mx = np.abs(rows[r]).max()
        e = int(exps[r])
        if mx == 0:
            assert e == 0 and np.all(codes[r] == 0)
            continue
        assert mx * 2.0 ** -e <= 448.0 < mx * 2.0 ** -(e - 1)
        for n in range(0, 576, 37):
            assert codes[r, n] == oracle.f64_to_e4m3(rows[r, n] * 2.0 ** -e)
    assert exps[8] == -3


def test_row_scale_exponent_floor_for_tiny_rows():
    """The exponent is kept at or above -126 (its scale 2^-e a normal float), so a row whose
    largest value is below 448 * 2^-126 is quantised with e = -126: its codes are those of
    the values times 2^126, which e4m3 still represents or flushes by its own rounding."""
    rows = np.zeros((3, 576))
    rows[0, :4] = [2.0 ** -130, -2.0 ** -131, 3 * 2.0 ** -133, 2.0 ** -140]
    rows[1, 0] = 448.0 * 2.0 ** -126   # exactly at the floor: e = -126 either way
    rows[2, 0] = 448.0 * 2.0 ** -125
    codes, exps = oracle.quantize_rows_fp8(rows)
    assert list(exps) == [-126, -126, -125]
    assert codes[0, 0] == oracle.f64_to_e4m3(2.0 ** -4)
    assert codes[0, 1] == oracle.f64_to_e4m3(-(2.0 ** -5))
    assert codes[0, 2] == oracle.f64_to_e4m3(3 * 2.0 ** -7)
    assert codes[0, 3] == 0  # 2^-14 is below half the smallest subnormal (2^-9)
    deq = oracle.dequantize_fp8(codes, exps)
    assert deq[0, 0] == 2.0 ** -130 and deq[0, 2] == 3 * 2.0 ** -133
    assert deq[1, 0] == rows[1, 0] and deq[2, 0] == rows[2, 0]


def test_dequantised_rows_are_exact_bf16_values():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, (64, 576))
    codes, exps = oracle.quantize_rows_fp8(x)
    deq = oracle.dequantize_fp8(codes, exps)
    bits = oracle.fp8_cache_as_bf16(codes, exps)
    assert np.array_equal(synth.bf16_bits_to_f64(bits), deq)
    # quantisation error within half a step of the row's scale (relative 2^-4 of |x| for
    # normal codes)
    e = exps.astype(np.int64)[:, None]
    step = np.where(np.abs(x) * 2.0 ** -e >= 2 ** -6,
                    2.0 ** (np.floor(np.log2(np.maximum(np.abs(x) * 2.0 ** -e, 2 ** -6))) - 3),
                    2.0 ** -9) * 2.0 ** e
    assert np.all(np.abs(deq - x) <= 0.5 * step + 1e-300)


def test_golden_fp8_decode():
    g = json.load(open(os.path.join(GOLDEN, "fp8_attention.json")))
    rows = np.array(g["rows_logical"])
    codes, exps = oracle.quantize_rows_fp8(rows)
    assert codes.tolist() == g["expected_codes"]
    assert exps.tolist() == g["expected_exps"]
    assert np.array_equal(oracle.dequantize_fp8(codes, exps), np.array(g["dequantised_rows"]))
    # paged: token 0, 1 in block 1; token 2 in block 0 slot 0; block 0 slot 1 poisoned
    kv_codes = np.zeros((2, 2, 4), dtype=np.uint8)
    kv_exps = np.zeros((2, 2), dtype=np.int8)
    kv_codes[1, 0], kv_exps[1, 0] = codes[0], exps[0]
    kv_codes[1, 1], kv_exps[1, 1] = codes[1], exps[1]
    kv_codes[0, 0], kv_exps[0, 0] = codes[2], exps[2]
    kv_codes[0, 1] = 0x7F
    q_lat = np.array([[[math.log(2), 0.0]]])
    q_rope = np.array([[[0.0, -math.log(3) / 0.1015625]]])
    out, lse = oracle.decode_absorbed(q_lat, q_rope,
                                      np.where(kv_codes == 0x7F, np.uint16(0x7FC0),
                                               oracle.fp8_cache_as_bf16(
                                                   np.where(kv_codes == 0x7F, 0, kv_codes),
                                                   kv_exps)),
                                      np.array([[1, 0]]), np.array([3]), g["scale"])
    np.testing.assert_allclose(out[0, 0], g["expected_out"], rtol=0, atol=1e-14)
    assert abs(lse[0, 0] - g["expected_lse"]) < 1e-14
    out2, lse2 = oracle.decode_absorbed_fp8(q_lat, q_rope, np.where(kv_codes == 0x7F, 0, kv_codes),
                                            kv_exps, np.array([[1, 0]]), np.array([3]), g["scale"])
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_append_kv_fp8_quantises_the_projected_row():
    rng = np.random.default_rng(3)
    B, dm, D = 3, 128, 576
    # integer-valued inputs at position 0 (RoPE is the identity): the fp64 row is exact
    h = rng.integers(-3, 4, (B, dm)).astype(np.float32)
    w = rng.integers(-2, 3, (D, dm)).astype(np.float32)
    hb, wb = synth.f32_to_bf16_bits(h), synth.f32_to_bf16_bits(w)
    bt = np.array([[2], [0], [1]], dtype=np.int32)
    codes = np.zeros((3, 64, D), dtype=np.uint8)
    exps = np.zeros((3, 64), dtype=np.int8)
    oracle.append_kv_fp8(hb, wb, np.zeros(B, dtype=np.int32), bt, codes, exps)
    x = h.astype(np.float64) @ w.astype(np.float64).T
    want_c, want_e = oracle.quantize_rows_fp8(x)
    for b in range(B):
        assert np.array_equal(codes[bt[b, 0], 0], want_c[b])
        assert exps[bt[b, 0], 0] == want_e[b]
    # a later position rotates only the rope part before quantising
    codes2 = np.zeros_like(codes)
    exps2 = np.zeros_like(exps)
    oracle.append_kv_fp8(hb, wb, np.full(B, 5, dtype=np.int32), np.array([[0], [1], [2]]),
                         codes2, exps2)
    xr = x.copy()
    xr[:, 512:] = oracle.rope(x[:, 512:], np.full(B, 5))
    want_c2, want_e2 = oracle.quantize_rows_fp8(xr)
    for b in range(B):
        assert np.array_equal(codes2[b, 5], want_c2[b]) and exps2[b, 5] == want_e2[b]
