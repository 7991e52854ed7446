"""GPU parity of the FP8 (e4m3) latent cache against the oracle, through the C ABI:
dequantisation of every code (bit-exact), quantisation of bf16 rows (bit-exact), the
FP8 append (bit-exact on integer inputs, one code step otherwise) and decode attention
over an FP8 cache against the oracle's attention over the dequantised rows."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_13_gb300 import synth
from tests.helpers import (assert_close_rows, assert_lse, dev_bf16, dev_i32, host_bits,
                           host_f64_from_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla as m
    return m


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_dequantise_every_code_bit_exact(mla):
    rng = np.random.default_rng(0)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    rows = 64
    codes = np.stack([np.roll(np.resize(finite, 576), 7 * r) for r in range(rows)])
    exps = rng.integers(-40, 20, rows).astype(np.int8)
    exps[0], exps[1] = -117, 118  # the extremes that keep every value a normal bf16
    out = mla.dequantize_kv_fp8(_dev_u8(codes), _dev_u8(exps))
    torch.cuda.synchronize()
    want = oracle.fp8_cache_as_bf16(codes, exps)
    assert np.array_equal(host_bits(out), want)


def test_quantise_bf16_rows_bit_exact(mla):
    rng = np.random.default_rng(1)
    rows = 300
    x = rng.normal(0, 1, (rows, 576)).astype(np.float32) * np.exp(
        rng.uniform(-20, 20, (rows, 1))).astype(np.float32)
    x[3] = 0.0
    x[4, :] = 0.0
    x[4, 100] = -448.0 * 2.0 ** 5   # max exactly at a power-of-two boundary
    x[5] = np.linspace(-500, 500, 576)  # ties and saturation-free spread
    x[6] = 0.0
    x[6, :3] = [2.0 ** -130, -(2.0 ** -131), 3 * 2.0 ** -133]  # subnormal row: e = -126
    bits = synth.f32_to_bf16_bits(x)
    codes, exps = mla.quantize_kv_fp8(dev_bf16(bits))
    torch.cuda.synchronize()
    want_c, want_e = oracle.quantize_rows_fp8(synth.bf16_bits_to_f64(bits))
    assert np.array_equal(exps.cpu().numpy(), want_e)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert want_e[6] == -126


def test_append_kv_fp8_integer_inputs_bit_exact_and_real_inputs_close(mla):
    rng = np.random.default_rng(2)
    B, dm, nb = 5, 512, 8
    bt = np.array([[3, 1], [0, 2], [5, 4], [7, 6], [2, 0]], dtype=np.int32)
    for integer in (True, False):
        if integer:
            h = rng.integers(-3, 4, (B, dm)).astype(np.float32)
            w = rng.integers(-2, 3, (576, dm)).astype(np.float32)
            pos = np.zeros(B, dtype=np.int32)
        else:
            h = rng.normal(0, 1, (B, dm)).astype(np.float32)
            w = (rng.normal(0, 0.02, (576, dm))).astype(np.float32)
            pos = np.array([0, 5, 63, 64, 100], dtype=np.int32)
        hb, wb = synth.f32_to_bf16_bits(h), synth.f32_to_bf16_bits(w)
        codes = np.zeros((nb, 64, 576), dtype=np.uint8)
        exps = np.zeros((nb, 64), dtype=np.int8)
        oracle.append_kv_fp8(hb, wb, pos, bt, codes, exps)
        dc, de = _dev_u8(np.zeros_like(codes)), _dev_u8(np.zeros_like(exps))
        ws = mla.append_kv_fp8(dev_bf16(hb), dev_bf16(wb), dev_i32(pos), dev_i32(bt), dc, de)
        assert mla.check_device_status(ws) == 0
        gc, ge = dc.cpu().numpy(), de.cpu().numpy()
        if integer:
            assert np.array_equal(gc, codes) and np.array_equal(ge, exps)
        else:
            # fp32 accumulation and fp32 RoPE against fp64: the same exponent and codes
            # at most one step apart (a rounding near a tie), values within 2 ulps
            for b in range(B):
                blk, slot = bt[b, pos[b] // 64], pos[b] % 64
                assert ge[blk, slot] == exps[blk, slot]
                g = oracle.dequantize_fp8(gc[blk, slot][None], ge[blk, slot][None])[0]
                o = oracle.dequantize_fp8(codes[blk, slot][None], exps[blk, slot][None])[0]
                step = np.maximum(np.abs(o), 2.0 ** (-6 + int(exps[blk, slot]))) * 2.0 ** -3
                assert np.all(np.abs(g - o) <= step * 1.0001)


def _fp8_case(B, H, L, seed):
    w = synth.Workload("fp8", B, H, tuple(L), None, True)
    d = synth.make_attention_inputs(w, seed=seed)
    codes, exps = oracle.quantize_rows_fp8(synth.bf16_bits_to_f64(d["kv_cache"]))
    return d, codes, exps


def _run_fp8(mla, d, codes, exps, splits, bt=None):
    bt = d["block_table"] if bt is None else bt
    max_len = int(np.max(d["seqlens"]))
    out, lse, ws = mla.decode_attention_fp8(dev_bf16(d["q_lat"]), dev_bf16(d["q_rope"]),
                                            _dev_u8(codes), _dev_u8(exps), dev_i32(bt),
                                            dev_i32(d["seqlens"]), max_len, d["scale"], splits)
    st = mla.check_device_status(ws)
    return host_f64_from_bf16(out), lse.cpu().numpy().astype(np.float64), st


@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_fp8_matches_oracle(mla, H, splits):
    d, codes, exps = _fp8_case(5, H, (100, 63, 65, 1, 900), seed=5)
    out, lse, st = _run_fp8(mla, d, codes, exps, splits)
    assert st == 0
    ref, lref = oracle.decode_absorbed_fp8(synth.bf16_bits_to_f64(d["q_lat"]),
                                           synth.bf16_bits_to_f64(d["q_rope"]), codes, exps,
                                           d["block_table"], d["seqlens"], d["scale"])
    assert_close_rows(out, ref)
    assert_lse(lse, lref)


def test_decode_fp8_equals_bf16_decode_of_the_dequantised_cache(mla):
    """The widening is exact, so the FP8 kernel and the bf16 kernel on the dequantised
    cache compute identical results."""
    d, codes, exps = _fp8_case(4, 128, (3000, 700, 1, 2222), seed=6)
    out8, lse8, st = _run_fp8(mla, d, codes, exps, 0)
    assert st == 0
    deq = oracle.fp8_cache_as_bf16(codes, exps)
    o16, l16, ws = mla.decode_attention(dev_bf16(d["q_lat"]), dev_bf16(d["q_rope"]),
                                        dev_bf16(deq), dev_i32(d["block_table"]),
                                        dev_i32(d["seqlens"]), 3000, d["scale"], 0)
    assert mla.check_device_status(ws) == 0
    assert np.array_equal(out8, host_f64_from_bf16(o16))
    assert np.array_equal(lse8, l16.cpu().numpy().astype(np.float64))


def test_decode_fp8_empty_sequences_and_poison(mla):
    d, codes, exps = _fp8_case(3, 64, (0, 130, 0), seed=7)
    codes = codes.copy()
    exps = exps.copy()
    bt = d["block_table"]
    # tokens past the end of sequence 1 and the spare block: NaN codes, huge exponents
    last = int(bt[1, 2])
    codes[last, 130 - 128:] = 0x7F
    exps[last, 130 - 128:] = 127
    codes[-1] = 0x7F
    out, lse, st = _run_fp8(mla, d, codes, exps, 1)
    assert st == 0
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))
    clean_c, clean_e = oracle.quantize_rows_fp8(synth.bf16_bits_to_f64(d["kv_cache"]))
    ref, lref = oracle.decode_absorbed_fp8(synth.bf16_bits_to_f64(d["q_lat"]),
                                           synth.bf16_bits_to_f64(d["q_rope"]), clean_c, clean_e,
                                           bt, d["seqlens"], d["scale"])
    assert_close_rows(out[1], ref[1])
    assert_lse(lse, lref)


def test_decode_fp8_long_sequences_sampled(mla):
    """64 heads over 32 sequences of 4096 tokens (a scaled-down long-context batch),
    checked on sampled sequences against the oracle."""
    d, codes, exps = _fp8_case(32, 64, (4096,) * 32, seed=8)
    out, lse, st = _run_fp8(mla, d, codes, exps, 0)
    assert st == 0
    rows = [0, 13, 31]
    ref, lref = oracle.decode_absorbed_fp8(synth.bf16_bits_to_f64(d["q_lat"][rows]),
                                           synth.bf16_bits_to_f64(d["q_rope"][rows]), codes, exps,
                                           d["block_table"][rows], d["seqlens"][rows], d["scale"])
    assert_close_rows(out[rows], ref)
    assert_lse(lse[rows], lref)


@pytest.mark.parametrize("H", [64, 128])
def test_decode_fp8_on_the_balanced_schedule(mla, H):
    """More sequences than resident clusters, so the default plan is the balanced schedule:
    clusters run several segments (the widening warps restart with every one) and
    sequences cut between clusters are merged."""
    rng = np.random.default_rng(9)
    L = rng.integers(1, 900, 100)
    L[:3] = (2000, 1, 64)
    d, codes, exps = _fp8_case(100, H, tuple(int(x) for x in L), seed=9)
    assert mla.decode_plan(100, H, int(L.max()), 0)[0] == 0
    out, lse, st = _run_fp8(mla, d, codes, exps, 0)
    assert st == 0
    rows = [0, 1, 2, 17, 50, 99]
    ref, lref = oracle.decode_absorbed_fp8(synth.bf16_bits_to_f64(d["q_lat"][rows]),
                                           synth.bf16_bits_to_f64(d["q_rope"][rows]), codes, exps,
                                           d["block_table"][rows], d["seqlens"][rows], d["scale"])
    assert_close_rows(out[rows], ref)
    assert_lse(lse[rows], lref)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
