"""GPU parity of mla_append_kv, mla_absorb_q and mla_out_absorb against the fp64
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_13_gb300 import synth
from tests.helpers import assert_close_rows, dev_bf16, dev_i32, host_bits, host_f64_from_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla as m
    return m


def bf16(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _append_both(mla, h, w, pos, bt, cache):
    c_gpu = dev_bf16(cache)
    ws = mla.append_kv(dev_bf16(h), dev_bf16(w), dev_i32(pos), dev_i32(bt), c_gpu)
    st = mla.check_device_status(ws)
    c_ref = cache.copy()
    oracle.append_kv(h, w, pos, bt, c_ref, allow_range=True)
    return host_bits(c_gpu), c_ref, st


# d_model 128: split-K partials and a finalize launch; 512 and 1024: the k-splits reduced in
# their cluster, rows written by its epilogue (1024 with 200 sequences: two row tiles)
@pytest.mark.parametrize("B,dm", [(7, 128), (7, 512), (200, 1024)])
def test_append_exact_on_integer_inputs(mla, B, dm):
    rng = np.random.default_rng(0)
    h = bf16(rng.integers(-1, 2, (B, dm)))
    w = bf16(rng.integers(-1, 2, (576, dm)))
    bt = np.arange(B * 2, dtype=np.int32).reshape(B, 2)[:, ::-1].copy()
    cache = bf16(rng.standard_normal((B * 2, 64, 576)))
    got, ref, st = _append_both(mla, h, w, np.zeros(B, np.int32), bt, cache)
    assert st == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("B,dm", [(5, 256), (200, 1024), (128, 7168)])
def test_append_real_inputs_within_fp32_summation_bound(mla, B, dm):
    rng = np.random.default_rng(1)
    h = bf16(rng.standard_normal((B, dm)))
    w = bf16(rng.standard_normal((576, dm)) * 0.02)
    nb = 3 * B
    bt = rng.permutation(nb).astype(np.int32).reshape(B, 3)
    pos = rng.integers(0, 192, B).astype(np.int32)
    cache = np.zeros((nb, 64, 576), np.uint16)
    got, ref, st = _append_both(mla, h, w, pos, bt, cache)
    assert st == 0
    _check_appended_rows(got, ref, h, w, pos, bt, dm)


def _check_appended_rows(got, ref, h, w, pos, bt, dm):
    B = h.shape[0]
    diff = np.abs(got.astype(np.int32) - ref.astype(np.int32))
    # bf16 bit patterns of same-sign values differ by the number of ulps between them
    assert (diff > 0).mean() < 0.01
    # The kernel sums the d_model products in fp32, in an order it does not fix; any order
    # is within dm * 2^-24 * sum |h_k w_k| of the exact sum (the standard bound for
    # recursive summation), and RoPE mixes each rotated pair with |cos|, |sin| <= 1. So the
    # stored bf16 value and the oracle's rounding of the exact value differ by at most one
    # bf16 ulp plus that bound.
    hf, wf = synth.bf16_bits_to_f64(h), synth.bf16_bits_to_f64(w)
    x = hf @ wf.T
    gam = dm * 2.0 ** -24 * (np.abs(hf) @ np.abs(wf).T)
    pair = gam[:, 512::2] + gam[:, 513::2] + 2.0 ** -21 * (np.abs(x[:, 512::2]) + np.abs(x[:, 513::2]))
    gam[:, 512::2] = pair
    gam[:, 513::2] = pair
    blk, slot = bt[np.arange(B), pos // 64], pos % 64
    g = synth.bf16_bits_to_f64(got[blk, slot])
    r = synth.bf16_bits_to_f64(ref[blk, slot])
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.maximum(np.abs(g), np.abs(r)), 2.0 ** -126))) - 7)
    assert np.all(np.abs(g - r) <= ulp + gam)
    mask = np.ones(got.shape[:2], dtype=bool)
    mask[blk, slot] = False
    assert np.array_equal(got[mask], ref[mask])  # nothing else written


@pytest.mark.parametrize("dm", [64, 256])  # finalize launch / cluster epilogue
def test_append_out_of_range_is_flagged_and_dropped(mla, dm):
    rng = np.random.default_rng(2)
    B = 3
    h = bf16(rng.standard_normal((B, dm)))
    w = bf16(rng.standard_normal((576, dm)))
    bt = np.array([[0], [1], [99]], np.int32)      # sequence 2 points outside the pool
    pos = np.array([3, 64, 0], np.int32)           # sequence 1 writes past its table
    cache = np.zeros((3, 64, 576), np.uint16)
    got, ref, st = _append_both(mla, h, w, pos, bt, cache)
    assert st == 4
    assert np.array_equal(got, ref)                # only sequence 0 was written


def _proj(B, dm, ql, H, seed):
    rng = np.random.default_rng(seed)
    s = 0.02
    return dict(h=bf16(rng.standard_normal((B, dm))),
                w_dq=bf16(rng.standard_normal((ql, dm)) * s),
                w_uq=bf16(rng.standard_normal((H * 128, ql)) * s),
                w_qr=bf16(rng.standard_normal((H * 64, ql)) * s),
                w_uk=bf16(rng.standard_normal((H, 128, 512)) * s),
                w_uv=bf16(rng.standard_normal((H, 128, 512)) * s),
                w_o=bf16(rng.standard_normal((dm, H * 128)) * s),
                pos=rng.integers(0, 9000, B).astype(np.int32))


# W_DQ's k-splits reduced in their cluster: 8 splits over 4 tiles with ragged rows (100);
# two row tiles (200), the second one 72 rows
# W_UQ + W_QR + RoPE in one launch: 128-column tiles at 16 and 32 heads, 192-column tiles
# (ragged last tile of each product) at 128 heads
@pytest.mark.parametrize("B,dm,ql,H,rows", [(3, 256, 128, 16, None),
                                           (100, 1024, 512, 32, None),
                                           (5, 512, 256, 128, None),
                                           # 256 row x column tiles: no cluster split fits,
                                           # W_DQ writes partials for a reduction launch
                                           (4096, 256, 1024, 16, [0, 2047, 4095]),
                                           (200, 2048, 1536, 16, [0, 127, 128, 150, 199]),
                                           (128, 7168, 1536, 128, [0, 61, 127])])
def test_absorb_q(mla, B, dm, ql, H, rows):
    p = _proj(B, dm, ql, H, 3)
    q_lat, q_rope, ws = mla.absorb_q(dev_bf16(p["h"]), dev_bf16(p["w_dq"]), dev_bf16(p["w_uq"]),
                                     dev_bf16(p["w_qr"]), dev_bf16(p["w_uk"]), dev_i32(p["pos"]))
    assert mla.check_device_status(ws) == 0
    rows = list(range(B)) if rows is None else rows
    rl, rr = oracle.absorb_q(p["h"][rows], p["w_dq"], p["w_uq"], p["w_qr"], p["w_uk"],
                             p["pos"][rows])
    assert_close_rows(host_f64_from_bf16(q_lat)[rows], rl, "q_lat")
    assert_close_rows(host_f64_from_bf16(q_rope)[rows], rr, "q_rope")


# W_O's k-splits reduced in their cluster: 128-column tiles with ragged rows (100), 256-column
# tiles over two row tiles (200)
@pytest.mark.parametrize("B,dm,H,rows", [(3, 256, 16, None), (100, 1024, 32, None),
                                         (4096, 512, 16, [0, 1000, 4095]),  # W_O: partials
                                         (200, 7168, 64, [0, 127, 128, 199]),
                                         (128, 7168, 128, [1, 64, 100])])
def test_out_absorb(mla, B, dm, H, rows):
    p = _proj(B, dm, 64, H, 4)
    o_lat = bf16(np.random.default_rng(5).standard_normal((B, H, 512)) * 0.05)
    y, ws = mla.out_absorb(dev_bf16(o_lat), dev_bf16(p["w_uv"]), dev_bf16(p["w_o"]))
    assert mla.check_device_status(ws) == 0
    rows = list(range(B)) if rows is None else rows
    ref = oracle.out_absorb(synth.bf16_bits_to_f64(o_lat)[rows], p["w_uv"], p["w_o"])
    assert_close_rows(host_f64_from_bf16(y)[rows], ref, "y")


def test_projection_launches_on_device(mla):
    """On a full-size part (148 or more SMs) the headline shapes' split-K products all fit as
    clusters: append, W_DQ and W_O each one launch (append 1, absorb_q 3, out_absorb 2), and
    W_DQ with W_DKR one launch in the combined call (3)."""
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count < 148:
        pytest.skip("a smaller part may plan partials")
    assert mla.projection_launches(128, 7168, 1536, 128) == (1, 3, 2, 3)
    # the large-batch parity cases above take the partial-writing paths
    assert mla.projection_launches(4096, 256, 1024, 16)[1] == 6  # W_DQ 2, W_UQ/W_QR/RoPE 3, W_UK 1
    assert mla.projection_launches(4096, 512, 128, 16)[2] == 3   # W_UV 1, W_O 2
    a, _, _, both = mla.projection_launches(2000, 256, 128, 16)
    assert a == 2 and both == 7  # the two calls: append 2, absorb_q 1 + 3 + 1



# append_kv and absorb_q in one call: W_DQ and W_DKR in one cluster-reduced launch (8 or 6
# splits over both products' tiles; 200 sequences: two row tiles)
@pytest.mark.parametrize("B,dm,ql,H,rows", [(3, 256, 128, 16, None),
                                           (100, 1024, 512, 32, None),
                                           (200, 2048, 1536, 16, [0, 127, 128, 199]),
                                           (128, 7168, 1536, 128, [0, 61, 127]),
                                           # 96 tiles: no cluster split fits, the two calls
                                           # run one after the other
                                           (2000, 256, 128, 16, [0, 999, 1999])])
def test_append_absorb_q(mla, B, dm, ql, H, rows):
    p = _proj(B, dm, ql, H, 6)
    rng = np.random.default_rng(7)
    w_dkr = bf16(rng.standard_normal((576, dm)) * 0.02)
    nb = 3 * B
    bt = rng.permutation(nb).astype(np.int32).reshape(B, 3)
    pos = rng.integers(0, 192, B).astype(np.int32)
    cache = np.zeros((nb, 64, 576), np.uint16)
    c_gpu = dev_bf16(cache)
    q_lat, q_rope, ws = mla.append_absorb_q(dev_bf16(p["h"]), dev_bf16(w_dkr), dev_i32(pos),
                                            dev_i32(bt), c_gpu, dev_bf16(p["w_dq"]),
                                            dev_bf16(p["w_uq"]), dev_bf16(p["w_qr"]),
                                            dev_bf16(p["w_uk"]))
    assert mla.check_device_status(ws) == 0
    c_ref = cache.copy()
    oracle.append_kv(p["h"], w_dkr, pos, bt, c_ref, allow_range=True)
    _check_appended_rows(host_bits(c_gpu), c_ref, p["h"], w_dkr, pos, bt, dm)
    rows = list(range(B)) if rows is None else rows
    # the query side takes the append's positions
    rl, rr = oracle.absorb_q(p["h"][rows], p["w_dq"], p["w_uq"], p["w_qr"], p["w_uk"], pos[rows])
    assert_close_rows(host_f64_from_bf16(q_lat)[rows], rl, "q_lat")
    assert_close_rows(host_f64_from_bf16(q_rope)[rows], rr, "q_rope")


def test_append_absorb_q_out_of_range_is_flagged_and_dropped(mla):
    """A row outside the cache is flagged and dropped by the combined launch's append side;
    the query side is computed for every row."""
    rng = np.random.default_rng(8)
    B, dm, ql, H = 3, 256, 128, 16
    p = _proj(B, dm, ql, H, 9)
    w_dkr = bf16(rng.standard_normal((576, dm)))
    bt = np.array([[0], [1], [99]], np.int32)
    pos = np.array([3, 64, 0], np.int32)
    cache = np.zeros((3, 64, 576), np.uint16)
    c_gpu = dev_bf16(cache)
    q_lat, q_rope, ws = mla.append_absorb_q(dev_bf16(p["h"]), dev_bf16(w_dkr), dev_i32(pos),
                                            dev_i32(bt), c_gpu, dev_bf16(p["w_dq"]),
                                            dev_bf16(p["w_uq"]), dev_bf16(p["w_qr"]),
                                            dev_bf16(p["w_uk"]))
    assert mla.check_device_status(ws) == 4
    c_ref = cache.copy()
    oracle.append_kv(p["h"], w_dkr, pos, bt, c_ref, allow_range=True)
    got = host_bits(c_gpu)
    written = np.zeros(got.shape[:2], bool)
    written[0, 3] = True
    assert np.array_equal(got[~written], c_ref[~written])  # only sequence 0 was written
    rl, rr = oracle.absorb_q(p["h"], p["w_dq"], p["w_uq"], p["w_qr"], p["w_uk"], pos)
    assert_close_rows(host_f64_from_bf16(q_lat), rl, "q_lat")
    assert_close_rows(host_f64_from_bf16(q_rope), rr, "q_rope")
