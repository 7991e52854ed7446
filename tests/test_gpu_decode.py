"""GPU parity of mla_decode_attention (and its split-KV combine) against the fp64
oracle, through the C ABI, on seeded inputs."""
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


def _to_dev(d):
    return dict(q_lat=dev_bf16(d["q_lat"]), q_rope=dev_bf16(d["q_rope"]),
                cache=dev_bf16(d["kv_cache"]), bt=dev_i32(d["block_table"]),
                seqlens=dev_i32(d["seqlens"]))


def _run(mla, d, num_splits=0, cache=None, bt=None):
    t = _to_dev(d)
    if cache is not None:
        t["cache"] = cache
    if bt is not None:
        t["bt"] = dev_i32(bt)
    max_len = int(np.max(d["seqlens"])) if len(d["seqlens"]) else 0
    out, lse, ws = mla.decode_attention(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                        t["seqlens"], max_len, d["scale"], num_splits)
    status = mla.check_device_status(ws)
    return host_f64_from_bf16(out), lse.cpu().numpy().astype(np.float64), status


def _oracle(d, rows=None, bt=None, cache=None):
    """Oracle on all sequences, or only on the listed rows (b indices)."""
    bt = d["block_table"] if bt is None else bt
    cache = d["kv_cache"] if cache is None else cache
    ql = synth.bf16_bits_to_f64(d["q_lat"])
    qr = synth.bf16_bits_to_f64(d["q_rope"])
    L = d["seqlens"]
    if rows is not None:
        ql, qr, bt, L = ql[rows], qr[rows], bt[rows], L[rows]
    return oracle.decode_absorbed(ql, qr, cache, bt, L, d["scale"])


def _case(B, H, seqlens, seed=0, shuffled=True):
    w = synth.Workload("case", B, H, tuple(seqlens), None, shuffled)
    return synth.make_attention_inputs(w, seed=seed)


def test_tiny_workload_full_parity(mla):
    d = synth.make_attention_inputs(synth.WORKLOADS["tiny"], seed=0)
    out, lse, st = _run(mla, d)
    assert st == 0
    ref, lref = _oracle(d)
    assert_close_rows(out, ref)
    assert_lse(lse, lref)


@pytest.mark.parametrize("H", [16, 32, 64, 128])
@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_ragged_lengths_and_splits(mla, H, splits):
    d = _case(5, H, (100, 63, 65, 1, 300), seed=1)
    out, lse, st = _run(mla, d, num_splits=splits)
    assert st == 0
    ref, lref = _oracle(d)
    assert_close_rows(out, ref)
    assert_lse(lse, lref)


def test_empty_sequence_gives_zero_and_neg_inf(mla):
    d = _case(3, 64, (0, 70, 0), seed=2)
    for splits in (1, 3):
        out, lse, st = _run(mla, d, num_splits=splits)
        assert st == 0
        assert np.all(out[0] == 0) and np.all(out[2] == 0)
        assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
        ref, lref = _oracle(d)
        assert_close_rows(out[1], ref[1])
        assert_lse(lse, lref)


def test_split_invariance(mla):
    d = _case(2, 128, (1000, 777), seed=3)
    outs = [_run(mla, d, num_splits=s)[:2] for s in (1, 2, 7, 0)]
    for o, l in outs[1:]:
        np.testing.assert_allclose(o, outs[0][0], rtol=1e-2, atol=2e-3)
        np.testing.assert_allclose(l, outs[0][1], atol=1e-4)


def test_poison_outside_sequences_is_never_read(mla):
    d = _case(3, 128, (100, 64, 130), seed=4)
    cache = d["kv_cache"].copy()
    bt = d["block_table"]
    nb = d["num_blocks"]
    used = {}
    for b, L in enumerate(d["seqlens"]):
        for t in range((L + 63) // 64):
            used.setdefault(int(bt[b, t]), 0)
            used[int(bt[b, t])] = max(used[int(bt[b, t])], min(64, L - 64 * t))
    for blk in range(nb):
        n = used.get(blk, 0)
        cache[blk, n:, :] = 0x7FC0 if blk % 2 else 0x7F80   # NaN / +inf
    bt2 = bt.copy()
    bt2[bt2 < 0] = 2 ** 30   # unused table entries: far out of range, must not be read
    out, lse, st = _run(mla, d, cache=dev_bf16(cache), bt=bt2)
    assert st == 0
    ref, lref = _oracle(d)
    assert_close_rows(out, ref)
    assert_lse(lse, lref)


def test_block_permutation_is_bit_identical(mla):
    d = _case(2, 64, (200, 129), seed=5, shuffled=False)
    out1, lse1, _ = _run(mla, d, num_splits=1)
    nb = d["num_blocks"]
    perm = np.random.default_rng(6).permutation(nb)
    cache2 = np.empty_like(d["kv_cache"])
    cache2[perm] = d["kv_cache"]
    bt2 = np.where(d["block_table"] >= 0, perm[np.maximum(d["block_table"], 0)], -1)
    out2, lse2, _ = _run(mla, d, num_splits=1, cache=dev_bf16(cache2), bt=bt2)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_constant_rows_return_the_row(mla):
    d = _case(2, 128, (333, 64), seed=7)
    c = synth.f32_to_bf16_bits(np.random.default_rng(8).standard_normal(576).astype(np.float32))
    cache = np.broadcast_to(c, d["kv_cache"].shape).copy()
    out, lse, st = _run(mla, d, cache=dev_bf16(cache))
    assert st == 0
    want = synth.bf16_bits_to_f64(c[:512])
    assert np.array_equal(out, np.broadcast_to(want, out.shape))


def test_out_of_range_block_sets_error_word(mla):
    d = _case(2, 64, (130, 64), seed=9)
    bt = d["block_table"].copy()
    bt[0, 1] = d["num_blocks"] + 1000
    out, lse, st = _run(mla, d, bt=bt)
    assert st == 4   # MLA_ERR_OUT_OF_RANGE
    assert np.all(np.isfinite(out))
    # the bad block is skipped: result equals the oracle that also skips it
    ref, lref = oracle.decode_absorbed(synth.bf16_bits_to_f64(d["q_lat"]),
                                       synth.bf16_bits_to_f64(d["q_rope"]), d["kv_cache"], bt,
                                       d["seqlens"], d["scale"], allow_range=True)
    assert_close_rows(out, ref)
    # the word was cleared by the read
    from mla_latent_kv_13_gb300 import mla as m
    assert m.check_device_status(m.alloc_workspace(256)) == 0


def test_combine_matches_oracle(mla):
    rng = np.random.default_rng(10)
    B, S, H = 3, 5, 16
    o = rng.standard_normal((B, S, H, 512)).astype(np.float32)
    l = (rng.standard_normal((B, S, H)) * 3).astype(np.float32)
    l[0, 1:, :] = -np.inf
    l[1, :, 3] = -np.inf
    out, lse = mla.decode_combine(torch.from_numpy(o).cuda(), torch.from_numpy(l).cuda())
    ref, lref = oracle.combine(o.astype(np.float64), l.astype(np.float64))
    assert_close_rows(host_f64_from_bf16(out), ref, norm_rtol=1e-2)
    assert_lse(lse.cpu().numpy(), lref, atol=1e-5)


@pytest.mark.parametrize("name,rows", [("v3", [0, 9]), ("mixed", [3, 77]), ("long", [5])])
def test_full_size_workloads_sampled(mla, name, rows):
    """Full-size workloads in the library's own split choice; the oracle checks the
    sampled sequences in full (every head, every latent column)."""
    w = synth.WORKLOADS[name]
    d = synth.make_attention_inputs(w, seed=0)
    out, lse, st = _run(mla, d)
    assert st == 0
    ref, lref = _oracle(d, rows=rows)
    assert_close_rows(out[rows], ref)
    assert_lse(lse[rows], lref)
    # property that holds at any size: every row is finite and lse >= max possible floor
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_balanced_schedule_many_ragged_sequences(mla):
    """The default schedule cuts the concatenated tiles of all sequences into equal
    ranges: sequences land whole in one range, cut across several, or are empty."""
    rng = np.random.default_rng(11)
    L = rng.integers(0, 700, 300)
    L[::17] = 0
    L[5] = 64
    d = _case(len(L), 64, tuple(int(x) for x in L), seed=12)
    out, lse, st = _run(mla, d, num_splits=0)
    assert st == 0
    ref, lref = _oracle(d)
    assert_close_rows(out, ref)
    assert_lse(lse, lref)


def test_balanced_schedule_matches_fixed_split(mla):
    # more sequences than resident clusters: the library's own choice is the schedule
    L = np.random.default_rng(13).integers(0, 5000, 100)
    L[:4] = (5000, 1, 0, 64)
    d = _case(100, 128, tuple(int(x) for x in L), seed=13)
    a = _run(mla, d, num_splits=0)
    b = _run(mla, d, num_splits=1)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-2, atol=2e-3)
    np.testing.assert_allclose(a[1], b[1], atol=1e-4)


@pytest.mark.parametrize("splits", [1, 0])
def test_reference_raised_by_one_half_mid_sequence(mla, splits):
    """The k_rope part of a few cached rows is scaled by 40, so that for many heads one
    token's score jumps far above the running reference in the middle of a sequence, inside
    one CTA's 32-token half of a tile (tokens 40 and 5 of their tiles lie in different
    halves); the rows' values (c_kv) keep their scale. The other half of the tile, the
    received half and the running output must all be brought to the new reference; results
    must still match the oracle."""
    d = _case(3, 128, (700, 333, 1000), seed=21)
    cache = d["kv_cache"].copy()
    bt = d["block_table"]
    spikes = [(0, 3 * 64 + 40), (1, 2 * 64 + 5), (2, 1 * 64 + 50), (2, 10 * 64 + 3)]
    for b, t in spikes:
        blk, r = bt[b][t // 64], t % 64
        rope = synth.bf16_bits_to_f64(cache[blk, r, 512:]) * 40.0
        cache[blk, r, 512:] = synth.f32_to_bf16_bits(rope.astype(np.float32))
    out, lse, st = _run(mla, d, num_splits=splits, cache=dev_bf16(cache))
    assert st == 0
    ref, lref = _oracle(d, cache=cache)
    assert_close_rows(out, ref)
    assert_lse(lse, lref)


@pytest.mark.parametrize("splits", [1, 0])
def test_seqlen_beyond_max_seqlen_is_reported_and_clamped(mla, splits):
    """A length above the call's max_seqlen (still inside the block table) is recorded as
    MLA_ERR_OUT_OF_RANGE and clamped to max_seqlen, on the fixed-split path and on the
    balanced schedule alike (so neither silently truncates to its own token ranges)."""
    B = 100 if splits == 0 else 3  # 100 sequences: more than one wave -> the schedule
    rng = np.random.default_rng(11)
    L = rng.integers(1, 300, size=B).astype(np.int32)
    L[1] = 700  # within the table (built for 700) but above the max_seqlen passed below
    d = _case(B, 64, tuple(int(x) for x in L), seed=12)
    max_len = 500
    if splits == 0:
        assert mla.decode_plan(B, 64, max_len, 0)[0] == 0
    t = _to_dev(d)
    out, lse, ws = mla.decode_attention(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                        t["seqlens"], max_len, d["scale"], splits)
    assert mla.check_device_status(ws) == 4  # MLA_ERR_OUT_OF_RANGE
    clamped = dict(d, seqlens=np.minimum(d["seqlens"], max_len))
    ref, lref = _oracle(clamped)
    assert_close_rows(host_f64_from_bf16(out), ref)
    assert_lse(lse.cpu().numpy(), lref)


@pytest.mark.parametrize("B", [100, 3])
def test_prepared_schedule_gives_the_same_bits(mla, B):
    """mla_decode_prepare once, then two mla_decode_attention_prepared calls (two layers
    over the same lengths), the first with the schedule prepared on another stream: the
    outputs equal mla_decode_attention's bit for bit, empty sequences included; B = 100
    runs the balanced schedule, B = 3 a fixed split (the prepare call does nothing)."""
    rng = np.random.default_rng(21 + B)
    L = rng.integers(1, 600, size=B).astype(np.int32)
    L[0] = 0
    if B > 3:
        L[57] = 0
    d = _case(B, 128, tuple(int(x) for x in L), seed=22)
    max_len = int(L.max())
    assert (mla.decode_plan(B, 128, max_len, 0)[0] == 0) == (B == 100)
    t = _to_dev(d)
    ref_out, ref_lse, _ = mla.decode_attention(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                               t["seqlens"], max_len, d["scale"], 0)
    ws = mla.alloc_workspace(mla.decode_workspace_size(B, 128, max_len, 0))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    mla.decode_prepare(t["seqlens"], B, 128, max_len, 0, ws, side)
    done = torch.cuda.Event()
    done.record(side)
    torch.cuda.current_stream().wait_event(done)
    for _ in range(2):
        out = torch.full_like(ref_out, 7.0)
        lse = torch.full_like(ref_lse, 7.0)
        mla.decode_attention_prepared(t["q_lat"], t["q_rope"], t["cache"], t["bt"], t["seqlens"],
                                      max_len, d["scale"], 0, out, lse, ws)
        assert mla.check_device_status(ws) == 0
        assert np.array_equal(host_bits(out), host_bits(ref_out))
        assert np.array_equal(lse.cpu().numpy(), ref_lse.cpu().numpy())
    o = host_f64_from_bf16(out)
    assert np.all(o[L == 0] == 0) and np.all(np.isneginf(lse.cpu().numpy()[L == 0]))


def test_balanced_schedule_without_cut_sequences(mla):
    """152 equal sequences: every share of the balanced schedule holds exactly two, so no
    sequence is cut and the merge kernel has no job (only its first CTA waits for the
    attention kernel); the outputs still match the oracle, and a second call gives the same
    bits."""
    B, H, L = 152, 64, 640
    d = _case(B, H, (L,) * B, seed=31)
    assert mla.decode_plan(B, H, L, 0)[0] == 0
    # with the 76 resident clusters of a GB300 the shares cut no sequence
    assert mla.decode_schedule(np.full(B, L, dtype=np.int32), d["block_table"].shape[1], 76)[1] == 0
    t = _to_dev(d)
    out1, lse1, ws = mla.decode_attention(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                          t["seqlens"], L, d["scale"], 0)
    assert mla.check_device_status(ws) == 0
    out2, lse2, _ = mla.decode_attention(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                         t["seqlens"], L, d["scale"], 0, workspace=ws)
    assert np.array_equal(host_bits(out1), host_bits(out2))
    rows = [0, 1, 75, 76, 151]
    ref, lref = _oracle(d, rows=rows)
    assert_close_rows(host_f64_from_bf16(out1)[rows], ref)
    assert_lse(lse1.cpu().numpy()[rows], lref)
