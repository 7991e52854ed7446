"""GPU parity of decode attention at the limits the C ABI accepts, through the C ABI:
the largest batch (4096 sequences: the schedule kernel's one-CTA scan at its capacity and
some fifty segments per cluster), the largest fixed split (256 token ranges merged per
row), and one long sequence cut by the balanced schedule into a part per cluster (a merge
over more than 32 parts). Sampled sequences against the fp64 oracle; properties that hold
at any size on every row."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_13_gb300 import synth
from tests.helpers import assert_close_rows, assert_lse, dev_bf16, dev_i32, host_f64_from_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla as m
    return m


def _case(H, seqlens, seed):
    L = np.asarray(seqlens, dtype=np.int32)
    w = synth.Workload("limits", len(L), H, tuple(int(x) for x in L), None, True)
    return synth.make_attention_inputs(w, seed=seed)


def _run(mla, d, num_splits):
    max_len = int(np.max(d["seqlens"]))
    out, lse, ws = mla.decode_attention(dev_bf16(d["q_lat"]), dev_bf16(d["q_rope"]),
                                        dev_bf16(d["kv_cache"]), dev_i32(d["block_table"]),
                                        dev_i32(d["seqlens"]), max_len, d["scale"], num_splits)
    st = mla.check_device_status(ws)
    return host_f64_from_bf16(out), lse.cpu().numpy().astype(np.float64), st


def _check_rows(d, out, lse, rows):
    rows = sorted(rows)
    ref, lref = oracle.decode_absorbed(synth.bf16_bits_to_f64(d["q_lat"][rows]),
                                       synth.bf16_bits_to_f64(d["q_rope"][rows]), d["kv_cache"],
                                       d["block_table"][rows], d["seqlens"][rows], d["scale"])
    assert_close_rows(out[rows], ref)
    assert_lse(lse[rows], lref)


def _check_all_rows_valid(d, out, lse):
    empty = d["seqlens"] == 0
    assert np.all(out[empty] == 0) and np.all(np.isneginf(lse[empty]))
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse[~empty]))


def test_largest_batch_on_the_balanced_schedule(mla):
    rng = np.random.default_rng(41)
    L = rng.integers(0, 130, 4096).astype(np.int32)
    L[::97] = 0
    L[1], L[2] = 129, 64
    d = _case(16, L, seed=41)
    assert mla.decode_plan(4096, 16, int(L.max()), 0)[0] == 0  # the balanced schedule
    out, lse, st = _run(mla, d, 0)
    assert st == 0
    rows = set(rng.choice(4096, 40, replace=False).tolist()) | {0, 1, 2, 97, 4095}
    _check_rows(d, out, lse, rows)
    _check_all_rows_valid(d, out, lse)


def test_largest_fixed_split(mla):
    """256 ranges of 2 tiles over a 32768-token sequence; the 700-token one fills 6 of its
    256 ranges, the other 250 are empty and merge with weight zero."""
    d = _case(16, (32768, 700), seed=42)
    out, lse, st = _run(mla, d, 256)
    assert st == 0
    _check_rows(d, out, lse, [0, 1])


def test_one_long_sequence_cut_into_a_part_per_cluster(mla):
    """77 sequences (one more than resident clusters on a GB300), so the balanced schedule
    runs; sequence 0 holds 131072 tokens, ~95% of all tiles, and is cut across every
    cluster, so its merge takes one part per cluster (more than 32)."""
    rng = np.random.default_rng(43)
    L = np.concatenate([[131072], rng.integers(1, 200, 76)]).astype(np.int32)
    d = _case(16, L, seed=43)
    assert mla.decode_plan(len(L), 16, int(L.max()), 0)[0] == 0
    out, lse, st = _run(mla, d, 0)
    assert st == 0
    _check_rows(d, out, lse, [0, 1, 40, 76])
    _check_all_rows_valid(d, out, lse)
