"""The full absorbed decode step (append -> absorb_q -> attention -> out_absorb) at
the full-step workload sizes, checked on sampled sequences against the oracle's
composition of the same four steps."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_13_gb300 import synth
from tests.helpers import assert_close_rows, dev_bf16, dev_i32, host_bits, host_f64_from_bf16

pytestmark = pytest.mark.gpu


def test_full_step_sampled():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla
    w = synth.WORKLOADS["step"]
    d = synth.make_step_inputs(w, seed=0)
    names = ["w_dkr", "w_dq", "w_uq", "w_qr", "w_uk", "w_uv", "w_o"]
    wt = {k: dev_bf16(d[k]) for k in names}
    cache = dev_bf16(d["kv_cache"])
    bt = dev_i32(d["block_table"])
    step = mla.DecodeStep(wt, d["B"], d["H"], int(d["seqlens_after"].max()))
    y = step(dev_bf16(d["h"]), dev_i32(d["pos"]), dev_i32(d["seqlens_after"]), bt, cache)
    assert step.check() == 0
    y_gpu = host_f64_from_bf16(y)
    assert np.all(np.isfinite(y_gpu))

    rows = [0, 77]
    ref_cache = d["kv_cache"]
    oracle.append_kv(d["h"][rows], d["w_dkr"], d["pos"][rows], d["block_table"][rows], ref_cache)
    # the appended rows themselves (<= 1 bf16 ulp)
    for b in rows:
        p = int(d["pos"][b])
        blk = int(d["block_table"][b, p // 64])
        got = host_bits(cache[blk, p % 64])
        diff = np.abs(got.astype(np.int32) - ref_cache[blk, p % 64].astype(np.int32))
        assert diff.max() <= 1
    q_lat, q_rope = oracle.absorb_q(d["h"][rows], d["w_dq"], d["w_uq"], d["w_qr"], d["w_uk"],
                                    d["pos"][rows])
    o_lat, _ = oracle.decode_absorbed(q_lat, q_rope, ref_cache, d["block_table"][rows],
                                      d["seqlens_after"][rows], d["scale"])
    y_ref = oracle.out_absorb(o_lat, d["w_uv"], d["w_o"])
    assert_close_rows(y_gpu[rows], y_ref, "y")


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_small_ragged_step_every_row(num_splits):
    """DecodeStep at 64 heads, d_model 1024, q_lora 512 on 20 sequences of ragged lengths
    (one whose only row is the appended one, block edges at 64 and 65, up to 1000): the
    combined append + query call, the schedule (or a fixed split: none, or three ranges
    merged), attention and the output projections, every row against the oracle's
    composition."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla
    lens = (1, 2, 63, 64, 65, 66, 127, 128, 129, 200, 300, 333, 400, 512, 513, 640, 700, 800,
            999, 1000)
    w = synth.Workload("step_small", len(lens), 64, lens, None, shuffled=True, full_step=True,
                       d_model=1024, q_lora=512)
    d = synth.make_step_inputs(w, seed=3)
    names = ["w_dkr", "w_dq", "w_uq", "w_qr", "w_uk", "w_uv", "w_o"]
    wt = {k: dev_bf16(d[k]) for k in names}
    cache = dev_bf16(d["kv_cache"])
    bt = dev_i32(d["block_table"])
    step = mla.DecodeStep(wt, d["B"], d["H"], int(d["seqlens_after"].max()),
                          num_splits=num_splits)
    y = step(dev_bf16(d["h"]), dev_i32(d["pos"]), dev_i32(d["seqlens_after"]), bt, cache)
    assert step.check() == 0
    y_gpu = host_f64_from_bf16(y)

    ref_cache = d["kv_cache"].copy()
    oracle.append_kv(d["h"], d["w_dkr"], d["pos"], d["block_table"], ref_cache)
    for b in range(d["B"]):  # the appended rows (<= 1 bf16 ulp)
        p = int(d["pos"][b])
        blk = int(d["block_table"][b, p // 64])
        got = host_bits(cache[blk, p % 64])
        diff = np.abs(got.astype(np.int32) - ref_cache[blk, p % 64].astype(np.int32))
        assert diff.max() <= 1
    q_lat, q_rope = oracle.absorb_q(d["h"], d["w_dq"], d["w_uq"], d["w_qr"], d["w_uk"], d["pos"])
    o_lat, _ = oracle.decode_absorbed(q_lat, q_rope, ref_cache, d["block_table"],
                                      d["seqlens_after"], d["scale"])
    y_ref = oracle.out_absorb(o_lat, d["w_uv"], d["w_o"])
    assert_close_rows(y_gpu, y_ref, "y")
