"""GPU parity of context-parallel decode, through the C ABI: G ranks' shares computed one
after another on this one GPU (mla_decode_attention_partial on each rank's token ranges,
nothing waits on another launch), stacked as an all-gather would leave them, merged by
mla_decode_combine_ranks, and compared with the fp64 oracle over the whole sequences."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_13_gb300 import context_parallel as cp
from mla_latent_kv_13_gb300 import synth
from tests.helpers import assert_close_rows, assert_lse, dev_bf16, dev_i32, host_f64_from_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla as m
    return m


def _ranks(mla, d, G, num_splits):
    q, r = dev_bf16(d["q_lat"]), dev_bf16(d["q_rope"])
    cache = dev_bf16(d["kv_cache"])
    ranges = cp.partition_ranges(d["seqlens"], G)
    parts, lses = [], []
    for g in range(G):
        lbt, lL = cp.local_block_table(d["block_table"], ranges[g])
        mx = int(lL.max())
        o, lse, ws = mla.decode_attention_partial(q, r, cache, dev_i32(lbt), dev_i32(lL), mx,
                                                  d["scale"], num_splits)
        assert mla.check_device_status(ws) == 0
        parts.append(o)
        lses.append(lse)
    return torch.stack(parts), torch.stack(lses), ranges


@pytest.mark.parametrize("G", [2, 3, 4])
@pytest.mark.parametrize("splits", [1, 0, 3])
def test_context_parallel_matches_oracle(mla, G, splits):
    w = synth.Workload("cp", 4, 128, (3000, 640, 65, 1), None, True)
    d = synth.make_attention_inputs(w, seed=31)
    go, gl, ranges = _ranks(mla, d, G, splits)
    ql, qr = synth.bf16_bits_to_f64(d["q_lat"]), synth.bf16_bits_to_f64(d["q_rope"])
    # each rank's fp32 part against the oracle over that rank's range
    for g in range(G):
        lbt, lL = cp.local_block_table(d["block_table"], ranges[g])
        ref_g, lref_g = oracle.decode_absorbed(ql, qr, d["kv_cache"], lbt, lL, d["scale"])
        assert_close_rows(go[g].cpu().numpy(), ref_g, f"rank {g} part")
        assert_lse(gl[g].cpu().numpy(), lref_g)
    out, lse = mla.decode_combine_ranks(go, gl)
    torch.cuda.synchronize()
    ref, lref = oracle.decode_absorbed(ql, qr, d["kv_cache"], d["block_table"], d["seqlens"],
                                       d["scale"])
    assert_close_rows(host_f64_from_bf16(out), ref)
    assert_lse(lse.cpu().numpy(), lref)


def test_partial_equals_full_attention_with_one_rank(mla):
    """G = 1: the partial result is the whole attention, in fp32."""
    w = synth.Workload("cp1", 3, 64, (1000, 77, 0), None, True)
    d = synth.make_attention_inputs(w, seed=32)
    t = dict(q=dev_bf16(d["q_lat"]), r=dev_bf16(d["q_rope"]), c=dev_bf16(d["kv_cache"]),
             bt=dev_i32(d["block_table"]), L=dev_i32(d["seqlens"]))
    o32, l32, _ = mla.decode_attention_partial(t["q"], t["r"], t["c"], t["bt"], t["L"], 1000,
                                               d["scale"], 0)
    o16, l16, _ = mla.decode_attention(t["q"], t["r"], t["c"], t["bt"], t["L"], 1000,
                                       d["scale"], 0)
    torch.cuda.synchronize()
    # the bf16 output is the fp32 one rounded to nearest
    assert torch.equal(o32.to(torch.bfloat16), o16)
    assert torch.equal(l32, l16)
    assert torch.all(o32[2] == 0) and torch.all(torch.isneginf(l32[2]))


def _cp_worker(rank, world, port, out):
    import os
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch
    import torch.distributed as dist
    from mla_latent_kv_13_gb300 import context_parallel as cpm
    from mla_latent_kv_13_gb300 import synth as sy
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = sy.Workload("cp2", 3, 64, (2000, 300, 40), None, True)
    d = sy.make_attention_inputs(w, seed=33)
    r = cpm.partition_ranges(d["seqlens"], world)
    lbt, lL = cpm.local_block_table(d["block_table"], r[rank])

    def dev(a, bf16=False):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else a).cuda()
        return t.view(torch.bfloat16) if bf16 else t

    o, lse = cpm.decode_context_parallel(dev(d["q_lat"], True), dev(d["q_rope"], True),
                                         dev(d["kv_cache"], True), dev(lbt), dev(lL),
                                         int(lL.max()), d["scale"])
    torch.cuda.synchronize()
    out[rank] = (o.view(torch.int16).cpu().numpy(), lse.cpu().numpy())
    dist.destroy_process_group()


def test_two_processes_exchange_over_gloo(mla):
    """Two ranks as two processes on this GPU, each with its own token ranges; the
    exchange runs on the host (gloo), so no kernel of one waits on the other's."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_cp_worker, args=(2, port, out), nprocs=2, join=True,
                       start_method="spawn")
    w = synth.Workload("cp2", 3, 64, (2000, 300, 40), None, True)
    d = synth.make_attention_inputs(w, seed=33)
    ref, lref = oracle.decode_absorbed(synth.bf16_bits_to_f64(d["q_lat"]),
                                       synth.bf16_bits_to_f64(d["q_rope"]), d["kv_cache"],
                                       d["block_table"], d["seqlens"], d["scale"])
    o0, l0 = out[0]
    o1, l1 = out[1]
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)  # every rank, the same result
    assert_close_rows(synth.bf16_bits_to_f64(o0.view(np.uint16)), ref)
    assert_lse(l0, lref)
