"""Host logic of context-parallel decode (CPU): the token-range partition, each rank's
block table, and the exchange of the ranks' partial results over torch.distributed
(gloo, world size 2) merged by the oracle's log-sum-exp combine, checked against the
oracle's attention over the whole sequences."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mla_latent_kv_13_gb300 import context_parallel as cp  # noqa: E402
from mla_latent_kv_13_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("G", [1, 2, 3, 4, 7])
def test_partition_covers_each_sequence_once_on_block_boundaries(G):
    L = np.array([0, 1, 63, 64, 65, 300, 4096, 5000], dtype=np.int32)
    r = cp.partition_ranges(L, G)
    assert r.shape == (G, len(L), 2)
    for b, n in enumerate(L):
        cover = np.zeros(n, dtype=int)
        for g in range(G):
            s, e = r[g, b]
            assert 0 <= s <= e <= n
            assert s % 64 == 0 or s == n
            cover[s:e] += 1
        assert np.all(cover == 1)
        nblk = [(r[g, b, 1] - r[g, b, 0] + 63) // 64 for g in range(G)]
        assert max(nblk) - min(nblk) <= 1  # balanced to one block


def test_local_block_table_maps_each_rank_to_its_blocks():
    L = np.array([300, 70, 0], dtype=np.int32)
    bt, _ = synth.make_block_table(L, shuffled=True, seed=3)
    r = cp.partition_ranges(L, 2)
    for g in range(2):
        lbt, lL = cp.local_block_table(bt, r[g])
        assert np.array_equal(lL, r[g, :, 1] - r[g, :, 0])
        for b in range(len(L)):
            s = r[g, b, 0] // 64
            n = (lL[b] + 63) // 64
            assert np.array_equal(lbt[b, :n], bt[b, s:s + n])
            assert np.all(lbt[b, n:] == -1)


def _inputs():
    w = synth.Workload("cp", 3, 16, (700, 129, 64), None, True)
    return synth.make_attention_inputs(w, seed=21)


def _rank_part(d, G, g):
    """Rank g's partial attention over its token ranges, computed by the oracle."""
    import oracle
    r = cp.partition_ranges(d["seqlens"], G)
    lbt, lL = cp.local_block_table(d["block_table"], r[g])
    return oracle.decode_absorbed(synth.bf16_bits_to_f64(d["q_lat"]),
                                  synth.bf16_bits_to_f64(d["q_rope"]), d["kv_cache"], lbt, lL,
                                  d["scale"])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from mla_latent_kv_13_gb300 import context_parallel as cpm
    dist.init_process_group("gloo", rank=rank, world_size=world)
    d = _inputs()
    o, lse = _rank_part(d, world, rank)
    go, gl = cpm.all_gather_parts(torch.from_numpy(o), torch.from_numpy(lse))
    out[rank] = (go.numpy(), gl.numpy())
    dist.destroy_process_group()


def test_two_ranks_exchange_and_merge_equals_whole_sequences():
    import oracle
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    d = _inputs()
    ref, lref = oracle.decode_absorbed(synth.bf16_bits_to_f64(d["q_lat"]),
                                       synth.bf16_bits_to_f64(d["q_rope"]), d["kv_cache"],
                                       d["block_table"], d["seqlens"], d["scale"])
    for rank in (0, 1):
        go, gl = out[rank]
        assert go.shape == (2, 3, 16, 512) and gl.shape == (2, 3, 16)
        # rank g's slot holds rank g's own part, on every rank
        for g in range(2):
            og, lg = _rank_part(d, 2, g)
            np.testing.assert_array_equal(go[g], og)
            np.testing.assert_array_equal(gl[g], lg)
        merged, lse = oracle.combine(np.transpose(go, (1, 0, 2, 3)), np.transpose(gl, (1, 0, 2)))
        np.testing.assert_allclose(merged, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lref, rtol=1e-12, atol=1e-12)
