"""Context-parallel decode: one batch's cached tokens spread over G ranks by token range.

"DeepSeek V3 MoE inference" §3 deploys decode attention as TP4 + SP4 + DP; "from the
memory wall to the compute wall" §2.3 explains why heads are the wrong axis to split
(every head reads the same compressed cache, so tensor parallelism over heads cuts
little of the traffic). Splitting the tokens does cut it: rank g holds the cache rows
of its token range of every sequence, computes attention over that range alone
(mla_decode_attention_partial: normalised fp32 output and log-sum-exp per head), the
ranks all-gather those (o_part [B, H, 512], lse [B, H]) -- 256 KB + 0.5 KB per sequence
at 128 heads -- and mla_decode_combine_ranks merges them by log-sum-exp, exactly.

This module holds the host side: the partition of each sequence's token blocks over
the ranks and the exchange over torch.distributed (NCCL for device tensors, gloo
through host memory). Every arithmetic step runs in libmla's kernels.
"""
from __future__ import annotations

import numpy as np

BLOCK = 64


def partition_ranges(seqlens, G: int) -> np.ndarray:
    """Token ranges of each sequence per rank: int32 [G, B, 2] of (start, end).

    Sequence b's T_b = ceil(L_b / 64) token blocks are cut into G contiguous runs of
    blocks, rank g taking blocks [floor(g T_b / G), floor((g + 1) T_b / G)); so every
    rank's range starts on a block boundary, ranges are disjoint, cover [0, L_b) and
    differ in length by at most one block. A rank may get an empty range."""
    L = np.asarray(seqlens, dtype=np.int64)
    if G < 1:
        raise ValueError("G must be >= 1")
    T = (L + BLOCK - 1) // BLOCK
    out = np.zeros((G, len(L), 2), dtype=np.int32)
    for g in range(G):
        t0 = (g * T) // G
        t1 = ((g + 1) * T) // G
        out[g, :, 0] = np.minimum(L, t0 * BLOCK)
        out[g, :, 1] = np.minimum(L, t1 * BLOCK)
    return out


def local_block_table(block_table, ranges_g) -> tuple[np.ndarray, np.ndarray]:
    """One rank's view of a global paged layout: for each sequence, the blocks of its
    range in logical order (the rank's own block table, -1 past its last block) and the
    range's length (the rank's seqlens). `ranges_g` is partition_ranges(...)[g]."""
    bt = np.asarray(block_table)
    B = bt.shape[0]
    starts, ends = ranges_g[:, 0], ranges_g[:, 1]
    nblk = (ends - starts + BLOCK - 1) // BLOCK
    mb = max(int(nblk.max()) if B else 0, 1)
    local = np.full((B, mb), -1, dtype=np.int32)
    for b in range(B):
        s0 = int(starts[b]) // BLOCK
        local[b, :nblk[b]] = bt[b, s0:s0 + nblk[b]]
    return local, (ends - starts).astype(np.int32)


def all_gather_parts(o_part, lse_part, group=None):
    """All-gather every rank's (o_part [B, H, 512], lse_part [B, H]) fp32 into
    ([G, B, H, 512], [G, B, H]) in rank order, over torch.distributed. With the gloo
    backend, device tensors travel through host memory; NCCL gathers device tensors
    directly. Returns tensors on the device of the inputs."""
    import torch
    import torch.distributed as dist
    G = dist.get_world_size(group)
    backend = dist.get_backend(group)
    dev = o_part.device
    via_host = backend == "gloo" and o_part.is_cuda
    o = o_part.contiguous().cpu() if via_host else o_part.contiguous()
    ls = lse_part.contiguous().cpu() if via_host else lse_part.contiguous()
    # gathered along the leading dimension (rank-major), then viewed as [G, ...]
    go = torch.empty((G * o.shape[0],) + tuple(o.shape[1:]), dtype=o.dtype, device=o.device)
    gl = torch.empty((G * ls.shape[0],) + tuple(ls.shape[1:]), dtype=ls.dtype, device=ls.device)
    dist.all_gather_into_tensor(go, o, group=group)
    dist.all_gather_into_tensor(gl, ls, group=group)
    go = go.view((G,) + tuple(o.shape))
    gl = gl.view((G,) + tuple(ls.shape))
    if via_host:
        go, gl = go.to(dev), gl.to(dev)
    return go, gl


def decode_context_parallel(q_lat, q_rope, kv_cache, block_table, seqlens, max_seqlen, scale,
                            num_splits=0, group=None, workspace=None, stream=None):
    """Decode attention with the tokens spread over the ranks of `group`: this rank's
    cache / block_table / seqlens hold its token ranges (see partition_ranges and
    local_block_table). Every rank passes the same queries and gets the same
    (out [B, H, 512] bf16, lse [B, H] fp32): its partial attention, the all-gather of
    all ranks' partials, their merge."""
    from mla_latent_kv_13_gb300 import mla
    o, lse, _ = mla.decode_attention_partial(q_lat, q_rope, kv_cache, block_table, seqlens,
                                             max_seqlen, scale, num_splits, workspace=workspace,
                                             stream=stream)
    go, gl = all_gather_parts(o, lse, group)
    return mla.decode_combine_ranks(go, gl, stream=stream)
