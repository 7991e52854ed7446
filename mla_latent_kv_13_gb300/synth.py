"""Seeded synthetic inputs for MLA latent-KV decode.

This module holds the workload table and the seeded generators that feed both
the CUDA path and the fp64 oracle. It contains none of the method's arithmetic:
it only draws numbers, rounds them to bf16 storage and lays out the paged cache
and its block table.

Recipe (all draws from numpy's PCG64 through ``SeedSequence(seed).spawn``; one
child stream per purpose, and large arrays are drawn in fixed-size chunks with
one grandchild stream per chunk, so the values do not depend on thread count):

* seqlens      child 0 (only the mixed-length workload draws them)
* block table  child 1: physical block ids are a permutation of the pool,
               sliced per sequence in logical order; unused entries are -1
* q_lat        child 2, N(0, sigma_q) rounded to bf16 (round-to-nearest-even)
* q_rope       child 3, same
* cache        child 4, N(0, sigma_kv) rounded to bf16, every physical block
* weights / h  children 5.. (full decode step only): weights N(0, 0.02), h N(0, 1)

The pool holds exactly sum(ceil(L_b / 64)) blocks plus one spare block that no
sequence uses; callers may poison it.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

D_C = 512          # latent width d_c
D_ROPE = 64        # decoupled-RoPE key width
D_QK = D_C + D_ROPE  # 576 cached values per token
BLOCK = 64         # tokens per cache page
D_NOPE = 128       # per-head query/key width without RoPE
D_V = 128          # per-head value width
SCALE_192 = 1.0 / np.sqrt(192.0)

_CHUNK = 1 << 22


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    seqlens: tuple | None      # fixed lengths, or None when drawn
    seqlen_range: tuple | None  # (lo, hi) inclusive when drawn
    shuffled: bool
    full_step: bool = False
    d_model: int = 7168
    q_lora: int = 1536
    s_q: int = 1  # query tokens per sequence; `heads` counts query rows (s_q x heads each)

    def describe(self) -> dict:
        d = {"workload": self.name, "batch": self.batch, "heads": self.heads // self.s_q,
             "d_c": D_C, "d_rope": D_ROPE, "block": BLOCK}
        if self.s_q > 1:
            d["query_tokens"] = self.s_q
        if self.seqlens is not None:
            d["seqlens"] = list(self.seqlens) if len(set(self.seqlens)) > 1 else self.seqlens[0]
        else:
            d["seqlen_range"] = list(self.seqlen_range)
        if self.full_step:
            d.update(d_model=self.d_model, q_lora=self.q_lora, d_nope=D_NOPE, d_v=D_V)
        return d


WORKLOADS = {
    "tiny": Workload("tiny", 2, 16, (64, 100), None, shuffled=False),
    "v3": Workload("v3", 16, 128, (4096,) * 16, None, shuffled=True),
    "mixed": Workload("mixed", 128, 128, None, (1024, 8192), shuffled=True),
    "long": Workload("long", 32, 64, (32768,) * 32, None, shuffled=True),
    # draft-token verification: 2 query tokens x 64 heads = 128 query rows per sequence
    "mtp": Workload("mtp", 128, 128, (8192,) * 128, None, shuffled=True, s_q=2),
    "step": Workload("step", 128, 128, (8192,) * 128, None, shuffled=True, full_step=True),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _normal_bf16(ss: np.random.SeedSequence, n: int, sigma: float) -> np.ndarray:
    """n values N(0, sigma) as bf16 bits, drawn chunk by chunk (thread-count independent)."""
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    kids = ss.spawn(nchunks)

    def work(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(kids[i]))
        v = g.standard_normal(hi - lo, dtype=np.float32)
        if sigma != 1.0:
            v *= np.float32(sigma)
        out[lo:hi] = f32_to_bf16_bits(v)

    if nchunks == 1:
        work(0)
    else:
        with _cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def draw_seqlens(w: Workload, seed: int = 0) -> np.ndarray:
    if w.seqlens is not None:
        return np.asarray(w.seqlens, dtype=np.int32)
    ss = np.random.SeedSequence(seed).spawn(8)[0]
    g = np.random.Generator(np.random.PCG64(ss))
    lo, hi = w.seqlen_range
    return g.integers(lo, hi, size=w.batch, endpoint=True).astype(np.int32)


def make_block_table(seqlens: np.ndarray, shuffled: bool, seed: int = 0,
                     max_blocks: int | None = None, reserve_tokens: int = 0):
    """Block table [B, max_blocks] int32 and the pool size (blocks incl. one spare).

    ``reserve_tokens`` extra token slots per sequence are allocated (for appends).
    """
    B = len(seqlens)
    need = [(int(L) + reserve_tokens + BLOCK - 1) // BLOCK for L in seqlens]
    total = int(sum(need))
    mb = max(max(need) if need else 0, 1) if max_blocks is None else max_blocks
    if shuffled:
        ss = np.random.SeedSequence(seed).spawn(8)[1]
        g = np.random.Generator(np.random.PCG64(ss))
        phys = g.permutation(total).astype(np.int32)
    else:
        phys = np.arange(total, dtype=np.int32)
    bt = np.full((B, mb), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        bt[b, :need[b]] = phys[o:o + need[b]]
        o += need[b]
    return bt, total + 1


def make_attention_inputs(w: Workload, seed: int = 0, sigma: float = 1.0,
                          seqlens: np.ndarray | None = None):
    """All decode-attention inputs of one workload as numpy arrays (bf16 as uint16 bits)."""
    kids = np.random.SeedSequence(seed).spawn(8)
    L = draw_seqlens(w, seed) if seqlens is None else np.asarray(seqlens, dtype=np.int32)
    bt, nblocks = make_block_table(L, w.shuffled, seed)
    B, H = w.batch, w.heads
    q_lat = _normal_bf16(kids[2], B * H * D_C, sigma).reshape(B, H, D_C)
    q_rope = _normal_bf16(kids[3], B * H * D_ROPE, sigma).reshape(B, H, D_ROPE)
    cache = _normal_bf16(kids[4], nblocks * BLOCK * D_QK, sigma).reshape(nblocks, BLOCK, D_QK)
    return dict(q_lat=q_lat, q_rope=q_rope, kv_cache=cache, block_table=bt,
                seqlens=L, num_blocks=nblocks, B=B, H=H, scale=float(SCALE_192))


def make_attention_queries(w: Workload, seed: int = 0, sigma: float = 1.0):
    """q_lat and q_rope of one workload, the same values make_attention_inputs draws
    (same streams), without drawing its cache."""
    kids = np.random.SeedSequence(seed).spawn(8)
    B, H = w.batch, w.heads
    q_lat = _normal_bf16(kids[2], B * H * D_C, sigma).reshape(B, H, D_C)
    q_rope = _normal_bf16(kids[3], B * H * D_ROPE, sigma).reshape(B, H, D_ROPE)
    return q_lat, q_rope


def make_step_inputs(w: Workload, seed: int = 0, prefilled: int | None = None):
    """Inputs of the full absorbed decode step: weights, hidden states, cache, tables.

    The cache holds ``prefilled`` tokens per sequence (default L-1) drawn like the
    attention workloads; the step appends one token at position ``prefilled``.
    Weight layouts ([out, in] row-major unless stated):
      w_dkr [576, d_model] (rows 0..511 = W_DKV, rows 512..575 = W_KR)
      w_dq  [q_lora, d_model]; w_uq [H*128, q_lora]; w_qr [H*64, q_lora]
      w_uk  [H, 128, 512];     w_uv [H, 128, 512];   w_o  [d_model, H*128]
    """
    kids = np.random.SeedSequence(seed).spawn(16)
    B, H, dm, ql = w.batch, w.heads, w.d_model, w.q_lora
    Lfull = np.asarray(w.seqlens, dtype=np.int32)
    pre = (Lfull - 1) if prefilled is None else np.full(B, prefilled, dtype=np.int32)
    bt, nblocks = make_block_table(pre, w.shuffled, seed, reserve_tokens=1)
    cache = _normal_bf16(kids[4], nblocks * BLOCK * D_QK, 1.0).reshape(nblocks, BLOCK, D_QK)
    s = 0.02
    d = dict(
        h=_normal_bf16(kids[5], B * dm, 1.0).reshape(B, dm),
        w_dkr=_normal_bf16(kids[6], D_QK * dm, s).reshape(D_QK, dm),
        w_dq=_normal_bf16(kids[7], ql * dm, s).reshape(ql, dm),
        w_uq=_normal_bf16(kids[8], H * D_NOPE * ql, s).reshape(H * D_NOPE, ql),
        w_qr=_normal_bf16(kids[9], H * D_ROPE * ql, s).reshape(H * D_ROPE, ql),
        w_uk=_normal_bf16(kids[10], H * D_NOPE * D_C, s).reshape(H, D_NOPE, D_C),
        w_uv=_normal_bf16(kids[11], H * D_V * D_C, s).reshape(H, D_V, D_C),
        w_o=_normal_bf16(kids[12], dm * H * D_V, s).reshape(dm, H * D_V),
        kv_cache=cache, block_table=bt, pos=pre.astype(np.int32),
        seqlens_after=(pre + 1).astype(np.int32), num_blocks=nblocks,
        B=B, H=H, d_model=dm, q_lora=ql, scale=float(SCALE_192), rope_theta=10000.0,
    )
    return d


def algorithmic_attention_bytes(seqlens, H: int, kv_bytes_per_value: int = 2) -> int:
    """Bytes a decode-attention pass must move at least once: the latent cache rows
    of every valid token (576 values: bf16, or e4m3 codes plus one exponent byte),
    q (576 bf16/head), out (512 bf16/head), lse (fp32/head)."""
    N = int(np.sum(seqlens))
    B = len(seqlens)
    row = D_QK * 2 if kv_bytes_per_value == 2 else D_QK + 1
    return N * row + B * H * (D_QK * 2 + D_C * 2 + 4)


def attention_flops(seqlens, H: int) -> int:
    """2*H*(576+512) multiply-adds' worth of flops per cached token (QK^T and PV)."""
    return int(np.sum(seqlens)) * 2 * H * (D_QK + D_C)
