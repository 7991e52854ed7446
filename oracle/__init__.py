"""fp64 CPU oracle for MLA latent-KV decode (ctypes over mla_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg may use this module; the product path never does. It shares no
code with the CUDA library and imports nothing from it.

Arrays cross the boundary as numpy: bf16 values as uint16 bit patterns, float
values as float64, indices as int32. Results are float64 (the cache rows written
by ``append_kv`` are bf16 bits, the cache's storage type).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libmla_oracle.so")

ERR_ARG = 1
ERR_RANGE = 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain IEEE fp64: no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i8p = ctypes.POINTER(ctypes.c_int8)
_i = ctypes.c_int
_d = ctypes.c_double


def _declare(L):
    L.mla_oracle_f64_to_bf16.argtypes = [_d]
    L.mla_oracle_f64_to_bf16.restype = ctypes.c_uint16
    L.mla_oracle_rope.argtypes = [_f64p, _i, _i, _i32p, _d]
    L.mla_oracle_rope.restype = None
    L.mla_oracle_kv_elements_mha.argtypes = [_i, _i, _i]
    L.mla_oracle_kv_elements_mha.restype = ctypes.c_longlong
    L.mla_oracle_kv_elements_mla.argtypes = [_i, _i, _i]
    L.mla_oracle_kv_elements_mla.restype = ctypes.c_longlong
    L.mla_oracle_append_kv.argtypes = [_u16p, _i, _i, _u16p, _i, _i, _i32p, _i32p, _i, _u16p,
                                       _i, _i, _d]
    L.mla_oracle_append_kv.restype = _i
    L.mla_oracle_decode_absorbed.argtypes = [_f64p, _f64p, _u16p, _i, _i, _i32p, _i, _i32p,
                                             _i, _i, _i, _i, _d, _f64p, _f64p, _f64p]
    L.mla_oracle_decode_absorbed.restype = _i
    L.mla_oracle_decode_expanded.argtypes = [_f64p, _f64p, _u16p, _i, _i, _i32p, _i, _i32p,
                                             _i, _i, _i, _i, _i, _i, _f64p, _f64p, _d, _f64p,
                                             _f64p]
    L.mla_oracle_decode_expanded.restype = _i
    L.mla_oracle_combine.argtypes = [_f64p, _f64p, _i, _i, _i, _i, _f64p, _f64p]
    L.mla_oracle_combine.restype = None
    L.mla_oracle_absorb_q.argtypes = [_u16p, _i, _i, _u16p, _i, _u16p, _u16p, _u16p, _i, _i,
                                      _i, _i, _i32p, _d, _f64p, _f64p, _f64p]
    L.mla_oracle_absorb_q.restype = _i
    L.mla_oracle_out_absorb.argtypes = [_f64p, _i, _i, _i, _i, _u16p, _u16p, _i, _f64p]
    L.mla_oracle_out_absorb.restype = _i
    L.mla_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    L.mla_oracle_e4m3_to_f64.restype = _d
    L.mla_oracle_f64_to_e4m3.argtypes = [_d]
    L.mla_oracle_f64_to_e4m3.restype = ctypes.c_uint8
    L.mla_oracle_quantize_rows_fp8.argtypes = [_f64p, ctypes.c_long, _i, _u8p, _i8p]
    L.mla_oracle_quantize_rows_fp8.restype = None
    L.mla_oracle_dequantize_rows_fp8.argtypes = [_u8p, _i8p, ctypes.c_long, _i, _f64p]
    L.mla_oracle_dequantize_rows_fp8.restype = None
    L.mla_oracle_append_kv_fp8.argtypes = [_u16p, _i, _i, _u16p, _i, _i, _i32p, _i32p, _i, _u8p,
                                           _i8p, _i, _i, _d]
    L.mla_oracle_append_kv_fp8.restype = _i


def _p(a, t):
    return a.ctypes.data_as(t)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle returned status {code}")
        self.code = code


def _check(rc, allow_range=False):
    if rc == 0 or (allow_range and rc == ERR_RANGE):
        return rc
    raise OracleError(rc)


# --------------------------------------------------------------- primitives

def f64_to_bf16(x: float) -> int:
    return int(lib().mla_oracle_f64_to_bf16(float(x)))


def rope(x, pos, theta=10000.0):
    """Rotate rows of x ([n, d_rope] float64) by their positions; returns a new array."""
    x = _f64(x).copy()
    n, d = x.shape
    pos = _i32(pos)
    lib().mla_oracle_rope(_p(x, _f64p), n, d, _p(pos, _i32p), float(theta))
    return x


def kv_elements_mha(layers, heads, head_dim):
    return int(lib().mla_oracle_kv_elements_mha(layers, heads, head_dim))


def kv_elements_mla(layers, d_c, d_rope):
    return int(lib().mla_oracle_kv_elements_mla(layers, d_c, d_rope))


# ------------------------------------------------------------------- steps

def append_kv(h, w_dkr, pos, block_table, kv_cache, d_c=512, rope_theta=10000.0,
              allow_range=False):
    """Project h into [c_kv | RoPE(k_rope)] and write it into kv_cache (modified in place)."""
    h, w_dkr, kv_cache = _u16(h), _u16(w_dkr), kv_cache
    assert kv_cache.flags.c_contiguous and kv_cache.dtype == np.uint16
    B, dm = h.shape
    D = w_dkr.shape[0]
    nb, bs, D2 = kv_cache.shape
    assert D2 == D
    bt, pos = _i32(block_table), _i32(pos)
    rc = lib().mla_oracle_append_kv(_p(h, _u16p), B, dm, _p(w_dkr, _u16p), d_c, D - d_c,
                                    _p(pos, _i32p), _p(bt, _i32p), bt.shape[1],
                                    _p(kv_cache, _u16p), nb, bs, float(rope_theta))
    return _check(rc, allow_range)


def decode_absorbed(q_lat, q_rope, kv_cache, block_table, seqlens, scale, want_probs=False,
                    allow_range=False):
    """Absorbed-form decode attention. Returns (out [B,H,d_c], lse [B,H][, probs of (0,0)])."""
    q_lat, q_rope = _f64(q_lat), _f64(q_rope)
    B, H, d_c = q_lat.shape
    d_r = q_rope.shape[2]
    kv_cache = _u16(kv_cache)
    nb, bs, D = kv_cache.shape
    assert D == d_c + d_r
    bt, L = _i32(block_table), _i32(seqlens)
    out = np.zeros((B, H, d_c))
    lse = np.zeros((B, H))
    probs = np.zeros(max(int(L[0]) if B else 1, 1)) if want_probs else None
    rc = lib().mla_oracle_decode_absorbed(
        _p(q_lat, _f64p), _p(q_rope, _f64p), _p(kv_cache, _u16p), nb, bs, _p(bt, _i32p),
        bt.shape[1], _p(L, _i32p), B, H, d_c, d_r, float(scale), _p(out, _f64p),
        _p(lse, _f64p), _p(probs, _f64p) if want_probs else None)
    _check(rc, allow_range)
    return (out, lse, probs) if want_probs else (out, lse)


def decode_absorbed_mq(q_lat, q_rope, kv_cache, block_table, seqlens, scale):
    """Decode attention for s_q query tokens per sequence (the draft tokens a main model
    verifies in one pass: "When MoE meets MLA" §5.3 item 3, "DeepSeek V3 MoE inference"
    §6). The draft rows are the last s_q of each sequence's seqlens[b] cached rows, and
    draft token t (0-based) attends causally: to the rows j < seqlens[b] - (s_q - 1 - t).
    Each (b, t) is therefore the absorbed decode of a sequence of that length over b's
    blocks. q_lat [B,s_q,H,d_c], q_rope [B,s_q,H,d_r] -> (out [B,s_q,H,d_c], lse [B,s_q,H])."""
    q_lat, q_rope = _f64(q_lat), _f64(q_rope)
    B, s_q, H, d_c = q_lat.shape
    d_r = q_rope.shape[3]
    bt, L = _i32(block_table), _i32(seqlens)
    visible = np.maximum(L[:, None] - (s_q - 1 - np.arange(s_q))[None, :], 0)
    out, lse = decode_absorbed(q_lat.reshape(B * s_q, H, d_c), q_rope.reshape(B * s_q, H, d_r),
                               kv_cache, np.repeat(bt, s_q, axis=0),
                               visible.reshape(-1).astype(np.int32), scale)
    return out.reshape(B, s_q, H, d_c), lse.reshape(B, s_q, H)


def decode_expanded(q_nope, q_rope, kv_cache, block_table, seqlens, w_uk, w_uv, scale):
    """Expanded (explicit K/V per head) decode attention. Returns (out_v [B,H,d_v], lse [B,H])."""
    q_nope, q_rope, w_uk, w_uv = _f64(q_nope), _f64(q_rope), _f64(w_uk), _f64(w_uv)
    B, H, d_h = q_nope.shape
    d_r = q_rope.shape[2]
    d_v = w_uv.shape[1]
    d_c = w_uk.shape[2]
    kv_cache = _u16(kv_cache)
    nb, bs, D = kv_cache.shape
    assert D == d_c + d_r and w_uk.shape == (H, d_h, d_c) and w_uv.shape == (H, d_v, d_c)
    bt, L = _i32(block_table), _i32(seqlens)
    out = np.zeros((B, H, d_v))
    lse = np.zeros((B, H))
    rc = lib().mla_oracle_decode_expanded(
        _p(q_nope, _f64p), _p(q_rope, _f64p), _p(kv_cache, _u16p), nb, bs, _p(bt, _i32p),
        bt.shape[1], _p(L, _i32p), B, H, d_c, d_r, d_h, d_v, _p(w_uk, _f64p), _p(w_uv, _f64p),
        float(scale), _p(out, _f64p), _p(lse, _f64p))
    _check(rc)
    return out, lse


def prefill_expanded(q_nope, q_rope, kv_cache, block_table_row, prefix, w_uk, w_uv, scale):
    """Chunked prefill of one sequence in the expanded (un-absorbed) form ("LLM inference:
    from the memory wall to the compute wall" §2.2: prefill is compute-bound, so the keys
    and values are projected back per head instead of absorbing the projections into the
    query). The chunk's C tokens sit at positions prefix .. prefix + C - 1 of the cache
    (already appended); query i attends causally to the positions j <= prefix + i:
      k_nope_j = W_UK[h] c_kv_j,  v_j = W_UV[h] c_kv_j,  s_j = scale (q_nope . k_nope_j +
      q_rope . k_rope_j),  out = sum_j softmax(s)_j v_j,  lse = ln sum_j exp(s_j),
    in fp64 from the bf16 inputs, each latent row projected once (numpy matmuls).
    q_nope [C,H,d_h], q_rope [C,H,d_r] -> (out_v [C,H,d_v], lse [C,H])."""
    q_nope, q_rope, w_uk, w_uv = _f64(q_nope), _f64(q_rope), _f64(w_uk), _f64(w_uv)
    C, H, _ = q_nope.shape
    bt = _i32(block_table_row).reshape(-1)
    cache = _u16(kv_cache)
    nb, bs, D = cache.shape
    d_c = w_uk.shape[2]
    T = int(prefix) + C
    blk = bt[np.arange(T) // bs]
    if np.any(blk < 0) or np.any(blk >= nb):
        raise ValueError("block id out of range")
    bits = cache[blk, np.arange(T) % bs].astype(np.uint32) << 16
    rows = bits.view(np.float32).astype(np.float64)          # [T][D], exact bf16 values
    ckv, kr = rows[:, :d_c], rows[:, d_c:]
    k_nope = np.einsum("hdc,tc->htd", w_uk, ckv)              # [H][T][d_h]
    v = np.einsum("hdc,tc->htd", w_uv, ckv)                   # [H][T][d_v]
    out = np.zeros((C, H, w_uv.shape[1]))
    lse = np.zeros((C, H))
    for i in range(C):
        n = int(prefix) + i + 1
        for h in range(H):
            s = scale * (k_nope[h, :n] @ q_nope[i, h] + kr[:n] @ q_rope[i, h])
            mx = s.max()
            e = np.exp(s - mx)
            den = e.sum()
            out[i, h] = (e / den) @ v[h, :n]
            lse[i, h] = mx + np.log(den)
    return out, lse


# ------------------------------------------------------------ fp8 cache

def e4m3_to_f64(code: int) -> float:
    """Value of an e4m3 code (1-4-3, bias 7, no infinities, all-ones = NaN)."""
    return float(lib().mla_oracle_e4m3_to_f64(int(code) & 0xFF))


def f64_to_e4m3(x: float) -> int:
    """Nearest e4m3 code, ties to the even mantissa, saturating at 448."""
    return int(lib().mla_oracle_f64_to_e4m3(float(x)))


def quantize_rows_fp8(x):
    """Rows of values [..., D] (float64) -> (codes uint8 [..., D], exps int8 [...]): per row
    the power-of-two scale 2^e with e the smallest integer such that max|x| 2^-e <= 448."""
    x = _f64(x)
    shp = x.shape
    D = shp[-1]
    rows = int(np.prod(shp[:-1])) if len(shp) > 1 else 1
    codes = np.zeros(shp, dtype=np.uint8)
    exps = np.zeros(shp[:-1], dtype=np.int8)
    lib().mla_oracle_quantize_rows_fp8(_p(x, _f64p), rows, D, _p(codes, _u8p), _p(exps, _i8p))
    return codes, exps


def dequantize_fp8(codes, exps):
    """codes [..., D] uint8, exps [...] int8 -> code * 2^e as float64."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    exps = np.ascontiguousarray(exps, dtype=np.int8)
    D = codes.shape[-1]
    rows = int(np.prod(codes.shape[:-1])) if codes.ndim > 1 else 1
    out = np.zeros(codes.shape)
    lib().mla_oracle_dequantize_rows_fp8(_p(codes, _u8p), _p(exps, _i8p), rows, D,
                                         _p(out, _f64p))
    return out


def fp8_cache_as_bf16(codes, exps):
    """The dequantised FP8 cache as bf16 bits. Every value code * 2^e has at most 4
    significant bits, so it is exactly a bf16 value (checked)."""
    v = dequantize_fp8(codes, exps).astype(np.float32)
    bits = v.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "dequantised value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def append_kv_fp8(h, w_dkr, pos, block_table, kv_codes, kv_exps, d_c=512, rope_theta=10000.0,
                  allow_range=False):
    """append_kv into an FP8 cache: the fp64 row is quantised (per-row power-of-two scale)
    and written into kv_codes [nb, bs, D] uint8 and kv_exps [nb, bs] int8 (in place)."""
    h, w_dkr = _u16(h), _u16(w_dkr)
    assert kv_codes.flags.c_contiguous and kv_codes.dtype == np.uint8
    assert kv_exps.flags.c_contiguous and kv_exps.dtype == np.int8
    B, dm = h.shape
    D = w_dkr.shape[0]
    nb, bs, D2 = kv_codes.shape
    assert D2 == D and kv_exps.shape == (nb, bs)
    bt, pos = _i32(block_table), _i32(pos)
    rc = lib().mla_oracle_append_kv_fp8(_p(h, _u16p), B, dm, _p(w_dkr, _u16p), d_c, D - d_c,
                                        _p(pos, _i32p), _p(bt, _i32p), bt.shape[1],
                                        _p(kv_codes, _u8p), _p(kv_exps, _i8p), nb, bs,
                                        float(rope_theta))
    return _check(rc, allow_range)


def decode_absorbed_fp8(q_lat, q_rope, kv_codes, kv_exps, block_table, seqlens, scale,
                        allow_range=False):
    """Absorbed decode attention over an FP8 cache: the attention of decode_absorbed over
    the dequantised rows code * 2^e (exactly bf16 values, so the bf16 routine applies)."""
    return decode_absorbed(q_lat, q_rope, fp8_cache_as_bf16(kv_codes, kv_exps), block_table,
                           seqlens, scale, allow_range=allow_range)


def combine(o_part, lse_part):
    """Merge split results: o_part [B,S,H,d], lse_part [B,S,H] -> (out [B,H,d], lse [B,H])."""
    o_part, lse_part = _f64(o_part), _f64(lse_part)
    B, S, H, d = o_part.shape
    out = np.zeros((B, H, d))
    lse = np.zeros((B, H))
    lib().mla_oracle_combine(_p(o_part, _f64p), _p(lse_part, _f64p), B, S, H, d,
                             _p(out, _f64p), _p(lse, _f64p))
    return out, lse


def absorb_q(h, w_dq, w_uq, w_qr, w_uk, pos, rope_theta=10000.0, want_nope=False):
    """Query side of the absorbed step. Returns (q_lat, q_rope[, q_nope]) as float64."""
    h, w_dq, w_uq, w_qr, w_uk = map(_u16, (h, w_dq, w_uq, w_qr, w_uk))
    B, dm = h.shape
    ql = w_dq.shape[0]
    H, d_h, d_c = w_uk.shape
    d_r = w_qr.shape[0] // H
    pos = _i32(pos)
    q_lat = np.zeros((B, H, d_c))
    q_rope = np.zeros((B, H, d_r))
    q_nope = np.zeros((B, H, d_h)) if want_nope else None
    rc = lib().mla_oracle_absorb_q(_p(h, _u16p), B, dm, _p(w_dq, _u16p), ql, _p(w_uq, _u16p),
                                   _p(w_qr, _u16p), _p(w_uk, _u16p), H, d_h, d_r, d_c,
                                   _p(pos, _i32p), float(rope_theta), _p(q_lat, _f64p),
                                   _p(q_rope, _f64p), _p(q_nope, _f64p) if want_nope else None)
    _check(rc)
    return (q_lat, q_rope, q_nope) if want_nope else (q_lat, q_rope)


def out_absorb(o_lat, w_uv, w_o):
    """Output side of the absorbed step: y [B, d_model] float64."""
    o_lat = _f64(o_lat)
    w_uv, w_o = _u16(w_uv), _u16(w_o)
    B, H, d_c = o_lat.shape
    d_v = w_uv.shape[1]
    dm = w_o.shape[0]
    y = np.zeros((B, dm))
    rc = lib().mla_oracle_out_absorb(_p(o_lat, _f64p), B, H, d_c, d_v, _p(w_uv, _u16p),
                                     _p(w_o, _u16p), dm, _p(y, _f64p))
    _check(rc)
    return y
