"""Thin Python binding of libmla (include/mla.h): argument marshalling only.

Every function takes torch tensors that live on the current CUDA device, passes
their data pointers and the current stream to the C ABI, and raises MLAError on a
non-zero status. Importing this module loads libmla.so and raises if it is
missing: there is no other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libmla.so not found at {LIB_PATH}; build it with "
        "`python -m mla_latent_kv_13_gb300.build` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

D_C, D_ROPE, D_QK, BLOCK, D_NOPE, D_V = 512, 64, 576, 64, 128, 128
WS_HEADER_BYTES = 256

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
          3: "MLA_ERR_WORKSPACE", 4: "MLA_ERR_OUT_OF_RANGE", 5: "MLA_ERR_TIMEOUT",
          6: "MLA_ERR_CUDA"}


class MLAError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
_szp = ctypes.POINTER(ctypes.c_size_t)

_SIGS = {
    "mla_status_string": ([_i], ctypes.c_char_p),
    "mla_append_kv_workspace_size": ([_i, _i, _szp], _i),
    "mla_append_kv": ([_vp, _i, _i, _vp, _vp, _vp, _i, _vp, _i, _f, _vp, _sz, _vp], _i),
    "mla_decode_workspace_size": ([_i, _i, _i, _i, _szp], _i),
    "mla_decode_plan": ([_i, _i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)], _i),
    "mla_projection_launches": ([_i, _i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i),
                                 ctypes.POINTER(_i), ctypes.POINTER(_i)], _i),
    "mla_decode_schedule": ([_vp, _i, _i, _i, _vp, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)],
                            _i),
    "mla_decode_attention": ([_vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _f, _i, _vp, _sz,
                              _vp, _vp, _vp], _i),
    "mla_decode_prepare": ([_vp, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "mla_decode_attention_prepared": ([_vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _f, _i, _vp,
                                       _sz, _vp, _vp, _vp], _i),
    "mla_decode_combine": ([_vp, _vp, _i, _i, _i, _vp, _vp, _vp], _i),
    "mla_decode_attention_partial": ([_vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _f, _i, _vp,
                                      _sz, _vp, _vp, _vp], _i),
    "mla_decode_combine_ranks": ([_vp, _vp, _i, _i, _i, _vp, _vp, _vp], _i),
    "mla_quantize_kv_fp8": ([_vp, ctypes.c_long, _vp, _vp, _vp], _i),
    "mla_dequantize_kv_fp8": ([_vp, _vp, ctypes.c_long, _vp, _vp], _i),
    "mla_append_kv_fp8": ([_vp, _i, _i, _vp, _vp, _vp, _i, _vp, _vp, _i, _f, _vp, _sz, _vp], _i),
    "mla_decode_attention_fp8": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _f, _i, _vp,
                                  _sz, _vp, _vp, _vp], _i),
    "mla_decode_mq_workspace_size": ([_i, _i, _i, _i, _i, _szp], _i),
    "mla_decode_attention_mq": ([_vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _i, _f, _i, _vp,
                                 _sz, _vp, _vp, _vp], _i),
    "mla_decode_attention_noalloc": ([_vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _f, _i, _vp,
                                      _vp, _vp], _i),
    "mla_absorb_q_workspace_size": ([_i, _i, _i, _i, _szp], _i),
    "mla_absorb_q": ([_vp, _i, _i, _vp, _i, _vp, _vp, _vp, _i, _vp, _f, _vp, _sz, _vp, _vp,
                      _vp], _i),
    "mla_append_absorb_q_workspace_size": ([_i, _i, _i, _i, _szp], _i),
    "mla_append_absorb_q": ([_vp, _i, _i, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _vp, _vp, _vp,
                             _i, _f, _vp, _sz, _vp, _vp, _vp], _i),
    "mla_out_absorb_workspace_size": ([_i, _i, _i, _szp], _i),
    "mla_out_absorb": ([_vp, _i, _i, _vp, _vp, _i, _vp, _sz, _vp, _vp], _i),
    "mla_clear_device_status": ([_vp, _vp], _i),
    "mla_selftest_wait_timeout": ([ctypes.c_uint, _vp, _sz, _vp], _i),
    "mla_prefill_workspace_size": ([_i, _i, _i, _szp], _i),
    "mla_prefill_attention": ([_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _vp, _f, _vp, _sz,
                               _vp, _vp, _vp], _i),
    "mla_check_device_status": ([_vp, _vp], _i),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

EXPORTED = tuple(_SIGS)


def lib():
    return _lib


def _ok(rc: int, where: str):
    if rc != 0:
        raise MLAError(rc, where)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensors pass as their 16-bit patterns; uint16/int16 views pass through."""
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected bf16 storage, got {t.dtype}")
    return t


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _size(fn, *args) -> int:
    out = ctypes.c_size_t(0)
    _ok(getattr(_lib, fn)(*args, ctypes.byref(out)), fn)
    return int(out.value)


def alloc_workspace(nbytes: int, device=None, stream=None) -> torch.Tensor:
    """Caller-owned workspace (256-byte aligned by the caching allocator), error word cleared."""
    ws = torch.empty(max(nbytes, WS_HEADER_BYTES), dtype=torch.uint8,
                     device=device or torch.cuda.current_device())
    assert ws.data_ptr() % 256 == 0
    _ok(_lib.mla_clear_device_status(_ptr(ws), _stream(stream)), "mla_clear_device_status")
    return ws


# ------------------------------------------------------------------ sizes

def append_kv_workspace_size(B, d_model):
    return _size("mla_append_kv_workspace_size", B, d_model)


def decode_workspace_size(B, H, max_seqlen, num_splits=0):
    return _size("mla_decode_workspace_size", B, H, max_seqlen, num_splits)


def decode_plan(B, H, max_seqlen, num_splits=0):
    """(splits, launches) of mla_decode_attention for these arguments: splits = 0 for the
    balanced schedule, else the fixed token ranges per sequence."""
    s, n = _i(0), _i(0)
    rc = _lib.mla_decode_plan(B, H, max_seqlen, num_splits, ctypes.byref(s), ctypes.byref(n))
    if rc != 0:
        raise MLAError(rc, "mla_decode_plan")
    return s.value, n.value


def projection_launches(B, d_model, q_lora, H):
    """(append, absorb_q, out_absorb, append_absorb_q): the kernels one call of each
    launches for these shapes on the current device."""
    a, q, o, aq = _i(0), _i(0), _i(0), _i(0)
    rc = _lib.mla_projection_launches(B, d_model, q_lora, H, ctypes.byref(a), ctypes.byref(q),
                                      ctypes.byref(o), ctypes.byref(aq))
    if rc != 0:
        raise MLAError(rc, "mla_projection_launches")
    return a.value, q.value, o.value, aq.value


def decode_schedule(seqlens, max_blocks, clusters):
    """The balanced schedule for these lengths, computed on the host: a list of segments
    (work unit, sequence, first block, end block, part or -1 when written directly) and
    the number of fp32 parts."""
    import numpy as np
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    cnt, parts = _i(0), _i(0)

    def call(buf, cap):
        rc = _lib.mla_decode_schedule(sl.ctypes.data_as(ctypes.c_void_p), len(sl), max_blocks,
                                      clusters, buf.ctypes.data_as(ctypes.c_void_p), cap,
                                      ctypes.byref(cnt), ctypes.byref(parts))
        if rc != 0:
            raise MLAError(rc, "mla_decode_schedule")

    call(np.zeros((1, 5), dtype=np.int32), 0)  # count only
    buf = np.zeros((max(cnt.value, 1), 5), dtype=np.int32)
    call(buf, cnt.value)
    return [tuple(int(x) for x in r) for r in buf[:cnt.value]], parts.value


def absorb_q_workspace_size(B, d_model, q_lora, H):
    return _size("mla_absorb_q_workspace_size", B, d_model, q_lora, H)


def append_absorb_q_workspace_size(B, d_model, q_lora, H):
    return _size("mla_append_absorb_q_workspace_size", B, d_model, q_lora, H)


def out_absorb_workspace_size(B, H, d_model):
    return _size("mla_out_absorb_workspace_size", B, H, d_model)


# ------------------------------------------------------------------ calls

def append_kv(h, w_dkr, pos, block_table, kv_cache, rope_theta=10000.0, workspace=None,
              stream=None):
    B, dm = h.shape
    nb = kv_cache.shape[0]
    if workspace is None:
        workspace = alloc_workspace(append_kv_workspace_size(B, dm), stream=stream)
    rc = _lib.mla_append_kv(_ptr(_bits(h)), B, dm, _ptr(_bits(w_dkr)), _ptr(pos),
                            _ptr(block_table), block_table.shape[1], _ptr(_bits(kv_cache)), nb,
                            float(rope_theta), _ptr(workspace), workspace.numel(),
                            _stream(stream))
    _ok(rc, "mla_append_kv")
    return workspace


def decode_attention(q_lat, q_rope, kv_cache, block_table, seqlens, max_seqlen, scale,
                     num_splits=0, out=None, lse=None, workspace=None, stream=None):
    """Returns (out [B,H,512] bf16, lse [B,H] fp32, workspace)."""
    B, H, _ = q_lat.shape
    dev = q_lat.device
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(decode_workspace_size(B, H, max_seqlen, num_splits),
                                    stream=stream)
    rc = _lib.mla_decode_attention(_ptr(_bits(q_lat)), _ptr(_bits(q_rope)),
                                   _ptr(_bits(kv_cache)), kv_cache.shape[0], _ptr(block_table),
                                   block_table.shape[1], _ptr(seqlens), B, H, int(max_seqlen),
                                   float(scale), int(num_splits), _ptr(workspace),
                                   workspace.numel(), _ptr(out), _ptr(lse), _stream(stream))
    _ok(rc, "mla_decode_attention")
    return out, lse, workspace


def decode_prepare(seqlens, B, H, max_seqlen, num_splits, workspace, stream=None):
    """mla_decode_prepare: the balanced schedule for these lengths into the workspace (nothing
    when the plan is a fixed split), for decode_attention_prepared calls over the same
    lengths and arguments."""
    rc = _lib.mla_decode_prepare(_ptr(seqlens), int(B), int(H), int(max_seqlen), int(num_splits),
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    _ok(rc, "mla_decode_prepare")
    return workspace


def decode_attention_prepared(q_lat, q_rope, kv_cache, block_table, seqlens, max_seqlen, scale,
                              num_splits, out, lse, workspace, stream=None):
    """mla_decode_attention_prepared: decode_attention over a workspace that decode_prepare
    filled for the same lengths and arguments. Returns (out, lse, workspace)."""
    B, H, _ = q_lat.shape
    rc = _lib.mla_decode_attention_prepared(
        _ptr(_bits(q_lat)), _ptr(_bits(q_rope)), _ptr(_bits(kv_cache)), kv_cache.shape[0],
        _ptr(block_table), block_table.shape[1], _ptr(seqlens), B, H, int(max_seqlen),
        float(scale), int(num_splits), _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
        _stream(stream))
    _ok(rc, "mla_decode_attention_prepared")
    return out, lse, workspace


def decode_mq_workspace_size(B, s_q, H, max_seqlen, num_splits=0):
    return _size("mla_decode_mq_workspace_size", B, s_q, H, max_seqlen, num_splits)


def decode_attention_mq(q_lat, q_rope, kv_cache, block_table, seqlens, max_seqlen, scale,
                        num_splits=0, out=None, lse=None, workspace=None, stream=None):
    """mla_decode_attention_mq: q_lat [B,s_q,H,512], q_rope [B,s_q,H,64] (draft tokens,
    causal among them). Returns (out [B,s_q,H,512] bf16, lse [B,s_q,H] fp32, workspace)."""
    B, s_q, H, _ = q_lat.shape
    dev = q_lat.device
    if out is None:
        out = torch.empty((B, s_q, H, D_C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(decode_mq_workspace_size(B, s_q, H, max_seqlen, num_splits),
                                    stream=stream)
    rc = _lib.mla_decode_attention_mq(_ptr(_bits(q_lat)), _ptr(_bits(q_rope)),
                                      _ptr(_bits(kv_cache)), kv_cache.shape[0],
                                      _ptr(block_table), block_table.shape[1], _ptr(seqlens), B,
                                      s_q, H, int(max_seqlen), float(scale), int(num_splits),
                                      _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
                                      _stream(stream))
    _ok(rc, "mla_decode_attention_mq")
    return out, lse, workspace


def decode_attention_noalloc(q_lat, q_rope, kv_cache, block_table, seqlens, max_seqlen, scale,
                             num_splits=0, out=None, lse=None, stream=None):
    """mla_decode_attention_noalloc: same results, scratch in the library's own device
    array (no workspace). Returns (out, lse)."""
    B, H, _ = q_lat.shape
    dev = q_lat.device
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    rc = _lib.mla_decode_attention_noalloc(_ptr(_bits(q_lat)), _ptr(_bits(q_rope)),
                                           _ptr(_bits(kv_cache)), kv_cache.shape[0],
                                           _ptr(block_table), block_table.shape[1],
                                           _ptr(seqlens), B, H, int(max_seqlen), float(scale),
                                           int(num_splits), _ptr(out), _ptr(lse),
                                           _stream(stream))
    _ok(rc, "mla_decode_attention_noalloc")
    return out, lse


def decode_combine(o_part, lse_part, out=None, lse=None, stream=None):
    B, S, H, _ = o_part.shape
    dev = o_part.device
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    rc = _lib.mla_decode_combine(_ptr(o_part), _ptr(lse_part), B, S, H, _ptr(out), _ptr(lse),
                                 _stream(stream))
    _ok(rc, "mla_decode_combine")
    return out, lse


def decode_attention_partial(q_lat, q_rope, kv_cache, block_table, seqlens, max_seqlen, scale,
                             num_splits=0, o_part=None, lse_part=None, workspace=None,
                             stream=None):
    """mla_decode_attention_partial: attention over this rank's token ranges only.
    Returns (o_part [B,H,512] fp32, lse_part [B,H] fp32, workspace)."""
    B, H, _ = q_lat.shape
    dev = q_lat.device
    if o_part is None:
        o_part = torch.empty((B, H, D_C), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((B, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(decode_workspace_size(B, H, max_seqlen, num_splits),
                                    stream=stream)
    rc = _lib.mla_decode_attention_partial(_ptr(_bits(q_lat)), _ptr(_bits(q_rope)),
                                           _ptr(_bits(kv_cache)), kv_cache.shape[0],
                                           _ptr(block_table), block_table.shape[1],
                                           _ptr(seqlens), B, H, int(max_seqlen), float(scale),
                                           int(num_splits), _ptr(workspace), workspace.numel(),
                                           _ptr(o_part), _ptr(lse_part), _stream(stream))
    _ok(rc, "mla_decode_attention_partial")
    return o_part, lse_part, workspace


def decode_combine_ranks(o_parts, lse_parts, out=None, lse=None, stream=None):
    """mla_decode_combine_ranks: o_parts [G,B,H,512] fp32, lse_parts [G,B,H] fp32 ->
    (out [B,H,512] bf16, lse [B,H] fp32)."""
    G, B, H, _ = o_parts.shape
    dev = o_parts.device
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    rc = _lib.mla_decode_combine_ranks(_ptr(o_parts), _ptr(lse_parts), G, B, H, _ptr(out),
                                       _ptr(lse), _stream(stream))
    _ok(rc, "mla_decode_combine_ranks")
    return out, lse


def _u8(t):
    if t.dtype not in (torch.uint8, torch.int8):
        raise TypeError(f"expected 8-bit storage, got {t.dtype}")
    return t


def quantize_kv_fp8(rows_bf16, codes=None, exps=None, stream=None):
    """mla_quantize_kv_fp8: bf16 rows [..., 576] -> (codes uint8 [..., 576], exps int8 [...])."""
    shp = rows_bf16.shape
    rows = rows_bf16.numel() // D_QK
    dev = rows_bf16.device
    if codes is None:
        codes = torch.empty(shp, dtype=torch.uint8, device=dev)
    if exps is None:
        exps = torch.empty(shp[:-1], dtype=torch.int8, device=dev)
    _ok(_lib.mla_quantize_kv_fp8(_ptr(_bits(rows_bf16)), rows, _ptr(_u8(codes)), _ptr(_u8(exps)),
                                 _stream(stream)), "mla_quantize_kv_fp8")
    return codes, exps


def dequantize_kv_fp8(codes, exps, out=None, stream=None):
    """mla_dequantize_kv_fp8: (codes [..., 576], exps [...]) -> bf16 rows [..., 576]."""
    rows = codes.numel() // D_QK
    if out is None:
        out = torch.empty(codes.shape, dtype=torch.bfloat16, device=codes.device)
    _ok(_lib.mla_dequantize_kv_fp8(_ptr(_u8(codes)), _ptr(_u8(exps)), rows, _ptr(_bits(out)),
                                   _stream(stream)), "mla_dequantize_kv_fp8")
    return out


def append_kv_fp8(h, w_dkr, pos, block_table, kv_codes, kv_exps, rope_theta=10000.0,
                  workspace=None, stream=None):
    B, dm = h.shape
    nb = kv_codes.shape[0]
    if workspace is None:
        workspace = alloc_workspace(append_kv_workspace_size(B, dm), stream=stream)
    rc = _lib.mla_append_kv_fp8(_ptr(_bits(h)), B, dm, _ptr(_bits(w_dkr)), _ptr(pos),
                                _ptr(block_table), block_table.shape[1], _ptr(_u8(kv_codes)),
                                _ptr(_u8(kv_exps)), nb, float(rope_theta), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _ok(rc, "mla_append_kv_fp8")
    return workspace


def decode_attention_fp8(q_lat, q_rope, kv_codes, kv_exps, block_table, seqlens, max_seqlen,
                         scale, num_splits=0, out=None, lse=None, workspace=None, stream=None):
    """mla_decode_attention_fp8. Returns (out [B,H,512] bf16, lse [B,H] fp32, workspace)."""
    B, H, _ = q_lat.shape
    dev = q_lat.device
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(decode_workspace_size(B, H, max_seqlen, num_splits),
                                    stream=stream)
    rc = _lib.mla_decode_attention_fp8(_ptr(_bits(q_lat)), _ptr(_bits(q_rope)),
                                       _ptr(_u8(kv_codes)), _ptr(_u8(kv_exps)), kv_codes.shape[0],
                                       _ptr(block_table), block_table.shape[1], _ptr(seqlens), B,
                                       H, int(max_seqlen), float(scale), int(num_splits),
                                       _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
                                       _stream(stream))
    _ok(rc, "mla_decode_attention_fp8")
    return out, lse, workspace


def absorb_q(h, w_dq, w_uq, w_qr, w_uk, pos, rope_theta=10000.0, q_lat=None, q_rope=None,
             workspace=None, stream=None):
    B, dm = h.shape
    ql = w_dq.shape[0]
    H = w_uk.shape[0]
    dev = h.device
    if q_lat is None:
        q_lat = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
    if q_rope is None:
        q_rope = torch.empty((B, H, D_ROPE), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = alloc_workspace(absorb_q_workspace_size(B, dm, ql, H), stream=stream)
    rc = _lib.mla_absorb_q(_ptr(_bits(h)), B, dm, _ptr(_bits(w_dq)), ql, _ptr(_bits(w_uq)),
                           _ptr(_bits(w_qr)), _ptr(_bits(w_uk)), H, _ptr(pos), float(rope_theta),
                           _ptr(workspace), workspace.numel(), _ptr(q_lat), _ptr(q_rope),
                           _stream(stream))
    _ok(rc, "mla_absorb_q")
    return q_lat, q_rope, workspace


def append_absorb_q(h, w_dkr, pos, block_table, kv_cache, w_dq, w_uq, w_qr, w_uk,
                    rope_theta=10000.0, q_lat=None, q_rope=None, workspace=None, stream=None):
    """append_kv and absorb_q in one call (both read h): the new rows go into kv_cache,
    returns (q_lat, q_rope, workspace)."""
    B, dm = h.shape
    ql = w_dq.shape[0]
    H = w_uk.shape[0]
    dev = h.device
    if q_lat is None:
        q_lat = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
    if q_rope is None:
        q_rope = torch.empty((B, H, D_ROPE), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = alloc_workspace(append_absorb_q_workspace_size(B, dm, ql, H), stream=stream)
    rc = _lib.mla_append_absorb_q(_ptr(_bits(h)), B, dm, _ptr(_bits(w_dkr)), _ptr(pos),
                                  _ptr(block_table), block_table.shape[1], _ptr(_bits(kv_cache)),
                                  kv_cache.shape[0], _ptr(_bits(w_dq)), ql, _ptr(_bits(w_uq)),
                                  _ptr(_bits(w_qr)), _ptr(_bits(w_uk)), H, float(rope_theta),
                                  _ptr(workspace), workspace.numel(), _ptr(q_lat), _ptr(q_rope),
                                  _stream(stream))
    _ok(rc, "mla_append_absorb_q")
    return q_lat, q_rope, workspace


def out_absorb(o_lat, w_uv, w_o, y=None, workspace=None, stream=None):
    B, H, _ = o_lat.shape
    dm = w_o.shape[0]
    if y is None:
        y = torch.empty((B, dm), dtype=torch.bfloat16, device=o_lat.device)
    if workspace is None:
        workspace = alloc_workspace(out_absorb_workspace_size(B, H, dm), stream=stream)
    rc = _lib.mla_out_absorb(_ptr(_bits(o_lat)), B, H, _ptr(_bits(w_uv)), _ptr(_bits(w_o)), dm,
                             _ptr(workspace), workspace.numel(), _ptr(y), _stream(stream))
    _ok(rc, "mla_out_absorb")
    return y, workspace


def check_device_status(workspace, stream=None) -> int:
    """Synchronise and return (and clear) the workspace's device error word."""
    return int(_lib.mla_check_device_status(_ptr(workspace), _stream(stream)))


def prefill_workspace_size(H, prefix, chunk):
    return _size("mla_prefill_workspace_size", H, prefix, chunk)


def prefill_attention(q_nope, q_rope, kv_cache, block_table_row, prefix, w_uk, w_uv, scale,
                      out=None, lse=None, workspace=None, stream=None):
    """mla_prefill_attention: q_nope [C,H,128], q_rope [C,H,64] of one sequence's chunk at
    positions prefix.. (already appended). Returns (out [C,H,128] bf16, lse [C,H] fp32,
    workspace)."""
    C, H, _ = q_nope.shape
    dev = q_nope.device
    if out is None:
        out = torch.empty((C, H, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((C, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(prefill_workspace_size(H, prefix, C), stream=stream)
    rc = _lib.mla_prefill_attention(_ptr(_bits(q_nope)), _ptr(_bits(q_rope)),
                                    _ptr(_bits(kv_cache)), kv_cache.shape[0],
                                    _ptr(block_table_row), block_table_row.numel(), int(prefix),
                                    C, H, _ptr(_bits(w_uk)), _ptr(_bits(w_uv)), float(scale),
                                    _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
                                    _stream(stream))
    _ok(rc, "mla_prefill_attention")
    return out, lse, workspace


def selftest_wait_timeout(limit_us, workspace, stream=None):
    """Run the failure-detection self-test; returns (status, detail) from the workspace
    header after it (expected: MLA_ERR_TIMEOUT and at least limit_us microseconds)."""
    _ok(_lib.mla_selftest_wait_timeout(int(limit_us), _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "mla_selftest_wait_timeout")
    torch.cuda.synchronize(workspace.device)
    hdr = workspace[:8].view(torch.int32).cpu().tolist()
    return hdr[0] & 0xFFFFFFFF, hdr[1] & 0xFFFFFFFF


def clear_device_status(workspace, stream=None):
    _ok(_lib.mla_clear_device_status(_ptr(workspace), _stream(stream)), "mla_clear_device_status")


class DecodeStep:
    """The absorbed MLA decode step for one layer: append the new token's latent,
    build the absorbed query, attend over the paged cache, project the latent
    output back. Holds caller-owned workspaces; every step runs in libmla kernels."""

    def __init__(self, weights: dict, B: int, H: int, max_seqlen: int, num_splits: int = 0,
                 rope_theta: float = 10000.0, scale: float | None = None):
        self.w = weights
        self.B, self.H = B, H
        self.dm = weights["w_dkr"].shape[1]
        self.ql = weights["w_dq"].shape[0]
        self.max_seqlen = max_seqlen
        self.num_splits = num_splits
        self.theta = rope_theta
        self.scale = (1.0 / (D_NOPE + D_ROPE) ** 0.5) if scale is None else scale
        dev = weights["w_dkr"].device
        self.ws_q = alloc_workspace(append_absorb_q_workspace_size(B, self.dm, self.ql, H))
        self.ws_att = alloc_workspace(decode_workspace_size(B, H, max_seqlen, num_splits))
        self.ws_out = alloc_workspace(out_absorb_workspace_size(B, H, self.dm))
        self.q_lat = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
        self.q_rope = torch.empty((B, H, D_ROPE), dtype=torch.bfloat16, device=dev)
        self.o_lat = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, H), dtype=torch.float32, device=dev)
        self.y = torch.empty((B, self.dm), dtype=torch.bfloat16, device=dev)

    def __call__(self, h, pos, seqlens_after, block_table, kv_cache, stream=None, out=None):
        """One step; the result y [B, d_model] bf16 goes to `out` if given, else to the
        step's own buffer (returned either way). One stream: the new cache rows and the
        absorbed query (one call: both read h), the attention schedule (it reads only the
        lengths, so it runs beside the last query projection), the attention, the output
        projections."""
        w = self.w
        y = self.y if out is None else out
        main = torch.cuda.current_stream() if stream is None else stream
        append_absorb_q(h, w["w_dkr"], pos, block_table, kv_cache, w["w_dq"], w["w_uq"],
                        w["w_qr"], w["w_uk"], self.theta, self.q_lat, self.q_rope, self.ws_q,
                        main)
        decode_prepare(seqlens_after, self.B, self.H, self.max_seqlen, self.num_splits,
                       self.ws_att, main)
        decode_attention_prepared(self.q_lat, self.q_rope, kv_cache, block_table, seqlens_after,
                                  self.max_seqlen, self.scale, self.num_splits, self.o_lat,
                                  self.lse, self.ws_att, main)
        out_absorb(self.o_lat, w["w_uv"], w["w_o"], y, self.ws_out, main)
        return y

    def check(self, stream=None) -> int:
        codes = [check_device_status(ws, stream) for ws in (self.ws_q, self.ws_att, self.ws_out)]
        return next((c for c in codes if c), 0)
