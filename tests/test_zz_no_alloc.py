"""mla_decode_attention_noalloc: the entry point for callers that cannot give the
library a workspace (graph capture, framework-owned memory, allocation-free serving
loops). Its split-KV scratch is the library's own device array; these checks compare
it, through the C ABI, with mla_decode_attention on the same inputs, two calls in a
row. Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

from mla_latent_kv_13_gb300 import synth
from tests.helpers import assert_close_rows, assert_lse, dev_bf16, dev_i32, host_f64_from_bf16

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, L):
    w = synth.Workload("noalloc", B, H, tuple(L), None, True)
    d = synth.make_attention_inputs(w, seed=seed)
    return d, dict(q_lat=dev_bf16(d["q_lat"]), q_rope=dev_bf16(d["q_rope"]),
                   cache=dev_bf16(d["kv_cache"]), bt=dev_i32(d["block_table"]),
                   seqlens=dev_i32(d["seqlens"]))


def test_noalloc_matches_workspace_path_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla
    cases = [(0, 4, 128, (3000, 700, 1, 2222), 4), (1, 3, 64, (5000, 64, 4100), 7)]
    for seed, B, H, L, splits in cases:   # two calls in a row, different inputs
        d, t = _inputs(seed, B, H, L)
        # the scratch is really used: these requests need split partials
        assert mla.decode_workspace_size(B, H, max(L), splits) > mla.WS_HEADER_BYTES
        ref_out, ref_lse, ws = mla.decode_attention(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                                    t["seqlens"], max(L), d["scale"], splits)
        assert mla.check_device_status(ws) == 0
        out, lse = mla.decode_attention_noalloc(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                                t["seqlens"], max(L), d["scale"], splits)
        torch.cuda.synchronize()
        assert_close_rows(host_f64_from_bf16(out), host_f64_from_bf16(ref_out), "noalloc out")
        assert_lse(lse.cpu().numpy(), ref_lse.cpu().numpy())


def test_noalloc_rejects_requests_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla
    B, H, L = 64, 128, 8192
    assert mla.decode_workspace_size(B, H, L, 64) > 32 << 20
    d, t = _inputs(2, 2, 128, (100, 100))
    with pytest.raises(mla.MLAError) as e:
        # B=64 with 64 splits needs far more than the fixed scratch: rejected on the host
        q = torch.zeros((B, H, 512), dtype=torch.bfloat16, device="cuda")
        r = torch.zeros((B, H, 64), dtype=torch.bfloat16, device="cuda")
        bt = torch.zeros((B, 128), dtype=torch.int32, device="cuda")
        sl = torch.zeros((B,), dtype=torch.int32, device="cuda")
        mla.decode_attention_noalloc(q, r, t["cache"], bt, sl, L, d["scale"], 64)
    assert e.value.code == 3   # MLA_ERR_WORKSPACE
