"""mla_decode_attention_noalloc: the entry point for callers that cannot give the
library a workspace -- code inside a CUDA-graph stream capture, plugins whose host
framework owns every device allocation, serving loops that must not call cudaMalloc on
their hot path. Its split-KV scratch is the library's own device array; these checks
compare it, through the C ABI, with mla_decode_attention on the same inputs, two calls
in a row (the array keeps the previous call's contents), for fixed splits and for the
balanced schedule, whose offsets, weights and parts all live in that array. Kept in a
file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

from mla_latent_kv_13_gb300 import synth
from tests.helpers import assert_close_rows, assert_lse, dev_bf16, dev_i32, host_f64_from_bf16

pytestmark = pytest.mark.gpu

SCRATCH = 40 << 20  # MLA_NOALLOC_SCRATCH_BYTES


def _inputs(seed, B, H, L):
    w = synth.Workload("noalloc", B, H, tuple(int(x) for x in L), None, True)
    d = synth.make_attention_inputs(w, seed=seed)
    return d, dict(q_lat=dev_bf16(d["q_lat"]), q_rope=dev_bf16(d["q_rope"]),
                   cache=dev_bf16(d["kv_cache"]), bt=dev_i32(d["block_table"]),
                   seqlens=dev_i32(d["seqlens"]))


def _compare_twice(cases):
    from mla_latent_kv_13_gb300 import mla
    for seed, B, H, L, splits in cases:  # consecutive calls share the scratch array
        d, t = _inputs(seed, B, H, L)
        ref_out, ref_lse, ws = mla.decode_attention(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                                    t["seqlens"], max(L), d["scale"], splits)
        assert mla.check_device_status(ws) == 0
        out, lse = mla.decode_attention_noalloc(t["q_lat"], t["q_rope"], t["cache"], t["bt"],
                                                t["seqlens"], max(L), d["scale"], splits)
        torch.cuda.synchronize()
        assert_close_rows(host_f64_from_bf16(out), host_f64_from_bf16(ref_out), "noalloc out")
        assert_lse(lse.cpu().numpy(), ref_lse.cpu().numpy())


def test_noalloc_matches_workspace_path_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla
    cases = [(0, 4, 128, (3000, 700, 1, 2222), 4), (1, 3, 64, (5000, 64, 4100), 7)]
    for _, B, H, L, splits in cases:  # the scratch is really used: split partials
        assert mla.decode_workspace_size(B, H, max(L), splits) > mla.WS_HEADER_BYTES
    _compare_twice(cases)


def test_noalloc_balanced_schedule_twice():
    """num_splits = 0 with more sequences than one wave of work units: the balanced
    schedule, whose tile offsets, weights, part indices and parts are all in the array."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla
    rng = np.random.default_rng(7)
    cases = []
    for seed, B in ((3, 100), (4, 90)):
        L = tuple(int(x) for x in rng.integers(1, 640, size=B))
        L = (0,) + L[1:]  # an empty sequence among them
        assert mla.decode_plan(B, 128, max(L), 0)[0] == 0  # the balanced schedule
        need = mla.decode_workspace_size(B, 128, max(L), 0)
        assert 32 << 20 < need <= SCRATCH
        cases.append((seed, B, 128, L, 0))
    _compare_twice(cases)
    # the headline serving shape's default plan fits as well
    assert mla.decode_workspace_size(128, 128, 8192, 0) <= SCRATCH


def test_noalloc_rejects_requests_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla
    B, H, L = 64, 128, 8192
    assert mla.decode_workspace_size(B, H, L, 64) > SCRATCH
    d, t = _inputs(2, 2, 128, (100, 100))
    q = torch.zeros((B, H, 512), dtype=torch.bfloat16, device="cuda")
    r = torch.zeros((B, H, 64), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, 128), dtype=torch.int32, device="cuda")
    sl = torch.zeros((B,), dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        # B=64 with 64 splits needs far more than the fixed scratch: rejected on the host
        mla.decode_attention_noalloc(q, r, t["cache"], bt, sl, L, d["scale"], 64)
    assert e.value.code == 3   # MLA_ERR_WORKSPACE
    with pytest.raises(mla.MLAError) as e:
        # an invalid argument is rejected before anything reaches the device
        mla.decode_attention_noalloc(q, r, t["cache"], bt, sl, L, -1.0, 1)
    assert e.value.code == 1   # MLA_ERR_INVALID_ARG
