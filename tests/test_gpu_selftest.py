"""Failure detection without a fault: a bounded wait that nothing satisfies gives up,
records MLA_ERR_TIMEOUT in the workspace, and the context stays usable."""
import numpy as np
import pytest
import torch

from mla_latent_kv_13_gb300 import synth
from tests.helpers import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla as m
    return m


@pytest.mark.parametrize("limit_us", [200, 2000])
def test_wait_that_nothing_satisfies_reports_timeout(mla, limit_us):
    ws = mla.alloc_workspace(256)
    mla.clear_device_status(ws)
    status, waited_us = mla.selftest_wait_timeout(limit_us, ws)
    assert status == 5  # MLA_ERR_TIMEOUT
    assert limit_us <= waited_us < limit_us + 100000
    assert mla.check_device_status(ws) == 5  # and clears
    assert mla.check_device_status(ws) == 0
    # the context is intact: a decode right after runs clean
    d = synth.make_attention_inputs(synth.WORKLOADS["tiny"], seed=0)
    out, lse, ws2 = mla.decode_attention(dev_bf16(d["q_lat"]), dev_bf16(d["q_rope"]),
                                         dev_bf16(d["kv_cache"]), dev_i32(d["block_table"]),
                                         dev_i32(d["seqlens"]), int(np.max(d["seqlens"])),
                                         d["scale"], 0)
    assert mla.check_device_status(ws2) == 0
    assert torch.isfinite(lse).all()
