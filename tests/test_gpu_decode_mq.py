"""GPU parity of mla_decode_attention_mq (s_q draft tokens per sequence, causal among
them) against the fp64 oracle, through the C ABI, on seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_13_gb300 import synth
from tests.helpers import (assert_close_rows, assert_lse, dev_bf16, dev_i32, host_bits,
                           host_f64_from_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla as m
    return m


def _case(B, s_q, H, seqlens, seed):
    """Inputs of B sequences with s_q x H query rows each (rows ordered token, head)."""
    w = synth.Workload("mq", B, s_q * H, tuple(seqlens), None, True)
    d = synth.make_attention_inputs(w, seed=seed)
    d["q_lat"] = d["q_lat"].reshape(B, s_q, H, 512)
    d["q_rope"] = d["q_rope"].reshape(B, s_q, H, 64)
    return d


def _run(mla, d, num_splits):
    max_len = int(np.max(d["seqlens"]))
    out, lse, ws = mla.decode_attention_mq(
        dev_bf16(d["q_lat"]), dev_bf16(d["q_rope"]), dev_bf16(d["kv_cache"]),
        dev_i32(d["block_table"]), dev_i32(d["seqlens"]), max_len, d["scale"], num_splits)
    return out, lse, mla.check_device_status(ws)


def _oracle(d):
    return oracle.decode_absorbed_mq(synth.bf16_bits_to_f64(d["q_lat"]),
                                     synth.bf16_bits_to_f64(d["q_rope"]), d["kv_cache"],
                                     d["block_table"], d["seqlens"], d["scale"])


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_draft_tokens_ragged_lengths(mla, splits):
    # lengths 1 and 3 leave the first draft tokens with nothing to attend to
    B, s_q, H = 6, 4, 16
    d = _case(B, s_q, H, (100, 3, 65, 1, 300, 64), seed=11)
    out, lse, st = _run(mla, d, splits)
    assert st == 0
    ref, lref = _oracle(d)
    got = host_f64_from_bf16(out).reshape(B * s_q * H, 512)
    assert_close_rows(got, ref.reshape(-1, 512))
    assert_lse(lse.cpu().numpy().astype(np.float64).reshape(-1), lref.reshape(-1))


@pytest.mark.parametrize("s_q,H", [(2, 64), (3, 32), (8, 16)])
def test_draft_rows_fill_the_tile(mla, s_q, H):
    B = 5
    d = _case(B, s_q, H, (700, 129, 64, 513, 2), seed=12)
    out, lse, st = _run(mla, d, 0)
    assert st == 0
    ref, lref = _oracle(d)
    assert_close_rows(host_f64_from_bf16(out).reshape(-1, 512), ref.reshape(-1, 512))
    assert_lse(lse.cpu().numpy().astype(np.float64).reshape(-1), lref.reshape(-1))


def test_single_query_token_is_plain_decode(mla):
    B, H = 4, 128
    d = _case(B, 1, H, (1000, 70, 5, 256), seed=13)
    out, lse, st = _run(mla, d, 0)
    max_len = int(np.max(d["seqlens"]))
    out1, lse1, ws = mla.decode_attention(
        dev_bf16(d["q_lat"].reshape(B, H, 512)), dev_bf16(d["q_rope"].reshape(B, H, 64)),
        dev_bf16(d["kv_cache"]), dev_i32(d["block_table"]), dev_i32(d["seqlens"]), max_len,
        d["scale"], 0)
    assert st == 0 and mla.check_device_status(ws) == 0
    assert np.array_equal(host_bits(out).reshape(B, H, 512), host_bits(out1))
    assert torch.equal(lse.reshape(B, H), lse1)
