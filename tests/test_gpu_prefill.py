"""GPU parity of mla_prefill_attention (chunked prefill, expanded form, causal over the
prefix and the chunk) against the fp64 oracle, through the C ABI, on seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_13_gb300 import synth
from tests.helpers import assert_close_rows, dev_bf16, dev_i32, host_f64_from_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_13_gb300 import mla as m
    return m


def _case(prefix, C, H, seed):
    d = synth.make_attention_inputs(synth.Workload("pf", 1, H, (prefix + C,), None, True),
                                    seed=seed)
    rng = np.random.default_rng(seed + 1000)
    d["q_nope"] = synth.f32_to_bf16_bits(rng.standard_normal((C, H, 128)).astype(np.float32))
    d["q_rope"] = synth.f32_to_bf16_bits(rng.standard_normal((C, H, 64)).astype(np.float32))
    # up-projections with the weight scale of the full-step workload
    d["w_uk"] = synth.f32_to_bf16_bits((rng.standard_normal((H, 128, 512)) * 0.02).astype(np.float32))
    d["w_uv"] = synth.f32_to_bf16_bits((rng.standard_normal((H, 128, 512)) * 0.02).astype(np.float32))
    return d


def _run(mla, d, prefix):
    out, lse, ws = mla.prefill_attention(dev_bf16(d["q_nope"]), dev_bf16(d["q_rope"]),
                                         dev_bf16(d["kv_cache"]), dev_i32(d["block_table"][0]),
                                         prefix, dev_bf16(d["w_uk"]), dev_bf16(d["w_uv"]),
                                         d["scale"])
    return out, lse, mla.check_device_status(ws)


@pytest.mark.parametrize("prefix,C,H", [(0, 64, 16), (100, 200, 16), (300, 130, 32),
                                        (5, 1, 16), (0, 257, 128)])
def test_prefill_matches_oracle(mla, prefix, C, H):
    d = _case(prefix, C, H, seed=prefix + C + H)
    out, lse, st = _run(mla, d, prefix)
    assert st == 0
    f = synth.bf16_bits_to_f64
    ref, lref = oracle.prefill_expanded(f(d["q_nope"]), f(d["q_rope"]), d["kv_cache"],
                                        d["block_table"][0], prefix, f(d["w_uk"]), f(d["w_uv"]),
                                        d["scale"])
    assert_close_rows(host_f64_from_bf16(out).reshape(-1, 128), ref.reshape(-1, 128))
    # lse: 1e-3 as for decode, plus what storing k_nope = W_UK c_kv in bf16 can move a score
    # by (round to nearest: |dk| <= 2^-9 |k|, and lse moves by at most the largest score
    # change): scale * 2^-9 * max_j sum_d |q_d| |k_jd| per query row
    qn = f(d["q_nope"])
    bt = d["block_table"][0]
    rows = np.stack([f(d["kv_cache"][bt[j // 64], j % 64, :512]) for j in range(prefix + C)])
    k = np.einsum("hdc,tc->htd", f(d["w_uk"]), rows)
    bound = np.empty((C, H))
    for i in range(C):
        n = prefix + i + 1
        bound[i] = d["scale"] * 2.0 ** -9 * np.array([np.max(np.abs(k[h, :n]) @ np.abs(qn[i, h]))
                                                      for h in range(H)])
    err = np.abs(lse.cpu().numpy().astype(np.float64) - lref)
    assert np.all(err <= 1e-3 + bound), f"lse: max err {err.max():.3e}, excess {(err - bound).max():.3e}"


def test_prefill_out_of_range_block_is_reported(mla):
    d = _case(64, 64, 16, seed=3)
    d["block_table"] = d["block_table"].copy()
    d["block_table"][0, 0] = d["num_blocks"] + 5
    _, _, st = _run(mla, d, 64)
    assert st == 4  # MLA_ERR_OUT_OF_RANGE
