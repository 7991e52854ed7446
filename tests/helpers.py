"""Shared test helpers: tensor conversion and the acceptance checks."""
import numpy as np
import torch

from mla_latent_kv_13_gb300 import synth

# acceptance: |err| <= ATOL + RTOL*|ref| elementwise; lse within LSE_ATOL; and the
# normwise relative error per (b, h) row at most NORM_RTOL (the elementwise bound is
# loose for small outputs, the normwise one is the sharp check).
ATOL, RTOL, LSE_ATOL, NORM_RTOL = 1e-2, 1e-2, 1e-3, 1e-2


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch.bfloat16)


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64_from_bf16(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits_to_f64(host_bits(t))


def assert_close_rows(got, ref, what="out", atol=ATOL, rtol=RTOL, norm_rtol=NORM_RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max():.3e}"
    g2 = got.reshape(-1, got.shape[-1])
    r2 = ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(r2, axis=1)
    en = np.linalg.norm(g2 - r2, axis=1)
    rel = np.where(rn > 0, en / np.maximum(rn, 1e-300), en)
    assert rel.max() <= norm_rtol, f"{what}: normwise rel err {rel.max():.3e}"
    return float(rel.max())


def assert_lse(got, ref, atol=LSE_ATOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), "lse: -inf pattern differs"
    d = np.abs(got[~inf_ref] - ref[~inf_ref])
    assert d.size == 0 or d.max() <= atol, f"lse: max err {d.max():.3e}"
