"""Shared helpers for the GPU-vs-oracle parity tests.

Error measure: err = max |gpu - oracle| / rms(oracle) over a tensor, as the
contract states it.  Tolerances: 2e-3 for bf16 inputs with fp32 state, 1e-5 for
fp32 inputs.  When the GPU writes a bf16 OUTPUT, storing the fp32 result in
bf16 rounds each element by up to 2^-8 of its magnitude (half an ulp), which
no kernel can avoid; that term is allowed per element on top of the
tolerance:  |gpu - oracle| <= tol * rms(oracle) + 2^-8 |oracle|.
"""
import numpy as np
import torch

TOL_BF16 = 2e-3
TOL_FP32 = 1e-5
BF16_HALF_ULP_REL = 2.0 ** -8


def to64(t):
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(gpu, ref, out_is_bf16=False):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    if rms == 0.0:
        rms = 1.0
    diff = np.abs(gpu - ref)
    if out_is_bf16:
        diff = np.maximum(diff - BF16_HALF_ULP_REL * np.abs(ref), 0.0)
    return float(diff.max() / rms) if diff.size else 0.0


def assert_close(gpu, ref, tol, what, out_is_bf16=False):
    e = rel_err(gpu, ref, out_is_bf16)
    assert np.isfinite(np.asarray(gpu, np.float64)).all(), f"{what}: non-finite values"
    assert e <= tol, f"{what}: max-abs/rms error {e:.3e} > {tol:.1e}"
    return e


def assert_gated_close(gpu, ref, out_is_bf16, what="o_gated"):
    """The gated output o^g = sigma(g) RMSNorm(o~) against the oracle with the plain bound:
    max |gpu - oracle| / rms(oracle) <= 2e-3 over the whole tensor (plus the bf16 half-ulp
    per element when the output is bf16).  RMSNorm divides each (token, head) row by its own
    RMS, which could in principle magnify an error of o~ on rows of small norm; measured, the
    errors of o~ scale with the row's own size, so no per-row allowance is needed."""
    return assert_close(gpu, ref, TOL_BF16, what, out_is_bf16)
