"""Shared test helpers: tensor conversion and the parity bars.

Bars, against the float64 oracle on the same inputs:
  * permutations and doc_start: bit-exact;
  * bf16 attention (fp32 accumulation): max |out - ref| <= 2e-2 and
    mean |out - ref| <= 2e-3;
  * fp32 attention: max |out - ref| <= 1e-5;
  * lse: max |lse - ref| <= 1e-3 (bf16), 1e-5 (fp32).
"""

import numpy as np
import torch

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-5
LSE_BF16 = 1e-3
LSE_F32 = 1e-5


def np32(t):
    return t.detach().float().cpu().numpy()


def npi(t):
    return t.detach().cpu().numpy()


def check_attention(out, lse, ref_out, ref_lse, dtype, what=""):
    """out/lse: numpy arrays from the GPU (already gathered to the rows the
    reference covers); ref_*: the oracle's float64 results."""
    err = np.abs(out.astype(np.float64) - ref_out)
    finite = np.isfinite(ref_lse)
    lerr = np.abs(np.where(finite, lse.astype(np.float64), 0.0) - np.where(finite, ref_lse, 0.0))
    assert np.array_equal(np.isfinite(lse), finite), f"{what}: -inf rows differ"
    lmax = lerr[finite].max() if finite.any() else 0.0
    if dtype == "bf16":
        assert err.max() <= BF16_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
        assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
        assert lmax <= LSE_BF16, f"{what}: lse err {lmax:.3e}"
    else:
        assert err.max() <= F32_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
        assert lmax <= LSE_F32, f"{what}: lse err {lmax:.3e}"
    return float(err.max()), float(err.mean()), float(lmax)


def torch_dtype(name):
    return torch.bfloat16 if name == "bf16" else torch.float32


# Gradients: errors normalised by max(1, max |ref|) of each tensor (gradient
# magnitudes grow with the number of contributing rows).  bf16 storage with
# fp32 accumulation: max <= 2e-2, mean <= 2e-3; fp32: max <= 1e-4 (sums of up
# to S fp32 products).
GRAD_BF16_MAX, GRAD_BF16_MEAN, GRAD_F32_MAX = 2e-2, 2e-3, 1e-4


def check_grad(got, ref, dtype, what=""):
    scale = max(1.0, float(np.abs(ref).max()))
    err = np.abs(got.astype(np.float64) - ref) / scale
    if dtype == "bf16":
        assert err.max() <= GRAD_BF16_MAX, f"{what}: max rel err {err.max():.3e}"
        assert err.mean() <= GRAD_BF16_MEAN, f"{what}: mean rel err {err.mean():.3e}"
    else:
        assert err.max() <= GRAD_F32_MAX, f"{what}: max rel err {err.max():.3e}"
    return float(err.max()), float(err.mean())
