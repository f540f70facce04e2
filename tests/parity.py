"""Shared helpers of the GPU parity tests: device copies and the tolerance check.

Tolerance (element by element against the fp64 oracle on the same bf16 inputs):
max |dO| <= 2e-2 and mean |dO| <= 2e-3; LSE error |dLSE| / max(1, |LSE|) <= 1e-3
(absolute near zero, where a relative bound is ill-posed: a causal first row
has LSE = s_00, which can be ~0).
"""
import numpy as np

MAX_ABS_O = 2e-2
MEAN_ABS_O = 2e-3
LSE_ERR = 1e-3


def to_dev(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def o_to_f64(o):
    return o.float().cpu().numpy().astype(np.float64)


def errors(o, lse, o_ref, lse_ref):
    do = np.abs(o - o_ref)
    dl = np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    return float(do.max()), float(do.mean()), float(dl.max())


def assert_close(o, lse, o_ref, lse_ref, what=""):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    mx, mean, le = errors(o, lse, o_ref, lse_ref)
    assert mx <= MAX_ABS_O and mean <= MEAN_ABS_O and le <= LSE_ERR, \
        f"{what}: max|dO|={mx:.3e} mean|dO|={mean:.3e} lse_err={le:.3e}"
    return mx, mean, le
