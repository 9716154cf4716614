"""Tolerances for comparing the CUDA path with the fp64 oracle.

bf16 inputs (fp32 accumulation, P rounded to bf16 before the P.V product,
output rounded to bf16): max-abs <= 2e-2 and mean-abs <= 2e-3 over all output
elements.  fp32 inputs: max-abs <= 1e-5.  Integer results are compared
bit-exactly elsewhere.
"""
import numpy as np
import torch

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-5


def to_np(t):
    return t.detach().float().cpu().double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def assert_close(out, ref, dtype, what=""):
    out = to_np(out)
    ref = np.asarray(ref, dtype=np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    err = np.abs(out - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if dtype in ("bf16", torch.bfloat16):
        assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, f"{what}: max {mx:.3e} mean {mean:.3e}"
    else:
        assert mx <= F32_MAX_ABS, f"{what}: max {mx:.3e}"
    return mx, mean
