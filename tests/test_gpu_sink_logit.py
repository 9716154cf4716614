"""Learned per-head sink logit ("Sliding Window and Sparse Attention, from
Longformer to CSA2", section 6, stage 3): the CUDA path against the fp64
oracle for prefill (tensor-core and fp32 kernels) and decode, element by
element, and the -inf logit reproducing the path without one bit for bit."""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close

PREFILL_CASES = [
    # B, H, Hkv, n, d, w, g
    (1, 4, 2, 513, 128, 200, 4),   # GQA pairs (two-head kernel), ragged tail
    (1, 3, 1, 300, 128, 64, 0),    # odd group: one-head kernel
    (2, 2, 2, 256, 64, 100, 2),    # d = 64
]


def logits(H, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(H, generator=g, dtype=torch.float64) * 6.0 - 2.0)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g", PREFILL_CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_sink_logit_matches_oracle(swa, oracle_mod, B, H, Hkv, n, d, w, g, dtype):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype=dtype, seed=n + d, sink_scale=4.0,
                                 device="cuda")
    sl = logits(H, n)
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    out = swa.prefill(x.Q, x.K, x.V, w, g, x.scale, lse=lse,
                      sink_logit=sl.float().cuda())
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    O, L = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale, sink_logit=sl.float().double())
    assert_close(out, O, dtype, f"prefill sink logit {B,H,Hkv,n,d,w,g}")
    tol = 2e-3 if dtype == "bf16" else 1e-5
    assert np.abs(lse.cpu().double().numpy() - L).max() < tol


@pytest.mark.gpu
def test_prefill_sink_logit_minus_inf_is_bit_exact(swa):
    x = synthetic.prefill_inputs(1, 4, 2, 400, 128, 150, 2, dtype="bf16", seed=4, device="cuda")
    plain = swa.prefill(x.Q, x.K, x.V, 150, 2, x.scale)
    none = swa.prefill(x.Q, x.K, x.V, 150, 2, x.scale,
                       sink_logit=torch.full((4,), -float("inf"), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(plain, none)


DECODE_CASES = [
    # B, H, Hkv, d, w, g, positions
    (2, 4, 1, 128, 64, 4, [200, 67]),
    (3, 8, 2, 128, 64, 4, [0, 5, 63]),
    (2, 2, 2, 64, 100, 0, [99, 1000]),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,d,w,g,pos", DECODE_CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_sink_logit_matches_oracle(swa, oracle_mod, B, H, Hkv, d, w, g, pos, dtype):
    x = synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, pos, dtype=dtype, seed=w + g + 1,
                                      sink_scale=4.0, device="cuda")
    sl = logits(H, w)
    O, L = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), w, g, x.scale,
                                   sink_logit=sl.float().double())
    for splits in (0, 1, 3):
        lse = torch.empty(B, H, dtype=torch.float32, device="cuda")
        out = swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale, lse=lse, num_splits=splits,
                         sink_logit=sl.float().cuda())
        torch.cuda.synchronize()
        assert_close(out, O, dtype, f"decode sink logit splits={splits}")
        tol = 2e-3 if dtype == "bf16" else 1e-5
        assert np.abs(lse.cpu().double().numpy() - L).max() < tol
    assert swa.device_status() == 0
