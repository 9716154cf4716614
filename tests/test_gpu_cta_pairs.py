"""The window-path prefill on the CTA-pair kernel (swa_debug_prefill_cta_pairs:
tcgen05 cta_group::2, two SMs per MMA of 256 rows) against the fp64 oracle,
and against the default kernel, whose output it reproduces bit for bit (the
same MMA k-steps and the same softmax code per row).  ("Sliding Window and
Sparse Attention, from Longformer to CSA2", sections 2 and 4.)"""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import BF16_MAX_ABS, BF16_MEAN_ABS, assert_close

CASES = [
    # B, H, Hkv, n, d, w, g
    (1, 4, 1, 256, 128, 128, 0),    # G = 4: one K/V stream for both halves
    (1, 4, 2, 300, 128, 100, 0),    # G = 2: a stream per half; ragged tail
    (1, 8, 2, 2000, 128, 500, 0),   # several items per cluster
    (2, 8, 4, 1500, 128, 700, 20),  # G = 2, a full 128-key sink tile
    (1, 8, 1, 1000, 128, 1000, 0),  # G = 8, full causal
    (3, 12, 6, 777, 128, 64, 0),    # window narrower than a tile, three sequences
    (1, 4, 1, 1, 128, 1, 0),        # one row, w = 1
    (1, 8, 2, 1200, 128, 300, 4),   # four sinks in a tile of their own, below the band
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g", CASES)
def test_cta_pairs_matches_oracle_and_default_kernel(swa, oracle_mod, B, H, Hkv, n, d, w, g):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=n + w + g,
                                 sink_scale=4.0, device="cuda")
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    out = swa.prefill_cta_pairs(x.Q, x.K, x.V, w, g, x.scale, lse=lse)
    ref = swa.prefill(x.Q, x.K, x.V, w, g, x.scale)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    O, L = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
    assert_close(out, O, "bf16", "CTA-pair prefill")
    assert np.abs(lse.double().cpu().numpy() - L).max() < 2e-3
    assert torch.equal(out, ref), "differs from the default kernel"


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mistral_like_prefill", "gemma3_local_prefill"])
def test_cta_pairs_full_size_sampled_rows(swa, oracle_mod, name):
    c = synthetic.WORKLOADS[name]
    B, H, Hkv, n, d, w, g = (c[k] for k in ("B", "H", "Hkv", "n", "d", "w", "g"))
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=0,
                                 sink_scale=c["sink_scale"], device="cuda")
    out = swa.prefill_cta_pairs(x.Q, x.K, x.V, w, g, x.scale)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    rows = synthetic.sample_rows(B, H, n, 64, seed=1).numpy()
    b_idx, h_idx, i_idx = (torch.as_tensor(rows[:, k], device="cuda") for k in range(3))
    got = out[b_idx, h_idx, i_idx].double().cpu().numpy()
    O, _ = oracle_mod.prefill_rows(x.Q[b_idx, h_idx, i_idx].cpu(), x.K.cpu(), x.V.cpu(), H, w, g,
                                   synthetic.default_scale(d), rows)
    err = np.abs(got - O)
    assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, \
        f"{name}: max {err.max():.3e} mean {err.mean():.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("H,Hkv,d,g", [(4, 1, 64, 0),    # d = 64
                                       (3, 1, 128, 0),   # odd group
                                       (2, 1, 128, 0)])  # H % 4 != 0
def test_cta_pairs_refuses_other_shapes(swa, H, Hkv, d, g):
    x = synthetic.prefill_inputs(1, H, Hkv, 256, d, 64, g, dtype="bf16", seed=0, device="cuda")
    with pytest.raises(swa.SwaError) as e:
        swa.prefill_cta_pairs(x.Q, x.K, x.V, 64, g, x.scale)
    assert e.value.status == -2
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_cta_pairs_wait_runs_out_and_recovers(swa, oracle_mod):
    """The bounded-wait path of the CTA pair: the injected launch leaves out its
    first key/value copy, CTA 0's issuer gives up after 1 ms, both CTAs' roles
    stop on the abort flag or their own limit and meet at the exit barrier; the
    status word reports the timeout and the next launches are exact."""
    assert swa.device_status() == 0
    B, H, Hkv, n, d, w, g = 1, 4, 1, 384, 128, 128, 0
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=7, device="cuda")
    swa.inject_stall("prefill", 1_000_000)
    swa.prefill_cta_pairs(x.Q, x.K, x.V, w, g, x.scale)
    assert swa.device_status() == -4  # SWA_ERR_DEVICE_TIMEOUT
    assert swa.device_status() == 0
    out = swa.prefill_cta_pairs(x.Q, x.K, x.V, w, g, x.scale)
    ref = swa.prefill(x.Q, x.K, x.V, w, g, x.scale)
    torch.cuda.synchronize()
    O, _ = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
    assert_close(out, O, "bf16", "CTA-pair prefill after recovery")
    assert torch.equal(out, ref)
    assert swa.device_status() == 0
