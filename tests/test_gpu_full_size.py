"""Prefill parity at the full workload sizes, in the launch configuration the
benchmark times: the whole layer runs on the GPU, and the fp64 oracle checks
64 query rows drawn without replacement (seed 1) plus the rows at the edges of
the band and the sinks, for the first and last query head of the last sequence.

Workloads (inputs seeded exactly as the benchmark seeds them):
  mistral_like_prefill   B=1 H=32 Hkv=8  n=16384  d=128 w=4096 g=0
  gemma3_local_prefill   B=2 H=32 Hkv=16 n=32768  d=128 w=1024 g=0
  long_sink_prefill      B=1 H=32 Hkv=8  n=131072 d=128 w=4096 g=4, sink keys x4
  gemma3_global_prefill  B=2 H=32 Hkv=16 n=32768  d=128 w=n (full causal) g=0
  mha_prefill            B=1 H=32 Hkv=32 n=16384  d=128 w=4096 g=0 (a group of one)
  dilated_prefill        B=1 H=32 Hkv=8  n=16384  d=128 dilated w=1024 r=4
  strided_prefill        B=1 H=32 Hkv=8  n=65536  d=128 strided r=256
  landmark_prefill       B=1 H=32 Hkv=8  n=16384  d=128 w=4096 g=4 landmarks r=64
"""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import BF16_MAX_ABS, BF16_MEAN_ABS

N_SAMPLED = 64


def edge_rows(B, H, n, w, g):
    cand = {0, 1, 3, g, w - 2, w - 1, w, w + 1, w + g - 1, w + g, w + g + 1, 4095, 4096, 4098,
            4099, 255, 256, 257, 1023, 1024, n // 2, n - 2, n - 1}
    rows = sorted(i for i in cand if 0 <= i < n)
    return [(B - 1, h, i) for h in (0, H - 1) for i in rows]


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mistral_like_prefill", "gemma3_local_prefill",
                                  "long_sink_prefill", "gemma3_global_prefill", "mha_prefill",
                                  "dilated_prefill", "strided_prefill", "landmark_prefill"])
def test_prefill_full_size_sampled_rows(swa, oracle_mod, name):
    c = synthetic.WORKLOADS[name]
    B, H, Hkv, n, d, w, g = (c[k] for k in ("B", "H", "Hkv", "n", "d", "w", "g"))
    pattern, r = c.get("pattern", "window"), c.get("r", 1)
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=0,
                                 sink_scale=c["sink_scale"], device="cuda")
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    if pattern == "window":
        out = swa.prefill(x.Q, x.K, x.V, w, g, x.scale, lse=lse)
    else:
        out = swa.prefill_pattern(x.Q, x.K, x.V, pattern, w, g, r, x.scale, lse=lse)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    rows = synthetic.sample_rows(B, H, n, N_SAMPLED, seed=1).numpy()
    rows = np.concatenate([rows, np.array(edge_rows(B, H, n, w, g), dtype=np.int64)])
    b_idx, h_idx, i_idx = (torch.as_tensor(rows[:, k], device="cuda") for k in range(3))
    q_rows = x.Q[b_idx, h_idx, i_idx].cpu()
    got = out[b_idx, h_idx, i_idx].double().cpu().numpy()
    got_lse = lse[b_idx, h_idx, i_idx].double().cpu().numpy()
    Kh, Vh = x.K.cpu(), x.V.cpu()
    del x, out, lse
    torch.cuda.empty_cache()
    if pattern == "window":
        O, L = oracle_mod.prefill_rows(q_rows, Kh, Vh, H, w, g, synthetic.default_scale(d), rows)
    else:
        O, L = oracle_mod.prefill_pattern_rows(q_rows, Kh, Vh, H, w, g, r, pattern,
                                               synthetic.default_scale(d), rows)
    assert np.isfinite(got).all()
    err = np.abs(got - O)
    assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, \
        f"{name}: max {err.max():.3e} mean {err.mean():.3e}"
    assert np.abs(got_lse - L).max() < 2e-3
