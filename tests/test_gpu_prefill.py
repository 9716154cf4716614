"""Prefill parity: the CUDA path (bf16 tensor-core kernel, fp32 CUDA-core
kernel) against the fp64 oracle, element by element, at sizes that span
several tiles with ragged tails, plus the degenerate cases."""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close

BF16_CASES = [
    # B, H, Hkv, n, d, w, g
    (1, 2, 1, 300, 128, 64, 0),      # ragged tail, window below one tile
    (1, 4, 2, 513, 128, 200, 4),     # sinks, ragged
    (2, 2, 2, 256, 64, 100, 0),      # d = 64
    (1, 1, 1, 1, 128, 4, 0),         # a single token
    (1, 2, 1, 400, 128, 1000, 0),    # window >= n: full causal attention
    (1, 8, 2, 1000, 128, 300, 3),    # GQA group of 4
    (1, 1, 1, 333, 128, 128, 130),   # more sinks than one key tile
    (1, 2, 1, 2048, 128, 512, 0),    # mostly full tiles
    (1, 2, 1, 130, 128, 129, 1),
    (3, 4, 1, 200, 64, 17, 2),       # several sequences, GQA 4, d = 64
    (1, 16, 1, 300, 128, 100, 2),    # group of 16: eight head pairs per kv head
    (2, 5, 1, 260, 128, 70, 1),      # odd group of 5: single-head kernel
    (2, 32, 16, 384, 128, 128, 0),   # the Gemma-3 head shape, window of one tile
    # the three mask rules of a partial tile: sinks reaching into the band's first
    # tile, a window far narrower than a tile beside sinks filling most of one,
    # and sinks spanning two tiles with a window of 5 (d = 64)
    (1, 2, 1, 600, 128, 100, 60),
    (1, 4, 2, 700, 128, 30, 120),
    (1, 2, 2, 500, 64, 5, 200),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g", BF16_CASES)
def test_prefill_bf16_matches_oracle(swa, oracle_mod, B, H, Hkv, n, d, w, g):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=n + w + g,
                                 sink_scale=4.0 if g else 1.0, device="cuda")
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    out = swa.prefill(x.Q, x.K, x.V, w, g, x.scale, lse=lse)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    O, L = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
    assert_close(out, O, "bf16", f"O {B,H,Hkv,n,d,w,g}")
    assert np.abs(lse.cpu().double().numpy() - L).max() < 2e-3


# A sink tile of its own: once the band of a 128-row query tile starts past
# key tile 0, the sinks 0..g-1 are read through key tile 0, masked to its first
# g keys.  Shapes with n well past w + 128, so most query tiles take it; a
# handful of sinks up to 17; odd groups (q-tile pairs) too.
SINK_TILE_CASES = [
    # B, H, Hkv, n, d, w, g
    (1, 4, 2, 900, 128, 100, 1),
    (2, 2, 1, 1000, 128, 64, 4),
    (1, 2, 1, 700, 64, 128, 16),
    (1, 2, 1, 700, 128, 128, 17),
    (1, 3, 1, 800, 128, 200, 4),     # a group of 3: q-tile pairs of one head
    (1, 1, 1, 1100, 64, 1, 5),       # window of one: only the sink tile and the diagonal
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g", SINK_TILE_CASES)
def test_prefill_sink_tile_below_band_matches_oracle(swa, oracle_mod, B, H, Hkv, n, d, w, g):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=n + g, sink_scale=4.0,
                                 device="cuda")
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    sink = torch.linspace(-2.0, 3.0, H, device="cuda", dtype=torch.float32)
    for sl in (None, sink):
        out = swa.prefill(x.Q, x.K, x.V, w, g, x.scale, lse=lse, sink_logit=sl)
        torch.cuda.synchronize()
        O, L = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale,
                                  sink_logit=None if sl is None else sl.cpu())
        assert_close(out, O, "bf16", f"O {B,H,Hkv,n,d,w,g} sink_logit={sl is not None}")
        assert np.abs(lse.cpu().double().numpy() - L).max() < 2e-3
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_prefill_bf16_window_one_is_value(swa):
    x = synthetic.prefill_inputs(1, 2, 1, 700, 128, 1, 0, dtype="bf16", seed=3, device="cuda")
    out = swa.prefill(x.Q, x.K, x.V, 1, 0, x.scale)
    torch.cuda.synchronize()
    ref = x.V.repeat_interleave(2, dim=1)
    assert torch.equal(out, ref)


@pytest.mark.gpu
def test_prefill_bf16_no_dependence_on_other_heads(swa):
    # the same head computed alone and inside a batch gives identical bits
    x = synthetic.prefill_inputs(2, 4, 2, 600, 128, 150, 2, dtype="bf16", seed=5, device="cuda")
    full = swa.prefill(x.Q, x.K, x.V, 150, 2, x.scale)
    one = swa.prefill(x.Q[1:2, 2:4].contiguous(), x.K[1:2, 1:2].contiguous(),
                      x.V[1:2, 1:2].contiguous(), 150, 2, x.scale)
    torch.cuda.synchronize()
    assert torch.equal(full[1:2, 2:4], one)


@pytest.mark.gpu
def test_prefill_tiny_fp32_workload(swa, oracle_mod):
    spec = synthetic.WORKLOADS["tiny_fp32_prefill"]
    x = synthetic.prefill_inputs(spec["B"], spec["H"], spec["Hkv"], spec["n"], spec["d"],
                                 spec["w"], spec["g"], dtype="f32", seed=0, device="cpu")
    Q, K, V = (t.cuda() for t in (x.Q, x.K, x.V))
    lse = torch.empty(1, 1, spec["n"], dtype=torch.float32, device="cuda")
    out = swa.prefill(Q, K, V, spec["w"], spec["g"], x.scale, lse=lse)
    torch.cuda.synchronize()
    O, L = oracle_mod.prefill(x.Q, x.K, x.V, spec["w"], spec["g"], x.scale)
    assert_close(out, O, "f32", "tiny fp32")
    assert np.abs(lse.cpu().double().numpy() - L).max() < 1e-5


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g", [(1, 4, 2, 333, 128, 50, 3), (2, 2, 1, 97, 64, 200, 0),
                                             (1, 1, 1, 64, 64, 1, 0), (1, 2, 2, 130, 64, 7, 9)])
def test_prefill_fp32_matches_oracle(swa, oracle_mod, B, H, Hkv, n, d, w, g):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="f32", seed=11, device="cuda")
    out = swa.prefill(x.Q, x.K, x.V, w, g, x.scale)
    torch.cuda.synchronize()
    O, _ = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
    assert_close(out, O, "f32", f"fp32 {B,H,Hkv,n,d,w,g}")
