"""The other fixed patterns (swa_prefill_pattern) against the fp64 oracle,
element by element: the dilated window, the Sparse Transformer's strided head
and landmarks, on the bf16 tensor-core kernels (head pairs and single heads)
and the fp32 kernel, at sizes that span several tiles with ragged tails,
lengths that are and are not multiples of the stride, strides longer than
the sequence, and landmarks that fall in the band, below the sinks and
before the band."""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close

CASES = [
    # pattern, B, H, Hkv, n, d, w, g, r
    ("dilated", 1, 4, 2, 700, 128, 50, 0, 4),       # n % r == 0, several tiles per class
    ("dilated", 2, 4, 2, 1001, 128, 100, 0, 3),     # n % r == 2: classes of two lengths
    ("dilated", 1, 3, 1, 515, 64, 7, 0, 5),         # single-head kernel, d = 64
    ("dilated", 1, 2, 2, 260, 128, 300, 0, 2),      # window longer than each class
    ("dilated", 1, 4, 2, 129, 128, 4, 0, 1),        # stride one: the plain window
    ("strided", 1, 4, 2, 1100, 128, 0, 0, 9),       # classes of 122/123 rows
    ("strided", 2, 4, 1, 384, 128, 0, 0, 128),      # classes of 3 rows (s = n / 3)
    ("strided", 1, 2, 2, 100, 128, 0, 0, 150),      # stride past the end: O = V
    ("strided", 1, 3, 3, 300, 64, 0, 0, 1),         # stride one: full causal
    ("landmark", 1, 4, 2, 1500, 128, 200, 0, 16),   # several landmark tiles
    ("landmark", 2, 4, 2, 900, 128, 64, 4, 50),     # with sinks; landmark 0 is a sink
    ("landmark", 1, 3, 1, 1300, 64, 128, 3, 2),     # a landmark every other position
    ("landmark", 1, 4, 2, 640, 128, 1000, 0, 7),    # window covers everything
    # many classes per q-tile level (class-major item order), classes of 129 and
    # 128 rows (two q tiles for some, one for the others)
    ("strided", 8, 16, 16, 644, 64, 0, 0, 5),       # single-head kernel
    ("dilated", 4, 32, 16, 1283, 64, 30, 0, 10),    # head pairs
    # items of four key tiles and more (window and class rows >= 512): the head-pair
    # kernel's skewed key/value protocol under the fixed patterns
    ("landmark", 1, 4, 2, 2100, 128, 600, 4, 32),
    ("dilated", 1, 4, 2, 2230, 128, 700, 0, 2),     # classes of 1115 rows
]


def inputs(B, H, Hkv, n, d, dtype, seed):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, 1, 0, dtype=dtype, seed=seed)
    return x.Q, x.K, x.V


@pytest.mark.gpu
@pytest.mark.parametrize("pattern,B,H,Hkv,n,d,w,g,r", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pattern_matches_oracle(swa, oracle_mod, pattern, B, H, Hkv, n, d, w, g, r, dtype):
    Q, K, V = inputs(B, H, Hkv, n, d, dtype, seed=n + r)
    scale = 1.0 / np.sqrt(d)
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    out = swa.prefill_pattern(Q.cuda(), K.cuda(), V.cuda(), pattern, w, g, r, scale, lse=lse)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    O, L = oracle_mod.prefill_pattern(Q, K, V, w, g, r, pattern, scale)
    assert_close(out, O, dtype, f"{pattern} {B,H,Hkv,n,d,w,g,r}")
    tol = 2e-3 if dtype == "bf16" else 1e-5
    assert np.abs(lse.cpu().double().numpy() - L).max() < tol


@pytest.mark.gpu
@pytest.mark.parametrize("pattern,w,g,r", [("dilated", 30, 0, 3), ("landmark", 100, 2, 32)])
def test_pattern_with_sink_logit(swa, oracle_mod, pattern, w, g, r):
    B, H, Hkv, n, d = 1, 4, 2, 600, 128
    Q, K, V = inputs(B, H, Hkv, n, d, "bf16", seed=3)
    sink = torch.tensor([1.0, -2.0, 0.5, 3.0])
    out = swa.prefill_pattern(Q.cuda(), K.cuda(), V.cuda(), pattern, w, g, r, 0.1,
                              sink_logit=sink.cuda())
    torch.cuda.synchronize()
    O, _ = oracle_mod.prefill_pattern(Q, K, V, w, g, r, pattern, 0.1, sink_logit=sink.double())
    assert_close(out, O, "bf16", f"{pattern} with sink logit")


@pytest.mark.gpu
def test_window_pattern_is_prefill(swa):
    B, H, Hkv, n, d = 1, 4, 2, 500, 128
    Q, K, V = (t.cuda() for t in inputs(B, H, Hkv, n, d, "bf16", seed=4))
    a = swa.prefill_pattern(Q, K, V, "window", 64, 3, 99)
    b = swa.prefill(Q, K, V, 64, 3)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
def test_dilated_and_strided_reject_sinks(swa):
    Q, K, V = (t.cuda() for t in inputs(1, 2, 2, 64, 64, "bf16", seed=5))
    for pat in ("dilated", "strided"):
        with pytest.raises(swa.SwaError):
            swa.prefill_pattern(Q, K, V, pat, 8, 2, 4)
    with pytest.raises(swa.SwaError):
        swa.prefill_pattern(Q, K, V, "landmark", 8, 0, 0)
