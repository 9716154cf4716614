"""The benchmark's useful-work counts (keys read per query position, for each
pattern) against the oracle's masks, on small shapes.  No GPU."""
import numpy as np
import pytest

import bench


@pytest.mark.parametrize("pattern,n,w,g,r", [
    ("window", 90, 7, 3, 1), ("window", 40, 50, 0, 1),
    ("dilated", 90, 5, 0, 4), ("dilated", 33, 40, 0, 3), ("dilated", 20, 3, 0, 25),
    ("strided", 90, 0, 0, 9), ("strided", 10, 0, 0, 1),
    ("landmark", 200, 16, 0, 8), ("landmark", 200, 16, 5, 4), ("landmark", 150, 9, 13, 6),
    ("landmark", 60, 100, 2, 5),
])
def test_row_keys_match_oracle_mask(oracle_mod, pattern, n, w, g, r):
    c = dict(n=n, w=w, g=g, pattern=pattern, r=r, B=1, H=1, d=1)
    ref = oracle_mod.pattern_mask(n, w, g, r, pattern).sum(axis=1)
    assert np.array_equal(bench.row_keys(np.arange(n), c), ref)
    assert bench.prefill_flops(c) == 4 * int(ref.sum())


def test_window_flops_match_pair_count(oracle_mod):
    for name in ("mistral_like_prefill", "gemma3_local_prefill"):
        c = dict(bench.PREFILL_WORKLOADS[name])
        small = dict(c, n=3000, w=min(c["w"], 700))
        assert bench.prefill_flops(small) == 4 * oracle_mod.count_pairs(
            small["n"], small["w"], small["g"]) * c["d"] * c["B"] * c["H"]


def test_roofline_bound_follows_the_larger_time():
    pk = dict(bf16=1718.7, bf16_sustained=1400.0, hbm=6507.5, src="test")
    # the Mistral-like layer is a dense contraction per tile: tensor-bound
    c = bench.PREFILL_WORKLOADS["mistral_like_prefill"]
    r = bench.prefill_roofline(c, bench.prefill_flops(c), 0.63, pk, None, "k")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - bench.prefill_flops(c) / 0.63e-3 / 1e12 / 1718.7) < 1e-12
    # the strided head at s = sqrt(n) reads ~n/2s keys per query: HBM-bound
    c = bench.PREFILL_WORKLOADS["strided_prefill"]
    r = bench.prefill_roofline(c, bench.prefill_flops(c), 0.33, pk, None, "k")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["algorithmic_bytes"] == 2 * (32 + 8) * 65536 * 128 * 2
    assert r["hbm_bound_ms"] > r["tensor_bound_ms"]
