"""Randomised properties of the oracle (hypothesis, CPU, fp64): invariants that
hold for any inputs, so that a mistake anywhere in the oracle's masking,
softmax or output assembly shows up on shapes the fixed pins do not cover.

- every output row is a convex combination of the value rows its mask row
  allows, so it lies inside their per-column range;
- LSE lies between the row's largest allowed score and that plus log(#keys);
- the output is affine in V: V -> aV + b gives O -> aO + b;
- a sink logit s rescales the plain output by exp(LSE_plain - LSE_sink), with
  LSE_sink = logaddexp(LSE_plain, s);
- the dilated pattern reads a subset of the window of (w-1)r+1 cells, and the
  landmark pattern a superset of the window.
No test here needs a GPU.
"""
import numpy as np
import pytest
import torch
from hypothesis import given, settings, strategies as st

shapes = st.fixed_dictionaries({
    "n": st.integers(1, 40),
    "d": st.sampled_from([4, 8]),
    "hkv": st.integers(1, 2),
    "grp": st.integers(1, 3),
    "w": st.integers(1, 45),
    "g": st.integers(0, 5),
    "seed": st.integers(0, 10_000),
})


def draw(n, d, H, Hkv, seed):
    gen = torch.Generator().manual_seed(seed)
    Q = torch.randn(1, H, n, d, generator=gen, dtype=torch.float64)
    K = torch.randn(1, Hkv, n, d, generator=gen, dtype=torch.float64)
    V = torch.randn(1, Hkv, n, d, generator=gen, dtype=torch.float64)
    return Q, K, V


@settings(max_examples=40, deadline=None)
@given(shapes)
def test_output_is_a_convex_combination_and_lse_is_bounded(oracle_mod, s):
    n, d, Hkv = s["n"], s["d"], s["hkv"]
    H = Hkv * s["grp"]
    Q, K, V = draw(n, d, H, Hkv, s["seed"])
    sc = 0.7
    O, L = oracle_mod.prefill(Q, K, V, s["w"], s["g"], sc)
    m = oracle_mod.mask(n, s["w"], s["g"]).astype(bool)
    for h in range(H):
        kvh = h // s["grp"]
        Vh = V[0, kvh].numpy()
        S = sc * (Q[0, h].numpy() @ K[0, kvh].numpy().T)
        for i in range(n):
            rows = Vh[m[i]]
            assert (O[0, h, i] >= rows.min(axis=0) - 1e-12).all()
            assert (O[0, h, i] <= rows.max(axis=0) + 1e-12).all()
            smax = S[i, m[i]].max()
            assert smax - 1e-12 <= L[0, h, i] <= smax + np.log(m[i].sum()) + 1e-12


@settings(max_examples=30, deadline=None)
@given(shapes, st.floats(-3, 3), st.floats(-2, 2))
def test_output_is_affine_in_v(oracle_mod, s, a, b):
    n, d, Hkv = s["n"], s["d"], s["hkv"]
    H = Hkv * s["grp"]
    Q, K, V = draw(n, d, H, Hkv, s["seed"])
    O1, L1 = oracle_mod.prefill(Q, K, V, s["w"], s["g"], 0.5)
    O2, L2 = oracle_mod.prefill(Q, K, a * V + b, s["w"], s["g"], 0.5)
    assert np.allclose(O2, a * O1 + b, atol=1e-10, rtol=0)
    assert np.array_equal(L1, L2)  # the weights do not depend on V


@settings(max_examples=30, deadline=None)
@given(shapes, st.lists(st.floats(-6, 6), min_size=6, max_size=6))
def test_sink_logit_rescales_the_plain_output(oracle_mod, s, sig):
    n, d, Hkv = s["n"], s["d"], s["hkv"]
    H = Hkv * s["grp"]
    Q, K, V = draw(n, d, H, Hkv, s["seed"])
    sink = np.array(sig[:H])
    O0, L0 = oracle_mod.prefill(Q, K, V, s["w"], s["g"], 0.5)
    O1, L1 = oracle_mod.prefill(Q, K, V, s["w"], s["g"], 0.5, sink_logit=sink)
    Ls = np.logaddexp(L0, sink[None, :, None])
    assert np.allclose(L1, Ls, atol=1e-12, rtol=0)
    assert np.allclose(O1, O0 * np.exp(L0 - Ls)[..., None], atol=1e-12, rtol=0)


@settings(max_examples=40, deadline=None)
@given(st.integers(1, 60), st.integers(1, 12), st.integers(1, 9), st.integers(0, 4))
def test_pattern_masks_nest_with_the_window(oracle_mod, n, w, r, g):
    dil = oracle_mod.pattern_mask(n, w, g, r, "dilated").astype(bool)
    wide = oracle_mod.mask(n, (w - 1) * r + 1, g).astype(bool)
    assert not (dil & ~wide).any()  # dilated reads inside the wider window
    lm = oracle_mod.pattern_mask(n, w, g, r, "landmark").astype(bool)
    win = oracle_mod.mask(n, w, g).astype(bool)
    assert not (win & ~lm).any()   # landmarks only add keys
    # every row reads at least itself, and nothing from the future
    for mk in (dil, lm, oracle_mod.pattern_mask(n, w, g, r, "strided").astype(bool)):
        assert mk.diagonal().all() and not np.triu(mk, 1).any()


@pytest.mark.parametrize("seed", [0, 1])
def test_decode_cache_equals_history_with_sink_logit(oracle_mod, seed):
    # the rolling-cache decode and the unbounded-history decode agree with a sink
    # logit too (the cache test without one is in test_oracle_pins.py)
    B, H, Hkv, d, w, g, P = 2, 4, 2, 8, 6, 2, 30
    gen = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, P, d, generator=gen, dtype=torch.float64)
    V = torch.randn(B, Hkv, P, d, generator=gen, dtype=torch.float64)
    q = torch.randn(B, H, d, generator=gen, dtype=torch.float64)
    sink = np.array([0.3, -1.0, 2.0, 0.0])
    for pos in (0, 3, 7, 8, 29):
        Kc = torch.zeros(B, Hkv, w + g, d, dtype=torch.float64)
        Vc = torch.zeros_like(Kc)
        for p in range(pos + 1):
            ring, sk = oracle_mod.cache_slots(p, w, g)
            Kc[:, :, ring], Vc[:, :, ring] = K[:, :, p], V[:, :, p]
            if sk >= 0:
                Kc[:, :, sk], Vc[:, :, sk] = K[:, :, p], V[:, :, p]
        posv = np.full(B, pos)
        O1, L1 = oracle_mod.decode_cache(q, Kc, Vc, posv, w, g, 0.4, sink_logit=sink)
        O2, L2 = oracle_mod.decode_history(q, K, V, posv, w, g, 0.4, sink_logit=sink)
        assert np.allclose(O1, O2, atol=1e-12, rtol=0) and np.allclose(L1, L2, atol=1e-12, rtol=0)
