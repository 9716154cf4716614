"""Pins for the oracle's other fixed patterns (dilated window, strided head,
landmarks).  Each checks the oracle against something other than itself: the
worked example the pages print, properties the pages state (the two-hop reach
of the Sparse Transformer, the cost and reach of a dilated window, landmarks
read once and never from the future), closed-form counts, and reductions to
cases already pinned (the window pattern, torch's causal attention) through
the residue-class decomposition that holds for any dilated or strided mask.

No test here needs a GPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


@pytest.fixture(scope="module")
def ex():
    with open(GOLDEN) as f:
        return json.load(f)


def reads(row):
    return [int(j) for j in np.nonzero(row)[0]]


def rand(*shape, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


# --------------------------------------------------------------------------
# worked examples and stated properties
# --------------------------------------------------------------------------

def test_landmarks_every_four(oracle_mod, ex):
    e = ex["landmarks_every_four"]
    m = oracle_mod.pattern_mask(e["n"], e["w"], e["g"], e["r"], "landmark")
    assert reads(m[7]) == e["row7_reads"]
    assert int(m[7].sum()) == e["row7_count"]
    # p4 is both in the window and designated, and is read once: the row is a
    # set of positions, five of them
    assert e["read_once_at_row7"] in reads(m[7])
    # no future position, designated or not
    assert m[3, e["row3_excludes_future_landmark"]] == 0
    assert not np.triu(m, k=1).any()


def test_landmarks_grow_with_context_anchor_does_not(oracle_mod):
    # the pages: adding the first position adds one key once the window has
    # moved on; adding every r-th position adds more keys as the context grows
    n, w, r = 200, 8, 16
    lm = oracle_mod.pattern_mask(n, w, 0, r, "landmark").sum(axis=1)
    anchor = oracle_mod.mask(n, w, 1).sum(axis=1)
    assert all(anchor[i] == w + 1 for i in range(w, n))
    for i in range(n):
        # the band, plus the landmarks 0, r, 2r, ... that lie before it
        expect = min(i + 1, w) + ((i - w) // r + 1 if i >= w else 0)
        assert lm[i] == expect, i
    assert lm[n - 1] > lm[w + r]


def test_landmark_limits_reduce_to_pinned_cases(oracle_mod):
    for n, w in [(30, 5), (17, 1), (64, 64)]:
        # one landmark only (position 0): the first-position rule of the figure,
        # i.e. the window with one sink
        assert np.array_equal(oracle_mod.pattern_mask(n, w, 0, n + 3, "landmark"),
                              oracle_mod.mask(n, w, 1))
        # every position a landmark: full causal attention
        assert np.array_equal(oracle_mod.pattern_mask(n, w, 0, 1, "landmark"),
                              np.tril(np.ones((n, n), dtype=np.uint8)))


def test_sparse_transformer_two_hops(oracle_mod, ex):
    e = ex["sparse_transformer_two_hops"]
    n, s = e["n"], e["s"]
    strided = oracle_mod.pattern_mask(n, s, 0, s, "strided").astype(np.int64)
    local = oracle_mod.mask(n, s, 0).astype(np.int64)
    causal = np.tril(np.ones((n, n), dtype=np.int64))
    # a strided hop then a local hop reaches every earlier position, and nothing
    # in the future
    reach = (strided @ local) > 0
    assert np.array_equal(reach, causal > 0)
    # one hop alone does not
    assert not np.array_equal(strided > 0, causal > 0)
    assert not np.array_equal(local > 0, causal > 0)
    # the strided head reads i, i-s, i-2s, ...: floor(i/s)+1 keys
    assert [int(c) for c in strided.sum(axis=1)] == [i // s + 1 for i in range(n)]
    # cost about n*sqrt(n) per head pair at s = sqrt(n)
    assert strided.sum() + local.sum() <= 2 * n * s


def test_dilated_cost_and_reach(oracle_mod, ex):
    e = ex["dilated_reach"]
    w, r = e["w"], e["r"]
    n = 60
    m = oracle_mod.pattern_mask(n, w, 0, r, "dilated")
    win = oracle_mod.mask(n, w, 0)
    for i in range(n):
        row = reads(m[i])
        assert len(row) == min(w, i // r + 1)
        if i >= (w - 1) * r:
            # the cost of a window of w ...
            assert len(row) == e["keys_per_row_far_from_start"] == int(win[i].sum())
            # ... and a reach r times as long
            assert i - row[0] == e["reach_factor"] * (w - 1)
        assert all((i - j) % r == 0 and j <= i for j in row)
    # stride one is the window itself
    assert np.array_equal(oracle_mod.pattern_mask(n, w, 0, 1, "dilated"), win)


def test_dilated_is_a_sum_of_shifted_diagonals(oracle_mod):
    # an independent construction: ones on the diagonals i - j = k r, k < w
    for n, w, r, g in [(40, 3, 5, 0), (33, 6, 2, 2), (25, 1, 4, 3), (50, 100, 7, 0)]:
        ref = np.zeros((n, n), dtype=np.uint8)
        for k in range(w):
            if k * r < n:
                ref += np.eye(n, k=-k * r, dtype=np.uint8)
        ref[:, :g] |= np.tril(np.ones((n, n), dtype=np.uint8))[:, :g]
        assert np.array_equal(oracle_mod.pattern_mask(n, w, g, r, "dilated"), ref), (n, w, r, g)
        assert oracle_mod.pattern_count_pairs(n, w, g, r, "dilated") == int(ref.sum())


def test_strided_is_dilated_without_limit(oracle_mod):
    n = 45
    for r in (1, 3, 7, 50):
        s = oracle_mod.pattern_mask(n, 0, 0, r, "strided")
        assert np.array_equal(s, oracle_mod.pattern_mask(n, n, 0, r, "dilated"))
    assert np.array_equal(oracle_mod.pattern_mask(n, 0, 0, 1, "strided"),
                          np.tril(np.ones((n, n), dtype=np.uint8)))


def test_window_code_is_the_window_mask(oracle_mod):
    for n, w, g in [(30, 4, 2), (9, 9, 0)]:
        assert np.array_equal(oracle_mod.pattern_mask(n, w, g, 5, "window"),
                              oracle_mod.mask(n, w, g))


# --------------------------------------------------------------------------
# attention under the patterns
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n,w,r,H,Hkv", [(50, 3, 4, 2, 1), (37, 5, 3, 4, 2), (20, 2, 7, 3, 3)])
def test_dilated_attention_is_window_attention_per_residue_class(oracle_mod, n, w, r, H, Hkv):
    # the keys of row i are the class of i mod r, at most w of them: row i of the
    # dilated pattern is the window pattern on that class's subsequence
    d = 16
    Q, K, V = rand(2, H, n, d, seed=1), rand(2, Hkv, n, d, seed=2), rand(2, Hkv, n, d, seed=3)
    sc = 0.4
    O, L = oracle_mod.prefill_pattern(Q, K, V, w, 0, r, "dilated", sc)
    for c in range(min(r, n)):
        idx = torch.arange(c, n, r)
        Oc, Lc = oracle_mod.prefill(Q[:, :, idx], K[:, :, idx], V[:, :, idx], w, 0, sc)
        assert np.allclose(O[:, :, idx.numpy()], Oc, atol=1e-12, rtol=0)
        assert np.allclose(L[:, :, idx.numpy()], Lc, atol=1e-12, rtol=0)


@pytest.mark.parametrize("n,r", [(41, 4), (32, 8), (9, 20)])
def test_strided_attention_is_causal_attention_per_residue_class(oracle_mod, n, r):
    d, H, Hkv = 12, 4, 2
    Q, K, V = rand(1, H, n, d, seed=4), rand(1, Hkv, n, d, seed=5), rand(1, Hkv, n, d, seed=6)
    sc = 1 / math.sqrt(d)
    O, _ = oracle_mod.prefill_pattern(Q, K, V, 0, 0, r, "strided", sc)
    for c in range(min(r, n)):
        idx = torch.arange(c, n, r)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[:, :, idx], K[:, :, idx].repeat_interleave(2, 1), V[:, :, idx].repeat_interleave(2, 1),
            is_causal=True, scale=sc)
        assert np.allclose(O[:, :, idx.numpy()], ref.numpy(), atol=1e-12, rtol=0)


def test_strided_beyond_length_returns_own_value(oracle_mod):
    # r > n - 1: each query reads only itself
    n, d = 13, 8
    Q, K, V = rand(1, 2, n, d, seed=7), rand(1, 1, n, d, seed=8), rand(1, 1, n, d, seed=9)
    for pat, w in [("strided", 0), ("dilated", 5)]:
        O, L = oracle_mod.prefill_pattern(Q, K, V, w, 0, n + 1, pat, 0.5)
        assert np.allclose(O, V.repeat_interleave(2, 1).numpy(), atol=1e-15, rtol=0)
        s = 0.5 * (Q * K.repeat_interleave(2, 1)).sum(-1)
        assert np.allclose(L, s.numpy(), atol=1e-12, rtol=0)


def test_landmark_attention_limits(oracle_mod):
    n, d, H, Hkv = 40, 16, 4, 2
    Q, K, V = rand(2, H, n, d, seed=10), rand(2, Hkv, n, d, seed=11), rand(2, Hkv, n, d, seed=12)
    sc = 0.25
    causal = torch.nn.functional.scaled_dot_product_attention(
        Q, K.repeat_interleave(2, 1), V.repeat_interleave(2, 1), is_causal=True, scale=sc)
    for w, r in [(5, 1), (n, 7), (n + 10, 3)]:
        O, _ = oracle_mod.prefill_pattern(Q, K, V, w, 0, r, "landmark", sc)
        assert np.allclose(O, causal.numpy(), atol=1e-12, rtol=0), (w, r)
    # a single landmark (position 0) is the window with one sink
    O, L = oracle_mod.prefill_pattern(Q, K, V, 6, 0, n, "landmark", sc)
    O1, L1 = oracle_mod.prefill(Q, K, V, 6, 1, sc)
    assert np.array_equal(O, O1) and np.array_equal(L, L1)


def test_landmark_attention_matches_sdpa_with_figure_mask(oracle_mod, ex):
    # the figure's rule at a larger size, with the mask taken row by row from
    # the stated read sets: the band of the last w cells plus every designated
    # position up to the query, each once
    n, w, r, d = 50, 6, 8, 16
    allow = torch.zeros(n, n, dtype=torch.bool)
    for i in range(n):
        allow[i, max(0, i - w + 1):i + 1] = True
        allow[i, torch.arange(0, i + 1, r)] = True
    Q, K, V = rand(1, 2, n, d, seed=13), rand(1, 2, n, d, seed=14), rand(1, 2, n, d, seed=15)
    O, _ = oracle_mod.prefill_pattern(Q, K, V, w, 0, r, "landmark", 0.3)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=allow, scale=0.3)
    assert np.allclose(O, ref.numpy(), atol=1e-12, rtol=0)


def test_pattern_rows_match_full(oracle_mod):
    n, d, H, Hkv = 70, 8, 4, 2
    Q, K, V = rand(2, H, n, d, seed=16), rand(2, Hkv, n, d, seed=17), rand(2, Hkv, n, d, seed=18)
    rows = np.array([[0, 0, 0], [1, 3, 69], [0, 2, 33], [1, 1, 8]], dtype=np.int64)
    q_rows = Q[rows[:, 0], rows[:, 1], rows[:, 2]]
    for pat, w, g, r in [("dilated", 4, 0, 3), ("strided", 0, 0, 9), ("landmark", 5, 2, 16)]:
        O, L = oracle_mod.prefill_pattern(Q, K, V, w, g, r, pat, 0.2)
        Or, Lr = oracle_mod.prefill_pattern_rows(q_rows, K, V, H, w, g, r, pat, 0.2, rows)
        assert np.array_equal(Or, O[rows[:, 0], rows[:, 1], rows[:, 2]])
        assert np.array_equal(Lr, L[rows[:, 0], rows[:, 1], rows[:, 2]])
