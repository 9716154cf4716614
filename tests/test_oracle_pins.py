"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- the numbers the pages print for their worked examples, closed
forms, textbook special cases and torch library routines (fp64, CPU).

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


def reads(mask_row):
    return [int(j) for j in np.nonzero(mask_row)[0]]


# --------------------------------------------------------------------------
# worked examples printed on the pages
# --------------------------------------------------------------------------

def test_window3_eight_tokens(oracle_mod, ex):
    e = ex["window3_eight_tokens"]
    m = oracle_mod.mask(e["n"], e["w"], e["g"])
    assert reads(m[7]) == e["row7_reads"]
    assert [int(c) for c in m.sum(axis=1)] == e["per_row_counts"]
    assert oracle_mod.count_pairs(e["n"], e["w"], e["g"]) == e["pairs"]
    assert oracle_mod.count_pairs(e["n"], e["n"], 0) == e["pairs_full_causal"]
    assert oracle_mod.count_pairs(e["n"], 1000, 0) == e["pairs_full_causal"]
    assert reads(oracle_mod.mask(e["n"], e["n"], 0)[7]) == e["full_causal_row7_reads"]
    # the window slides: with a ninth token, p8 reads p6..p8
    assert reads(oracle_mod.mask(9, e["w"], 0)[8]) == e["row8_reads_when_n9"]


def test_anchor_plus_window(oracle_mod, ex):
    e = ex["anchor_plus_window"]
    row7 = oracle_mod.mask(e["n"], e["w"], e["g"])[7]
    assert reads(row7) == e["row7_reads"]
    assert all(row7[j] == 0 for j in e["row7_excludes"])
    # derived from the same rule: rows 0..3 read 1,2,3,4 keys, rows 4..7 read 3+1
    assert oracle_mod.count_pairs(8, 3, 1) == 1 + 2 + 3 + 4 * 5


def test_no_future_reads(oracle_mod, ex):
    e = ex["no_future_reads"]
    # even with every position designated a sink, query 3 cannot read key 4
    m = oracle_mod.mask(8, 3, 8)
    assert m[e["query"], e["key"]] == 0
    assert reads(m[3]) == [0, 1, 2, 3]
    for n, w, g in [(17, 4, 3), (33, 1, 40), (5, 9, 2)]:
        mm = oracle_mod.mask(n, w, g)
        assert not np.triu(mm, k=1).any()


# --------------------------------------------------------------------------
# the mask against torch's own construction (tril / triu, as the Q&A page's
# example builds it) plus sink columns
# --------------------------------------------------------------------------

def torch_mask(n, w, g):
    ones = torch.ones(n, n, dtype=torch.int64)
    causal = torch.tril(ones)
    band = torch.triu(causal, diagonal=-w + 1)
    sinks = causal.clone()
    sinks[:, g:] = 0
    return ((band + sinks) > 0).numpy().astype(np.uint8)


@pytest.mark.parametrize("n,w,g", [(6, 3, 0), (1, 1, 0), (9, 2, 0), (40, 7, 3), (64, 64, 4),
                                   (50, 100, 0), (31, 1, 31), (23, 5, 9), (70, 16, 1)])
def test_mask_matches_torch_construction(oracle_mod, n, w, g):
    assert np.array_equal(oracle_mod.mask(n, w, g), torch_mask(n, w, g))


def test_mask_row_matches_full_mask(oracle_mod):
    m = oracle_mod.mask(57, 11, 3)
    for i in (0, 3, 10, 11, 12, 56):
        assert np.array_equal(oracle_mod.mask_row(i, 57, 11, 3), m[i])


# --------------------------------------------------------------------------
# connection counts: closed form vs brute force
# --------------------------------------------------------------------------

def pairs_closed_form(n, w, g):
    """Per row i: the window holds min(i+1, w) keys; the sinks add the ones
    that have left the window, min(g, max(0, i-w+1))."""
    total = 0
    for i in range(n):
        left = max(0, i - w + 1)
        total += (i - left + 1) + min(g, left)
    return total


def pairs_aggregate(n, w, g):
    """Sum over rows in closed form for n >= w."""
    assert n >= w
    s = w * (w + 1) // 2 + (n - w) * w
    # sink contribution: rows i >= w gain min(g, i-w+1)
    m = n - w  # rows w..n-1, their i-w+1 runs 1..m
    s += sum(min(g, t) for t in range(1, m + 1)) if m <= 100000 else (
        g * (g + 1) // 2 + (m - g) * g if m >= g else m * (m + 1) // 2)
    return s


def test_pairs_closed_form_small(oracle_mod):
    for n in range(1, 65, 3):
        for w in (1, 2, 3, 5, 8, 13, 31, 64, 70):
            for g in (0, 1, 2, 4, 8):
                assert oracle_mod.count_pairs(n, w, g) == pairs_closed_form(n, w, g), (n, w, g)


def test_pairs_workload_sizes(oracle_mod):
    # per-head connection counts of the benchmark workloads
    assert pairs_closed_form(512, 64, 0) == 30752
    assert pairs_aggregate(16384, 4096, 0) == 58722304
    assert pairs_aggregate(32768, 1024, 0) == 33030656
    assert pairs_aggregate(131072, 4096, 4) == 528992250
    assert oracle_mod.count_pairs(512, 64, 0) == 30752
    assert oracle_mod.count_pairs(16384, 4096, 0) == 58722304


# --------------------------------------------------------------------------
# tile classes: brute force from a torch-built mask
# --------------------------------------------------------------------------

def torch_tiles(n, w, g, BM, BN):
    m = torch.from_numpy(torch_mask(n, w, g)).to(torch.int64)
    nq, nk = -(-n // BM), -(-n // BN)
    pad = torch.zeros(nq * BM, nk * BN, dtype=torch.int64)
    real = torch.zeros_like(pad)
    pad[:n, :n] = m
    real[:n, :] = 1  # rows that exist; columns past n count as blocked cells
    t = pad.view(nq, BM, nk, BN).sum(dim=(1, 3))
    cells = real.view(nq, BM, nk, BN).sum(dim=(1, 3))
    out = torch.zeros(nq, nk, dtype=torch.int32)
    out[t > 0] = 1
    out[(t == cells) & (cells > 0)] = 2
    return out.numpy()


@pytest.mark.parametrize("n,w,g,BM,BN", [
    (300, 64, 0, 64, 64), (300, 100, 4, 64, 128), (257, 3, 1, 16, 16),
    (200, 1000, 0, 128, 64), (129, 128, 130, 128, 128), (333, 17, 5, 16, 64),
])
def test_tiles_match_bruteforce(oracle_mod, n, w, g, BM, BN):
    assert np.array_equal(oracle_mod.tiles(n, w, g, BM, BN), torch_tiles(n, w, g, BM, BN))


# --------------------------------------------------------------------------
# attention: textbook special cases and torch SDPA (fp64, CPU)
# --------------------------------------------------------------------------

def rand(*shape, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


def sdpa(Q, K, V, mask_bool, scale):
    """torch's scaled_dot_product_attention with a boolean mask (True = attend);
    K/V expanded over the query heads of each group."""
    G = Q.shape[1] // K.shape[1]
    Ke = K.repeat_interleave(G, dim=1)
    Ve = V.repeat_interleave(G, dim=1)
    return torch.nn.functional.scaled_dot_product_attention(
        Q, Ke, Ve, attn_mask=torch.as_tensor(mask_bool, dtype=torch.bool), scale=scale)


def test_full_window_is_causal_attention(oracle_mod):
    B, H, Hkv, n, d = 2, 4, 2, 37, 16
    Q, K, V = rand(B, H, n, d, seed=1), rand(B, Hkv, n, d, seed=2), rand(B, Hkv, n, d, seed=3)
    sc = 1 / math.sqrt(d)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, K.repeat_interleave(2, 1), V.repeat_interleave(2, 1), is_causal=True, scale=sc)
    for w, g in [(n, 0), (n + 5, 0), (3, n), (1, n + 2)]:
        O, _ = oracle_mod.prefill(Q, K, V, w, g, sc)
        assert np.allclose(O, ref.numpy(), atol=1e-12, rtol=0), (w, g)


@pytest.mark.parametrize("n,w,g,H,Hkv", [(45, 7, 0, 2, 1), (64, 16, 4, 4, 2), (33, 5, 2, 3, 3),
                                         (20, 2, 1, 8, 2)])
def test_matches_sdpa_with_torch_mask(oracle_mod, n, w, g, H, Hkv):
    d = 24
    Q, K, V = rand(1, H, n, d, seed=4), rand(1, Hkv, n, d, seed=5), rand(1, Hkv, n, d, seed=6)
    sc = 0.3
    O, _ = oracle_mod.prefill(Q, K, V, w, g, sc)
    ref = sdpa(Q, K, V, torch_mask(n, w, g).astype(bool), sc)
    assert np.allclose(O, ref.numpy(), atol=1e-12, rtol=0)


def test_lse_matches_torch_logsumexp(oracle_mod):
    n, w, g, d = 29, 6, 2, 8
    Q, K, V = rand(1, 1, n, d, seed=7), rand(1, 1, n, d, seed=8), rand(1, 1, n, d, seed=9)
    sc = 0.7
    _, L = oracle_mod.prefill(Q, K, V, w, g, sc)
    s = (Q[0, 0] @ K[0, 0].T) * sc
    s = s.masked_fill(~torch.as_tensor(torch_mask(n, w, g).astype(bool)), float("-inf"))
    assert np.allclose(L[0, 0], torch.logsumexp(s, dim=1).numpy(), atol=1e-12, rtol=0)


def test_window_one_returns_own_value(oracle_mod):
    n, d = 40, 12
    Q, K, V = rand(1, 2, n, d, seed=10), rand(1, 2, n, d, seed=11), rand(1, 2, n, d, seed=12)
    O, L = oracle_mod.prefill(Q, K, V, 1, 0, 0.5)
    assert np.array_equal(O, V.numpy())
    own = 0.5 * (Q * K).sum(-1)
    assert np.allclose(L, own.numpy(), atol=1e-12, rtol=0)


def test_constant_values_pass_through(oracle_mod):
    n, d = 50, 8
    Q, K = rand(1, 1, n, d, seed=13), rand(1, 1, n, d, seed=14)
    c = rand(d, seed=15)
    V = c.expand(1, 1, n, d).contiguous()
    O, _ = oracle_mod.prefill(Q, K, V, 9, 2, 1.3)
    assert np.allclose(O, np.broadcast_to(c.numpy(), O.shape), atol=1e-13, rtol=0)


def test_identical_keys_average_the_allowed_values(oracle_mod):
    n, w, g, d = 30, 5, 3, 6
    Q, V = rand(1, 1, n, d, seed=16), rand(1, 1, n, d, seed=17)
    K = rand(d, seed=18).expand(1, 1, n, d).contiguous()
    O, L = oracle_mod.prefill(Q, K, V, w, g, 0.9)
    for i in range(n):
        # the allowed set written out from the rule: window i-w+1..i plus sinks < g, causal
        allowed = sorted(set(range(max(0, i - w + 1), i + 1)) | set(range(min(g, i + 1))))
        mean = V[0, 0, allowed].mean(0).numpy()
        assert np.allclose(O[0, 0, i], mean, atol=1e-12, rtol=0)
        s = 0.9 * float((Q[0, 0, i] * K[0, 0, 0]).sum())
        assert math.isclose(L[0, 0, i], s + math.log(len(allowed)), abs_tol=1e-12)


def test_minus_inf_masking_differs_from_zero_scores(oracle_mod):
    n, d = 24, 8
    Q, K, V = rand(1, 1, n, d, seed=19), rand(1, 1, n, d, seed=20), rand(1, 1, n, d, seed=21)
    O_inf, _ = oracle_mod.prefill(Q, K, V, 4, 1, 0.4)
    O_zero, _ = oracle_mod.prefill(Q, K, V, 4, 1, 0.4, zero_score=True)
    assert np.abs(O_inf - O_zero).max() > 1e-2
    # zero scores: the blocked keys (future included) keep positive weight
    s = (Q[0, 0] @ K[0, 0].T) * 0.4
    allowed = torch.as_tensor(torch_mask(n, 4, 1).astype(bool))
    s = torch.where(allowed, s, torch.zeros_like(s))
    ref = torch.softmax(s, dim=1) @ V[0, 0]
    assert np.allclose(O_zero[0, 0], ref.numpy(), atol=1e-12, rtol=0)


def test_window_differs_from_full_attention(oracle_mod):
    n, d = 32, 8
    Q, K, V = rand(1, 1, n, d, seed=22), rand(1, 1, n, d, seed=23), rand(1, 1, n, d, seed=24)
    O_w, _ = oracle_mod.prefill(Q, K, V, 4, 0, 0.35)
    O_f, _ = oracle_mod.prefill(Q, K, V, n, 0, 0.35)
    assert np.array_equal(O_w[0, 0, :4], O_f[0, 0, :4])  # rows that see everything anyway
    assert np.abs(O_w[0, 0, 4:] - O_f[0, 0, 4:]).max() > 1e-3


def test_sampled_rows_match_full(oracle_mod):
    B, H, Hkv, n, d = 2, 4, 2, 41, 8
    Q, K, V = rand(B, H, n, d, seed=25), rand(B, Hkv, n, d, seed=26), rand(B, Hkv, n, d, seed=27)
    rows = np.array([[0, 0, 0], [1, 3, 40], [0, 2, 7], [1, 1, 20]], dtype=np.int64)
    qr = np.stack([Q[b, h, i].numpy() for b, h, i in rows])
    Or, Lr = oracle_mod.prefill_rows(qr, K, V, H, 6, 2, 0.5, rows)
    ref = sdpa(Q, K, V, torch_mask(n, 6, 2).astype(bool), 0.5).numpy()
    for t, (b, h, i) in enumerate(rows):
        assert np.allclose(Or[t], ref[b, h, i], atol=1e-12, rtol=0)


# --------------------------------------------------------------------------
# decode and the rolling cache
# --------------------------------------------------------------------------

def test_cache_slots_eviction_example(oracle_mod, ex):
    e = ex["rolling_cache_eviction"]
    w = e["w"]
    ring = [None] * w
    for p in range(8):
        r, s = oracle_mod.cache_slots(p, w, 0)
        assert s == -1
        ring[r] = p
    assert sorted(ring) == e["kept_at_7"]
    r8, _ = oracle_mod.cache_slots(8, w, 0)
    evicted = ring[r8]
    ring[r8] = 8
    assert evicted == e["evicted_when_8_arrives"]
    assert sorted(ring) == e["kept_at_8"]


def test_cache_slots_sinks(oracle_mod):
    assert oracle_mod.cache_slots(0, 4096, 4) == (0, 4096)
    assert oracle_mod.cache_slots(3, 4096, 4) == (3, 4099)
    assert oracle_mod.cache_slots(4, 4096, 4) == (4, -1)
    assert oracle_mod.cache_slots(100000, 4096, 4) == (100000 % 4096, -1)


def test_decode_history_is_last_prefill_row(oracle_mod):
    B, H, Hkv, d, P = 2, 4, 2, 16, 30
    K, V = rand(B, Hkv, P, d, seed=28), rand(B, Hkv, P, d, seed=29)
    q = rand(B, H, d, seed=30)
    pos = np.array([29, 13])
    for w, g in [(5, 0), (5, 2), (40, 0), (1, 3)]:
        O, L = oracle_mod.decode_history(q, K, V, pos, w, g, 0.25)
        for b in range(B):
            p = int(pos[b])
            n = p + 1
            Q = torch.zeros(1, H, n, d, dtype=torch.float64)
            Q[0, :, p] = q[b]
            ref = sdpa(Q, K[b:b + 1, :, :n], V[b:b + 1, :, :n],
                       torch_mask(n, w, g).astype(bool), 0.25)
            assert np.allclose(O[b], ref[0, :, p].numpy(), atol=1e-12, rtol=0)


def place(Kc, Vc, oracle_mod, b, kvh, p, k, v, w, g):
    r, s = oracle_mod.cache_slots(p, w, g)
    Kc[b, kvh, r] = k
    Vc[b, kvh, r] = v
    if s >= 0:
        Kc[b, kvh, s] = k
        Vc[b, kvh, s] = v


@pytest.mark.parametrize("w,g", [(8, 2), (3, 1), (4, 0), (1, 2), (6, 6)])
def test_streaming_cache_matches_unbounded_history(oracle_mod, w, g):
    B, H, Hkv, d, P = 1, 2, 1, 8, 41
    K, V = rand(B, Hkv, P, d, seed=31), rand(B, Hkv, P, d, seed=32)
    q = rand(P, B, H, d, seed=33)
    Kc = np.full((B, Hkv, w + g, d), np.nan)  # unwritten slots are never read
    Vc = np.full((B, Hkv, w + g, d), np.nan)
    for p in range(P):
        place(Kc, Vc, oracle_mod, 0, 0, p, K[0, 0, p].numpy(), V[0, 0, p].numpy(), w, g)
        pos = np.array([p])
        Oc, Lc = oracle_mod.decode_cache(q[p], Kc, Vc, pos, w, g, 0.6)
        Oh, Lh = oracle_mod.decode_history(q[p], K, V, pos, w, g, 0.6)
        assert np.allclose(Oc, Oh, atol=1e-12, rtol=0), p
        assert np.allclose(Lc, Lh, atol=1e-12, rtol=0), p


# --------------------------------------------------------------------------
# learned per-head sink logit ("Sliding Window and Sparse Attention, from
# Longformer to CSA2", section 6, stage 3): one more softmax entry per head
# with score sink_h and a zero value vector
# --------------------------------------------------------------------------
def sdpa_with_sink(Q, K, V, mask_bool, scale, sink):
    """torch SDPA over the keys plus one extra zero key/zero value whose
    additive mask entry is sink[h]; also returns the log-sum-exp."""
    B, H, n, d = Q.shape
    G = H // K.shape[1]
    Ke = torch.cat([K.repeat_interleave(G, dim=1), torch.zeros(B, H, 1, d, dtype=Q.dtype)], dim=2)
    Ve = torch.cat([V.repeat_interleave(G, dim=1), torch.zeros(B, H, 1, d, dtype=Q.dtype)], dim=2)
    bias = torch.full((B, H, n, n + 1), -math.inf, dtype=Q.dtype)
    bias[..., :n][:, :, torch.as_tensor(mask_bool, dtype=torch.bool)] = 0.0
    bias[..., n] = torch.as_tensor(sink, dtype=Q.dtype).view(1, H, 1)
    O = torch.nn.functional.scaled_dot_product_attention(Q, Ke, Ve, attn_mask=bias, scale=scale)
    L = torch.logsumexp(scale * Q @ Ke.transpose(-1, -2) + bias, dim=-1)
    return O, L


@pytest.mark.parametrize("n,w,g,H,Hkv", [(40, 7, 2, 2, 1), (33, 50, 0, 4, 2), (25, 1, 3, 2, 2)])
def test_sink_logit_is_an_extra_zero_value_entry(oracle_mod, n, w, g, H, Hkv):
    B, d, scale = 2, 16, 0.3
    Q, K, V = rand(B, H, n, d, seed=40), rand(B, Hkv, n, d, seed=41), rand(B, Hkv, n, d, seed=42)
    sink = np.linspace(-2.0, 3.0, H)
    O, L = oracle_mod.prefill(Q, K, V, w, g, scale, sink_logit=sink)
    ref, refL = sdpa_with_sink(Q, K, V, torch_mask(n, w, g).astype(bool), scale, sink)
    assert np.allclose(O, ref.numpy(), atol=1e-12, rtol=0)
    assert np.allclose(L, refL.numpy(), atol=1e-12, rtol=0)


def test_sink_logit_window_one_is_a_sigmoid(oracle_mod):
    # w = 1: the only key is the row itself, so O_i = V_i * sigmoid(s_ii - sink)
    B, H, n, d, scale = 1, 3, 20, 8, 0.5
    Q, K, V = rand(B, H, n, d, seed=43), rand(B, H, n, d, seed=44), rand(B, H, n, d, seed=45)
    sink = np.array([-1.0, 0.0, 2.5])
    O, L = oracle_mod.prefill(Q, K, V, 1, 0, scale, sink_logit=sink)
    s_ii = scale * (Q * K).sum(-1).numpy()
    sig = 1.0 / (1.0 + np.exp(-(s_ii - sink.reshape(1, H, 1))))
    assert np.allclose(O, V.numpy() * sig[..., None], atol=1e-13, rtol=0)
    assert np.allclose(L, np.logaddexp(s_ii, sink.reshape(1, H, 1)), atol=1e-13, rtol=0)


def test_sink_logit_minus_inf_and_huge(oracle_mod):
    B, H, Hkv, n, d = 1, 2, 1, 30, 8
    Q, K, V = rand(B, H, n, d, seed=46), rand(B, Hkv, n, d, seed=47), rand(B, Hkv, n, d, seed=48)
    O0, L0 = oracle_mod.prefill(Q, K, V, 6, 2, 0.4)
    O1, L1 = oracle_mod.prefill(Q, K, V, 6, 2, 0.4, sink_logit=np.full(H, -np.inf))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)  # no sink: the plain softmax
    O2, L2 = oracle_mod.prefill(Q, K, V, 6, 2, 0.4, sink_logit=np.full(H, 800.0))
    assert np.abs(O2).max() < 1e-300  # the sink takes all the mass
    assert np.allclose(L2, 800.0, atol=1e-12, rtol=0)


def test_sink_logit_decode_matches_prefill_rows(oracle_mod):
    B, H, Hkv, d, P, w, g = 2, 4, 2, 16, 30, 6, 2
    K, V = rand(B, Hkv, P, d, seed=49), rand(B, Hkv, P, d, seed=50)
    q = rand(B, H, d, seed=51)
    sink = np.array([0.5, -0.5, 1.5, -3.0])
    pos = np.array([29, 11])
    Oh, Lh = oracle_mod.decode_history(q, K, V, pos, w, g, 0.25, sink_logit=sink)
    for b in range(B):
        p = int(pos[b])
        Q = torch.zeros(1, H, p + 1, d, dtype=torch.float64)
        Q[0, :, p] = q[b]
        ref, refL = sdpa_with_sink(Q, K[b:b + 1, :, :p + 1], V[b:b + 1, :, :p + 1],
                                   torch_mask(p + 1, w, g).astype(bool), 0.25, sink)
        assert np.allclose(Oh[b], ref[0, :, p].numpy(), atol=1e-12, rtol=0)
        assert np.allclose(Lh[b], refL[0, :, p].numpy(), atol=1e-12, rtol=0)
    # the rolling cache gives the same as the unbounded history
    Kc = np.zeros((B, Hkv, w + g, d))
    Vc = np.zeros((B, Hkv, w + g, d))
    for b in range(B):
        for p in range(int(pos[b]) + 1):
            for kvh in range(Hkv):
                place(Kc, Vc, oracle_mod, b, kvh, p, K[b, kvh, p].numpy(), V[b, kvh, p].numpy(), w, g)
    Oc, Lc = oracle_mod.decode_cache(q, Kc, Vc, pos, w, g, 0.25, sink_logit=sink)
    assert np.allclose(Oc, Oh, atol=1e-12, rtol=0)
    assert np.allclose(Lc, Lh, atol=1e-12, rtol=0)
