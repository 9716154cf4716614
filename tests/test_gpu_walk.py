"""The tile walk the prefill kernels actually take, logged by their producers
(swa_debug_prefill_walk), against the tile set of the method as the fp64
oracle defines it: every 128-row query tile of every head is visited by
exactly one work item, which loads exactly the key tiles holding at least one
allowed (query, key) pair, sink tiles before band tiles, each once; tiles the
kernel treats as mask-free are those the oracle finds full.  ("Sliding Window and Sparse
Attention, from Longformer to CSA2", section 4: block-sparse attention reads
only the tiles that meet the band; "Local and Sparse Attention: Reading Fewer
Token Positions", Figures 1-2.)"""
import collections

import numpy as np
import pytest

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close

BM = BN = 128
FULL, LAND = 1, 2


def group_items(entries):
    """{(b, kvh, unit, qtile, cls): [(k0, flags), ...] in load order}, after
    checking that each such item is one work item (one rank)."""
    items, ranks = collections.OrderedDict(), {}
    for e in entries.tolist():
        t, b, kvh, u, qt, cls, k0, fl = e
        key = (b, kvh, u, qt, cls)
        assert ranks.setdefault(key, t) == t, f"item {key} loaded by two work items"
        items.setdefault(key, []).append((k0, fl))
    return items


def check_window_walk(items, B, H, Hkv, n, w, g, oracle_mod):
    G = H // Hkv
    pairs = G % 2 == 0
    cls = oracle_mod.tiles(n, w, g, BM, BN)
    n_qt = cls.shape[0]
    n_items_qt = n_qt if pairs else -(-n_qt // 2)
    units = G // 2 if pairs else G
    expect = {(b, k, u, q, 0) for b in range(B) for k in range(Hkv) for u in range(units)
              for q in range(n_items_qt)}
    assert set(items) == expect, "work items missing or extra"
    for (b, k, u, q, _), tiles in items.items():
        kts = [k0 // BN for k0, _ in tiles]
        assert all(k0 % BN == 0 for k0, _ in tiles)
        assert len(kts) == len(set(kts)), f"a key tile loaded twice in item {(b, k, u, q)}"
        rows = [q] if pairs else [qq for qq in (2 * q, 2 * q + 1) if qq < n_qt]
        want = set()
        for qq in rows:
            want |= set(np.nonzero(cls[qq])[0].tolist())
        assert set(kts) == want, (f"item {(b, k, u, q)}: kernel tiles {sorted(kts)} "
                                  f"oracle tiles {sorted(want)}")
        # sink tiles below the band first, then the band in ascending order
        assert kts == sorted(kts), f"tiles out of order in item {(b, k, u, q)}"
        if pairs:  # mask-free tiles are exactly the oracle's full ones
            for k0, fl in tiles:
                assert bool(fl & FULL) == (cls[q, k0 // BN] == 2), (q, k0, fl)
        for k0, fl in tiles:  # no flag outside full and landmark
            assert fl & ~(FULL | LAND) == 0, (q, k0, fl)


CASES = [
    # B, H, Hkv, n, d, w, g
    (2, 4, 2, 700, 128, 200, 4),      # even group, 4 sinks in a tile below the band
    (1, 3, 1, 900, 64, 300, 0),       # group of 3: q-tile pairs
    (1, 2, 1, 600, 128, 100, 20),     # 20 sinks: a full 128-key sink tile
    (1, 2, 2, 1000, 128, 1000, 0),    # multi-head attention, full causal
    (1, 8, 2, 333, 128, 64, 1),       # group of 4, ragged tail
    (1, 32, 8, 16384, 128, 4096, 0),  # the Mistral-like layer, full size
    (2, 32, 16, 32768, 128, 1024, 0), # the Gemma-3-like layer, full size
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g", CASES)
def test_window_walk_matches_oracle_tiles(swa, oracle_mod, B, H, Hkv, n, d, w, g):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=n + w, sink_scale=4.0,
                                 device="cuda")
    out, entries = swa.prefill_walk(x.Q, x.K, x.V, "window", w, g, 1, x.scale)
    items = group_items(entries)
    check_window_walk(items, B, H, Hkv, n, w, g, oracle_mod)
    if n <= 1000:  # the logged run is a normal prefill
        O, _ = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
        assert_close(out, O, "bf16", "walk run output")
    assert swa.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("n,w,g,r", [(1500, 256, 4, 16), (2100, 600, 4, 32)])
def test_landmark_walk_matches_oracle_mask(swa, oracle_mod, n, w, g, r):
    B, H, Hkv, d = 1, 4, 2, 128
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=3, sink_scale=4.0,
                                 device="cuda")
    out, entries = swa.prefill_walk(x.Q, x.K, x.V, "landmark", w, g, r, x.scale)
    items = group_items(entries)
    band = oracle_mod.tiles(n, w, g, BM, BN)
    n_qt = band.shape[0]
    assert set(items) == {(0, k, u, q, 0) for k in range(Hkv) for u in range(1) for q in range(n_qt)}
    for (_, _, _, q, _), tiles in items.items():
        # landmark tiles: the landmarks (j mod r == 0) some row of the q tile reads
        # outside its band and sinks, as landmark-list tiles, from the oracle's mask
        want_land = set()
        for i in range(q * BM, min(n, q * BM + BM)):
            row = oracle_mod.pattern_mask_row(i, n, w, g, r, "landmark")
            for j in np.nonzero(row)[0]:
                if j < g or j >= i - w + 1:
                    continue
                assert j % r == 0
                want_land.add((j // r) // BN)
        got_land = {k0 // BN for k0, fl in tiles if fl & LAND}
        assert got_land == want_land, (q, sorted(got_land), sorted(want_land))
        got_band = {k0 // BN for k0, fl in tiles if not fl & LAND}
        assert got_band == set(np.nonzero(band[q])[0].tolist()), q
        kinds = [bool(fl & LAND) for _, fl in tiles]
        assert kinds == sorted(kinds, reverse=True), "landmark tiles are loaded first"
    O, _ = oracle_mod.prefill_pattern(x.Q, x.K, x.V, w, g, r, "landmark", x.scale)
    assert_close(out, O, "bf16", "landmark walk run output")


@pytest.mark.gpu
@pytest.mark.parametrize("H,Hkv", [(2, 1), (3, 1)])
def test_dilated_walk_covers_every_class(swa, oracle_mod, H, Hkv):
    B, n, d, w, r = 1, 1000, 128, 100, 3
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, 0, dtype="bf16", seed=4, device="cuda")
    out, entries = swa.prefill_walk(x.Q, x.K, x.V, "dilated", w, 0, r, x.scale)
    items = group_items(entries)
    G = H // Hkv
    units = G // 2 if G % 2 == 0 else G
    seen = set()
    for (b, k, u, q, c), tiles in items.items():
        n_c = (n - c + r - 1) // r                 # rows of residue class c
        cls = oracle_mod.tiles(n_c, w, 0, BM, BN)  # a window of w inside the class
        assert {k0 // BN for k0, _ in tiles} == set(np.nonzero(cls[q])[0].tolist()), (c, q)
        seen.add((b, k, u, q, c))
    want = {(0, k, u, q, c) for k in range(Hkv) for u in range(units) for c in range(r)
            for q in range(-(-((n - c + r - 1) // r) // BM))}
    assert seen == want
    O, _ = oracle_mod.prefill_pattern(x.Q, x.K, x.V, w, 0, r, "dilated", x.scale)
    assert_close(out, O, "bf16", "dilated walk run output")
