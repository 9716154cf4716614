"""The C-ABI boundary without a GPU: the library loads, exports every symbol
the header declares, validates arguments on the host, and its host helpers
(connection counts, tile classes, cache slots) agree bit-exactly with the
oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "swa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("swa_prefill", "swa_decode", "swa_cache_append"):
        assert required in names


def test_library_exports_every_declared_symbol(swa):
    lib = ctypes.CDLL(swa.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(swa.SIGNATURES)


def test_debug_library_exports_every_declared_symbol(swa):
    """libswa_debug.so (the kernels with their bounds checks) offers the same
    boundary; the product build has no checks to shrink."""
    lib = ctypes.CDLL(swa._LIB_DEBUG_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert swa.lib.swa_debug_shrink_bounds() == -2  # SWA_ERR_UNSUPPORTED
    with swa.debug_build():
        assert swa.lib.swa_version() >= 100
        assert swa.lib.swa_status_string(-7).decode() == "SWA_ERR_DEVICE_BOUNDS"


def test_version_and_status_strings(swa):
    assert swa.lib.swa_version() >= 100
    for code, name in swa.STATUS.items():
        assert swa.lib.swa_status_string(code).decode() == name


def test_count_pairs_matches_oracle(swa, oracle_mod):
    for n in (1, 2, 7, 8, 9, 63, 64, 65, 300):
        for w in (1, 2, 3, 8, 64, 500):
            for g in (0, 1, 4, 9):
                assert swa.count_pairs(n, w, g) == oracle_mod.count_pairs(n, w, g), (n, w, g)
    assert swa.count_pairs(8, 3, 0) == 21 and swa.count_pairs(8, 8, 0) == 36
    assert swa.count_pairs(16384, 4096, 0) == oracle_mod.count_pairs(16384, 4096, 0)
    assert swa.count_pairs(131072, 4096, 4) == 528992250
    assert swa.count_pairs(-1, 3, 0) == -1


@pytest.mark.parametrize("BM,BN", [(128, 128), (64, 32), (16, 16), (128, 64), (32, 128)])
def test_tile_classes_match_oracle(swa, oracle_mod, BM, BN):
    rng = np.random.default_rng(BM * 1000 + BN)
    cases = [(1, 1, 0), (300, 64, 0), (300, 100, 4), (257, 3, 1), (200, 1000, 0), (129, 128, 130),
             (333, 17, 5), (1000, 129, 1), (512, 64, 0), (700, 256, 300)]
    cases += [(int(rng.integers(1, 700)), int(rng.integers(1, 400)), int(rng.integers(0, 20)))
              for _ in range(12)]
    for n, w, g in cases:
        mine = swa.enumerate_tiles(n, w, g, BM, BN).numpy()
        ref = oracle_mod.tiles(n, w, g, BM, BN)
        assert np.array_equal(mine, ref), (n, w, g, BM, BN)


def test_tile_classes_workload_counts(swa):
    # partial/full tile counts per head at 128x128 tiles for the benchmark shapes
    t = swa.enumerate_tiles(16384, 4096, 0, 128, 128).numpy()
    assert (t == 2).sum() == 3472 and (t == 1).sum() == 224
    t = swa.enumerate_tiles(32768, 1024, 0, 128, 128).numpy()
    assert (t == 2).sum() == 1764 and (t == 1).sum() == 504


def test_cache_slot_matches_oracle(swa, oracle_mod):
    for w, g in [(3, 0), (3, 1), (4096, 4), (8, 2), (1, 5)]:
        for p in list(range(0, 20)) + [4095, 4096, 100000]:
            assert swa.cache_slot(p, w, g) == oracle_mod.cache_slots(p, w, g), (p, w, g)
    with pytest.raises(swa.SwaError):
        swa.cache_slot(-1, 3, 0)
    with pytest.raises(swa.SwaError):  # w + g past INT32_MAX: the sink slot w + p would wrap
        swa.cache_slot(5, 2**31 - 10, 20)


def test_chunk_key_positions_refuses_lists_past_int32(swa):
    """The row count is the return value: a list of more than INT32_MAX rows is
    refused before anything is written (the buffer here holds one row)."""
    import ctypes
    one = ctypes.c_int64(7)
    off = ctypes.c_int32(0)
    rc = swa.lib.swa_chunk_key_positions(0, 2**31 - 200, 0, 2**30, ctypes.addressof(one), 2**62,
                                         ctypes.byref(off))
    assert rc == -1 and one.value == 7


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


def test_host_validation_rejects_before_launch(swa):
    L = swa.lib
    ok_args = dict(B=1, H=4, Hkv=2, n=16, d=128, w=4, g=0, scale=0.1)

    def prefill(**kw):
        a = dict(ok_args, **kw)
        return L.swa_prefill_ex(FAKE, FAKE, FAKE, FAKE, None, a["B"], a["H"], a["Hkv"], a["n"],
                                a["d"], a["w"], a["g"], a["scale"], 0, None)

    assert prefill(d=96) == -2          # unsupported head size
    assert prefill(H=3) == -1           # H not a multiple of Hkv
    assert prefill(w=0) == -1
    assert prefill(g=-1) == -1
    assert prefill(n=0) == -1
    assert prefill(scale=0.0) == -1
    assert prefill(scale=float("nan")) == -1
    assert L.swa_prefill_ex(FAKE + 8, FAKE, FAKE, FAKE, None, 1, 4, 2, 16, 128, 4, 0, 0.1, 0,
                            None) == -1  # misaligned Q
    assert L.swa_prefill_ex(None, FAKE, FAKE, FAKE, None, 1, 4, 2, 16, 128, 4, 0, 0.1, 0,
                            None) == -1  # null Q
    # decode: any group size is accepted (a group of 3 here; the missing
    # workspace is what is refused), bad split count, missing workspace
    assert L.swa_decode_ex(FAKE, FAKE, FAKE, FAKE, 1, 6, 2, 128, 8, 0, 0.1, FAKE, None, 0, 0,
                           None, 0, None) == -6
    assert L.swa_decode_ex(FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 128, 8, 0, 0.1, FAKE, None, 0, 2000,
                           None, 0, None) == -1
    assert L.swa_decode_ex(FAKE, FAKE, FAKE, FAKE, 2, 4, 2, 128, 8, 0, 0.1, FAKE, None, 0, 4,
                           None, 0, None) == -6
    # one partial (m, l, o[d]) per head of the group for each of the
    # num_splits*B*Hkv CTAs plus one per (sequence, kv head) segment boundary
    assert L.swa_decode_workspace_bytes(2, 4, 2, 128, 8, 0, 4) == (16 + 4) * 2 * 130 * 4
    assert L.swa_decode_workspace_bytes(2, 4, 2, 128, 8, 0, 1) == (4 + 4) * 2 * 130 * 4
    # more CTAs than cache rows are not used: at most one row per CTA
    assert L.swa_decode_workspace_bytes(1, 2, 1, 64, 3, 1, 1000) == (4 + 1) * 2 * 66 * 4
    # a group of 3 is scored as a padded group of 4
    assert L.swa_decode_workspace_bytes(2, 6, 2, 128, 8, 0, 4) == (16 + 4) * 4 * 130 * 4
    # a group of 16 is two sub-groups of 8: B * Hkv * 2 segments
    assert L.swa_decode_workspace_bytes(2, 16, 1, 128, 8, 0, 1) == (4 + 4) * 8 * 130 * 4
    # a group of 12 is two sub-groups of 6, each padded to 8
    assert L.swa_decode_workspace_bytes(1, 12, 1, 64, 8, 0, 2) == (4 + 2) * 8 * 66 * 4
    # append: negative T, misaligned cache; T == 0 is a no-op
    assert L.swa_cache_append(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 1, 2, 128, 8, 0, 0, None) == -1
    assert L.swa_cache_append(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 1, 1, 2, 128, 8, 0, 0, None) == -1
    assert L.swa_cache_append(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 2, 128, 8, 0, 0, None) == 0


def test_pattern_and_chunk_validation_rejects_before_launch(swa):
    L = swa.lib

    def pattern(pat, w=8, g=0, r=4, n=64, d=128, H=4, Hkv=2, scale=0.1):
        return L.swa_prefill_pattern(FAKE, FAKE, FAKE, FAKE, None, None, 1, H, Hkv, n, d, pat, w,
                                     g, r, scale, 0, None)

    assert pattern(7) == -1                   # no such pattern
    assert pattern(1, r=0) == -1              # stride below one
    assert pattern(2, r=-3) == -1
    assert pattern(1, g=2) == -2              # the class patterns take no sinks
    assert pattern(2, g=1) == -2
    assert pattern(3, r=0) == -1
    assert pattern(3, w=0) == -1
    assert pattern(1, d=96) == -2
    assert pattern(3, n=0) == -1
    assert pattern(1, scale=float("inf")) == -1
    assert pattern(0, w=0) == -1              # the window code is swa_prefill_sink_logit

    B, H, Hkv, T, d, w, g = 2, 4, 2, 50, 128, 64, 4
    need = L.swa_prefill_chunk_workspace_bytes(B, Hkv, T, d, w, g, 0)
    # key lists of roundup(g+w-1, 128) + roundup(T, 128) rows for K and V, bf16
    assert need == 2 * B * Hkv * (128 + 128) * d * 2
    assert L.swa_prefill_chunk_workspace_bytes(B, Hkv, 0, d, w, g, 0) == 0

    def chunk(T=T, ws=FAKE, ws_bytes=need, pos0=FAKE, append=1):
        return L.swa_prefill_chunk(FAKE, FAKE, FAKE, FAKE, FAKE, pos0, FAKE, None, None, B, H,
                                   Hkv, T, d, w, g, 0.1, append, 0, ws, ws_bytes, None)

    assert chunk(T=0) == -1
    assert chunk(pos0=None) == -1
    assert chunk(pos0=FAKE + 2) == -1         # pos0 not 4-byte aligned
    assert chunk(ws=None) == -6
    assert chunk(ws_bytes=need - 1) == -6
    assert chunk(ws=FAKE + 8) == -6           # workspace not 16-byte aligned


@pytest.mark.parametrize("n,w,g,r,BM,BN", [
    (300, 20, 0, 4, 32, 16), (500, 64, 3, 7, 64, 32), (257, 8, 9, 2, 16, 16),
    (1000, 100, 1, 50, 128, 128), (90, 200, 2, 5, 32, 8), (400, 30, 40, 8, 32, 32),
])
def test_landmark_tiles_cover_the_oracle_mask(swa, oracle_mod, n, w, g, r, BM, BN):
    # the kernels' landmark tiles (swa_enumerate_landmark_tiles) carry exactly the
    # landmark pairs the window tiles do not: mask(landmark) = mask(window) + those
    full = oracle_mod.pattern_mask(n, w, g, r, "landmark").astype(bool)
    win = oracle_mod.mask(n, w, g).astype(bool)
    assert not (win & ~full).any()
    extra = full & ~win                                   # pairs only the landmarks give
    cols = np.arange(0, n, r)                             # landmark m sits at position r*m
    assert not extra[:, np.setdiff1d(np.arange(n), cols)].any()
    need = extra[:, cols]                                 # [n rows, ceil(n/r) landmarks]
    nq, nk = -(-n // BM), -(-len(cols) // BN)
    pad = np.zeros((nq * BM, nk * BN), dtype=bool)
    pad[:n, :len(cols)] = need
    rows_exist = np.zeros(nq * BM, dtype=bool)
    rows_exist[:n] = True
    ref = np.zeros((nq, nk), dtype=np.int32)
    for qt in range(nq):
        for lt in range(nk):
            blk = pad[qt * BM:(qt + 1) * BM, lt * BN:(lt + 1) * BN]
            ex = rows_exist[qt * BM:(qt + 1) * BM]
            cnt = blk[ex].sum()
            ref[qt, lt] = 0 if cnt == 0 else (2 if cnt == ex.sum() * BN else 1)
    got = swa.enumerate_landmark_tiles(n, w, g, r, BM, BN).numpy()
    # the last row of a query tile needs every landmark from ceil(g/r) up to its
    # own limit, so the visited range holds no empty tile: classes match exactly
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("pos0,w,g,T", [
    (0, 64, 4, 50), (3, 64, 4, 50), (70, 64, 4, 50), (1000, 100, 2, 130), (99, 100, 2, 130),
    (200, 37, 5, 1), (5, 37, 5, 1), (600, 300, 3, 257), (1, 1, 2, 40), (10, 1, 2, 40),
    (300, 128, 0, 150), (50, 128, 0, 150), (100000, 4096, 4, 300), (4099, 4096, 4, 20),
    (4, 8, 4, 3), (12, 8, 4, 1),
])
def test_chunk_key_list_reads_the_oracle_positions(swa, oracle_mod, pos0, w, g, T):
    # the key list of a chunked prefill (the layout the gather kernel writes and the
    # prefill kernels index): with the prefill mask applied to list indices, chunk
    # query t reads exactly the positions the oracle's mask row pos0+t allows, each
    # once, and never a padding row
    pos, off = swa.chunk_key_positions(pos0, w, g, T)
    pos = pos.numpy()
    assert len(pos) % 128 == 0 and off + T <= len(pos)
    for t in range(T):
        i = t + off
        j = np.arange(i + 1)
        take = (j >= i - w + 1) | (j < g)
        got = pos[j[take]]
        assert (got >= 0).all(), (t, "reads a padding row")
        assert len(set(got.tolist())) == len(got), (t, "reads a key twice")
        want = np.nonzero(oracle_mod.mask_row(pos0 + t, pos0 + t + 1, w, g))[0]
        assert sorted(got.tolist()) == want.tolist(), t
    # the query offset is a multiple of the 128-row tile once the window has left the sinks
    if pos0 >= g and pos0 - w + 1 >= g:
        assert off % 128 == 0
