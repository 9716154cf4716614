"""The kernels' bounds checks (libswa_debug.so, built with SWA_DEBUG; see
include/swa.h): every kernel on tiny shapes (n <= 64; w in {1, 2, 3, >= n};
g in {0, 1, 4, > w}; groups of 1 to 4; positions before, at and past the
window), checked against the oracle with every check passing; and one check
made to fail on purpose (swa_debug_shrink_bounds), which must report
SWA_ERR_DEVICE_BOUNDS and skip exactly the store it guards.  Nothing traps."""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close

SWA_ERR_DEVICE_BOUNDS = -7


@pytest.fixture
def dbg(swa):
    with swa.debug_build():
        assert swa.device_status() == 0
        yield swa
        assert swa.device_status() == 0


TINY_PREFILL = [
    # B, H, Hkv, n, d, w, g
    (1, 1, 1, 1, 64, 1, 0),
    (1, 2, 1, 17, 128, 1, 0),
    (2, 2, 2, 33, 64, 2, 1),
    (1, 3, 1, 40, 128, 3, 4),
    (1, 4, 2, 64, 128, 80, 0),     # w >= n: full causal
    (2, 4, 1, 50, 128, 5, 9),      # g > w
    (1, 6, 3, 64, 64, 3, 1),
    (1, 8, 2, 61, 128, 16, 4),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g", TINY_PREFILL)
def test_tiny_prefill_passes_every_check(dbg, oracle_mod, B, H, Hkv, n, d, w, g):
    for dtype in ("bf16", "f32"):
        x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype=dtype, seed=n + w + g,
                                     sink_scale=4.0, device="cuda")
        lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
        out = dbg.prefill(x.Q, x.K, x.V, w, g, x.scale, lse=lse)
        assert dbg.device_status() == 0
        O, L = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
        assert_close(out, O, dtype, f"{dtype} prefill {B, H, Hkv, n, d, w, g}")
        assert np.abs(lse.double().cpu().numpy() - L).max() < 2e-3


@pytest.mark.gpu
@pytest.mark.parametrize("pattern,w,g,r", [("dilated", 3, 0, 2), ("strided", 0, 0, 8),
                                           ("landmark", 4, 1, 5), ("landmark", 2, 4, 3)])
def test_tiny_patterns_pass_every_check(dbg, oracle_mod, pattern, w, g, r):
    for H, Hkv in ((2, 1), (3, 1)):
        x = synthetic.prefill_inputs(1, H, Hkv, 60, 128, w, g, dtype="bf16", seed=r, device="cuda")
        out = dbg.prefill_pattern(x.Q, x.K, x.V, pattern, w, g, r, x.scale)
        assert dbg.device_status() == 0
        O, _ = oracle_mod.prefill_pattern(x.Q, x.K, x.V, w, g, r, pattern, x.scale)
        assert_close(out, O, "bf16", f"{pattern} H={H}")


def _with_tokens(Kc, Vc, kn, vn, p0, upto, w, g, oracle_mod):
    """CPU copies of the caches after tokens 0..upto-1 of kn/vn were written
    at positions p0, p0+1, ... (their ring slots, and sink slots below g)."""
    Kt, Vt = Kc.clone(), Vc.clone()
    for u in range(upto):
        ring, sink = oracle_mod.cache_slots(p0 + u, w, g)
        for slot in (ring, sink):
            if slot >= 0:
                Kt[:, :, slot] = kn[:, :, u]
                Vt[:, :, slot] = vn[:, :, u]
    return Kt, Vt


@pytest.mark.gpu
@pytest.mark.parametrize("w,g", [(1, 0), (3, 1), (16, 4), (8, 9)])
def test_tiny_append_decode_chunk_pass_every_check(dbg, oracle_mod, w, g):
    B, H, Hkv, d, T = 2, 4, 2, 128, 5
    for pos in sorted({0, w - 1, w + g + 2}):
        c = synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, pos, seed=pos + 1, sink_scale=4.0,
                                          device="cuda")
        # a cache as appends leave it: a position below g still in the window
        # has the same key and value in its ring slot and its sink slot
        for q in range(min(g, pos + 1)):
            if pos - q < w:
                c.Kc[:, :, w + q] = c.Kc[:, :, q % w]
                c.Vc[:, :, w + q] = c.Vc[:, :, q % w]
        p = torch.full((B,), pos, dtype=torch.int32, device="cuda")
        out = dbg.decode(c.q, c.Kc, c.Vc, p, w, g, c.scale)
        assert dbg.device_status() == 0
        O, _ = oracle_mod.decode_cache(c.q, c.Kc, c.Vc, np.full(B, pos), w, g, c.scale)
        assert_close(out, O, "bf16", f"decode pos={pos}")
        # append T tokens at pos+1 .., exactly into their slots
        kn, vn = synthetic.token_stream(B, Hkv, d, T, seed=pos + 2)
        Kt, Vt = _with_tokens(c.Kc.cpu(), c.Vc.cpu(), kn, vn, pos + 1, T, w, g, oracle_mod)
        p1 = torch.full((B,), pos + 1, dtype=torch.int32, device="cuda")
        dbg.cache_append(c.Kc, c.Vc, kn.cuda(), vn.cuda(), p1, w, g)
        assert dbg.device_status() == 0
        assert torch.equal(c.Kc.cpu(), Kt) and torch.equal(c.Vc.cpu(), Vt)
        # a chunk of T more at pos+1+T, appended in the same call: row t sees
        # the cache with the chunk's tokens 0..t in it
        qc = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(pos)).to(torch.bfloat16)
        kc, vc = synthetic.token_stream(B, Hkv, d, T, seed=pos + 3)
        p2 = pos + 1 + T
        o3 = dbg.prefill_chunk(qc.cuda(), kc.cuda(), vc.cuda(), c.Kc, c.Vc,
                               torch.full((B,), p2, dtype=torch.int32, device="cuda"), w, g,
                               c.scale, append=True)
        assert dbg.device_status() == 0
        for t in (0, T - 1):
            Kq, Vq = _with_tokens(Kt, Vt, kc, vc, p2, t + 1, w, g, oracle_mod)
            O3, _ = oracle_mod.decode_cache(qc[:, :, t], Kq, Vq, np.full(B, p2 + t), w, g, c.scale)
            assert_close(o3[:, :, t], O3, "bf16", f"chunk row {t} pos={p2 + t}")


@pytest.mark.gpu
def test_shrunk_bound_fails_reports_and_skips_its_store(dbg, oracle_mod):
    """The last output row of the last head of the last sequence fails its
    check: it is left as it was (NaN here), every other row is exact, and the
    status word says SWA_ERR_DEVICE_BOUNDS."""
    B, H, Hkv, n, d, w, g = 2, 4, 2, 100, 128, 30, 4
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=11, device="cuda")
    out = torch.full_like(x.Q, float("nan"))
    dbg.shrink_bounds()
    dbg.prefill(x.Q, x.K, x.V, w, g, x.scale, out=out)
    assert dbg.device_status() == SWA_ERR_DEVICE_BOUNDS
    got = out.float().cpu()
    assert torch.isnan(got[B - 1, H - 1, n - 1]).all()
    O, _ = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
    mask = torch.ones(B, H, n, dtype=torch.bool)
    mask[B - 1, H - 1, n - 1] = False
    assert_close(got[mask].numpy(), O[mask.numpy()], "bf16", "rows that passed their checks")
    # the setting was used once: the next launch writes every row
    out2 = dbg.prefill(x.Q, x.K, x.V, w, g, x.scale)
    assert dbg.device_status() == 0
    assert_close(out2, O, "bf16", "after the shrunk launch")
