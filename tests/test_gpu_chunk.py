"""Chunked prefill into the rolling cache (swa_prefill_chunk): T new tokens
at positions pos0 .. pos0+T-1 attend to what the rolling cache keeps of the
earlier positions and to themselves.  Compared element by element with the
fp64 oracle over the unbounded history of positions (which knows nothing of
slots), for empty caches, caches still inside the sinks, wrapped rings,
single tokens, odd and even GQA groups, and a prompt fed in chunks."""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close


def build_cache(oracle_mod, K, V, pos0, w, g):
    """Rolling caches holding positions 0 .. pos0[b]-1 of each sequence, placed
    with the oracle's slot map; slots never written hold NaN (never read)."""
    B, Hkv, P, d = K.shape
    Kc = torch.full((B, Hkv, w + g, d), float("nan"), dtype=K.dtype)
    Vc = torch.full_like(Kc, float("nan"))
    for b in range(B):
        for p in range(int(pos0[b])):
            ring, sink = oracle_mod.cache_slots(p, w, g)
            Kc[b, :, ring] = K[b, :, p]
            Vc[b, :, ring] = V[b, :, p]
            if sink >= 0:
                Kc[b, :, sink] = K[b, :, p]
                Vc[b, :, sink] = V[b, :, p]
    return Kc, Vc


def oracle_chunk(oracle_mod, q, K, V, pos0, w, g, scale, sink=None):
    B, H, T, d = q.shape
    O = np.empty((B, H, T, d))
    L = np.empty((B, H, T))
    for t in range(T):
        o, l = oracle_mod.decode_history(q[:, :, t], K, V, np.asarray(pos0) + t, w, g, scale,
                                         sink_logit=sink)
        O[:, :, t] = o
        L[:, :, t] = l
    return O, L


CASES = [
    # B, H, Hkv, d, w, g, T, pos0 per sequence
    (3, 4, 2, 128, 64, 4, 50, [0, 3, 70]),      # empty cache, inside the sinks, wrapped ring
    (2, 3, 1, 128, 100, 2, 130, [1000, 99]),    # one-head kernel (odd group), T > one tile
    (2, 2, 2, 64, 37, 5, 1, [200, 5]),          # a single token (a decode step), d = 64
    (1, 8, 2, 128, 300, 3, 257, [600]),         # group of 4, ragged tiles
    (2, 2, 1, 64, 1, 2, 40, [1, 10]),           # window one: only the token itself and sinks
    (2, 4, 2, 128, 128, 0, 150, [300, 50]),     # no sinks, a window of one whole tile
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,d,w,g,T,pos0", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunk_prefill_matches_oracle(swa, oracle_mod, B, H, Hkv, d, w, g, T, pos0, dtype):
    P = max(pos0) + T
    K, V = synthetic.token_stream(B, Hkv, d, P, dtype=dtype, seed=P + w, g=g, sink_scale=4.0)
    gen = torch.Generator().manual_seed(T + d)
    q = torch.randn(B, H, T, d, generator=gen).to(synthetic.torch_dtype(dtype))
    Kc, Vc = build_cache(oracle_mod, K, V, pos0, w, g)
    kn = torch.stack([K[b, :, pos0[b]:pos0[b] + T] for b in range(B)])
    vn = torch.stack([V[b, :, pos0[b]:pos0[b] + T] for b in range(B)])
    scale = 1.0 / np.sqrt(d)
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    out = swa.prefill_chunk(q.cuda(), kn.cuda(), vn.cuda(), Kc.cuda(), Vc.cuda(),
                            torch.tensor(pos0, dtype=torch.int32, device="cuda"), w, g, scale,
                            lse=lse)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    O, L = oracle_chunk(oracle_mod, q, K, V, pos0, w, g, scale)
    assert_close(out, O, dtype, f"chunk {B,H,Hkv,d,w,g,T,pos0}")
    tol = 2e-3 if dtype == "bf16" else 1e-5
    assert np.abs(lse.cpu().double().numpy() - L).max() < tol


@pytest.mark.gpu
def test_chunk_prefill_with_sink_logit(swa, oracle_mod):
    B, H, Hkv, d, w, g, T, pos0 = 2, 4, 2, 128, 80, 4, 70, [150, 30]
    P = max(pos0) + T
    K, V = synthetic.token_stream(B, Hkv, d, P, dtype="bf16", seed=5, g=g, sink_scale=4.0)
    q = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    Kc, Vc = build_cache(oracle_mod, K, V, pos0, w, g)
    kn = torch.stack([K[b, :, pos0[b]:pos0[b] + T] for b in range(B)])
    vn = torch.stack([V[b, :, pos0[b]:pos0[b] + T] for b in range(B)])
    sink = torch.tensor([0.5, -1.0, 2.0, 0.0])
    out = swa.prefill_chunk(q.cuda(), kn.cuda(), vn.cuda(), Kc.cuda(), Vc.cuda(),
                            torch.tensor(pos0, dtype=torch.int32, device="cuda"), w, g, 0.1,
                            sink_logit=sink.cuda())
    torch.cuda.synchronize()
    O, _ = oracle_chunk(oracle_mod, q, K, V, pos0, w, g, 0.1, sink=sink.double())
    assert_close(out, O, "bf16", "chunk with sink logit")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fused", [False, True])
def test_prompt_in_chunks_then_decode(swa, oracle_mod, dtype, fused):
    # a prompt of 300 tokens taken in chunks of 64 (prefill_chunk with append, or
    # prefill_chunk then cache_append), then one decode step: every output against
    # the unbounded history
    B, H, Hkv, d, w, g, Lp, T = 2, 4, 2, 128, 100, 4, 300, 64
    K, V = synthetic.token_stream(B, Hkv, d, Lp + 1, dtype=dtype, seed=9, g=g, sink_scale=4.0)
    gen = torch.Generator().manual_seed(10)
    q = torch.randn(B, H, Lp + 1, d, generator=gen).to(synthetic.torch_dtype(dtype))
    Kc = torch.zeros(B, Hkv, w + g, d, dtype=K.dtype, device="cuda")
    Vc = torch.zeros_like(Kc)
    scale = 1.0 / np.sqrt(d)
    for p0 in range(0, Lp, T):
        t = min(T, Lp - p0)
        pos0 = torch.full((B,), p0, dtype=torch.int32, device="cuda")
        kn = K[:, :, p0:p0 + t].contiguous().cuda()
        vn = V[:, :, p0:p0 + t].contiguous().cuda()
        out = swa.prefill_chunk(q[:, :, p0:p0 + t].contiguous().cuda(), kn, vn, Kc, Vc, pos0, w, g,
                                scale, append=fused)
        if not fused:
            swa.cache_append(Kc, Vc, kn, vn, pos0, w, g)
        torch.cuda.synchronize()
        O, _ = oracle_chunk(oracle_mod, q[:, :, p0:p0 + t], K, V, [p0] * B, w, g, scale)
        assert_close(out, O, dtype, f"chunk at {p0}")
    # the next token, decoded from the cache the chunks built
    pos = torch.full((B,), Lp, dtype=torch.int32, device="cuda")
    swa.cache_append(Kc, Vc, K[:, :, Lp:Lp + 1].contiguous().cuda(),
                     V[:, :, Lp:Lp + 1].contiguous().cuda(), pos, w, g)
    o = swa.decode(q[:, :, Lp].contiguous().cuda(), Kc, Vc, pos, w, g, scale, num_splits=2)
    torch.cuda.synchronize()
    O, _ = oracle_mod.decode_history(q[:, :, Lp], K, V, np.full(B, Lp), w, g, scale)
    assert_close(o, O, dtype, "decode after chunks")
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_fused_append_writes_the_cache_bit_exact(swa, oracle_mod):
    # prefill_chunk(append=True) leaves the cache byte for byte as cache_append
    # does, including wrap-around (chunk longer than the window) and the sinks
    B, Hkv, H, d, w, g, T = 2, 2, 4, 128, 48, 3, 70
    pos0 = [0, 130]
    P = max(pos0) + T
    K, V = synthetic.token_stream(B, Hkv, d, P, dtype="bf16", seed=3, g=g)
    q = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    Kc, Vc = build_cache(oracle_mod, K, V, pos0, w, g)
    Kc, Vc = torch.nan_to_num(Kc).cuda(), torch.nan_to_num(Vc).cuda()
    kn = torch.stack([K[b, :, pos0[b]:pos0[b] + T] for b in range(B)]).cuda()
    vn = torch.stack([V[b, :, pos0[b]:pos0[b] + T] for b in range(B)]).cuda()
    p0 = torch.tensor(pos0, dtype=torch.int32, device="cuda")
    K2, V2 = Kc.clone(), Vc.clone()
    out = swa.prefill_chunk(q.cuda(), kn, vn, Kc, Vc, p0, w, g, append=True)
    ref = swa.prefill_chunk(q.cuda(), kn, vn, K2, V2, p0, w, g)  # reads the old cache
    swa.cache_append(K2, V2, kn, vn, p0, w, g)
    torch.cuda.synchronize()
    assert torch.equal(Kc.view(torch.int16), K2.view(torch.int16))
    assert torch.equal(Vc.view(torch.int16), V2.view(torch.int16))
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_chunk_full_size_sampled_rows(swa, oracle_mod):
    # the chunked-prefill workload at full size, in the call the benchmark times
    # (append on): sampled rows against the oracle's decode over the rolling cache
    # advanced to each row's position, and the appended cache bit for bit
    c = synthetic.WORKLOADS["chunked_prefill_stream"]
    B, H, Hkv, d, w, g, T, pos0 = (c[k] for k in ("B", "H", "Hkv", "d", "w", "g", "T", "pos0"))
    x = synthetic.chunk_inputs(B, H, Hkv, d, w, g, T, pos0, seed=0, sink_scale=c["sink_scale"],
                               device="cuda")
    Kc0, Vc0 = x.Kc.cpu(), x.Vc.cpu()
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    out = swa.prefill_chunk(x.q, x.k_new, x.v_new, x.Kc, x.Vc, x.pos0, w, g, x.scale, lse=lse,
                            append=True)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    kn, vn, q = x.k_new.cpu(), x.v_new.cpu(), x.q.cpu()
    slot = [oracle_mod.cache_slots(pos0 + t, w, g)[0] for t in range(T)]

    # the cache after the call: every ring slot now holds a chunk position, sinks untouched
    Kexp, Vexp = Kc0.clone(), Vc0.clone()
    for t in range(T):
        Kexp[:, :, slot[t]] = kn[:, :, t]
        Vexp[:, :, slot[t]] = vn[:, :, t]
    assert torch.equal(x.Kc.cpu().view(torch.int16), Kexp.view(torch.int16))
    assert torch.equal(x.Vc.cpu().view(torch.int16), Vexp.view(torch.int16))

    gen = np.random.default_rng(1)
    picks = [(B - 1, t) for t in (0, 1, 127, 128, T // 2, T - 1)]
    picks += [(int(gen.integers(B)), int(gen.integers(T))) for _ in range(10)]
    got, got_lse = out.cpu(), lse.cpu()
    for b, t in picks:
        Kb, Vb = Kc0[b].clone(), Vc0[b].clone()
        for u in range(t + 1):
            Kb[:, slot[u]] = kn[b, :, u]
            Vb[:, slot[u]] = vn[b, :, u]
        O, L = oracle_mod.decode_cache(q[b:b + 1, :, t], Kb[None], Vb[None],
                                       np.array([pos0 + t]), w, g, x.scale)
        assert_close(got[b, :, t], O[0], "bf16", f"chunk row b={b} t={t}")
        assert np.abs(got_lse[b, :, t].double().numpy() - L[0]).max() < 2e-3
