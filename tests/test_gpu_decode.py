"""Decode and cache-append parity: the CUDA path against the fp64 oracle.
The rolling cache is checked against the unbounded history at every decode
position; slot placement is checked bit-exactly."""
import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close


@pytest.mark.gpu
def test_decode_streaming_workload_full_size(swa, oracle_mod):
    s = synthetic.WORKLOADS["streaming_decode_sinks"]
    x = synthetic.decode_cache_inputs(s["B"], s["H"], s["Hkv"], s["d"], s["w"], s["g"], s["pos"],
                                      dtype="bf16", seed=0, sink_scale=s["sink_scale"],
                                      device="cuda")
    out = swa.decode(x.q, x.Kc, x.Vc, x.pos, x.w, x.g, x.scale)  # library workspace path
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    O, _ = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), x.w, x.g, x.scale)
    assert_close(out, O, "bf16", "streaming decode full size")


DEC_CASES = [
    # B, H, Hkv, d, w, g, positions
    (2, 4, 1, 128, 64, 4, [200, 67]),        # sinks out of the window / just left
    (3, 8, 2, 128, 64, 4, [0, 5, 63]),       # partly filled ring
    (2, 2, 2, 64, 100, 0, [99, 1000]),
    (1, 8, 1, 128, 33, 5, [35]),             # sinks still inside the window for some
    (4, 16, 2, 128, 300, 2, [301, 302, 1, 299]),
    (2, 32, 16, 128, 128, 0, [500, 127]),    # GQA group of 2 (the Gemma-3 shape)
    (3, 6, 3, 64, 40, 3, [2, 41, 3000]),     # group of 2, d = 64
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,d,w,g,pos", DEC_CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_matches_oracle(swa, oracle_mod, B, H, Hkv, d, w, g, pos, dtype):
    x = synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, pos, dtype=dtype, seed=w + g,
                                      sink_scale=4.0, device="cuda")
    O, L = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), w, g, x.scale)
    for splits in (1, 2, 3, 7, 16):
        lse = torch.empty(B, H, dtype=torch.float32, device="cuda")
        out = swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale, lse=lse, num_splits=splits)
        torch.cuda.synchronize()
        assert_close(out, O, dtype, f"decode splits={splits}")
        tol = 2e-3 if dtype == "bf16" else 1e-5
        assert np.abs(lse.cpu().double().numpy() - L).max() < tol
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_decode_result_does_not_depend_on_split_count(swa):
    x = synthetic.decode_cache_inputs(4, 8, 2, 128, 1000, 4, 5000, seed=9, sink_scale=4.0,
                                      device="cuda")
    outs = [swa.decode(x.q, x.Kc, x.Vc, x.pos, 1000, 4, x.scale, num_splits=s).float()
            for s in (1, 2, 5, 13, 64, 250)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2e-2


@pytest.mark.gpu
@pytest.mark.parametrize("w,g", [(8, 2), (3, 1), (5, 0), (4, 6)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_streaming_append_then_decode_matches_history(swa, oracle_mod, w, g, dtype):
    B, H, Hkv, d, P = 2, 4, 2, 128, 41
    K, V = synthetic.token_stream(B, Hkv, d, P, dtype=dtype, seed=7, device="cuda", g=g,
                                  sink_scale=4.0)
    gen = torch.Generator(device="cuda").manual_seed(8)
    qs = torch.randn(P, B, H, d, generator=gen, device="cuda").to(synthetic.torch_dtype(dtype))
    Kc = torch.zeros(B, Hkv, w + g, d, dtype=K.dtype, device="cuda")
    Vc = torch.zeros_like(Kc)
    scale = 0.125
    for p in range(P):
        pos = torch.full((B,), p, dtype=torch.int32, device="cuda")
        swa.cache_append(Kc, Vc, K[:, :, p:p + 1].contiguous(), V[:, :, p:p + 1].contiguous(),
                         pos, w, g)
        out = swa.decode(qs[p], Kc, Vc, pos, w, g, scale, num_splits=2)
        torch.cuda.synchronize()
        O, _ = oracle_mod.decode_history(qs[p], K, V, np.full(B, p), w, g, scale)
        assert_close(out, O, dtype, f"stream p={p}")
    assert swa.device_status() == 0


def expected_cache(oracle_mod, K, pos0, T, w, g, init):
    """Cache contents after appending positions pos0..pos0+T-1 onto `init`,
    placed with the oracle's slot map (ring: only the last w positions)."""
    C = init.clone()
    B = K.shape[0]
    for b in range(B):
        for t in range(T):
            p = int(pos0[b]) + t
            ring, sink = oracle_mod.cache_slots(p, w, g)
            if t >= T - w:
                C[b, :, ring] = K[b, :, t]
            if sink >= 0:
                C[b, :, sink] = K[b, :, t]
    return C


@pytest.mark.gpu
@pytest.mark.parametrize("T,w,g,pos0", [(5, 8, 2, [0, 6]), (20, 8, 3, [0, 100]), (1, 3, 1, [8, 2]),
                                        (7, 7, 7, [3, 0])])
def test_chunked_append_slots_bit_exact(swa, oracle_mod, T, w, g, pos0):
    B, Hkv, d = 2, 2, 64
    gen = torch.Generator(device="cuda").manual_seed(T * 31 + w)
    Kn = torch.randn(B, Hkv, T, d, generator=gen, device="cuda").to(torch.bfloat16)
    Vn = torch.randn(B, Hkv, T, d, generator=gen, device="cuda").to(torch.bfloat16)
    Kc = torch.randn(B, Hkv, w + g, d, generator=gen, device="cuda").to(torch.bfloat16)
    Vc = torch.randn(B, Hkv, w + g, d, generator=gen, device="cuda").to(torch.bfloat16)
    expK = expected_cache(oracle_mod, Kn.cpu(), pos0, T, w, g, Kc.cpu())
    expV = expected_cache(oracle_mod, Vn.cpu(), pos0, T, w, g, Vc.cpu())
    swa.cache_append(Kc, Vc, Kn, Vn, torch.tensor(pos0, dtype=torch.int32, device="cuda"), w, g)
    torch.cuda.synchronize()
    assert torch.equal(Kc.cpu(), expK)
    assert torch.equal(Vc.cpu(), expV)


@pytest.mark.gpu
def test_negative_position_is_reported(swa):
    x = synthetic.decode_cache_inputs(2, 4, 2, 64, 16, 0, [5, -3], seed=1, device="cuda")
    assert swa.device_status() == 0
    out = swa.decode(x.q, x.Kc, x.Vc, x.pos, 16, 0, x.scale, num_splits=2)
    assert swa.device_status() == -1  # SWA_ERR_INVALID_ARG, read from the device
    assert torch.isfinite(out.float()).all()
    assert swa.device_status() == 0   # cleared


# groups the kernels are not built for directly: padded sub-groups (3 -> 4,
# 5/6/7 -> 8) and groups split into sub-groups of at most 8 heads (12, 16, 24)
ANY_G_CASES = [
    # B, H, Hkv, d, w, g, positions
    (2, 6, 2, 128, 64, 4, [200, 5]),          # group of 3
    (2, 5, 1, 128, 100, 2, [99, 3000]),       # group of 5
    (3, 12, 2, 64, 50, 3, [0, 51, 777]),      # group of 6, d = 64
    (1, 7, 1, 128, 33, 0, [40]),              # group of 7
    (2, 24, 2, 128, 128, 4, [130, 1000]),     # group of 12: two sub-groups of 6
    (2, 16, 1, 128, 256, 4, [300, 17]),       # group of 16: two sub-groups of 8
    (1, 24, 1, 64, 70, 1, [500]),             # group of 24: three sub-groups of 8
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,d,w,g,pos", ANY_G_CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_any_group_matches_oracle(swa, oracle_mod, B, H, Hkv, d, w, g, pos, dtype):
    x = synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, pos, dtype=dtype, seed=H + w,
                                      sink_scale=4.0, device="cuda")
    O, L = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), w, g, x.scale)
    for splits in (0, 1, 3):
        lse = torch.empty(B, H, dtype=torch.float32, device="cuda")
        out = torch.full_like(x.q, float("nan"))
        swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale, out=out, lse=lse, num_splits=splits)
        torch.cuda.synchronize()
        assert_close(out, O, dtype, f"decode G={H // Hkv} splits={splits}")
        tol = 2e-3 if dtype == "bf16" else 1e-5
        assert np.abs(lse.cpu().double().numpy() - L).max() < tol
    if dtype == "bf16":  # the library-workspace entry point too
        out = swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale)
        torch.cuda.synchronize()
        assert_close(out, O, dtype, f"swa_decode G={H // Hkv}")
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_streaming_group_of_three_matches_history(swa, oracle_mod):
    B, H, Hkv, d, P, w, g = 2, 6, 2, 128, 30, 8, 2
    K, V = synthetic.token_stream(B, Hkv, d, P, seed=17, device="cuda", g=g, sink_scale=4.0)
    gen = torch.Generator(device="cuda").manual_seed(18)
    qs = torch.randn(P, B, H, d, generator=gen, device="cuda").to(torch.bfloat16)
    Kc = torch.zeros(B, Hkv, w + g, d, dtype=K.dtype, device="cuda")
    Vc = torch.zeros_like(Kc)
    for p in range(P):
        pos = torch.full((B,), p, dtype=torch.int32, device="cuda")
        swa.cache_append(Kc, Vc, K[:, :, p:p + 1].contiguous(), V[:, :, p:p + 1].contiguous(),
                         pos, w, g)
        out = swa.decode(qs[p], Kc, Vc, pos, w, g, 0.125)
        torch.cuda.synchronize()
        O, _ = oracle_mod.decode_history(qs[p], K, V, np.full(B, p), w, g, 0.125)
        assert_close(out, O, "bf16", f"stream G=3 p={p}")
    assert swa.device_status() == 0
