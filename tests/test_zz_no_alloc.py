"""swa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (plugins handed only their buffers, processes whose memory
belongs to another allocator, loops where cudaMalloc/cudaFree are not
allowed).  It keeps its split partials in a fixed array inside the library.

Called through the C ABI and compared with swa_decode (the entry point that
allocates its workspace) on two calls in a row, since the array is shared and
keeps the previous call's contents; bit for bit with swa_decode_ex given a
NaN-filled workspace of its own, for smaller calls after a large one; and with
the fp64 oracle.  This file is collected last on purpose.
"""
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close

SWA_ERR_WORKSPACE = -6


def call_noalloc(swa, x, out, w, g):
    B, H, d = x.q.shape
    Hkv = x.Kc.shape[1]
    return swa.lib.swa_decode_noalloc(
        x.q.data_ptr(), x.Kc.data_ptr(), x.Vc.data_ptr(), x.pos.data_ptr(), B, H, Hkv, d, w, g,
        x.scale, out.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
def test_noalloc_decode_matches_swa_decode_twice(swa):
    cases = [
        # the streaming-decode workload: B=32 H=32 Hkv=8 d=128 w=4096 g=4, pos=100000
        dict(B=32, H=32, Hkv=8, d=128, w=4096, g=4, pos=100000, seed=0),
        # a different shape second, so the shared array holds another call's data
        dict(B=3, H=8, Hkv=2, d=128, w=300, g=2, pos=[5, 299, 1000], seed=1),
    ]
    for c in cases:
        x = synthetic.decode_cache_inputs(c["B"], c["H"], c["Hkv"], c["d"], c["w"], c["g"],
                                          c["pos"], dtype="bf16", seed=c["seed"], sink_scale=4.0,
                                          device="cuda")
        ref = swa.decode(x.q, x.Kc, x.Vc, x.pos, c["w"], c["g"], x.scale)  # swa_decode
        torch.cuda.synchronize()
        for _ in range(2):
            out = torch.full_like(x.q, float("nan"))
            assert call_noalloc(swa, x, out, c["w"], c["g"]) == 0
            torch.cuda.synchronize()
            assert_close(out, ref.double().cpu().numpy(), "bf16", f"noalloc {c}")
    assert swa.device_status() == 0


def call_decode_ex_fresh_workspace(swa, x, out, w, g):
    """swa_decode_ex with the automatic split count (the one swa_decode_noalloc
    uses) and a workspace of its own, filled with NaN, so that any partial the
    merge reads without the split pass having written it shows up."""
    B, H, d = x.q.shape
    Hkv = x.Kc.shape[1]
    nbytes = swa.decode_workspace_bytes(B, H, Hkv, d, w, g)
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    rc = swa.lib.swa_decode_ex(
        x.q.data_ptr(), x.Kc.data_ptr(), x.Vc.data_ptr(), x.pos.data_ptr(), B, H, Hkv, d, w, g,
        x.scale, out.data_ptr(), None, 0, 0, ws.data_ptr(), nbytes,
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0


@pytest.mark.gpu
def test_noalloc_is_bit_exact_after_a_larger_call(swa, oracle_mod):
    """A large call fills much of the shared array; smaller calls after it must
    read none of what it left: they equal, bit for bit, swa_decode_ex run with a
    NaN-filled workspace of its own (same kernels, same split count)."""
    cases = [
        dict(B=32, H=32, Hkv=8, d=128, w=4096, g=4, pos=100000, seed=2),   # the large one
        dict(B=2, H=8, Hkv=2, d=128, w=64, g=4, pos=[70, 3], seed=3),
        dict(B=1, H=2, Hkv=1, d=64, w=1000, g=0, pos=[5000], seed=4),
        dict(B=5, H=16, Hkv=2, d=128, w=512, g=2, pos=[1, 511, 512, 513, 90000], seed=5),
    ]
    for c in cases:
        x = synthetic.decode_cache_inputs(c["B"], c["H"], c["Hkv"], c["d"], c["w"], c["g"],
                                          c["pos"], dtype="bf16", seed=c["seed"], sink_scale=4.0,
                                          device="cuda")
        ref = torch.full_like(x.q, float("nan"))
        call_decode_ex_fresh_workspace(swa, x, ref, c["w"], c["g"])
        out = torch.full_like(x.q, float("nan"))
        assert call_noalloc(swa, x, out, c["w"], c["g"]) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"noalloc differs from swa_decode_ex for {c}"
        # and independently of the other entry points: the fp64 oracle
        O, _ = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), c["w"], c["g"],
                                       x.scale)
        assert_close(out, O, "bf16", f"noalloc vs oracle {c}")
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_the_array(swa):
    # 256 sequences x 8 kv heads: at least 2048 partials x 8 heads x (128+2) fp32 = 8.5 MB > 4 MiB
    B, H, Hkv, d, w, g = 256, 64, 8, 128, 65536, 0
    need = swa.decode_workspace_bytes(B, H, Hkv, d, w, g)
    assert need > (4 << 20)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    rc = swa.lib.swa_decode_noalloc(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                    pos.data_ptr(), B, H, Hkv, d, w, g, 0.1, dummy.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == SWA_ERR_WORKSPACE
