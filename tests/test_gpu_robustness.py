"""Failure paths and concurrency of the library, on the GPU, made without a
GPU fault:

* the kernels' bounded waits: swa_debug_inject_stall makes one launch leave
  out its first key/value copy, so a wait runs out after a short limit; the
  kernel must stop cleanly (copies drained, tensor memory freed), the status
  word must say SWA_ERR_DEVICE_TIMEOUT, and the next normal launches on the
  same context must match the oracle;
* a workspace allocation that fails (a request larger than the GPU) returns
  SWA_ERR_ALLOC and leaves the library usable;
* swa_decode on two streams at once, and from two host threads whose shapes
  make their workspaces grow, match the oracle;
* positions at the end of the int32 range: an append that would pass
  INT32_MAX writes nothing and is reported; a decode at INT32_MAX - 1 is
  exact;
* a process that uses two GPUs sets each kernel's shared-memory limit on both.
"""
import threading

import numpy as np
import pytest
import torch

from sink_sparse_attention_swa_b300 import synthetic
from tests.parity import assert_close

SWA_ERR_INVALID_ARG = -1
SWA_ERR_DEVICE_TIMEOUT = -4
SWA_ERR_ALLOC = -5
INT32_MAX = 2**31 - 1


def _prefill_ok(swa, oracle_mod, B, H, Hkv, n, d, w, g, pattern=None, r=1, seed=0):
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=seed, sink_scale=4.0,
                                 device="cuda")
    if pattern is None:
        out = swa.prefill(x.Q, x.K, x.V, w, g, x.scale)
        O, _ = oracle_mod.prefill(x.Q, x.K, x.V, w, g, x.scale)
    else:
        out = swa.prefill_pattern(x.Q, x.K, x.V, pattern, w, g, r, x.scale)
        O, _ = oracle_mod.prefill_pattern(x.Q, x.K, x.V, w, g, r, pattern, x.scale)
    torch.cuda.synchronize()
    assert_close(out, O, "bf16", f"prefill after recovery {B, H, Hkv, n, d, w, g, pattern}")


# (B, H, Hkv, n, d, w, g, pattern, r): the head-pair kernel (even group), the
# q-tile-pair kernel (group of one) and the single-head kernel (a fixed
# pattern with an odd group)
STALL_PREFILL = [
    (1, 2, 1, 256, 128, 64, 4, None, 1),
    (1, 1, 1, 384, 64, 100, 0, None, 1),
    (1, 3, 1, 300, 128, 16, 0, "dilated", 3),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Hkv,n,d,w,g,pattern,r", STALL_PREFILL)
def test_prefill_wait_runs_out_and_recovers(swa, oracle_mod, B, H, Hkv, n, d, w, g, pattern, r):
    assert swa.device_status() == 0
    x = synthetic.prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=3, device="cuda")
    swa.inject_stall("prefill", 1_000_000)  # 1 ms per bounded wait
    if pattern is None:
        swa.prefill(x.Q, x.K, x.V, w, g, x.scale)
    else:
        swa.prefill_pattern(x.Q, x.K, x.V, pattern, w, g, r, x.scale)
    assert swa.device_status() == SWA_ERR_DEVICE_TIMEOUT
    assert swa.device_status() == 0  # read and cleared
    # the context is intact: tensor memory was freed, later launches are exact
    _prefill_ok(swa, oracle_mod, B, H, Hkv, n, d, w, g, pattern, r, seed=4)
    _prefill_ok(swa, oracle_mod, 1, 4, 2, 300, 128, 64, 4, seed=5)
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_decode_wait_runs_out_and_recovers(swa, oracle_mod):
    assert swa.device_status() == 0
    B, H, Hkv, d, w, g = 2, 8, 2, 128, 256, 4
    x = synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, [300, 1000], seed=6, sink_scale=4.0,
                                      device="cuda")
    swa.inject_stall("decode", 1_000_000)
    swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale, num_splits=3)
    assert swa.device_status() == SWA_ERR_DEVICE_TIMEOUT
    assert swa.device_status() == 0
    O, _ = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), w, g, x.scale)
    for splits in (0, 3):
        out = swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale, num_splits=splits)
        torch.cuda.synchronize()
        assert_close(out, O, "bf16", f"decode after recovery, splits={splits}")
    _prefill_ok(swa, oracle_mod, 1, 4, 2, 300, 128, 64, 4, seed=7)
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_injection_is_one_shot_and_can_be_cancelled(swa, oracle_mod):
    swa.inject_stall("prefill", 1_000_000)
    swa.lib.swa_debug_inject_stall(0, 0)  # cancelled before any launch
    _prefill_ok(swa, oracle_mod, 1, 2, 1, 200, 64, 32, 2, seed=8)
    assert swa.device_status() == 0
    with pytest.raises(swa.SwaError):
        swa.inject_stall("prefill", 10)  # below the accepted range


@pytest.mark.gpu
def test_workspace_allocation_failure_is_reported(swa, oracle_mod):
    # a decode whose library workspace would be several TB: cudaMalloc fails
    B, H, Hkv, d, w, g = 1 << 24, 512, 64, 128, 1, 0
    assert swa.decode_workspace_bytes(B, H, Hkv, d, w, g) > (1 << 40)
    dummy = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = swa.lib.swa_decode(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), pos.data_ptr(),
                            B, H, Hkv, d, w, g, 0.1, dummy.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    assert rc == SWA_ERR_ALLOC
    # nothing was enqueued and the next calls (launch error checks included) work
    x = synthetic.decode_cache_inputs(2, 4, 2, 128, 64, 4, [70, 5], seed=9, sink_scale=4.0,
                                      device="cuda")
    out = swa.decode(x.q, x.Kc, x.Vc, x.pos, 64, 4, x.scale)
    torch.cuda.synchronize()
    O, _ = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), 64, 4, x.scale)
    assert_close(out, O, "bf16", "decode after a failed allocation")
    _prefill_ok(swa, oracle_mod, 1, 4, 2, 300, 128, 64, 4, seed=10)
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_swa_decode_on_two_streams_at_once(swa, oracle_mod):
    """Two swa_decode calls (the library-workspace entry point) with different
    inputs on two streams, not serialised: each stream has its own workspace."""
    B, H, Hkv, d, w, g = 32, 32, 8, 128, 4096, 4
    xs = [synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, 100000 + k, seed=20 + k,
                                        sink_scale=4.0, device="cuda") for k in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(x.q) for x in xs]
    torch.cuda.synchronize()
    for rep in range(3):
        for x, s, o in zip(xs, streams, outs):
            swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale, out=o, stream=s)
        torch.cuda.synchronize()
        for x, o in zip(xs, outs):
            O, _ = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), w, g, x.scale)
            assert_close(o, O, "bf16", f"two streams, repetition {rep}")
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_swa_decode_from_two_threads_growing_workspaces(swa, oracle_mod):
    """Two host threads, each on its own stream, call swa_decode with growing
    batch sizes, so each stream's library workspace is outgrown and replaced
    while the other thread's kernels run."""
    w, g, H, Hkv, d = 512, 4, 16, 4, 128
    sizes = [1, 3, 9, 27, 64]
    inputs = {(t, B): synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, 700 + 13 * t, seed=40 + t + B,
                                                    sink_scale=4.0, device="cuda")
              for t in range(2) for B in sizes}
    results, errors = {}, []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for rep in range(2):
                    for B in sizes:
                        x = inputs[(t, B)]
                        results[(t, B, rep)] = swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale,
                                                          stream=s)
            s.synchronize()
        except Exception as e:  # noqa: BLE001 - surfaced below
            errors.append(e)

    torch.cuda.synchronize()
    th = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for (t, B, rep), out in results.items():
        x = inputs[(t, B)]
        O, _ = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, x.pos.cpu().numpy(), w, g, x.scale)
        assert_close(out, O, "bf16", f"thread {t} B={B} rep={rep}")
    assert swa.device_status() == 0


@pytest.mark.gpu
def test_append_past_int32_max_is_refused(swa):
    B, Hkv, d, w, g, T = 2, 2, 128, 64, 4, 4
    gen = torch.Generator(device="cuda").manual_seed(11)
    Kc = torch.randn(B, Hkv, w + g, d, generator=gen, device="cuda").to(torch.bfloat16)
    Vc = torch.randn(B, Hkv, w + g, d, generator=gen, device="cuda").to(torch.bfloat16)
    kn = torch.randn(B, Hkv, T, d, generator=gen, device="cuda").to(torch.bfloat16)
    vn = torch.randn(B, Hkv, T, d, generator=gen, device="cuda").to(torch.bfloat16)
    K0, V0 = Kc.clone(), Vc.clone()
    # sequence 0 would pass INT32_MAX; sequence 1 starts at the last accepted
    # start, INT32_MAX - T (its positions end at INT32_MAX - 1)
    pos0 = torch.tensor([INT32_MAX - 1, INT32_MAX - T], dtype=torch.int32, device="cuda")
    swa.cache_append(Kc, Vc, kn, vn, pos0, w, g)
    assert swa.device_status() == SWA_ERR_INVALID_ARG
    assert torch.equal(Kc[0], K0[0]) and torch.equal(Vc[0], V0[0])
    for t in range(T):  # the valid sequence is written where the slot rule puts it
        slot = (INT32_MAX - T + t) % w
        assert torch.equal(Kc[1, :, slot], kn[1, :, t]) and torch.equal(Vc[1, :, slot], vn[1, :, t])
    assert swa.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_at_the_end_of_the_int32_range(swa, oracle_mod, dtype):
    B, H, Hkv, d, w, g = 3, 8, 2, 128, 300, 4
    pos = [INT32_MAX - 1, INT32_MAX, 5]
    x = synthetic.decode_cache_inputs(B, H, Hkv, d, w, g, pos, dtype=dtype, seed=12,
                                      sink_scale=4.0, device="cuda")
    O, _ = oracle_mod.decode_cache(x.q, x.Kc, x.Vc, np.array(pos, dtype=np.int64), w, g, x.scale)
    for splits in (0, 2):
        out = swa.decode(x.q, x.Kc, x.Vc, x.pos, w, g, x.scale, num_splits=splits)
        torch.cuda.synchronize()
        assert_close(out, O, dtype, f"decode near INT32_MAX, splits={splits}")
    assert swa.device_status() == 0


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs two GPUs")
def test_second_device_after_the_first(swa, oracle_mod):
    """Each kernel's shared-memory limit is a per-device setting: after launches
    on device 0, the same kernels must launch on device 1 too."""
    for dev in (0, 1):
        with torch.cuda.device(dev):
            x = synthetic.prefill_inputs(1, 4, 2, 300, 128, 64, 4, dtype="bf16", seed=dev,
                                         device=f"cuda:{dev}")
            out = swa.prefill(x.Q, x.K, x.V, 64, 4, x.scale)
            torch.cuda.synchronize(dev)
            O, _ = oracle_mod.prefill(x.Q, x.K, x.V, 64, 4, x.scale)
            assert_close(out, O, "bf16", f"prefill on device {dev}")
            c = synthetic.decode_cache_inputs(2, 8, 2, 128, 64, 4, [70, 9], seed=dev,
                                              device=f"cuda:{dev}")
            o2 = swa.decode(c.q, c.Kc, c.Vc, c.pos, 64, 4, c.scale)
            torch.cuda.synchronize(dev)
            O2, _ = oracle_mod.decode_cache(c.q, c.Kc, c.Vc, c.pos.cpu().numpy(), 64, 4, c.scale)
            assert_close(o2, O2, "bf16", f"decode on device {dev}")
            assert swa.device_status() == 0


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs two GPUs")
def test_binding_runs_on_the_tensors_device(swa, oracle_mod):
    """The library launches on the current device; the binding makes the device
    of a call's tensors current for the call, and refuses tensors or a stream
    on another device before anything is launched."""
    with torch.cuda.device(0):
        x = synthetic.prefill_inputs(1, 4, 2, 300, 128, 64, 4, dtype="bf16", seed=5,
                                     device="cuda:1")
        out = swa.prefill(x.Q, x.K, x.V, 64, 4, x.scale)
        assert out.device == torch.device("cuda:1")
        torch.cuda.synchronize(1)
        O, _ = oracle_mod.prefill(x.Q, x.K, x.V, 64, 4, x.scale)
        assert_close(out, O, "bf16", "prefill with its tensors on device 1")
        with pytest.raises(ValueError):
            swa.prefill(x.Q, x.K.to("cuda:0"), x.V, 64, 4, x.scale)
        with pytest.raises(ValueError):
            swa.prefill(x.Q, x.K, x.V, 64, 4, x.scale, stream=torch.cuda.Stream(device=0))
    with torch.cuda.device(1):
        assert swa.device_status() == 0
