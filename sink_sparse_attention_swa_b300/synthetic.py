"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random tensors with a
seeded generator and names the workloads by their shapes.  Both the CUDA path
and the CPU oracle consume what it produces (the oracle after an exact widening
of the same bf16/fp32 values to fp64).

Workloads (the shapes come from the model families the pages quote):
  tiny_fp32_prefill       B=1 H=Hkv=1 n=512 d=64 w=64 g=0, fp32
  mistral_like_prefill    B=1 H=32 Hkv=8 n=16384 d=128 w=4096 g=0, bf16
  streaming_decode_sinks  B=32 H=32 Hkv=8 d=128 w=4096 g=4, pos=100000, bf16,
                          the four sink keys scaled x4
  gemma3_local_prefill    B=2 H=32 Hkv=16 n=32768 d=128 w=1024 g=0, bf16
  long_sink_prefill       B=1 H=32 Hkv=8 n=131072 d=128 w=4096 g=4, bf16,
                          sink keys (positions 0..3) scaled x4
  gemma3_global_prefill   B=2 H=32 Hkv=16 n=32768 d=128 w=n (full causal) g=0,
                          bf16: the global layer between the local ones
  mha_prefill             B=1 H=Hkv=32 n=16384 d=128 w=4096 g=0, bf16: plain
                          multi-head attention (a group of one)
  dilated_prefill         B=1 H=32 Hkv=8 n=16384 d=128, dilated window w=1024
                          r=4 (the reach of a 4096 window at a quarter of it)
  strided_prefill         B=1 H=32 Hkv=8 n=65536 d=128, Sparse Transformer
                          strided head r=256 (s = sqrt(n))
  landmark_prefill        B=1 H=32 Hkv=8 n=16384 d=128 w=4096 g=4 (sink keys
                          x4), landmarks every r=64 positions
  chunked_prefill_stream  B=4 H=32 Hkv=8 d=128 w=4096 g=4, a chunk of T=4096
                          prompt tokens at positions 100000 .. 104095 against
                          a full rolling cache (sink keys x4), bf16
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

WORKLOADS = {
    "tiny_fp32_prefill": dict(kind="prefill", B=1, H=1, Hkv=1, n=512, d=64, w=64, g=0,
                              dtype="f32", sink_scale=1.0),
    "mistral_like_prefill": dict(kind="prefill", B=1, H=32, Hkv=8, n=16384, d=128, w=4096,
                                 g=0, dtype="bf16", sink_scale=1.0),
    "streaming_decode_sinks": dict(kind="decode", B=32, H=32, Hkv=8, d=128, w=4096, g=4,
                                   pos=100000, dtype="bf16", sink_scale=4.0),
    "gemma3_local_prefill": dict(kind="prefill", B=2, H=32, Hkv=16, n=32768, d=128, w=1024,
                                 g=0, dtype="bf16", sink_scale=1.0),
    "long_sink_prefill": dict(kind="prefill", B=1, H=32, Hkv=8, n=131072, d=128, w=4096,
                              g=4, dtype="bf16", sink_scale=4.0),
    "gemma3_global_prefill": dict(kind="prefill", B=2, H=32, Hkv=16, n=32768, d=128, w=32768,
                                  g=0, dtype="bf16", sink_scale=1.0),
    "mha_prefill": dict(kind="prefill", B=1, H=32, Hkv=32, n=16384, d=128, w=4096, g=0,
                        dtype="bf16", sink_scale=1.0),
    "dilated_prefill": dict(kind="prefill", B=1, H=32, Hkv=8, n=16384, d=128, w=1024, g=0,
                            dtype="bf16", sink_scale=1.0, pattern="dilated", r=4),
    "strided_prefill": dict(kind="prefill", B=1, H=32, Hkv=8, n=65536, d=128, w=0, g=0,
                            dtype="bf16", sink_scale=1.0, pattern="strided", r=256),
    "landmark_prefill": dict(kind="prefill", B=1, H=32, Hkv=8, n=16384, d=128, w=4096, g=4,
                             dtype="bf16", sink_scale=4.0, pattern="landmark", r=64),
    "chunked_prefill_stream": dict(kind="chunk", B=4, H=32, Hkv=8, d=128, w=4096, g=4, T=4096,
                                   pos0=100000, dtype="bf16", sink_scale=4.0),
}

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclass
class PrefillInputs:
    Q: torch.Tensor
    K: torch.Tensor
    V: torch.Tensor
    w: int
    g: int
    scale: float
    meta: dict = field(default_factory=dict)


def prefill_inputs(B, H, Hkv, n, d, w, g, dtype="bf16", seed=0, sink_scale=1.0,
                   device="cpu", scale=None) -> PrefillInputs:
    """Q [B,H,n,d], K/V [B,Hkv,n,d], i.i.d. N(0,1) drawn in the order Q, K, V from
    one generator seeded with `seed` on `device`; key rows 0..g-1 multiplied by
    `sink_scale`; then cast to `dtype`."""
    gen = _gen(seed, device)
    Q = torch.randn(B, H, n, d, generator=gen, device=device, dtype=torch.float32)
    K = torch.randn(B, Hkv, n, d, generator=gen, device=device, dtype=torch.float32)
    V = torch.randn(B, Hkv, n, d, generator=gen, device=device, dtype=torch.float32)
    if g > 0 and sink_scale != 1.0:
        K[:, :, : min(g, n)] *= sink_scale
    dt = torch_dtype(dtype)
    return PrefillInputs(Q.to(dt), K.to(dt), V.to(dt), w, g,
                         default_scale(d) if scale is None else scale,
                         dict(B=B, H=H, Hkv=Hkv, n=n, d=d, dtype=dtype, seed=seed))


@dataclass
class DecodeInputs:
    q: torch.Tensor
    Kc: torch.Tensor
    Vc: torch.Tensor
    pos: torch.Tensor
    w: int
    g: int
    scale: float
    meta: dict = field(default_factory=dict)


def decode_cache_inputs(B, H, Hkv, d, w, g, pos, dtype="bf16", seed=0, sink_scale=1.0,
                        device="cpu", scale=None) -> DecodeInputs:
    """A filled rolling cache Kc/Vc [B,Hkv,w+g,d] (ring slots 0..w-1, then g sink
    slots), i.i.d. N(0,1) with the sink-slot keys multiplied by `sink_scale`;
    one query q [B,H,d]; pos [B] int32 (an int or a per-sequence list).
    Draw order from one generator: Kc, Vc, q."""
    gen = _gen(seed, device)
    S = w + g
    Kc = torch.randn(B, Hkv, S, d, generator=gen, device=device, dtype=torch.float32)
    Vc = torch.randn(B, Hkv, S, d, generator=gen, device=device, dtype=torch.float32)
    q = torch.randn(B, H, d, generator=gen, device=device, dtype=torch.float32)
    if g > 0 and sink_scale != 1.0:
        Kc[:, :, w:] *= sink_scale
    if isinstance(pos, int):
        pos_t = torch.full((B,), pos, dtype=torch.int32, device=device)
    else:
        pos_t = torch.as_tensor(pos, dtype=torch.int32, device=device)
    dt = torch_dtype(dtype)
    return DecodeInputs(q.to(dt), Kc.to(dt), Vc.to(dt), pos_t, w, g,
                        default_scale(d) if scale is None else scale,
                        dict(B=B, H=H, Hkv=Hkv, d=d, dtype=dtype, seed=seed))


def token_stream(B, Hkv, d, T, dtype="bf16", seed=0, device="cpu", sink_scale=1.0, g=0):
    """K/V for T consecutive positions [B,Hkv,T,d] (positions 0..T-1), keys of
    positions < g multiplied by `sink_scale`."""
    gen = _gen(seed, device)
    K = torch.randn(B, Hkv, T, d, generator=gen, device=device, dtype=torch.float32)
    V = torch.randn(B, Hkv, T, d, generator=gen, device=device, dtype=torch.float32)
    if g > 0 and sink_scale != 1.0:
        K[:, :, : min(g, T)] *= sink_scale
    dt = torch_dtype(dtype)
    return K.to(dt), V.to(dt)


def sample_rows(B, H, n, count, seed=1):
    """`count` distinct (b, h, i) rows drawn without replacement with a CPU
    generator seeded with `seed`; int64 tensor [count, 3]."""
    gen = _gen(seed, "cpu")
    total = B * H * n
    idx = torch.randperm(total, generator=gen)[:count]
    i = idx % n
    h = (idx // n) % H
    b = idx // (n * H)
    return torch.stack([b, h, i], dim=1).to(torch.int64)


@dataclass
class ChunkInputs:
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    Kc: torch.Tensor
    Vc: torch.Tensor
    pos0: torch.Tensor
    w: int
    g: int
    scale: float


def chunk_inputs(B, H, Hkv, d, w, g, T, pos0, dtype="bf16", seed=0, sink_scale=1.0,
                 device="cpu", scale=None) -> ChunkInputs:
    """A chunk of T tokens at positions pos0 .. pos0+T-1 (the same pos0 for every
    sequence) against a filled rolling cache: the cache and the chunk's queries
    come from decode_cache_inputs-style draws (Kc, Vc, then q [B,H,T,d]), the
    chunk's keys and values from a second generator seeded seed+1 (k_new,
    v_new [B,Hkv,T,d])."""
    gen = _gen(seed, device)
    S = w + g
    Kc = torch.randn(B, Hkv, S, d, generator=gen, device=device, dtype=torch.float32)
    Vc = torch.randn(B, Hkv, S, d, generator=gen, device=device, dtype=torch.float32)
    q = torch.randn(B, H, T, d, generator=gen, device=device, dtype=torch.float32)
    if g > 0 and sink_scale != 1.0:
        Kc[:, :, w:] *= sink_scale
    kn, vn = token_stream(B, Hkv, d, T, dtype=dtype, seed=seed + 1, device=device)
    dt = torch_dtype(dtype)
    pos_t = torch.full((B,), pos0, dtype=torch.int32, device=device)
    return ChunkInputs(q.to(dt), kn, vn, Kc.to(dt), Vc.to(dt), pos_t, w, g,
                       default_scale(d) if scale is None else scale)
