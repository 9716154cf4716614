"""Causal sliding-window attention with attention sinks on B300 (sm_103a).

A thin ctypes binding over ``libswa.so`` (C ABI in ``include/swa.h``).  The
functions here only marshal arguments -- shapes, dtypes, pointers, the stream
-- and call the library; every step of the computation runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch is used for device memory
and streams only), all on one device, which each call makes current while it
runs.  The library is loaded on first use; if it is missing that first call
raises ImportError: there is no fallback.

    prefill(q, k, v, w, g=0, scale=None, out=None, lse=None)        -> out
    prefill_pattern(q, k, v, pattern, w, g=0, r=1, ...)             -> out
    prefill_chunk(q, k_new, v_new, k_cache, v_cache, pos0, w, g=0,
                  append=False, ...)                                -> out
    decode(q, k_cache, v_cache, pos, w, g=0, scale=None, ...)        -> out
    cache_append(k_cache, v_cache, k_new, v_new, pos0, w, g=0)

The library is ``libswa.so`` next to this file, built in place by
``build.py``; the environment variable SWA_LIBRARY names another copy.
"""
from __future__ import annotations

import contextlib
import ctypes
import functools
import math
import os

import torch

__all__ = [
    "SwaError", "prefill", "prefill_pattern", "prefill_chunk", "prefill_chunk_workspace_bytes",
    "PATTERNS", "decode", "cache_append", "decode_workspace_bytes",
    "count_pairs", "enumerate_tiles", "enumerate_landmark_tiles", "chunk_key_positions",
    "cache_slot", "device_status", "inject_stall", "prefill_walk",
    "selftest_umma",
    "library_path", "lib",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.environ.get("SWA_LIBRARY", os.path.join(_PKG, "libswa.so"))
_LIB_DEBUG_PATH = os.path.join(_PKG, "libswa_debug.so")

STATUS = {0: "SWA_OK", -1: "SWA_ERR_INVALID_ARG", -2: "SWA_ERR_UNSUPPORTED", -3: "SWA_ERR_CUDA",
          -4: "SWA_ERR_DEVICE_TIMEOUT", -5: "SWA_ERR_ALLOC", -6: "SWA_ERR_WORKSPACE",
          -7: "SWA_ERR_DEVICE_BOUNDS"}
SWA_BF16, SWA_F32 = 0, 1
# fixed patterns of swa_prefill_pattern
PATTERNS = {"window": 0, "dilated": 1, "strided": 2, "landmark": 3}
_DT = {torch.bfloat16: SWA_BF16, torch.float32: SWA_F32}

# Every function the C header declares, with its ctypes signature.
_i, _i64, _f, _p, _sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
SIGNATURES = {
    "swa_prefill": (_i, [_p, _p, _p, _p] + [_i] * 7 + [_f, _p]),
    "swa_prefill_ex": (_i, [_p, _p, _p, _p, _p] + [_i] * 7 + [_f, _i, _p]),
    "swa_prefill_sink_logit": (_i, [_p, _p, _p, _p, _p, _p] + [_i] * 7 + [_f, _i, _p]),
    "swa_prefill_pattern": (_i, [_p] * 6 + [_i] * 5 + [_i] * 4 + [_f, _i, _p]),
    "swa_prefill_chunk_workspace_bytes": (_sz, [_i] * 7),
    "swa_prefill_chunk": (_i, [_p] * 9 + [_i] * 7 + [_f, _i, _i, _p, _sz, _p]),
    "swa_decode": (_i, [_p, _p, _p, _p] + [_i] * 6 + [_f, _p, _p]),
    "swa_decode_workspace_bytes": (_sz, [_i] * 7),
    "swa_decode_ex": (_i, [_p, _p, _p, _p] + [_i] * 6 + [_f, _p, _p, _i, _i, _p, _sz, _p]),
    "swa_decode_sink_logit": (_i, [_p, _p, _p, _p, _p] + [_i] * 6 + [_f, _p, _p, _i, _i, _p, _sz,
                                                                    _p]),
    "swa_decode_noalloc": (_i, [_p, _p, _p, _p] + [_i] * 6 + [_f, _p, _p]),
    "swa_cache_append": (_i, [_p, _p, _p, _p, _p] + [_i] * 6 + [_i, _p]),
    "swa_count_pairs": (_i64, [_i64, _i64, _i64]),
    "swa_enumerate_tiles": (_i, [_i64, _i64, _i64, _i, _i, _p, _sz]),
    "swa_enumerate_landmark_tiles": (_i, [_i64, _i64, _i64, _i64, _i, _i, _p, _sz]),
    "swa_chunk_key_positions": (_i, [_i64, _i, _i, _i, _p, _sz, _p]),
    "swa_cache_slot": (_i, [_i64, _i, _i, _p, _p]),
    "swa_get_device_status": (_i, [_p]),
    "swa_debug_inject_stall": (_i, [_i, _i64]),
    "swa_debug_prefill_walk": (_i, [_p] * 4 + [_i] * 5 + [_i] * 4 + [_f, _p, _i64, _p]),
    "swa_debug_prefill_cta_pairs": (_i, [_p, _p, _p, _p, _p] + [_i] * 7 + [_f, _p]),
    "swa_debug_shrink_bounds": (_i, []),
    "swa_status_string": (ctypes.c_char_p, [_i]),
    "swa_version": (_i, []),
    "swa_selftest_umma": (_i, [_p, _p, _p, _p, _p, _p]),
}


class SwaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({STATUS.get(status, 'unknown')})")
        self.status = status


_LIB = None


def _bind(path):
    if not os.path.exists(path):
        raise ImportError(
            f"{os.path.basename(path)} not found at {path}; build it with "
            "`python -m sink_sparse_attention_swa_b300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _load():
    global _LIB
    if _LIB is None:
        _LIB = _bind(_LIB_PATH)
    return _LIB


@contextlib.contextmanager
def debug_build():
    """Within the block every entry point of this module calls libswa_debug.so
    (the same kernels with their bounds checks compiled in; see include/swa.h)
    instead of libswa.so.  Each library keeps its own device status word."""
    global _LIB
    prev = _load()
    _LIB = _bind(_LIB_DEBUG_PATH)
    try:
        yield
    finally:
        _LIB = prev


def shrink_bounds() -> None:
    """swa_debug_shrink_bounds: in a debug build, the next bf16 prefill checks
    its output rows against a limit one row short (raises SwaError with
    SWA_ERR_UNSUPPORTED in a product build)."""
    _check("swa_debug_shrink_bounds", _load().swa_debug_shrink_bounds())


def __getattr__(name):
    if name == "lib":
        return _load()
    raise AttributeError(name)


def library_path() -> str:
    return _LIB_PATH


def _check(name: str, rc: int) -> None:
    if rc != 0:
        raise SwaError(name, rc)


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif isinstance(stream, torch.cuda.Stream) and device is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _on_device(fn):
    """Runs an entry point with the device of its first tensor argument as the
    current CUDA device: the library launches on the current device, and every
    tensor of the call must live there (checked by _need)."""
    @functools.wraps(fn)
    def call(*args, **kwargs):
        t = args[0] if args else None
        if isinstance(t, torch.Tensor) and t.is_cuda:
            with torch.cuda.device(t.device):
                return fn(*args, **kwargs)
        return fn(*args, **kwargs)
    return call


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not on cuda:{torch.cuda.current_device()} "
                         "with the call's other tensors")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


@_on_device
def prefill(q, k, v, w: int, g: int = 0, scale: float | None = None, out=None, lse=None,
            stream=None, sink_logit=None):
    """q [B,H,n,d], k/v [B,Hkv,n,d] (bf16 or fp32, CUDA) -> out [B,H,n,d].
    lse: optional fp32 [B,H,n] output (natural-log log-sum-exp per row).
    sink_logit: optional fp32 [H] CUDA tensor of learned per-head sink logits
    (swa_prefill_sink_logit)."""
    _need(q, "q")
    B, H, n, d = q.shape
    Hkv = k.shape[1]
    _need(k, "k", q.dtype, (B, Hkv, n, d))
    _need(v, "v", q.dtype, (B, Hkv, n, d))
    if q.dtype not in _DT:
        raise TypeError("q must be bfloat16 or float32")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, n))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, (H,))
        rc = _load().swa_prefill_sink_logit(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                            _ptr(sink_logit), B, H, Hkv, n, d, int(w), int(g),
                                            scale, _DT[q.dtype], _stream(stream, q.device))
        _check("swa_prefill_sink_logit", rc)
        return out
    rc = _load().swa_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, n, d,
                            int(w), int(g), scale, _DT[q.dtype], _stream(stream, q.device))
    _check("swa_prefill_ex", rc)
    return out


@_on_device
def prefill_pattern(q, k, v, pattern: str, w: int = 1, g: int = 0, r: int = 1,
                    scale: float | None = None, out=None, lse=None, sink_logit=None, stream=None):
    """Prefill under a fixed pattern (swa_prefill_pattern): "window" (w, g),
    "dilated" (keys i, i-r, ..., i-(w-1)r), "strided" (every j with (i-j) mod r
    == 0) or "landmark" (the window and sinks plus every j with j mod r == 0).
    Shapes and dtypes as prefill()."""
    _need(q, "q")
    B, H, n, d = q.shape
    Hkv = k.shape[1]
    _need(k, "k", q.dtype, (B, Hkv, n, d))
    _need(v, "v", q.dtype, (B, Hkv, n, d))
    if q.dtype not in _DT:
        raise TypeError("q must be bfloat16 or float32")
    if pattern not in PATTERNS:
        raise ValueError(f"pattern must be one of {sorted(PATTERNS)}")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, n))
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, (H,))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = _load().swa_prefill_pattern(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                     _ptr(sink_logit), B, H, Hkv, n, d, PATTERNS[pattern], int(w),
                                     int(g), int(r), scale, _DT[q.dtype], _stream(stream, q.device))
    _check("swa_prefill_pattern", rc)
    return out


@_on_device
def prefill_chunk(q, k_new, v_new, k_cache, v_cache, pos0, w: int, g: int = 0,
                  scale: float | None = None, out=None, lse=None, sink_logit=None,
                  append: bool = False, workspace=None, stream=None):
    """Chunked prefill (swa_prefill_chunk): q [B,H,T,d] at positions
    pos0[b] .. pos0[b]+T-1 (pos0 int32 [B], CUDA) against the rolling caches
    [B,Hkv,w+g,d] and the chunk's own k_new/v_new [B,Hkv,T,d] -> out [B,H,T,d].
    append=False only reads the caches; append=True also writes the chunk into
    them (as cache_append does) in the same call."""
    _need(q, "q")
    B, H, T, d = q.shape
    Hkv = k_new.shape[1]
    _need(k_new, "k_new", q.dtype, (B, Hkv, T, d))
    _need(v_new, "v_new", q.dtype, (B, Hkv, T, d))
    _need(k_cache, "k_cache", q.dtype, (B, Hkv, w + g, d))
    _need(v_cache, "v_cache", q.dtype, (B, Hkv, w + g, d))
    _need(pos0, "pos0", torch.int32, (B,))
    if q.dtype not in _DT:
        raise TypeError("q must be bfloat16 or float32")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, T))
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, (H,))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = int(_load().swa_prefill_chunk_workspace_bytes(B, Hkv, T, d, int(w), int(g),
                                                           _DT[q.dtype]))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = _load().swa_prefill_chunk(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(pos0), _ptr(out), _ptr(lse),
                                   _ptr(sink_logit), B, H, Hkv, T, d, int(w), int(g), scale,
                                   int(bool(append)), _DT[q.dtype], _ptr(workspace), ws_bytes,
                                   _stream(stream, q.device))
    _check("swa_prefill_chunk", rc)
    return out


def prefill_chunk_workspace_bytes(B, Hkv, T, d, w, g, dtype=torch.bfloat16) -> int:
    return int(_load().swa_prefill_chunk_workspace_bytes(B, Hkv, T, d, int(w), int(g),
                                                         _DT[dtype]))


def decode_workspace_bytes(B, H, Hkv, d, w, g, num_splits=0) -> int:
    return int(_load().swa_decode_workspace_bytes(B, H, Hkv, d, w, g, num_splits))


@_on_device
def decode(q, k_cache, v_cache, pos, w: int, g: int = 0, scale: float | None = None, out=None,
           lse=None, num_splits: int = 0, workspace=None, stream=None, sink_logit=None):
    """q [B,H,d]; k_cache/v_cache [B,Hkv,w+g,d]; pos int32 [B] (CUDA) -> out [B,H,d].
    With workspace=None and lse=None and bf16 inputs this is swa_decode (library
    workspace); otherwise swa_decode_ex with a workspace allocated here if needed."""
    _need(q, "q")
    B, H, d = q.shape
    Hkv = k_cache.shape[1]
    _need(k_cache, "k_cache", q.dtype, (B, Hkv, w + g, d))
    _need(v_cache, "v_cache", q.dtype, (B, Hkv, w + g, d))
    _need(pos, "pos", torch.int32, (B,))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.shape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = _stream(stream, q.device)
    if (workspace is None and lse is None and num_splits == 0 and q.dtype == torch.bfloat16
            and sink_logit is None):
        rc = _load().swa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(pos), B, H, Hkv, d,
                            int(w), int(g), scale, _ptr(out), st)
        _check("swa_decode", rc)
        return out
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H))
    nbytes = decode_workspace_bytes(B, H, Hkv, d, w, g, num_splits)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if workspace is not None:
        _need(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, (H,))
        rc = _load().swa_decode_sink_logit(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(pos),
                                           _ptr(sink_logit), B, H, Hkv, d, int(w), int(g), scale,
                                           _ptr(out), _ptr(lse), _DT[q.dtype], int(num_splits),
                                           _ptr(workspace), ws_bytes, st)
        _check("swa_decode_sink_logit", rc)
        return out
    rc = _load().swa_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(pos), B, H, Hkv, d,
                           int(w), int(g), scale, _ptr(out), _ptr(lse), _DT[q.dtype],
                           int(num_splits), _ptr(workspace), ws_bytes, st)
    _check("swa_decode_ex", rc)
    return out


@_on_device
def cache_append(k_cache, v_cache, k_new, v_new, pos0, w: int, g: int = 0, stream=None):
    """Write k_new/v_new [B,Hkv,T,d] at positions pos0[b] .. pos0[b]+T-1 into the
    rolling caches [B,Hkv,w+g,d] (ring slot p mod w; sink slot w+p for p < g)."""
    _need(k_cache, "k_cache")
    B, Hkv, S, d = k_cache.shape
    if S != w + g:
        raise ValueError(f"cache has {S} slots, expected w+g = {w + g}")
    _need(v_cache, "v_cache", k_cache.dtype, k_cache.shape)
    T = k_new.shape[2]
    _need(k_new, "k_new", k_cache.dtype, (B, Hkv, T, d))
    _need(v_new, "v_new", k_cache.dtype, (B, Hkv, T, d))
    _need(pos0, "pos0", torch.int32, (B,))
    rc = _load().swa_cache_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(pos0),
                              T, B, Hkv, d, int(w), int(g), _DT[k_cache.dtype],
                              _stream(stream, k_cache.device))
    _check("swa_cache_append", rc)


def count_pairs(n: int, w: int, g: int) -> int:
    return int(_load().swa_count_pairs(n, w, g))


def enumerate_tiles(n: int, w: int, g: int, BM: int, BN: int):
    """Tile classes [ceil(n/BM), ceil(n/BN)] as a torch int32 CPU tensor."""
    nq, nk = -(-n // BM), -(-n // BN)
    out = torch.zeros(nq, nk, dtype=torch.int32)
    _check("swa_enumerate_tiles", _load().swa_enumerate_tiles(n, w, g, BM, BN, out.data_ptr(), out.numel()))
    return out


def enumerate_landmark_tiles(n: int, w: int, g: int, r: int, BM: int, BN: int):
    """Landmark tile classes [ceil(n/BM), ceil(ceil(n/r)/BN)] int32 (0/1/2), host-only."""
    nq, nk = -(-n // BM), -(-(-(-n // r)) // BN)
    out = torch.zeros((nq, nk), dtype=torch.int32)
    rc = _load().swa_enumerate_landmark_tiles(n, w, g, r, BM, BN, out.data_ptr(), out.numel())
    _check("swa_enumerate_landmark_tiles", rc)
    return out


def chunk_key_positions(pos0: int, w: int, g: int, T: int):
    """(positions int64 [rows] with -1 for padding, query offset) of the key list a
    chunked prefill builds; host-only."""
    cap = ((g + w - 1 + 127) // 128 + (T + 127) // 128) * 128
    pos = torch.empty(cap, dtype=torch.int64)
    off = ctypes.c_int32(0)
    rc = _load().swa_chunk_key_positions(int(pos0), int(w), int(g), int(T), pos.data_ptr(), cap,
                                         ctypes.byref(off))
    _check("swa_chunk_key_positions", rc if rc < 0 else 0)
    return pos[:rc], int(off.value)


def cache_slot(p: int, w: int, g: int):
    r, s = ctypes.c_int32(), ctypes.c_int32()
    _check("swa_cache_slot", _load().swa_cache_slot(p, w, g, ctypes.byref(r), ctypes.byref(s)))
    return r.value, s.value


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status code."""
    return int(_load().swa_get_device_status(_stream(stream, None)))


WALK_FIELDS = ("item", "b", "kvh", "unit", "qtile", "cls", "k0", "flags")


@_on_device
def prefill_cta_pairs(q, k, v, w: int, g: int = 0, scale: float | None = None, out=None,
                      lse=None, stream=None):
    """The bf16 window-path prefill on the CTA-pair kernel
    (swa_debug_prefill_cta_pairs): same arguments and result as prefill();
    raises SwaError (SWA_ERR_UNSUPPORTED) unless d == 128, H / Hkv is even and
    H % 4 == 0."""
    _need(q, "q", torch.bfloat16)
    B, H, n, d = q.shape
    Hkv = k.shape[1]
    _need(k, "k", torch.bfloat16, (B, Hkv, n, d))
    _need(v, "v", torch.bfloat16, (B, Hkv, n, d))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, n))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = _load().swa_debug_prefill_cta_pairs(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                             Hkv, n, d, int(w), int(g), scale,
                                             _stream(stream, q.device))
    _check("swa_debug_prefill_cta_pairs", rc)
    return out


@_on_device
def prefill_walk(q, k, v, pattern: str, w: int, g: int = 0, r: int = 1,
                 scale: float | None = None, max_entries: int = 1 << 20, stream=None):
    """Diagnostic (swa_debug_prefill_walk): runs the bf16 prefill and returns
    (out, entries) where entries is an int32 CPU tensor [m, 8] of the key tiles
    the kernels loaded, columns WALK_FIELDS, and m the number loaded."""
    _need(q, "q", torch.bfloat16)
    B, H, n, d = q.shape
    Hkv = k.shape[1]
    _need(k, "k", torch.bfloat16, (B, Hkv, n, d))
    _need(v, "v", torch.bfloat16, (B, Hkv, n, d))
    out = torch.empty_like(q)
    log = torch.zeros(8 + 8 * max_entries, dtype=torch.int32, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = _stream(stream, q.device)
    rc = _load().swa_debug_prefill_walk(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Hkv, n, d,
                                        PATTERNS[pattern], int(w), int(g), int(r), scale,
                                        _ptr(log), max_entries, st)
    _check("swa_debug_prefill_walk", rc)
    torch.cuda.synchronize(q.device)
    m = int(log[0].item())
    if m > max_entries:
        raise RuntimeError(f"the walk has {m} tiles, more than max_entries={max_entries}")
    return out, log[8:8 + 8 * m].view(m, 8).cpu()


STALL_KINDS = {"prefill": 1, "decode": 2}


def inject_stall(kind: str, wait_ns: int = 1_000_000) -> None:
    """Test aid (swa_debug_inject_stall): the next prefill ("prefill") or decode
    split pass ("decode") launched on the current device leaves out its first
    key/value copy and waits at most wait_ns per bounded wait, so its timeout
    path runs; device_status() then returns -4 (SWA_ERR_DEVICE_TIMEOUT)."""
    _check("swa_debug_inject_stall", _load().swa_debug_inject_stall(STALL_KINDS[kind], int(wait_ns)))


@_on_device
def selftest_umma(A, Bk, Bn, stream=None):
    """Diagnostic: (A @ Bk^T, A @ Bn) computed by the tensor-core operand paths
    the prefill kernel uses; A/Bk/Bn [128,128] bf16 CUDA."""
    for t, nm in ((A, "A"), (Bk, "Bk"), (Bn, "Bn")):
        _need(t, nm, torch.bfloat16, (128, 128))
    D1 = torch.empty(128, 128, dtype=torch.float32, device=A.device)
    D2 = torch.empty_like(D1)
    _check("swa_selftest_umma", _load().swa_selftest_umma(_ptr(A), _ptr(Bk), _ptr(Bn), _ptr(D1),
                                                      _ptr(D2), _stream(stream, A.device)))
    return D1, D2
