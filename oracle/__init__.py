"""The CPU oracle for causal sliding-window attention with attention sinks.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product library never imports this
package, and this package imports nothing from the product library.

The arithmetic lives in ``swa_oracle.c`` (plain C, fp64, OpenMP), compiled on
first use with gcc into ``oracle/_build/``.  This module only marshals numpy
arrays into it.  See the C file for the definitions and the page passages each
routine follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libswa_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP).  Returns its path."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
        ):
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(
                ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                 "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
            )
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_mask_row.argtypes = [_i64, _i64, _i64, _i64, _ptr]
        lib.oracle_mask.argtypes = [_i64, _i64, _i64, _ptr]
        lib.oracle_count_pairs.argtypes = [_i64, _i64, _i64]
        lib.oracle_count_pairs.restype = _i64
        lib.oracle_tiles.argtypes = [_i64, _i64, _i64, _i64, _i64, _ptr]
        lib.oracle_prefill.argtypes = [_ptr] * 5 + [_i64] * 7 + [_dbl, ctypes.c_int, _ptr]
        lib.oracle_prefill_rows.argtypes = [_ptr] * 3 + [_i64] * 7 + [_dbl, _ptr, _i64, _ptr, _ptr,
                                                                    _ptr]
        lib.oracle_decode_history.argtypes = [_ptr] * 4 + [_i64] * 7 + [_dbl, _ptr, _ptr, _ptr]
        lib.oracle_cache_slots.argtypes = [_i64, _i64, _i64, _ptr, _ptr]
        lib.oracle_decode_cache.argtypes = [_ptr] * 4 + [_i64] * 6 + [_dbl, _ptr, _ptr, _ptr]
        lib.oracle_pattern_mask_row.argtypes = [_i64] * 5 + [ctypes.c_int, _ptr]
        lib.oracle_pattern_mask.argtypes = [_i64] * 4 + [ctypes.c_int, _ptr]
        lib.oracle_pattern_count_pairs.argtypes = [_i64] * 4 + [ctypes.c_int]
        lib.oracle_pattern_count_pairs.restype = _i64
        lib.oracle_prefill_pattern.argtypes = ([_ptr] * 5 + [_i64] * 8 +
                                               [ctypes.c_int, _dbl, _ptr])
        lib.oracle_prefill_pattern_rows.argtypes = ([_ptr] * 3 + [_i64] * 8 +
                                                    [ctypes.c_int, _dbl, _ptr, _i64, _ptr, _ptr,
                                                     _ptr])
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    """Widen to a C-contiguous float64 numpy array (exact for bf16/fp32 input)."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _sinks(sink_logit, H):
    """Per-head sink logits as float64 [H] (None: no sink logit)."""
    if sink_logit is None:
        return None
    a = _f64(sink_logit).reshape(-1)
    assert a.shape == (H,), (a.shape, H)
    return a


def _pn(a):
    return None if a is None else _p(a)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(t: int) -> None:
    _load().oracle_set_num_threads(int(t))


def mask_row(i: int, n: int, w: int, g: int) -> np.ndarray:
    row = np.zeros(n, dtype=np.uint8)
    _load().oracle_mask_row(i, n, w, g, _p(row))
    return row


def mask(n: int, w: int, g: int) -> np.ndarray:
    """Explicit n x n mask, uint8 (1 = attend)."""
    m = np.zeros((n, n), dtype=np.uint8)
    _load().oracle_mask(n, w, g, _p(m))
    return m


def count_pairs(n: int, w: int, g: int) -> int:
    return int(_load().oracle_count_pairs(n, w, g))


# Fixed patterns (see oracle_pattern_mask_row in the C source).
PATTERNS = {"window": 0, "dilated": 1, "strided": 2, "landmark": 3}


def _pat(pattern) -> int:
    return PATTERNS[pattern] if isinstance(pattern, str) else int(pattern)


def pattern_mask_row(i: int, n: int, w: int, g: int, r: int, pattern) -> np.ndarray:
    row = np.zeros(n, dtype=np.uint8)
    _load().oracle_pattern_mask_row(i, n, w, g, r, _pat(pattern), _p(row))
    return row


def pattern_mask(n: int, w: int, g: int, r: int, pattern) -> np.ndarray:
    m = np.zeros((n, n), dtype=np.uint8)
    _load().oracle_pattern_mask(n, w, g, r, _pat(pattern), _p(m))
    return m


def pattern_count_pairs(n: int, w: int, g: int, r: int, pattern) -> int:
    return int(_load().oracle_pattern_count_pairs(n, w, g, r, _pat(pattern)))


def prefill_pattern(Q, K, V, w: int, g: int, r: int, pattern, scale: float, sink_logit=None):
    """prefill() under a fixed pattern (window, dilated, strided, landmark)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, n, d = Q.shape
    Hkv = K.shape[1]
    assert K.shape == (B, Hkv, n, d) and V.shape == K.shape and H % Hkv == 0
    O = np.empty_like(Q)
    L = np.empty((B, H, n), dtype=np.float64)
    sl = _sinks(sink_logit, H)
    _load().oracle_prefill_pattern(_p(Q), _p(K), _p(V), _p(O), _p(L), B, H, Hkv, n, d, w, g, r,
                                   _pat(pattern), float(scale), _pn(sl))
    return O, L


def prefill_pattern_rows(q_rows, K, V, H: int, w: int, g: int, r: int, pattern, scale: float,
                         rows, sink_logit=None):
    """prefill_rows() under a fixed pattern."""
    q_rows, K, V = _f64(q_rows), _f64(K), _f64(V)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    B, Hkv, n, d = K.shape
    m = rows.shape[0]
    assert rows.shape == (m, 3) and q_rows.shape == (m, d)
    O = np.empty((m, d), dtype=np.float64)
    L = np.empty(m, dtype=np.float64)
    sl = _sinks(sink_logit, H)
    _load().oracle_prefill_pattern_rows(_p(q_rows), _p(K), _p(V), B, H, Hkv, n, d, w, g, r,
                                        _pat(pattern), float(scale), _p(rows), m, _p(O), _p(L),
                                        _pn(sl))
    return O, L


def tiles(n: int, w: int, g: int, BM: int, BN: int) -> np.ndarray:
    """Tile classes [ceil(n/BM), ceil(n/BN)] int32: 0 empty, 1 partial, 2 full."""
    nq, nk = -(-n // BM), -(-n // BN)
    out = np.zeros((nq, nk), dtype=np.int32)
    _load().oracle_tiles(n, w, g, BM, BN, _p(out))
    return out


def prefill(Q, K, V, w: int, g: int, scale: float, zero_score: bool = False, sink_logit=None):
    """Q [B,H,n,d], K/V [B,Hkv,n,d] -> (O [B,H,n,d], LSE [B,H,n]) in float64.
    sink_logit: optional per-head sink logits [H] (see the C source)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, n, d = Q.shape
    Hkv = K.shape[1]
    assert K.shape == (B, Hkv, n, d) and V.shape == K.shape and H % Hkv == 0
    O = np.empty_like(Q)
    L = np.empty((B, H, n), dtype=np.float64)
    sl = _sinks(sink_logit, H)
    _load().oracle_prefill(_p(Q), _p(K), _p(V), _p(O), _p(L), B, H, Hkv, n, d, w, g,
                           float(scale), int(bool(zero_score)), _pn(sl))
    return O, L


def prefill_rows(q_rows, K, V, H: int, w: int, g: int, scale: float, rows, sink_logit=None):
    """Sampled prefill rows.  rows: int array [m,3] of (b, h, i); q_rows [m,d] the
    matching query rows; K/V [B,Hkv,n,d].  Returns (O_rows [m,d], LSE_rows [m])."""
    q_rows, K, V = _f64(q_rows), _f64(K), _f64(V)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    B, Hkv, n, d = K.shape
    m = rows.shape[0]
    assert rows.shape == (m, 3) and q_rows.shape == (m, d)
    O = np.empty((m, d), dtype=np.float64)
    L = np.empty(m, dtype=np.float64)
    sl = _sinks(sink_logit, H)
    _load().oracle_prefill_rows(_p(q_rows), _p(K), _p(V), B, H, Hkv, n, d, w, g,
                                float(scale), _p(rows), m, _p(O), _p(L), _pn(sl))
    return O, L


def decode_history(q, Khist, Vhist, pos, w: int, g: int, scale: float, sink_logit=None):
    """q [B,H,d]; Khist/Vhist [B,Hkv,P,d] indexed by position; pos [B]."""
    q, Kh, Vh = _f64(q), _f64(Khist), _f64(Vhist)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    B, H, d = q.shape
    Hkv, P = Kh.shape[1], Kh.shape[2]
    assert Kh.shape == (B, Hkv, P, d) and Vh.shape == Kh.shape and pos.shape == (B,)
    assert int(pos.max()) < P
    O = np.empty_like(q)
    L = np.empty((B, H), dtype=np.float64)
    sl = _sinks(sink_logit, H)
    _load().oracle_decode_history(_p(q), _p(Kh), _p(Vh), _p(pos), P, B, H, Hkv, d, w, g,
                                  float(scale), _p(O), _p(L), _pn(sl))
    return O, L


def cache_slots(p: int, w: int, g: int):
    """(ring slot, sink slot or -1) where the rolling cache keeps position p."""
    r, s = _i64(), _i64()
    _load().oracle_cache_slots(p, w, g, ctypes.byref(r), ctypes.byref(s))
    return int(r.value), int(s.value)


def decode_cache(q, Kc, Vc, pos, w: int, g: int, scale: float, sink_logit=None):
    """q [B,H,d]; Kc/Vc [B,Hkv,w+g,d] rolling cache; pos [B]."""
    q, Kc, Vc = _f64(q), _f64(Kc), _f64(Vc)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    B, H, d = q.shape
    Hkv = Kc.shape[1]
    assert Kc.shape == (B, Hkv, w + g, d) and Vc.shape == Kc.shape and pos.shape == (B,)
    O = np.empty_like(q)
    L = np.empty((B, H), dtype=np.float64)
    sl = _sinks(sink_logit, H)
    _load().oracle_decode_cache(_p(q), _p(Kc), _p(Vc), _p(pos), B, H, Hkv, d, w, g,
                                float(scale), _p(O), _p(L), _pn(sl))
    return O, L
