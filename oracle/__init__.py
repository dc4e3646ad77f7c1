"""The CPU oracle for decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it, and it never imports the CUDA library: the two share no code.

The arithmetic lives in ``dkv_oracle.cpp`` (plain C++17, fp64 accumulation),
written from the pages' definitions:

* "TinyServe: Query-Aware Cache Selection for Efficient LLM Serving" --
  page layout, page metadata (m_j, M_j), the bound score r(q, phi_j), top-K page
  selection and attention over the selected pages (Algorithm 1, steps 1-4).
* "论文阅读：HeadInfer" -- exact per-head attention Softmax(q K^T / sqrt(d)) V.
* "FlexGen: High-Throughput Generative Inference of Large Language Models with a
  Single GPU" (解读) -- 4-bit group-of-64 min/max KV quantisation.

This module only marshals numpy arrays into that library.  16-bit floats travel
as their raw bit patterns (``numpy.uint16``) with an ``is_fp16`` flag
(0 = bfloat16, 1 = IEEE half).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dkv_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libdkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library with g++ if it is missing or stale."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_get_threads.restype = i32
            lib.oracle_value16.argtypes = [ctypes.c_uint16, i32]
            lib.oracle_value16.restype = dbl
            lib.oracle_fp16_round.argtypes = [dbl]
            lib.oracle_fp16_round.restype = ctypes.c_uint16
            lib.oracle_meta.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P]
            lib.oracle_scores.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P]
            lib.oracle_topk.argtypes = [i32, i32, i32, P, P]
            lib.oracle_attention.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                             P, P, P, dbl, P, i32, P]
            lib.oracle_meta8.argtypes = [i64, i32, i32, P, P, P, P, P, P]
            lib.oracle_scores8.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P]
            lib.oracle_quant4.argtypes = [i64, i32, P, P, P, P]
            lib.oracle_dequant4.argtypes = [i64, i32, P, P, P, P]
            lib.oracle_q4_step.argtypes = [ctypes.c_uint16, ctypes.c_uint16,
                                           ctypes.POINTER(ctypes.c_int)]
            lib.oracle_q4_step.restype = dbl
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def set_threads(n: int) -> None:
    """Threads used by every oracle routine (0 = all host cores)."""
    _load().oracle_set_threads(int(n))


def threads() -> int:
    return int(_load().oracle_get_threads())


def value16(bits: np.ndarray, is_fp16: int) -> np.ndarray:
    """Exact value (float64) of each 16-bit float bit pattern."""
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.array([lib.oracle_value16(int(b), int(is_fp16)) for b in flat])
    return out.reshape(np.shape(bits))


def fp16_round(x) -> np.ndarray:
    """Round each float64 to the nearest IEEE half (ties to even); bit patterns."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float64).ravel()
    out = np.array([lib.oracle_fp16_round(float(v)) for v in flat], dtype=np.uint16)
    return out.reshape(np.shape(x))


def meta(K: np.ndarray, S: int, is_fp16: int):
    """Page metadata (m_j, M_j): channel-wise min / max of each page's keys.

    K: uint16 bits [B, Hkv, N, d].  Returns (meta_min, meta_max) uint16 bits
    [B, Hkv, P, d] with P = ceil(N / S).
    """
    K = _c(K, np.uint16)
    B, H, N, d = K.shape
    P = (N + S - 1) // S
    mn = np.empty((B, H, P, d), np.uint16)
    mx = np.empty((B, H, P, d), np.uint16)
    _load().oracle_meta(B, H, N, d, S, int(is_fp16), _ptr(K), _ptr(mn), _ptr(mx))
    return mn, mx


def scores(q: np.ndarray, meta_min: np.ndarray, meta_max: np.ndarray, is_fp16: int):
    """Bound scores r(q, phi_j) in float64, [B, Hq, P]."""
    q = _c(q, np.uint16)
    meta_min = _c(meta_min, np.uint16)
    meta_max = _c(meta_max, np.uint16)
    B, Hq, d = q.shape
    _, Hkv, P, _ = meta_min.shape
    out = np.empty((B, Hq, P), np.float64)
    _load().oracle_scores(B, Hq, Hkv, P, d, int(is_fp16), _ptr(q), _ptr(meta_min),
                          _ptr(meta_max), _ptr(out))
    return out


def group_scores(q: np.ndarray, meta_min: np.ndarray, meta_max: np.ndarray, is_fp16: int):
    """One selection per kv head group (GQA), float64 [B, Hkv, P].

    Page j's group score is the sum over the group's query heads h of the
    bound score r(q_h, phi_j) ("TinyServe", 相关性函数实例化).  The pages define
    r for one query vector and are silent on grouped heads; the sum is the
    reading used for one shared selection, and it stays an upper bound:
    sum_h r(q_h, phi_j) >= max over the page's keys k of sum_h q_h . k.
    """
    r = scores(q, meta_min, meta_max, is_fp16)  # [B, Hq, P]
    B, Hq, P = r.shape
    Hkv = meta_min.shape[1]
    return r.reshape(B, Hkv, Hq // Hkv, P).sum(axis=2)


def meta8(meta_min: np.ndarray, meta_max: np.ndarray, is_fp16: int):
    """8-bit page metadata from (m_j, M_j): (code_min, code_max) uint8
    [B, Hkv, P, d] and (lo, step) float32 [B, Hkv, P], with
    dec(c) = fma(c, step, lo) rounded outward: dec(code_min) <= m and
    dec(code_max) >= M channel by channel (definition in dkv_oracle.cpp)."""
    meta_min = _c(meta_min, np.uint16)
    meta_max = _c(meta_max, np.uint16)
    B, Hkv, P, d = meta_min.shape
    cmin = np.empty((B, Hkv, P, d), np.uint8)
    cmax = np.empty((B, Hkv, P, d), np.uint8)
    lo = np.empty((B, Hkv, P), np.float32)
    step = np.empty((B, Hkv, P), np.float32)
    _load().oracle_meta8(B * Hkv * P, d, int(is_fp16), _ptr(meta_min), _ptr(meta_max),
                         _ptr(cmin), _ptr(cmax), _ptr(lo), _ptr(step))
    return cmin, cmax, lo, step


def scores8(q: np.ndarray, cmin: np.ndarray, cmax: np.ndarray, lo: np.ndarray,
            step: np.ndarray, is_fp16: int):
    """Bound scores over 8-bit metadata in float64, [B, Hq, P]: r with the
    decoded dec(code_max) / dec(code_min) in place of M / m."""
    q = _c(q, np.uint16)
    cmin, cmax = _c(cmin, np.uint8), _c(cmax, np.uint8)
    lo, step = _c(lo, np.float32), _c(step, np.float32)
    B, Hq, d = q.shape
    _, Hkv, P, _ = cmin.shape
    out = np.empty((B, Hq, P), np.float64)
    _load().oracle_scores8(B, Hq, Hkv, P, d, int(is_fp16), _ptr(q), _ptr(cmin), _ptr(cmax),
                           _ptr(lo), _ptr(step), _ptr(out))
    return out


def topk(r: np.ndarray, K: int) -> np.ndarray:
    """Top-K page indices per row of r [..., P], ascending; ties -> lower index."""
    r = _c(r, np.float64)
    P = r.shape[-1]
    BH = int(np.prod(r.shape[:-1]))
    kk = min(int(K), P)
    sel = np.empty(r.shape[:-1] + (kk,), np.int32)
    _load().oracle_topk(BH, P, int(K), _ptr(r), _ptr(sel))
    return sel


def attention(q, K, V, S: int, scale: float, is_fp16: int, sel=None):
    """Decode attention in float64, [B, Hq, d].

    sel is None for exact attention over all N tokens, else int32 [B, Hq, n]
    page indices whose tokens (in the order given) form the attended set.
    """
    q = _c(q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    B, Hq, d = q.shape
    _, Hkv, N, _ = K.shape
    out = np.empty((B, Hq, d), np.float64)
    if sel is None:
        sel_p, nsel = ctypes.c_void_p(0), 0
    else:
        sel = _c(sel, np.int32)
        sel_p, nsel = _ptr(sel), sel.shape[-1]
    _load().oracle_attention(B, Hq, Hkv, N, d, S, int(is_fp16), _ptr(q), _ptr(K),
                             _ptr(V), float(scale), sel_p, nsel, _ptr(out))
    return out


def quant4(x: np.ndarray):
    """4-bit group-of-64 quantisation of fp16 rows [..., d].

    Returns (codes uint8 [..., d/2], gmin uint16 [..., d/64], gmax uint16 [..., d/64]).
    """
    x = _c(x, np.uint16)
    d = x.shape[-1]
    rows = int(np.prod(x.shape[:-1]))
    codes = np.empty(x.shape[:-1] + (d // 2,), np.uint8)
    gmin = np.empty(x.shape[:-1] + (d // 64,), np.uint16)
    gmax = np.empty(x.shape[:-1] + (d // 64,), np.uint16)
    _load().oracle_quant4(rows, d, _ptr(x), _ptr(codes), _ptr(gmin), _ptr(gmax))
    return codes, gmin, gmax


def dequant4(codes: np.ndarray, gmin: np.ndarray, gmax: np.ndarray) -> np.ndarray:
    """Inverse of quant4: fp16 bit patterns [..., d]."""
    codes = _c(codes, np.uint8)
    gmin = _c(gmin, np.uint16)
    gmax = _c(gmax, np.uint16)
    d = codes.shape[-1] * 2
    rows = int(np.prod(codes.shape[:-1]))
    x = np.empty(codes.shape[:-1] + (d,), np.uint16)
    _load().oracle_dequant4(rows, d, _ptr(codes), _ptr(gmin), _ptr(gmax), _ptr(x))
    return x


def q4_step(mn: int, mx: int):
    """The 4-bit format's step for a group with fp16 min / max bits (mn, mx).

    Returns (step as a float, tiny) where tiny is True for groups whose range is
    below 451 * 2^-24 (the step then lies on a finer grid than fp16 offers).
    """
    tiny = ctypes.c_int(0)
    s = _load().oracle_q4_step(int(mn), int(mx), ctypes.byref(tiny))
    return float(s), bool(tiny.value)
