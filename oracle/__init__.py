"""CPU oracle for the hyper-connection mix-statistics path (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference legs
import this package. The CUDA product path never does, and the two share no code.

The arithmetic lives in hcmix_oracle.c (plain C, compiled here with gcc and
-ffp-contract=off); this module only compiles it, loads it with ctypes and
marshals numpy arrays. Parity status of each function is stated in its C
comment and in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hcmix_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libhcmix_oracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle library with gcc (no fused multiply-add contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            L.oracle_chunk_dot.restype = F
            L.oracle_chunk_dot.argtypes = [P, P, I]
            L.oracle_chunk_dot_seq_f32.restype = F
            L.oracle_chunk_dot_seq_f32.argtypes = [P, P, I]
            L.oracle_sq_tree.restype = F
            L.oracle_sq_tree.argtypes = [P]
            L.oracle_stats.restype = None
            L.oracle_stats.argtypes = [P, I64, P, I64, I64, I64, I64, I, P, P]
            L.oracle_stats_seq_f32.restype = None
            L.oracle_stats_seq_f32.argtypes = [P, I64, P, I64, I64, I64, I64, I, P]
            L.oracle_stats_f64.restype = None
            L.oracle_stats_f64.argtypes = [P, I64, P, I64, I64, I64, I64, I, P, P]
            L.oracle_mix_unsplit_f64.restype = None
            L.oracle_mix_unsplit_f64.argtypes = [P, I64, P, I64, I64, I64, I64, I, P]
            L.oracle_sinkhorn.restype = None
            L.oracle_sinkhorn.argtypes = [P, I, I, F]
            L.oracle_epilogue.restype = None
            L.oracle_epilogue.argtypes = [P, P, I64, I64, I64, I, I, P, P, I, F, F, P, P, P]
            L.oracle_epilogue_f64.restype = None
            L.oracle_epilogue_f64.argtypes = [P, P, I64, I64, I64, I, I, P, P, I,
                                              ctypes.c_double, ctypes.c_double, P, P, P]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_x(x: np.ndarray) -> np.ndarray:
    assert x.dtype == np.uint16 and x.ndim == 2 and x.strides[1] == 2
    return x


def _check_w(W: np.ndarray) -> np.ndarray:
    assert W.dtype == np.float32 and W.ndim == 2 and W.strides[1] == 4
    return W


def _rows_parallel(fn, M: int, threads: int):
    """Run fn(row0, row1) over contiguous row blocks on `threads` host threads.

    Rows are independent, so the result is identical to one thread.
    """
    threads = max(1, min(threads, M))
    if threads == 1:
        fn(0, M)
        return
    bounds = [M * t // threads for t in range(threads + 1)]
    ts = [threading.Thread(target=fn, args=(bounds[t], bounds[t + 1])) for t in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()


def stats(x: np.ndarray, W: np.ndarray, K: int | None = None, threads: int = 1,
          rows: tuple[int, int] | None = None):
    """(mix[M, mix] fp32, sq[M] fp32) with the page's slice order."""
    _check_x(x); _check_w(W)
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    mixn = W.shape[0]
    mix = np.zeros((M, mixn), np.float32)
    sq = np.zeros(M, np.float32)
    L = lib()
    xs, ws = x.strides[0] // 2, W.strides[0] // 4

    def run(r0, r1):
        L.oracle_stats(_ptr(x), xs, _ptr(W), ws, r0, r1, K, mixn, _ptr(mix), _ptr(sq))
    if rows is None:
        _rows_parallel(run, M, threads)
    else:
        run(*rows)
    return mix, sq


def stats_seq_f32(x: np.ndarray, W: np.ndarray):
    _check_x(x); _check_w(W)
    M, K = x.shape
    mix = np.zeros((M, W.shape[0]), np.float32)
    lib().oracle_stats_seq_f32(_ptr(x), x.strides[0] // 2, _ptr(W), W.strides[0] // 4,
                               0, M, K, W.shape[0], _ptr(mix))
    return mix


def stats_f64(x: np.ndarray, W: np.ndarray):
    _check_x(x); _check_w(W)
    M, K = x.shape
    mix = np.zeros((M, W.shape[0]), np.float64)
    sq = np.zeros(M, np.float64)
    lib().oracle_stats_f64(_ptr(x), x.strides[0] // 2, _ptr(W), W.strides[0] // 4,
                           0, M, K, W.shape[0], _ptr(mix), _ptr(sq))
    return mix, sq


def mix_unsplit_f64(x: np.ndarray, W: np.ndarray):
    _check_x(x); _check_w(W)
    M, K = x.shape
    mix = np.zeros((M, W.shape[0]), np.float64)
    lib().oracle_mix_unsplit_f64(_ptr(x), x.strides[0] // 2, _ptr(W), W.strides[0] // 4,
                                 0, M, K, W.shape[0], _ptr(mix))
    return mix


def chunk_dot(x: np.ndarray, w: np.ndarray) -> np.float32:
    x = np.ascontiguousarray(x, np.uint16); w = np.ascontiguousarray(w, np.float32)
    return np.float32(lib().oracle_chunk_dot(_ptr(x), _ptr(w), len(x)))


def chunk_dot_seq_f32(x: np.ndarray, w: np.ndarray) -> np.float32:
    x = np.ascontiguousarray(x, np.uint16); w = np.ascontiguousarray(w, np.float32)
    return np.float32(lib().oracle_chunk_dot_seq_f32(_ptr(x), _ptr(w), len(x)))


def sq_tree(x64: np.ndarray) -> np.float32:
    x64 = np.ascontiguousarray(x64, np.uint16)
    assert x64.shape == (64,)
    return np.float32(lib().oracle_sq_tree(_ptr(x64)))


def sinkhorn(c: np.ndarray, iters: int, hc_eps: float = 0.0) -> np.ndarray:
    c = np.array(c, np.float32, copy=True, order="C")
    hc = c.shape[0]
    lib().oracle_sinkhorn(_ptr(c), hc, iters, hc_eps)
    return c


def epilogue(mix: np.ndarray, sq: np.ndarray, K: int, hc_scale: np.ndarray, hc_base: np.ndarray,
             iters: int = 20, rms_eps: float = 1e-6, hc_eps: float = 0.0, hc: int = 4,
             threads: int = 1):
    """(pre[M,hc], post[M,hc], comb[M,hc,hc]) fp32."""
    mix = np.ascontiguousarray(mix, np.float32)
    sq = np.ascontiguousarray(sq, np.float32)
    sc = np.ascontiguousarray(hc_scale, np.float32)
    bs = np.ascontiguousarray(hc_base, np.float32)
    M, mixn = mix.shape
    pre = np.zeros((M, hc), np.float32)
    post = np.zeros((M, hc), np.float32)
    comb = np.zeros((M, hc, hc), np.float32)
    L = lib()

    def run(r0, r1):
        L.oracle_epilogue(_ptr(mix), _ptr(sq), r0, r1, K, mixn, hc, _ptr(sc), _ptr(bs),
                          iters, rms_eps, hc_eps, _ptr(pre), _ptr(post), _ptr(comb))
    _rows_parallel(run, M, threads)
    return pre, post, comb


def epilogue_f64(mix: np.ndarray, sq: np.ndarray, K: int, hc_scale: np.ndarray,
                 hc_base: np.ndarray, iters: int = 20, rms_eps: float = 1e-6,
                 hc_eps: float = 0.0, hc: int = 4):
    mix = np.ascontiguousarray(mix, np.float64)
    sq = np.ascontiguousarray(sq, np.float64)
    sc = np.ascontiguousarray(hc_scale, np.float32)
    bs = np.ascontiguousarray(hc_base, np.float32)
    M, mixn = mix.shape
    pre = np.zeros((M, hc), np.float64)
    post = np.zeros((M, hc), np.float64)
    comb = np.zeros((M, hc, hc), np.float64)
    lib().oracle_epilogue_f64(_ptr(mix), _ptr(sq), 0, M, K, mixn, hc, _ptr(sc), _ptr(bs), iters,
                              rms_eps, hc_eps, _ptr(pre), _ptr(post), _ptr(comb))
    return pre, post, comb


def fused(x: np.ndarray, W: np.ndarray, hc_scale, hc_base, iters: int = 20,
          rms_eps: float = 1e-6, hc_eps: float = 0.0, threads: int = 1):
    """Whole path: (pre, post, comb, mix, sq)."""
    mix, sq = stats(x, W, threads=threads)
    pre, post, comb = epilogue(mix, sq, x.shape[1], hc_scale, hc_base, iters, rms_eps, hc_eps,
                               threads=threads)
    return pre, post, comb, mix, sq
