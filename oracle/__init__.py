"""CPU oracle for DeepSelect row-wise top-k -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It shares no code with the CUDA library and never calls it.
The arithmetic lives in ``oracle.c`` (compiled here with gcc on first use); this module
only marshals numpy arrays.  See ``oracle.c`` for what each function computes and the
passages it follows.

Values travel as raw bit patterns: ``uint16`` arrays for bf16, ``float32`` (or
``uint32``) arrays for fp32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16 = 0
FP32 = 1

NSTAT = 8
STAT_A, STAT_R, STAT_W, STAT_MAXC, STAT_M, STAT_FLAGS, STAT_TUPD = range(7)

F_CAP = 1
F_BLOCKSTART = 2
F_TDECR = 4
F_READS = 8
F_RB2 = 16
F_WSUM = 32
F_FINAL_SHORT = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP over rows)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, u32, u64, vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                                  ctypes.c_uint64, ctypes.c_void_p)
        lib.oracle_key.argtypes = [u32, ctypes.c_int]
        lib.oracle_key.restype = u32
        lib.oracle_philox4x32_10.argtypes = [vp, vp, vp]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_block_draw.argtypes = [u64, i64, i64]
        lib.oracle_block_draw.restype = u32
        lib.oracle_block_permutation.argtypes = [u64, i64, i64, vp]
        lib.oracle_block_permutation.restype = ctypes.c_int
        lib.oracle_topk_sort.argtypes = [vp, ctypes.c_int, i64, i64, i64, i32, vp, vp, i32]
        lib.oracle_topk_sort.restype = ctypes.c_int
        lib.oracle_deepselect.argtypes = [vp, ctypes.c_int, i64, i64, i64, i32, i32, i32, u64,
                                          vp, vp, vp, vp, i32]
        lib.oracle_deepselect.restype = ctypes.c_int
        lib.oracle_topk_sample.argtypes = [vp, ctypes.c_int, i64, i64, i64, i32, ctypes.c_double, vp, vp,
                                           vp, vp, i32]
        lib.oracle_topk_sample.restype = ctypes.c_int
        lib.oracle_work_bound.argtypes = [i64, i32, i32, i32]
        lib.oracle_work_bound.restype = ctypes.c_double
        lib.oracle_num_threads_max.argtypes = []
        lib.oracle_num_threads_max.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == BF16:
        if x.dtype != np.uint16:
            raise TypeError("bf16 input must be a uint16 bit-pattern array")
        return x
    if x.dtype == np.float32:
        return x.view(np.uint32)
    if x.dtype != np.uint32:
        raise TypeError("fp32 input must be float32 or uint32 bits")
    return x


def _rows_view(x: np.ndarray, N: int | None, stride: int | None):
    if x.ndim == 1:
        x = x.reshape(1, -1)
    if x.ndim != 2:
        raise ValueError("x must be 1-D or 2-D")
    if not x.flags.c_contiguous:
        raise ValueError("x must be C-contiguous (rows of `stride` elements)")
    rows, width = x.shape
    N = width if N is None else int(N)
    stride = width if stride is None else int(stride)
    if stride != width or N > width:
        raise ValueError("N must not exceed the row width, and stride must equal it")
    return x, rows, N, stride


def max_threads() -> int:
    return int(_load().oracle_num_threads_max())


def key(bits: int, dtype: int) -> int:
    """Order-preserving integer key of one raw value."""
    return int(_load().oracle_key(ctypes.c_uint32(int(bits)), dtype))


def philox4x32_10(counter, key_) -> tuple:
    c = np.asarray(counter, dtype=np.uint32).copy()
    k = np.asarray(key_, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return tuple(int(v) for v in out)


def block_draw(seed: int, row: int, b: int) -> int:
    return int(_load().oracle_block_draw(seed, row, b))


def block_permutation(seed: int, row: int, m: int) -> np.ndarray:
    perm = np.zeros(max(m, 1), dtype=np.int64)
    if _load().oracle_block_permutation(seed, row, m, _ptr(perm)) != 0:
        raise MemoryError("oracle_block_permutation failed")
    return perm[:m]


def topk_sort(x: np.ndarray, dtype: int, k: int, N: int | None = None, threads: int = 1):
    """Row-wise top-k by a full stable sort (key desc, column asc).

    Returns (vals, idx) of shape (rows, k), in that sorted order.  ``vals`` holds the
    raw bit patterns (uint16 for bf16, uint32 for fp32)."""
    bits = _as_bits(x, dtype)
    bits, rows, N, stride = _rows_view(bits, N, None)
    vals = np.zeros((rows, k), dtype=np.uint16 if dtype == BF16 else np.uint32)
    idx = np.zeros((rows, k), dtype=np.int32)
    rc = _load().oracle_topk_sort(_ptr(bits), dtype, rows, N, stride, k, _ptr(vals), _ptr(idx),
                                  threads)
    if rc != 0:
        raise ValueError(f"oracle_topk_sort rejected its arguments (rc={rc})")
    return vals, idx


def deepselect(x: np.ndarray, dtype: int, k: int, B: int, B2: int, seed: int,
               N: int | None = None, perm: np.ndarray | None = None, threads: int = 1):
    """The DeepSelectTopk transcription.

    Returns (vals, idx, stats): vals/idx of shape (rows, k) in final-buffer order, and
    stats of shape (rows, NSTAT) with A, R, W, max|C|, m, flags, T-updates."""
    bits = _as_bits(x, dtype)
    bits, rows, N, stride = _rows_view(bits, N, None)
    vals = np.zeros((rows, k), dtype=np.uint16 if dtype == BF16 else np.uint32)
    idx = np.zeros((rows, k), dtype=np.int32)
    stats = np.zeros((rows, NSTAT), dtype=np.int64)
    pptr = None
    if perm is not None:
        m = -(-N // B)
        perm = np.ascontiguousarray(perm, dtype=np.int64)
        if perm.shape != (m,):
            raise ValueError(f"perm must have ceil(N/B) = {m} entries")
        pptr = _ptr(perm)
    rc = _load().oracle_deepselect(_ptr(bits), dtype, rows, N, stride, k, B, B2, seed, pptr,
                                   _ptr(vals), _ptr(idx), _ptr(stats), threads)
    if rc != 0:
        raise ValueError(f"oracle_deepselect rejected its arguments (rc={rc})")
    return vals, idx, stats


def topk_sample(x: np.ndarray, dtype: int, k: int, temperature: float, uniforms, N: int | None = None,
                threads: int = 1):
    """Top-k sampling (see oracle.c): returns (token, prob, cdf) -- the sampled column and
    its probability per row, and the normalised running sums (rows, k) of the weights in
    the sorted top-k order."""
    bits = _as_bits(x, dtype)
    bits, rows, N, stride = _rows_view(bits, N, None)
    u = np.ascontiguousarray(np.asarray(uniforms, dtype=np.float64).reshape(rows))
    token = np.zeros(rows, dtype=np.int32)
    prob = np.zeros(rows, dtype=np.float64)
    cdf = np.zeros((rows, k), dtype=np.float64)
    rc = _load().oracle_topk_sample(_ptr(bits), dtype, rows, N, stride, k, float(temperature), _ptr(u),
                                    _ptr(token), _ptr(prob), _ptr(cdf), threads)
    if rc != 0:
        raise ValueError(f"oracle_topk_sample rejected its arguments (rc={rc})")
    return token, prob, cdf


def work_bound(N: int, k: int, B: int, B2: int) -> float:
    """(1 + k/B2) (k+B+B2) H_m with m = ceil(N/B)."""
    return float(_load().oracle_work_bound(N, k, B, B2))
