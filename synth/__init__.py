"""Seeded synthetic inputs for the DeepSelect top-k workloads.

This module only draws input rows; it holds none of the method's arithmetic, so both
the oracle tests and the CUDA tests may use it.  Rows are numpy arrays of raw bit
patterns: ``uint16`` for bf16 (rounded from fp32 to nearest-even) and ``float32`` for
fp32.  The random block order the method draws is not generated here: it is a function
of the ``seed`` argument of the top-k call.

Workloads (the shapes of the DeepSeek indexer and sampler top-k the DeepSelect pages
describe; all values are synthetic):

  row65536_f32        1 x 65,536 fp32, N(0,1); k=512, B=B2=1024
  indexer_bf16        64 x 131,072 bf16, N(0,1); k=512, B=B2=4096
  sampler_f32         256 x 129,280 fp32, 2*N(0,1) with 32 spikes per row drawn
                      from U(8,12) at distinct random columns; k in {1,64,512,4096};
                      B=8192, B2=4096
  longctx_bf16        4 x 1,048,576 bf16; kind "iid" (N(0,1)), "ascending" (sorted
                      N(0,1) draws) or "levels" (256 values (2j-255)/64, j uniform);
                      k in {512, 2048}; B=B2=4096
  huge_f32            1 x 268,435,456 fp32, U(-1,1) on the 2^24-point grid
                      r/2^23 - 1; k in {32, 4096}; B=8192, B2=4096

Every generator takes ``rows`` / ``N`` overrides so the tests can draw the same
distributions at sizes the oracle finishes quickly, and a ``stride`` that pads rows.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16 = 0
FP32 = 1
DTYPE_NAMES = {BF16: "bf16", FP32: "fp32"}
ESIZE = {BF16: 2, FP32: 4}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    name: str
    dtype: int
    x: np.ndarray            # (rows, stride) raw values; columns >= N are padding
    rows: int
    N: int
    stride: int
    k: int
    ks: list = field(default_factory=list)
    B: int = 1024
    B2: int = 1024
    desc: str = ""

    @property
    def esize(self) -> int:
        return ESIZE[self.dtype]

    @property
    def input_bytes(self) -> int:
        return self.rows * self.N * self.esize


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(int(seed)))


def _padded(vals: np.ndarray, stride: int, pad_value) -> np.ndarray:
    rows, n = vals.shape
    if stride == n:
        return np.ascontiguousarray(vals)
    out = np.full((rows, stride), pad_value, dtype=vals.dtype)
    out[:, :n] = vals
    return out


def _normal_rows(rng, rows, N, scale=1.0) -> np.ndarray:
    out = np.empty((rows, N), dtype=np.float32)
    for r in range(rows):
        out[r] = rng.standard_normal(N, dtype=np.float32)
    if scale != 1.0:
        out *= np.float32(scale)
    return out


def normal(rows: int, N: int, dtype: int, seed: int, stride: int | None = None,
           scale: float = 1.0, name: str = "normal", k: int = 8, B: int = 1024,
           B2: int = 1024) -> Workload:
    stride = N if stride is None else stride
    rng = _rng(seed)
    v = _normal_rows(rng, rows, N, scale)
    x = f32_to_bf16_bits(v) if dtype == BF16 else v
    pad = np.uint16(0) if dtype == BF16 else np.float32(0)
    return Workload(name, dtype, _padded(x, stride, pad), rows, N, stride, k, [k], B, B2,
                    f"{rows}x{N} {DTYPE_NAMES[dtype]} N(0,{scale}^2)")


def row65536_f32(seed: int = 1001, rows: int = 1, N: int = 65536) -> Workload:
    w = normal(rows, N, FP32, seed, name="row65536_f32", k=512, B=1024, B2=1024)
    w.desc = f"{rows}x{N} fp32 i.i.d. N(0,1)"
    return w


def indexer_bf16(seed: int = 2001, rows: int = 64, N: int = 131072,
                 stride: int | None = None) -> Workload:
    if stride is None:
        stride = -(-N // 512) * 512      # rows padded to a multiple of 1024 bytes
    w = normal(rows, N, BF16, seed, stride=stride, name="indexer_bf16", k=512, B=4096, B2=4096)
    w.desc = f"{rows}x{N} bf16 i.i.d. N(0,1), row stride {stride} elements"
    return w


def sampler_f32(seed: int = 3001, rows: int = 256, N: int = 129280, spikes: int = 32,
                k: int = 512) -> Workload:
    rng = _rng(seed)
    v = _normal_rows(rng, rows, N, scale=2.0)
    s = min(spikes, N)
    for r in range(rows):
        cols = rng.choice(N, size=s, replace=False)
        v[r, cols] = rng.uniform(8.0, 12.0, size=s).astype(np.float32)
    return Workload("sampler_f32", FP32, np.ascontiguousarray(v), rows, N, N, k,
                    [1, 64, 512, 4096], 8192, 4096,
                    f"{rows}x{N} fp32 2*N(0,1) + {s} spikes U(8,12) per row")


def longctx_bf16(kind: str = "iid", seed: int = 4001, rows: int = 4, N: int = 1048576,
                 k: int = 512) -> Workload:
    rng = _rng(seed + {"iid": 0, "ascending": 10, "levels": 20}[kind])
    if kind == "iid":
        x = f32_to_bf16_bits(_normal_rows(rng, rows, N))
    elif kind == "ascending":
        x = f32_to_bf16_bits(np.sort(_normal_rows(rng, rows, N), axis=1))
    elif kind == "levels":
        j = rng.integers(0, 256, size=(rows, N), dtype=np.int32)
        x = f32_to_bf16_bits(((2 * j - 255).astype(np.float32) / np.float32(64.0)))
    else:
        raise ValueError(f"unknown row kind {kind!r}")
    return Workload(f"longctx_bf16_{kind}", BF16, np.ascontiguousarray(x), rows, N, N, k,
                    [512, 2048], 4096, 4096, f"{rows}x{N} bf16 {kind}")


def huge_f32(seed: int = 5001, rows: int = 1, N: int = 268435456, k: int = 32) -> Workload:
    rng = _rng(seed)
    x = np.empty((rows, N), dtype=np.float32)
    chunk = 1 << 24
    for r in range(rows):
        for c0 in range(0, N, chunk):
            c1 = min(N, c0 + chunk)
            u = rng.integers(0, 1 << 24, size=c1 - c0, dtype=np.uint32)
            x[r, c0:c1] = u.astype(np.float32) * np.float32(2.0 ** -23) - np.float32(1.0)
    return Workload("huge_f32", FP32, x, rows, N, N, k, [32, 4096], 8192, 4096,
                    f"{rows}x{N} fp32 U(-1,1) on a 2^24-point grid")


def block_ordered(N: int, B: int, order: str, dtype: int = FP32, seed: int = 7) -> np.ndarray:
    """One row whose blocks of B are value-ordered: 'ascending' (every value of block b
    exceeds every value of block b-1), 'descending', or 'staircase' (block-ordered
    ascending with the values inside each block shuffled)."""
    rng = _rng(seed)
    base = np.arange(N, dtype=np.float64)
    if order == "ascending":
        v = base
    elif order == "descending":
        v = base[::-1].copy()
    elif order == "staircase":
        v = base.copy()
        for lo in range(0, N, B):
            seg = v[lo:lo + B]
            rng.shuffle(seg)
            v[lo:lo + B] = seg
    else:
        raise ValueError(order)
    v = (v / N * 2.0 - 1.0).astype(np.float32)   # distinct, exact in fp32 for N <= 2^23
    if dtype == BF16:
        raise ValueError("block_ordered rows are fp32 (bf16 cannot hold N distinct values)")
    return v
