"""GB300-native DeepSelect row-wise top-k.

A thin ctypes binding over ``libds_topk.so`` (built in-tree from ``csrc/`` by
``top_selection_gb300.build``).  Functions carry the C ABI's names and do argument
marshalling only: every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback; when the library has not been built every call raises.

The C ABI (``include/ds_topk.h``) documents the operation, the argument layout, the
ownership rules and the error codes.  ``topk()`` is a convenience wrapper that takes and
returns torch tensors (PyTorch supplies device memory and streams only).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "DS_BF16", "DS_FP32", "DS_NSTAT", "DSError", "ds_topk", "ds_topk_ex", "ds_get_plan",
    "ds_workspace_bytes", "ds_get_device_status", "ds_status_string", "ds_version",
    "ds_block_order", "ds_wait_probe", "ds_topk_noalloc", "ds_noalloc_scratch_bytes", "topk",
    "library_path", "load",
]

DS_BF16 = 0
DS_FP32 = 1
DS_NSTAT = 8

STATUS_NAMES = {
    0: "DS_OK", 1: "DS_ERR_INVALID_ARG", 2: "DS_ERR_ALIGNMENT", 3: "DS_ERR_UNSUPPORTED",
    4: "DS_ERR_CUDA", 5: "DS_ERR_TIMEOUT", 6: "DS_ERR_INTERNAL", 7: "DS_ERR_WORKSPACE",
}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libds_topk.so")
_lock = threading.Lock()
_lib = None


class DSError(RuntimeError):
    def __init__(self, status: int, what: str = "ds_topk"):
        self.status = int(status)
        super().__init__(f"{what} failed: {STATUS_NAMES.get(self.status, self.status)} "
                         f"({ds_status_string(self.status) if _lib else ''})")


class ds_options(ctypes.Structure):
    _fields_ = [("parts", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("stats", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("input_ready", ctypes.c_int32),
                ("sorted", ctypes.c_int32)]


class ds_plan(ctypes.Structure):
    _fields_ = [("parts", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("chunk_elems", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("ctas_per_sm", ctypes.c_int32), ("merge_launch", ctypes.c_int32),
                ("B", ctypes.c_int32), ("B2", ctypes.c_int32), ("spec_k", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libds_topk.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m top_selection_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        i32, i64, u64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t
        lib.ds_topk.argtypes = [vp, i32, i64, i64, i64, i32, i32, i32, u64, vp, vp, vp]
        lib.ds_topk.restype = ctypes.c_int
        lib.ds_topk_ex.argtypes = [vp, i32, i64, i64, i64, i32, i32, i32, u64, vp, vp,
                                   ctypes.POINTER(ds_options), vp]
        lib.ds_topk_ex.restype = ctypes.c_int
        lib.ds_get_plan.argtypes = [i32, i64, i64, i32, i32, i32, ctypes.POINTER(ds_options),
                                    ctypes.POINTER(ds_plan)]
        lib.ds_get_plan.restype = ctypes.c_int
        lib.ds_workspace_bytes.argtypes = [i32, i64, i64, i32, i32, i32, ctypes.POINTER(ds_options),
                                           ctypes.POINTER(sz)]
        lib.ds_workspace_bytes.restype = ctypes.c_int
        lib.ds_get_device_status.argtypes = [vp]
        lib.ds_get_device_status.restype = ctypes.c_int
        lib.ds_status_string.argtypes = [ctypes.c_int]
        lib.ds_status_string.restype = ctypes.c_char_p
        lib.ds_version.argtypes = []
        lib.ds_version.restype = ctypes.c_char_p
        lib.ds_block_order.argtypes = [u64, i64, i64, i32, vp, vp]
        lib.ds_block_order.restype = ctypes.c_int
        lib.ds_wait_probe.argtypes = [i64, vp]
        lib.ds_wait_probe.restype = ctypes.c_int
        lib.ds_topk_noalloc.argtypes = [vp, i32, i64, i64, i64, i32, i32, i32, u64, vp, vp, i32, i32, vp]
        lib.ds_topk_noalloc.restype = ctypes.c_int
        lib.ds_topk_sample.argtypes = [vp, i32, i64, i64, i64, i32, i32, i32, u64, ctypes.c_float, vp, vp, vp,
                                       vp, vp, vp]
        lib.ds_topk_sample.restype = ctypes.c_int
        lib.ds_noalloc_scratch_bytes.argtypes = []
        lib.ds_noalloc_scratch_bytes.restype = ctypes.c_size_t
        _lib = lib
        return lib


def _opts(parts=0, cluster=0, stats=0, workspace=0, workspace_bytes=0, input_ready=False, sorted=False):
    return ds_options(int(parts), int(cluster), int(stats) or None, int(workspace) or None,
                      int(workspace_bytes), 1 if input_ready else 0, 1 if sorted else 0)


# ------------------------------------------------------------------ C ABI mirror ----

def ds_topk(x, dtype, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, stream=0) -> int:
    """Raw C call with device pointers (ints); returns the ds_status code."""
    return load().ds_topk(int(x) or None, dtype, rows, N, row_stride, k, B, B2, seed,
                          int(out_vals) or None, int(out_idx) or None, int(stream) or None)


def ds_topk_ex(x, dtype, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx,
               parts=0, cluster=0, stats=0, workspace=0, workspace_bytes=0, input_ready=False,
               stream=0, sorted=False) -> int:
    o = _opts(parts, cluster, stats, workspace, workspace_bytes, input_ready, sorted)
    return load().ds_topk_ex(int(x) or None, dtype, rows, N, row_stride, k, B, B2, seed,
                             int(out_vals) or None, int(out_idx) or None, ctypes.byref(o),
                             int(stream) or None)


def ds_get_plan(dtype, rows, N, k, B, B2, parts=0, cluster=0, stats=False) -> dict:
    o = _opts(parts, cluster, 1 if stats else 0)
    p = ds_plan()
    st = load().ds_get_plan(dtype, rows, N, k, B, B2, ctypes.byref(o), ctypes.byref(p))
    if st != 0:
        raise DSError(st, "ds_get_plan")
    return p.as_dict()


def ds_workspace_bytes(dtype, rows, N, k, B, B2, parts=0, cluster=0) -> int:
    o = _opts(parts, cluster)
    out = ctypes.c_size_t(0)
    st = load().ds_workspace_bytes(dtype, rows, N, k, B, B2, ctypes.byref(o), ctypes.byref(out))
    if st != 0:
        raise DSError(st, "ds_workspace_bytes")
    return int(out.value)


def ds_get_device_status(stream=0) -> int:
    return load().ds_get_device_status(int(stream) or None)


def ds_status_string(status: int) -> str:
    return load().ds_status_string(int(status)).decode()


def ds_version() -> str:
    return load().ds_version().decode()


def ds_block_order(seed, row, first_block, nblocks, out_perm, stream=0) -> int:
    return load().ds_block_order(seed, row, first_block, nblocks, int(out_perm), int(stream) or None)


def ds_wait_probe(cycles, stream=0) -> int:
    return load().ds_wait_probe(int(cycles), int(stream) or None)


def ds_topk_noalloc(x, dtype, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, parts=0, cluster=0,
                    stream=0) -> int:
    """ds_topk for callers that cannot allocate: scratch comes from a fixed array in the
    library (see include/ds_topk.h).  Raw device pointers; returns the ds_status code."""
    return load().ds_topk_noalloc(int(x) or None, dtype, rows, N, row_stride, k, B, B2, seed,
                                  int(out_vals) or None, int(out_idx) or None, parts, cluster,
                                  int(stream) or None)


def ds_noalloc_scratch_bytes() -> int:
    return int(load().ds_noalloc_scratch_bytes())


# ------------------------------------------------------------------ torch helper ----

def _torch_dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16 or t.dtype in (torch.int16, torch.uint16):
        return DS_BF16
    if t.dtype in (torch.float32, torch.int32):
        return DS_FP32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 (or 16-bit patterns) and fp32 only")


def topk(x, k: int, B: int, B2: int, seed: int = 0x5EED, N: int | None = None,
         out=None, parts: int = 0, cluster: int = 0, stats=None, workspace=None, stream=None,
         input_ready: bool = False, sorted: bool = False):
    """Row-wise DeepSelect top-k of a CUDA tensor ``x`` of shape (rows, stride).

    Returns (values, indices), each (rows, k), unordered within a row unless ``sorted``
    (then by value descending, equal values by column ascending).  ``N`` (default:
    the row length) may be shorter than the stride.  ``stats`` is an optional int64
    CUDA tensor (rows, DS_NSTAT) filled when each row is one part.  ``input_ready`` states
    that ``x`` was complete before the previous kernel on the stream started, which lets
    the call start reading it while that kernel finishes."""
    import torch
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (there is no CPU path)")
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    dtype = _torch_dtype_code(x)
    rows = x.shape[0]
    n = x.shape[1] if N is None else int(N)
    stride = x.stride(0) if rows > 1 else x.shape[1]
    if out is None:
        vals = torch.empty((rows, k), dtype=x.dtype, device=x.device)
        idx = torch.empty((rows, k), dtype=torch.int32, device=x.device)
    else:
        vals, idx = out
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = ds_topk_ex(x.data_ptr(), dtype, rows, n, stride, k, B, B2, seed, vals.data_ptr(),
                    idx.data_ptr(), parts=parts, cluster=cluster,
                    stats=0 if stats is None else stats.data_ptr(), workspace=ws_ptr,
                    workspace_bytes=ws_bytes, input_ready=input_ready, stream=stream, sorted=sorted)
    if st != 0:
        raise DSError(st)
    return vals, idx


def ds_topk_sample(x, dtype, rows, N, row_stride, k, B, B2, seed, temperature, uniforms, out_vals, out_idx,
                   out_token, out_prob=0, stream=0) -> int:
    """Raw C call (device pointers as ints); returns the ds_status code."""
    return load().ds_topk_sample(int(x) or None, dtype, rows, N, row_stride, k, B, B2, seed, float(temperature),
                                 int(uniforms) or None, int(out_vals) or None, int(out_idx) or None,
                                 int(out_token) or None, int(out_prob) or None, int(stream) or None)


def topk_sample(x, k: int, temperature: float, uniforms, B: int = 0, B2: int = 0, seed: int = 0x5EED,
                N: int | None = None, stream=None):
    """Top-k sampling of each row of the CUDA logits tensor ``x`` (rows, stride): the
    sorted top-k (values, columns), then one column drawn per row from the softmax of the
    k values at ``temperature`` with the row's uniform draw from ``uniforms`` (a CUDA
    float32 tensor of rows values in [0, 1)).  Returns (token, prob, values, indices)."""
    import torch
    if not x.is_cuda or not uniforms.is_cuda:
        raise ValueError("x and uniforms must be CUDA tensors (there is no CPU path)")
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    if uniforms.dtype != torch.float32 or uniforms.numel() != x.shape[0] or not uniforms.is_contiguous():
        raise ValueError("uniforms must be a contiguous float32 tensor with one value per row")
    dtype = _torch_dtype_code(x)
    rows = x.shape[0]
    n = x.shape[1] if N is None else int(N)
    stride = x.stride(0) if rows > 1 else x.shape[1]
    vals = torch.empty((rows, k), dtype=x.dtype, device=x.device)
    idx = torch.empty((rows, k), dtype=torch.int32, device=x.device)
    token = torch.empty(rows, dtype=torch.int32, device=x.device)
    prob = torch.empty(rows, dtype=torch.float32, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    st = ds_topk_sample(x.data_ptr(), dtype, rows, n, stride, k, B, B2, seed, temperature, uniforms.data_ptr(),
                        vals.data_ptr(), idx.data_ptr(), token.data_ptr(), prob.data_ptr(), stream)
    if st != 0:
        raise DSError(st, "ds_topk_sample")
    return token, prob, vals, idx
