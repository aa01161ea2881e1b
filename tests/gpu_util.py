"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and check a
result against the oracle's full stable sort."""
import numpy as np

import oracle
import synth


def bits_of(x, dtype):
    return x.view(np.uint16) if dtype == synth.BF16 else x.view(np.uint32)


def pad_rows(x_np, dtype):
    """Copy of x with each row padded to a 16-byte multiple; the padding holds the
    largest value of the dtype's order (+NaN with full payload), so a kernel that read
    past N would return it."""
    rows, n = x_np.shape
    mult = 8 if dtype == synth.BF16 else 4
    stride = -(-n // mult) * mult
    if dtype == synth.BF16:
        out = np.full((rows, stride), 0x7FFF, dtype=np.uint16)
    else:
        out = np.full((rows, stride), 0x7FFFFFFF, dtype=np.uint32).view(np.float32)
    out[:, :n] = x_np
    return out, n


def to_device(x_np, dtype):
    import torch
    if dtype == synth.BF16:
        return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x_np).view(np.float32)).cuda()


def run_gpu(x_np, dtype, k, B, B2, seed, N=None, parts=0, cluster=0, stats=False, workspace=None, sorted=False):
    """Returns (vals_bits, idx, stats-or-None) as numpy arrays."""
    import torch
    import top_selection_gb300 as ds
    xt = to_device(x_np, dtype)
    rows = x_np.shape[0]
    st = torch.zeros((rows, ds.DS_NSTAT), dtype=torch.int64, device="cuda") if stats else None
    vals, idx = ds.topk(xt, k, B, B2, seed=seed, N=N, parts=parts, cluster=cluster, stats=st,
                        workspace=workspace, sorted=sorted)
    status = ds.ds_get_device_status(torch.cuda.current_stream().cuda_stream)
    assert status == 0, f"device status {status}"
    v = vals.cpu().numpy()
    v = v.view(np.uint16) if dtype == synth.BF16 else v.view(np.uint32)
    return v, idx.cpu().numpy(), (st.cpu().numpy() if stats else None)


def check_topk(x_np, dtype, k, vals, idx, N=None, threads=8):
    """The value multiset equals the oracle's top-k exactly (bitwise); the indices are
    distinct, inside the row, and point at their values; and every column whose key is
    strictly above the k-th key is returned (so the index sets agree whenever no tie
    crosses the k-th value)."""
    bits = bits_of(x_np, dtype)
    n = bits.shape[1] if N is None else N
    ref_v, ref_i = oracle.topk_sort(np.ascontiguousarray(bits[:, :n]), dtype, k, threads=threads)
    for r in range(bits.shape[0]):
        assert sorted(vals[r].tolist()) == sorted(ref_v[r].tolist()), f"row {r}: value multiset differs"
        ir = idx[r].astype(np.int64)
        assert len(set(ir.tolist())) == k, f"row {r}: repeated index"
        assert ir.min() >= 0 and ir.max() < n, f"row {r}: index outside the row"
        assert np.array_equal(bits[r][ir], vals[r]), f"row {r}: index does not point at its value"
        kth = oracle.key(int(ref_v[r][-1]), dtype)
        keys = np.array([oracle.key(int(v), dtype) for v in ref_v[r]], dtype=np.int64)
        must = set(ref_i[r][keys > kth].tolist())
        assert must <= set(ir.tolist()), f"row {r}: a value above the k-th is missing"


def check_topk_by_counts(x_f32_row, k, vals_f32, idx):
    """Top-k check that holds at any size, for finite rows without -0: with v the
    smallest returned value, the returned values above v are exactly the row's values
    above v, and the returned copies of v exist in the row."""
    x = x_f32_row
    assert len(np.unique(idx)) == k
    assert idx.min() >= 0 and idx.max() < x.size
    assert np.array_equal(x[idx].view(np.uint32), vals_f32.view(np.uint32))
    v = vals_f32.min()
    assert int((vals_f32 > v).sum()) == int((x > v).sum())
    assert int((vals_f32 == v).sum()) <= int((x == v).sum())


def check_sorted(x_np, dtype, k, vals, idx, N=None, threads=8):
    """Sorted output: check_topk, and the sequence is the oracle's order -- values (bit
    patterns) position by position, and the columns at every position whose key is above
    the k-th key (values equal to the k-th may come from other columns, by column)."""
    check_topk(x_np, dtype, k, vals, idx, N=N, threads=threads)
    bits = bits_of(x_np, dtype)
    n = bits.shape[1] if N is None else N
    ref_v, ref_i = oracle.topk_sort(np.ascontiguousarray(bits[:, :n]), dtype, k, threads=threads)
    for r in range(bits.shape[0]):
        assert np.array_equal(vals[r], ref_v[r]), f"row {r}: value sequence differs from the oracle's"
        kth = oracle.key(int(ref_v[r][-1]), dtype)
        above = np.array([oracle.key(int(v), dtype) > kth for v in ref_v[r]], dtype=bool)
        assert np.array_equal(idx[r][above], ref_i[r][above]), f"row {r}: column order differs above the k-th"
        eq = ~above
        cols = idx[r][eq].astype(np.int64)
        assert np.all(np.diff(cols) > 0), f"row {r}: equal values not in column order"
