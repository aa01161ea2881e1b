"""ds_topk_noalloc: the entry point for callers that cannot allocate device memory
(inside a graph capture, in allocation-free serving loops, or when a caching allocator
already holds the device's memory).  It must give the same top-k as ds_topk_ex on the
split-over-clusters launch, which is the one that needs scratch, on two calls in a row:
the second call reuses the fixed scratch array the first one left behind.

This file is collected last so that a run stopping at its first failure has already run
every other test."""
import numpy as np
import pytest

import synth
from gpu_util import check_topk, to_device

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _values(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint16) if dtype == synth.BF16 else a.view(np.uint32)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_noalloc_matches_existing_entry_point(dtype):
    import top_selection_gb300 as ds
    rng = np.random.default_rng(77 + dtype)
    rows, N, k, B, B2 = 3, 300000, 512, 4096, 4096
    parts, cluster = 8, 2                      # four clusters per row: needs scratch
    x = rng.standard_normal((rows, N)).astype(np.float32)
    if dtype == synth.BF16:
        x = synth.f32_to_bf16_bits(x)
    need = ds.ds_workspace_bytes(dtype, rows, N, k, B, B2, parts=parts, cluster=cluster)
    assert 0 < need <= ds.ds_noalloc_scratch_bytes()
    xt = to_device(x, dtype)
    s = torch.cuda.current_stream().cuda_stream
    ref_v = torch.empty((rows, k), dtype=xt.dtype, device="cuda")
    ref_i = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for call in range(2):
        st = ds.ds_topk_ex(xt.data_ptr(), dtype, rows, N, N, k, B, B2, 5 + call, ref_v.data_ptr(),
                           ref_i.data_ptr(), parts=parts, cluster=cluster, workspace=ws.data_ptr(),
                           workspace_bytes=need, stream=s)
        assert st == 0
        out_v = torch.empty((rows, k), dtype=xt.dtype, device="cuda")
        out_i = torch.empty((rows, k), dtype=torch.int32, device="cuda")
        st = ds.ds_topk_noalloc(xt.data_ptr(), dtype, rows, N, N, k, B, B2, 5 + call, out_v.data_ptr(),
                                out_i.data_ptr(), parts=parts, cluster=cluster, stream=s)
        assert st == 0
        assert ds.ds_get_device_status(s) == 0
        rv, nv = _values(ref_v, dtype), _values(out_v, dtype)
        ni = out_i.cpu().numpy()
        for r in range(rows):
            # exact: the same value multiset as the existing entry point
            assert sorted(nv[r].tolist()) == sorted(rv[r].tolist())
        check_topk(x, dtype, k, nv, ni)


def test_noalloc_rejects_scratch_beyond_its_maximum():
    import top_selection_gb300 as ds
    # 64 clusters per row x 64 rows x k=4096 x 8 bytes is far above the fixed array
    rows, N, k = 64, 4 * 1024 * 1024, 4096
    need = ds.ds_workspace_bytes(synth.FP32, rows, N, k, 8192, 4096, parts=128, cluster=2)
    assert need > ds.ds_noalloc_scratch_bytes()
    x = torch.empty(16, dtype=torch.float32, device="cuda")   # never read: rejected first
    v = torch.empty(16, dtype=torch.float32, device="cuda")
    i = torch.empty(16, dtype=torch.int32, device="cuda")
    st = ds.ds_topk_noalloc(x.data_ptr(), synth.FP32, rows, N, N, k, 8192, 4096, 1, v.data_ptr(),
                            i.data_ptr(), parts=128, cluster=2, stream=torch.cuda.current_stream().cuda_stream)
    assert st == 7          # DS_ERR_WORKSPACE
