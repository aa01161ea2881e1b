"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Literal single-CTA rows must reproduce the oracle transcription's schedule exactly
(A, R, W, max|C| for the same block order); every result must pass check_topk (value
multiset bit-exact, indices distinct and pointing at their values, all columns above the
k-th key present)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import bits_of, check_sorted, check_topk, check_topk_by_counts, pad_rows, run_gpu, to_device

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


# ---------------------------------------------------------------- block order ------

@pytest.mark.parametrize("seed,row,b0,n", [(0, 0, 0, 1), (0x5EED, 0, 0, 64), (123, 7, 40, 300),
                                           (2**63 + 5, 2**31 + 3, 1000, 1024), (9, 1, 0, 17)])
def test_block_order_matches_oracle(seed, row, b0, n):
    import top_selection_gb300 as ds
    out = torch.zeros(n, dtype=torch.int32, device="cuda")
    assert ds.ds_block_order(seed, row, b0, n, out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    got = out.cpu().numpy().tolist()
    draws = {b: oracle.block_draw(seed, row, b) for b in range(b0, b0 + n)}
    want = sorted(draws, key=lambda b: (draws[b], b))
    assert got == want
    if b0 == 0:
        assert got == oracle.block_permutation(seed, row, n).tolist()


# ---------------------------------------------------------------- literal schedule -

def _literal_case(x, dtype, k, B, B2, seed):
    xp, n = pad_rows(x, dtype)
    v, i, st = run_gpu(xp, dtype, k, B, B2, seed, N=n, parts=1, stats=True)
    ov, oi, ost = oracle.deepselect(x, dtype, k, B, B2, seed, threads=8)
    assert (ost[:, oracle.STAT_FLAGS] == 0).all()
    for col in (oracle.STAT_A, oracle.STAT_R, oracle.STAT_W, oracle.STAT_MAXC, oracle.STAT_M):
        assert np.array_equal(st[:, col], ost[:, col]), f"stat {col}: gpu {st[:, col]} oracle {ost[:, col]}"
    check_topk(x, dtype, k, v, i)


def test_literal_single_row_f32():
    w = synth.row65536_f32()
    _literal_case(w.x, w.dtype, 512, 1024, 1024, 0x5EED)


@pytest.mark.parametrize("order", ["ascending", "descending", "staircase"])
def test_literal_block_ordered(order):
    N, k, B, B2 = 262144, 512, 1024, 1024
    x = synth.block_ordered(N, B, order).reshape(1, -1)
    for seed in (0, 1, 77):
        _literal_case(x, synth.FP32, k, B, B2, seed)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_literal_random_shapes(dtype):
    rng = np.random.default_rng(10 + dtype)
    for trial in range(12):
        rows = int(rng.integers(1, 6))
        N = int(rng.integers(1, 40000))
        k = int(rng.integers(1, min(N, 4096) + 1))
        B = int(rng.integers(1, 600)) * 8
        B = max(B, -(-N // 1024 // 8) * 8 + 8)          # one CTA visits at most 1024 blocks
        B2 = int(rng.integers(1, 3000))
        x = rng.standard_normal((rows, N)).astype(np.float32)
        if trial % 3 == 1:
            x = np.round(x * 4) / 4                     # ties
        if dtype == synth.BF16:
            x = synth.f32_to_bf16_bits(x)
        try:
            _literal_case(x, dtype, k, B, B2, int(rng.integers(0, 2**63)))
        except Exception as e:
            raise AssertionError(f"trial {trial}: rows={rows} N={N} k={k} B={B} B2={B2}") from e


# ---------------------------------------------------------------- edge cases -------

def test_edge_values():
    """Signed zeros, NaNs of both signs, infinities and denormals, in both dtypes."""
    specials32 = np.array([0x00000000, 0x80000000, 0x7FC00000, 0xFFC00000, 0x7F800000, 0xFF800000,
                           0x00000001, 0x80000001, 0x7F7FFFFF, 0xFF7FFFFF, 0x3F800000, 0xBF800000],
                          dtype=np.uint32)
    rng = np.random.default_rng(3)
    row = specials32[rng.integers(0, len(specials32), size=5000)].reshape(1, -1)
    for k in (1, 7, 100, 2000, 4096, 5000):
        if k > 4096:
            continue
        v, i, _ = run_gpu(row.view(np.float32), synth.FP32, k, 256, 256, 4)
        check_topk(row.view(np.float32), synth.FP32, k, v, i)
    specials16 = np.array([0x0000, 0x8000, 0x7FC0, 0xFFC0, 0x7F80, 0xFF80, 0x0001, 0x8001, 0x3F80, 0xBF80],
                          dtype=np.uint16)
    row16 = specials16[rng.integers(0, len(specials16), size=3001)].reshape(1, -1)
    for k in (1, 3, 500, 3001):
        v, i, _ = run_gpu(row16, synth.BF16, k, 64, 64, 5)
        check_topk(row16, synth.BF16, k, v, i)


@pytest.mark.parametrize("N", [1, 2, 7, 8, 9, 15, 16, 17, 1023, 1025, 4097])
@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_ragged_lengths(N, dtype):
    rng = np.random.default_rng(N)
    x = rng.standard_normal((3, N)).astype(np.float32)
    if dtype == synth.BF16:
        x = synth.f32_to_bf16_bits(x)
    xp, n = pad_rows(x, dtype)
    for k in sorted({1, max(1, N // 2), min(N, 4096)}):
        v, i, _ = run_gpu(xp, dtype, k, 8, 8, 11, N=n)
        check_topk(x, dtype, k, v, i)
        v, i, _ = run_gpu(xp, dtype, k, 8, 8, 11, N=n, parts=1)
        check_topk(x, dtype, k, v, i)


def test_padded_stride():
    w = synth.indexer_bf16(rows=5, N=131000, stride=131072)
    v, i, _ = run_gpu(w.x, w.dtype, 512, 4096, 4096, 3, N=w.N)
    check_topk(w.x, w.dtype, 512, v, i, N=w.N)


def test_k_equals_n_and_k_max():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 4096)).astype(np.float32)
    v, i, _ = run_gpu(x, synth.FP32, 4096, 1024, 1024, 1)
    check_topk(x, synth.FP32, 4096, v, i)
    w = synth.sampler_f32(rows=3, N=129280)
    v, i, _ = run_gpu(w.x, w.dtype, 4096, 8192, 4096, 2)
    check_topk(w.x, w.dtype, 4096, v, i)


# ---------------------------------------------------------------- split rows -------

@pytest.mark.parametrize("parts,cluster", [(2, 2), (4, 4), (8, 8), (4, 1), (8, 2), (16, 4), (16, 16)])
@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_split_rows(parts, cluster, dtype):
    rng = np.random.default_rng(parts * 10 + cluster)
    rows, N = 3, 200000
    x = rng.standard_normal((rows, N)).astype(np.float32)
    if dtype == synth.BF16:
        x = synth.f32_to_bf16_bits(x)
    for k in (1, 64, 512, 2048):
        v, i, _ = run_gpu(x, dtype, k, 2048, 2048, 99, parts=parts, cluster=cluster)
        check_topk(x, dtype, k, v, i)


def test_split_rows_tie_heavy():
    w = synth.longctx_bf16("levels", rows=2, N=300000)
    for parts, cluster in [(4, 4), (8, 1), (16, 8)]:
        v, i, _ = run_gpu(w.x, w.dtype, 2048, 4096, 4096, 5, parts=parts, cluster=cluster)
        check_topk(w.x, w.dtype, 2048, v, i)


def test_caller_workspace():
    import top_selection_gb300 as ds
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 300000)).astype(np.float32)
    nb = ds.ds_workspace_bytes(synth.FP32, 2, 300000, 512, 4096, 4096, parts=8, cluster=2)
    assert nb > 0
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        v, i, _ = run_gpu(x, synth.FP32, 512, 4096, 4096, 7, parts=8, cluster=2, workspace=ws)
        check_topk(x, synth.FP32, 512, v, i)


# ---------------------------------------------------------------- workloads --------

def _auto(w, k):
    v, i, _ = run_gpu(w.x, w.dtype, k, w.B, w.B2, 0x5EED, N=w.N)
    check_topk(w.x, w.dtype, k, v, i, N=w.N, threads=16)


def test_workload_row65536_f32():
    _auto(synth.row65536_f32(), 512)


def test_workload_indexer_bf16():
    _auto(synth.indexer_bf16(), 512)


@pytest.mark.parametrize("k", [1, 64, 512, 4096])
def test_workload_sampler_f32(k):
    _auto(synth.sampler_f32(), k)


@pytest.mark.parametrize("k,ties", [(64, 3), (512, 8), (512, 40)])
def test_sampler_rows_ties_at_the_kth_value(k, ties):
    """Sampler rows (one CTA each) where `ties` more elements, the next ones below the k-th
    largest value, are set to that value: the final select's pivot bin holds a few keys
    (ranked in one warp when they number at most 32, counted in further passes
    otherwise) with several copies of the pivot, of which exactly the quota is taken."""
    w = synth.sampler_f32()
    x = w.x[:, : w.N].copy()
    for r in range(w.rows):
        order = np.argsort(-x[r], kind="stable")
        x[r, order[k: k + ties]] = x[r, order[k - 1]]
    v, i, _ = run_gpu(x, w.dtype, k, w.B, w.B2, 0x5EED, N=w.N)
    check_topk(x, w.dtype, k, v, i, N=w.N, threads=16)


@pytest.mark.parametrize("kind", ["iid", "ascending", "levels"])
@pytest.mark.parametrize("k", [512, 2048])
def test_workload_longctx_bf16(kind, k):
    _auto(synth.longctx_bf16(kind), k)


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_longctx_ascending_compactions_make_progress(seed):
    # On ascending rows every element passes the threshold, so compactions follow one
    # another and each must leave room for a whole pass; the block order decides which
    # keys the cuts meet.
    w = synth.longctx_bf16("ascending")
    v, i, _ = run_gpu(w.x, w.dtype, 2048, w.B, w.B2, seed, N=w.N)
    check_topk(w.x, w.dtype, 2048, v, i, N=w.N, threads=16)


@pytest.mark.parametrize("shape,k", [("row65536", 512), ("row65536", 2048), ("indexer", 512), ("indexer", 2048)])
@pytest.mark.parametrize("seed", [1, 0x5EED])
def test_sorted_rows_held_whole_share_dense_passes(shape, k, seed):
    """Rows held whole whose values ascend along the row: every chunk above the edge is a
    dense pass (all its elements pass), several in one CTA on the single row, so warps
    share passes out in slices, help from their waits and contend for the one open job."""
    import top_selection_gb300 as ds
    w = {"row65536": synth.row65536_f32, "indexer": synth.indexer_bf16}[shape]()
    assert ds.ds_get_plan(w.dtype, w.rows, w.N, k, w.B, w.B2)["spec_k"] > 0  # held whole
    x = w.x[:, : w.N]
    xs = np.sort(synth.bf16_bits_to_f32(x) if w.dtype == synth.BF16 else x, axis=1)
    xs = synth.f32_to_bf16_bits(xs) if w.dtype == synth.BF16 else np.ascontiguousarray(xs, dtype=np.float32)
    v, i, _ = run_gpu(xs, w.dtype, k, w.B, w.B2, seed, N=w.N)
    check_topk(xs, w.dtype, k, v, i, N=w.N, threads=16)


# ---------------------------------------------------------------- hot sampled blocks -

def _spikes_in_sampled_blocks(w, k, seed):
    """w's rows with spikes U(8, 12) in the first block each part of the planned split
    visits (that block is always in the warm-up's sample), k - 32 of them per row in all:
    the sample holds nearly all of the row's largest values, fewer than k, and its group
    maxima overstate how many large values the rest of the row holds.  On rows held whole
    the speculative edge then lands among the spikes, fewer than k keys reach it, and the
    kernel must filter the row again from the proven edge."""
    import top_selection_gb300 as ds
    plan = ds.ds_get_plan(w.dtype, w.rows, w.N, k, w.B, w.B2)
    assert plan["spec_k"] > 0, plan
    parts = plan["parts"]
    m = -(-w.N // w.B)
    x = w.x[:, : w.N].copy()
    xf = synth.bf16_bits_to_f32(x) if w.dtype == synth.BF16 else x
    rng = np.random.default_rng(0xB10C)
    per = (k - 32) // parts
    for r in range(w.rows):
        for p in range(parts):  # part p holds blocks p, p + parts, ...
            first = min((oracle.block_draw(seed, r, b), b) for b in range(p, m, parts))[1]
            lo, hi = first * w.B, min(first * w.B + w.B, w.N)
            cols = lo + rng.choice(hi - lo, size=per, replace=False)
            xf[r, cols] = rng.uniform(8.0, 12.0, size=per).astype(np.float32)
    return synth.f32_to_bf16_bits(xf) if w.dtype == synth.BF16 else xf


@pytest.mark.parametrize("shape,k", [("indexer", 512), ("indexer", 2048), ("row65536", 512), ("longctx", 512),
                                     ("longctx", 2048)])
def test_spikes_in_every_sampled_block(shape, k):
    w = {"indexer": synth.indexer_bf16, "row65536": synth.row65536_f32,
         "longctx": lambda: synth.longctx_bf16("iid")}[shape]()
    seed = 0x5EED
    x = _spikes_in_sampled_blocks(w, k, seed)
    v, i, _ = run_gpu(x, w.dtype, k, w.B, w.B2, seed)
    check_topk(x, w.dtype, k, v, i, threads=16)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_one_hot_block_per_row(seed):
    # One block per row with k - 32 spikes, at a random position: the warm-up samples the
    # hot block in some rows and not in others.
    w = synth.indexer_bf16()
    x = synth.bf16_bits_to_f32(w.x[:, : w.N].copy())
    rng = np.random.default_rng(seed)
    for r in range(w.rows):
        b = int(rng.integers(0, w.N // w.B))
        cols = b * w.B + rng.choice(w.B, size=480, replace=False)
        x[r, cols] = rng.uniform(8.0, 12.0, size=480).astype(np.float32)
    x = synth.f32_to_bf16_bits(x)
    v, i, _ = run_gpu(x, w.dtype, 512, w.B, w.B2, seed)
    check_topk(x, w.dtype, 512, v, i, threads=16)


@pytest.mark.parametrize("k", [32, 4096])
def test_workload_huge_f32(k):
    w = synth.huge_f32()
    v, i, _ = run_gpu(w.x, w.dtype, k, w.B, w.B2, 0x5EED)
    check_topk_by_counts(w.x[0], k, v[0].view(np.float32), i[0].astype(np.int64))
    # the oracle on a sampled slice of the same row, through the same launch shape
    sl = np.ascontiguousarray(w.x[:, : 1 << 22])
    v2, i2, _ = run_gpu(sl, w.dtype, k, w.B, w.B2, 0x5EED)
    check_topk(sl, w.dtype, k, v2, i2)


# ---------------------------------------------------------------- failure path -----

def test_wait_timeout_is_reported_and_context_survives():
    import top_selection_gb300 as ds
    s = torch.cuda.current_stream().cuda_stream
    assert ds.ds_get_device_status(s) == 0
    assert ds.ds_wait_probe(2_000_000, s) == 0
    assert ds.ds_get_device_status(s) == 5          # DS_ERR_TIMEOUT
    assert ds.ds_get_device_status(s) == 0          # cleared
    w = synth.row65536_f32(rows=2)
    v, i, _ = run_gpu(w.x, w.dtype, 512, 1024, 1024, 1)
    check_topk(w.x, w.dtype, 512, v, i)


def test_graph_capture_replay():
    import top_selection_gb300 as ds
    w = synth.indexer_bf16(rows=8, N=131072)
    xt = to_device(w.x, w.dtype)
    vals = torch.empty((8, 512), dtype=xt.dtype, device="cuda")
    idx = torch.empty((8, 512), dtype=torch.int32, device="cuda")
    ds.topk(xt, 512, 4096, 4096, seed=1, out=(vals, idx))     # first call outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ds.topk(xt, 512, 4096, 4096, seed=1, out=(vals, idx))
    vals.zero_()
    g.replay()
    torch.cuda.synchronize()
    v = vals.cpu().numpy().view(np.uint16)
    check_topk(w.x, w.dtype, 512, v, idx.cpu().numpy())


# ------------------------------------------------- consecutive calls on one stream -----
# Calls on a stream may overlap their edges (programmatic dependent launch): a call starts
# its scan while the previous call finishes, and writes its outputs only once the previous
# call has completed.

@pytest.mark.parametrize("ready", [False, True])
def test_back_to_back_calls_same_outputs(ready):
    """A graph of consecutive calls on different inputs into the same outputs: the outputs
    hold the last call's result, and intermediate results (copied out between calls)
    are each correct -- also when the calls state that their inputs were complete before
    the previous call started (and so overlap it)."""
    import top_selection_gb300 as ds
    ws = [synth.indexer_bf16(seed=600 + i, rows=16, N=131072) for i in range(6)]
    xs = [to_device(w.x, w.dtype) for w in ws]
    vals = torch.empty((16, 512), dtype=xs[0].dtype, device="cuda")
    idx = torch.empty((16, 512), dtype=torch.int32, device="cuda")
    keep_v = [torch.empty_like(vals) for _ in xs]
    keep_i = [torch.empty_like(idx) for _ in xs]
    ds.topk(xs[0], 512, 4096, 4096, seed=3, out=(vals, idx))
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i, x in enumerate(xs):
                ds.topk(x, 512, 4096, 4096, seed=3, out=(vals, idx), input_ready=ready)
                if i % 2 == 1:
                    keep_v[i].copy_(vals)
                    keep_i[i].copy_(idx)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert ds.ds_get_device_status() == 0
    check_topk(ws[-1].x, ws[-1].dtype, 512, vals.cpu().numpy().view(np.uint16), idx.cpu().numpy())
    for i in (1, 3):
        check_topk(ws[i].x, ws[i].dtype, 512, keep_v[i].cpu().numpy().view(np.uint16), keep_i[i].cpu().numpy())


def test_input_written_right_before_each_call():
    """The input of every call is written by a copy kernel just before the call, on the same
    stream; every result matches its own input."""
    import top_selection_gb300 as ds
    ws = [synth.indexer_bf16(seed=700 + i, rows=16, N=131072) for i in range(4)]
    srcs = [to_device(w.x, w.dtype) for w in ws]
    x = torch.empty_like(srcs[0])
    outs = [(torch.empty((16, 512), dtype=x.dtype, device="cuda"), torch.empty((16, 512), dtype=torch.int32,
                                                                                device="cuda")) for _ in ws]
    for rep in range(2):
        for i in range(len(ws)):
            x.copy_(srcs[i])
            ds.topk(x, 512, 4096, 4096, seed=5, out=outs[i])
        torch.cuda.synchronize()
        assert ds.ds_get_device_status() == 0
        for i, w in enumerate(ws):
            check_topk(w.x, w.dtype, 512, outs[i][0].cpu().numpy().view(np.uint16), outs[i][1].cpu().numpy())


@pytest.mark.parametrize("parts", [0, 1])
def test_input_is_previous_calls_output(parts):
    """A call whose input is the output of the call just before it on the stream (which
    lets its successor start early) reads that output only once it is complete: the top-64
    of each row's top-512 values is the row's top-64."""
    import top_selection_gb300 as ds
    ws = [synth.indexer_bf16(seed=900 + i, rows=64, N=131072) for i in range(3)]
    xs = [to_device(w.x, w.dtype) for w in ws]
    mid = torch.empty((64, 512), dtype=xs[0].dtype, device="cuda")
    mid_i = torch.empty((64, 512), dtype=torch.int32, device="cuda")
    outs = [(torch.empty((64, 64), dtype=mid.dtype, device="cuda"),
             torch.empty((64, 64), dtype=torch.int32, device="cuda")) for _ in range(20)]
    for j in range(len(outs)):
        mid.fill_(-1)  # every value -1.0: a stale read returns only -1.0
        ds.topk(xs[j % 3], 512, 4096, 4096, seed=5, out=(mid, mid_i))
        ds.topk(mid, 64, 256, 256, seed=6, out=outs[j], parts=parts)
    torch.cuda.synchronize()
    assert ds.ds_get_device_status() == 0
    want = [oracle.topk_sort(bits_of(w.x, w.dtype), w.dtype, 64, threads=8)[0] for w in ws]
    for j, (v, _) in enumerate(outs):
        got = np.sort(v.cpu().numpy().view(np.uint16).astype(np.int64), axis=1)
        assert np.array_equal(got, np.sort(want[j % 3].astype(np.int64), axis=1)), f"call {j}"


@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_many_rows_one_part_each(dtype):
    """Rows that already cover the SMs run one per CTA in the split-row kernel when k is
    small against a chunk (no cluster, k + one chunk of candidates); a ragged row length
    leaves a tail in the last block."""
    import top_selection_gb300 as ds
    rng = np.random.default_rng(31 + dtype)
    rows, N = 200, 19997
    x = rng.standard_normal((rows, N)).astype(np.float32)
    if dtype == synth.BF16:
        x = synth.f32_to_bf16_bits(x)
    xp, n = pad_rows(x, dtype)
    plan = ds.ds_get_plan(dtype, rows, n, 64, 1024, 1024)
    assert plan["parts"] == 1 and plan["threads"] == 256
    for k in (1, 64, 256):
        v, i, _ = run_gpu(xp, dtype, k, 1024, 1024, 17, N=n)
        check_topk(x, dtype, k, v, i)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
@pytest.mark.parametrize("k", [1, 1000, 2048])
def test_many_short_rows_k_up_to_n(dtype, k):
    """One CTA per row in the split-row kernel with k up to the row length: 8 blocks per
    row (the fewest the plan splits this way), ties from rounding."""
    import top_selection_gb300 as ds
    rng = np.random.default_rng(77 + k + dtype)
    rows, N, B = 160, 2048, 256
    x = np.round(rng.standard_normal((rows, N)) * 8).astype(np.float32) / 8
    if dtype == synth.BF16:
        x = synth.f32_to_bf16_bits(x)
    plan = ds.ds_get_plan(dtype, rows, N, k, B, B)
    assert plan["parts"] == 1 and plan["threads"] == 256
    v, i, _ = run_gpu(x, dtype, k, B, B, 23)
    check_topk(x, dtype, k, v, i)


def test_many_rows_special_values_and_input_ready():
    """One CTA per row in the split-row kernel on rows full of signed zeros, infinities,
    NaNs of both signs and denormals; the same calls stating their inputs were ready
    before the previous call started give the same results."""
    import top_selection_gb300 as ds
    specials = np.array([0x00000000, 0x80000000, 0x7FC00000, 0xFFC00000, 0x7F800000, 0xFF800000,
                         0x00000001, 0x80000001, 0x3F800000, 0xBF800000, 0x40000000, 0xC0000000],
                        dtype=np.uint32)
    rng = np.random.default_rng(91)
    rows, N, k, B = 160, 8192, 300, 512
    x = specials[rng.integers(0, len(specials), size=(rows, N))].view(np.float32)
    x[:, ::7] = rng.standard_normal((rows, len(range(0, N, 7)))).astype(np.float32)
    plan = ds.ds_get_plan(synth.FP32, rows, N, k, B, B)
    assert plan["parts"] == 1 and plan["threads"] == 256
    xt = to_device(x, synth.FP32)
    outs = []
    for ready in (False, True):
        vals = torch.empty((rows, k), dtype=torch.float32, device="cuda")
        idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
        ds.topk(xt, k, B, B, seed=4, out=(vals, idx), input_ready=ready)
        ds.topk(xt, k, B, B, seed=4, out=(vals, idx), input_ready=ready)
        torch.cuda.synchronize()
        assert ds.ds_get_device_status() == 0
        v, i = vals.cpu().numpy().view(np.uint32), idx.cpu().numpy()
        check_topk(x, synth.FP32, k, v, i)
        outs.append(np.sort(v, axis=1))
    assert np.array_equal(outs[0], outs[1])


def test_concurrent_streams_multi_cluster_rows():
    """Rows split over several clusters use a library workspace; calls on two streams at
    the same time (no ordering between them) each get their own, so both results are
    right.  A larger call on one stream then grows that stream's workspace while work
    enqueued earlier may still use the old one."""
    import top_selection_gb300 as ds
    rng = np.random.default_rng(404)
    xa = rng.standard_normal((3, 400000)).astype(np.float32)
    xb = rng.standard_normal((3, 400000)).astype(np.float32)
    ta, tb = to_device(xa, synth.FP32), to_device(xb, synth.FP32)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = {}
    torch.cuda.synchronize()
    for rep in range(4):
        for name, t, s in (("a", ta, sa), ("b", tb, sb)):
            with torch.cuda.stream(s):
                v = torch.empty((3, 512), dtype=torch.float32, device="cuda")
                i = torch.empty((3, 512), dtype=torch.int32, device="cuda")
                ds.topk(t, 512, 4096, 4096, seed=rep, out=(v, i), parts=16, cluster=4, stream=s.cuda_stream)
                outs[(name, rep)] = (v, i)
    with torch.cuda.stream(sa):   # more rows: stream a's workspace grows
        xc = rng.standard_normal((9, 400000)).astype(np.float32)
        tc = to_device(xc, synth.FP32)
        vc = torch.empty((9, 512), dtype=torch.float32, device="cuda")
        ic = torch.empty((9, 512), dtype=torch.int32, device="cuda")
        ds.topk(tc, 512, 4096, 4096, seed=9, out=(vc, ic), parts=16, cluster=4, stream=sa.cuda_stream)
    torch.cuda.synchronize()
    assert ds.ds_get_device_status() == 0
    for (name, rep), (v, i) in outs.items():
        x = xa if name == "a" else xb
        check_topk(x, synth.FP32, 512, v.cpu().numpy().view(np.uint32), i.cpu().numpy())
    check_topk(xc, synth.FP32, 512, vc.cpu().numpy().view(np.uint32), ic.cpu().numpy())


@pytest.mark.parametrize("shape", ["row65536", "indexer", "sampler", "longctx", "huge"])
def test_library_chosen_block_sizes(shape):
    """B = B2 = 0 lets the library choose the block size and compaction slack; results
    match the oracle on every workload shape (the 268M-element row by the count identity
    and on a 4M-element slice)."""
    import top_selection_gb300 as ds
    if shape == "huge":
        w = synth.huge_f32()
        for k in (32, 4096):
            v, i, _ = run_gpu(w.x, w.dtype, k, 0, 0, 0x5EED)
            check_topk_by_counts(w.x[0], k, v[0].view(np.float32), i[0].astype(np.int64))
        sl = np.ascontiguousarray(w.x[:, : 1 << 22])
        v, i, _ = run_gpu(sl, w.dtype, 4096, 0, 0, 0x5EED)
        check_topk(sl, w.dtype, 4096, v, i)
        return
    w = {"row65536": synth.row65536_f32, "indexer": synth.indexer_bf16, "sampler": synth.sampler_f32,
         "longctx": lambda: synth.longctx_bf16("ascending")}[shape]()
    plan = ds.ds_get_plan(w.dtype, w.rows, w.N, 512, 0, 0)
    waves = -(-w.rows // torch.cuda.get_device_properties(0).multi_processor_count)
    assert (plan["B"], plan["B2"]) == ((8192 if waves == 1 else 4096), 4096)
    for k in (1, 512, 4096 if w.N >= 4096 else w.N):
        v, i, _ = run_gpu(w.x, w.dtype, k, 0, 0, 0x5EED, N=w.N)
        check_topk(w.x, w.dtype, k, v, i, N=w.N, threads=16)



# ---------------------------------------------------------------- sorted output ----

@pytest.mark.parametrize("shape", ["row65536", "indexer", "sampler", "longctx", "huge_slice"])
def test_sorted_output_workloads(shape):
    """options.sorted: each row's k results come in the oracle's order (value descending,
    equal values by column ascending) on every workload shape, k from 1 to 4096."""
    if shape == "huge_slice":
        w = synth.huge_f32()
        x = np.ascontiguousarray(w.x[:, : 1 << 22])
        for k in (32, 4096):
            v, i, _ = run_gpu(x, w.dtype, k, w.B, w.B2, 0x5EED, sorted=True)
            check_sorted(x, w.dtype, k, v, i)
        return
    w = {"row65536": synth.row65536_f32, "indexer": lambda: synth.indexer_bf16(rows=16),
         "sampler": lambda: synth.sampler_f32(rows=24), "longctx": lambda: synth.longctx_bf16("levels")}[shape]()
    for k in (1, 2, 100, 512, 4096):
        v, i, _ = run_gpu(w.x, w.dtype, k, w.B, w.B2, 0x5EED, N=w.N, sorted=True)
        check_sorted(w.x, w.dtype, k, v, i, N=w.N, threads=16)


@pytest.mark.parametrize("parts,cluster", [(1, 1), (0, 0), (16, 4)])
@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_sorted_output_every_path(parts, cluster, dtype):
    """The one-CTA schedule, the split-row kernel and rows over several clusters (merge
    kernel) all give sorted results with the option; ties and special values included."""
    rng = np.random.default_rng(123 + parts + dtype)
    rows, N = 3, 300000
    x = np.round(rng.standard_normal((rows, N)) * 16).astype(np.float32) / 16   # many ties
    x[0, ::1001] = np.float32(np.inf)
    x[1, ::997] = -0.0
    if dtype == synth.BF16:
        x = synth.f32_to_bf16_bits(x)
    B = 4096
    for k in (7, 777, 4096):
        v, i, _ = run_gpu(x, dtype, k, B, B, 5, parts=parts, cluster=cluster, sorted=True)
        check_sorted(x, dtype, k, v, i)


# ---------------------------------------------------------------- top-k sampling ----

@pytest.mark.parametrize("shape,k,temperature", [
    ("sampler", 1, 1.0), ("sampler", 64, 0.7), ("sampler", 512, 1.0), ("sampler", 512, 2.5),
    ("sampler", 4096, 1.0), ("indexer", 512, 1.0)])
def test_topk_sample_matches_oracle(shape, k, temperature):
    """ds_topk_sample: the sorted top-k matches the oracle's sequence, and the sampled
    column is the oracle's, except where the row's uniform draw lies within the fp32
    rounding bound of a boundary of the oracle's running sums (the GPU sums weights in
    fp32, the oracle in fp64); the reported probability matches within that bound."""
    import top_selection_gb300 as ds
    w = synth.sampler_f32(rows=48) if shape == "sampler" else synth.indexer_bf16(rows=16)
    rng = np.random.default_rng(k * 7 + int(temperature * 10))
    u = rng.random(w.rows).astype(np.float32)
    u[0], u[1] = 0.0, np.float32(0.99999994)
    xt = to_device(w.x, w.dtype)
    tok, prob, vals, idx = ds.topk_sample(xt, k, temperature, torch.from_numpy(u).cuda(), B=w.B, B2=w.B2, N=w.N)
    assert ds.ds_get_device_status() == 0
    v = vals.cpu().numpy()
    v = v.view(np.uint16) if w.dtype == synth.BF16 else v.view(np.uint32)
    i = idx.cpu().numpy()
    check_sorted(w.x, w.dtype, k, v, i, N=w.N, threads=16)
    bits = bits_of(w.x, w.dtype)
    otok, oprob, ocdf = oracle.topk_sample(np.ascontiguousarray(bits[:, :w.N]), w.dtype, k, temperature,
                                           u.astype(np.float64), threads=16)
    tok, prob = tok.cpu().numpy(), prob.cpu().numpy()
    tol = (k + 8) * 2.0 ** -22
    for r in range(w.rows):
        pos = np.nonzero(i[r] == tok[r])[0]
        assert pos.size == 1, f"row {r}: sampled column is not one of the row's top-k"
        p = int(pos[0])
        if tok[r] != otok[r]:
            lo = ocdf[r, p - 1] if p > 0 else 0.0
            assert lo - tol <= u[r] <= ocdf[r, p] + tol, f"row {r}: token {tok[r]} vs oracle {otok[r]}"
        else:
            assert abs(prob[r] - oprob[r]) <= tol + 1e-6 * oprob[r], f"row {r}: probability"
    if k == 1:
        assert np.array_equal(tok, i[:, 0])


@pytest.mark.slow
def test_workload_huge_f32_full_row_against_the_oracle():
    """The whole 268,435,456-element row (not a slice): the GPU's top 32 and top 4096, in
    the launch the planner picks for it (256 parts over clusters of 8 and the merge
    kernel), against the oracle's full stable sort of the same row (a few minutes of CPU)."""
    w = synth.huge_f32()
    got = {k: run_gpu(w.x, w.dtype, k, w.B, w.B2, 0x5EED)[:2] for k in (32, 4096)}
    bits = w.x.view(np.uint32)
    ref_v, ref_i = oracle.topk_sort(bits, w.dtype, 4096, threads=1)
    for k, (v, i) in got.items():
        rv, ri = ref_v[:, :k], ref_i[:, :k]
        assert sorted(v[0].tolist()) == sorted(rv[0].tolist()), f"k={k}: value multiset differs"
        ir = i[0].astype(np.int64)
        assert len(set(ir.tolist())) == k and np.array_equal(bits[0][ir], v[0])
        kth = oracle.key(int(rv[0][-1]), w.dtype)
        keys = np.array([oracle.key(int(x), w.dtype) for x in rv[0]], dtype=np.int64)
        assert set(ri[0][keys > kth].tolist()) <= set(ir.tolist()), f"k={k}: a value above the k-th is missing"
