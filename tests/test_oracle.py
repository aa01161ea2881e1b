"""Pins for the CPU oracle: it is checked against things other than itself.

- published Philox4x32-10 known-answer vectors;
- the float order (numpy) for the key mapping, exhaustively over bf16;
- brute force (Python sorting of the float values) on tiny inputs;
- the block-order experiment table and the complexity tables of the DeepSelect TopK
  tutorial (sections 2.3, 3.7, 1.3, 6.3);
- the closed form for block-ordered inputs (each block accepted whole or not at all);
- the harmonic-number expectation of that closed form over many seeds;
- the invariants and the expected-work bound of DeepSelect-deep-dive.md.
"""
import itertools
import math

import numpy as np
import pytest

import synth
from conftest import golden_rows


# ------------------------------------------------------------------ Philox ----------

def test_philox_known_answers(oracle_lib):
    rows = golden_rows("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        vals = [int(v, 16) for v in r]
        ctr, key, want = vals[0:4], vals[4:6], tuple(vals[6:10])
        assert oracle_lib.philox4x32_10(ctr, key) == want


def test_block_draw_is_philox_word0(oracle_lib):
    seed, row, b = 0x0123456789ABCDEF, 7, 12345
    want = oracle_lib.philox4x32_10([b, row, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])[0]
    assert oracle_lib.block_draw(seed, row, b) == want


def test_block_permutation_is_sorted_draws(oracle_lib):
    seed, row, m = 42, 3, 200
    perm = oracle_lib.block_permutation(seed, row, m)
    assert sorted(perm.tolist()) == list(range(m))
    draws = [oracle_lib.block_draw(seed, row, b) for b in range(m)]
    want = sorted(range(m), key=lambda b: (draws[b], b))
    assert perm.tolist() == want


def test_block_permutation_uniform_positions(oracle_lib):
    # position of block 0 among m=8 blocks over many seeds: uniform (chi-square, 7 dof)
    m, trials = 8, 4000
    counts = np.zeros(m)
    for s in range(trials):
        perm = oracle_lib.block_permutation(s, 0, m)
        counts[int(np.nonzero(perm == 0)[0][0])] += 1
    exp = trials / m
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 24.3  # p ~ 0.001 for 7 degrees of freedom


def test_rows_get_different_orders(oracle_lib):
    a = oracle_lib.block_permutation(5, 0, 64)
    b = oracle_lib.block_permutation(5, 1, 64)
    c = oracle_lib.block_permutation(6, 0, 64)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


# ------------------------------------------------------------------ keys ------------

def _float_rank_key(v):
    """Python ordering of a non-NaN float: by value, -0 below +0."""
    return (float(v), 0 if math.copysign(1.0, float(v)) < 0 else 1)


def test_key_order_bf16_exhaustive(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32)
    keys = np.array([oracle_lib.key(int(b), oracle_lib.BF16) for b in bits], dtype=np.int64)
    assert len(set(keys.tolist())) == 65536 and keys.min() == 0 and keys.max() == 65535
    f = synth.bf16_bits_to_f32(bits.astype(np.uint16)).astype(np.float64)
    nan = np.isnan(f)
    order_by_key = np.argsort(keys)
    non_nan = [int(b) for b in order_by_key if not nan[b]]
    want = sorted(non_nan, key=lambda b: _float_rank_key(f[b]))
    assert non_nan == want
    # NaNs: sign-clear NaNs above +inf, sign-set NaNs below -inf
    k_pinf = keys[0x7F80]
    k_ninf = keys[0xFF80]
    for b in np.nonzero(nan)[0]:
        if b & 0x8000:
            assert keys[b] < k_ninf
        else:
            assert keys[b] > k_pinf


def test_key_order_fp32_sampled(oracle_lib):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=3000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x00000001,
                        0x80000001, 0x3F800000, 0xBF800000, 0x7F7FFFFF, 0xFF7FFFFF], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    f = bits.view(np.float32).astype(np.float64)
    keep = ~np.isnan(f)
    bits, f = bits[keep], f[keep]
    keys = [oracle_lib.key(int(b), oracle_lib.FP32) for b in bits]
    by_key = [int(i) for i in np.argsort(np.array(keys, dtype=np.int64), kind="stable")]
    by_float = sorted(range(len(bits)), key=lambda i: _float_rank_key(f[i]))
    # equal floats have equal bits here except +-0, which the rank key separates
    assert [int(bits[i]) for i in by_key] == [int(bits[i]) for i in by_float]


# ------------------------------------------------------------ brute force -----------

def _brute_topk(vals_f32, k):
    """k largest by float value (-0 below +0), smaller column first on ties."""
    n = len(vals_f32)
    order = sorted(range(n), key=lambda j: (_float_rank_key(vals_f32[j]), -j), reverse=True)
    return order[:k]


def _alphabet_rows(alphabet, n):
    for combo in itertools.product(alphabet, repeat=n):
        yield np.array(combo, dtype=np.float32)


def test_topk_sort_bruteforce_small_alphabet(oracle_lib):
    alphabet = [-1.5, -0.0, 0.0, 2.0, 2.0 ** -140]   # ties, signed zeros, a denormal
    for n in range(1, 6):
        for x in _alphabet_rows(alphabet, n):
            for k in range(1, n + 1):
                vals, idx = oracle_lib.topk_sort(x, oracle_lib.FP32, k)
                want = _brute_topk(x, k)
                assert idx[0].tolist() == want
                assert vals[0].tolist() == [int(v) for v in x.view(np.uint32)[want]]


def test_topk_sort_bruteforce_bf16_random(oracle_lib):
    rng = np.random.default_rng(1)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        x = synth.f32_to_bf16_bits(rng.integers(-4, 5, size=n).astype(np.float32) / 4)
        k = int(rng.integers(1, n + 1))
        vals, idx = oracle_lib.topk_sort(x, oracle_lib.BF16, k)
        want = _brute_topk(synth.bf16_bits_to_f32(x), k)
        assert idx[0].tolist() == want


def test_topk_sort_special_cases(oracle_lib):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 500)).astype(np.float32)
    x[1, 17] = x[1].max() + 1.0
    v, i = oracle_lib.topk_sort(x, oracle_lib.FP32, 1)
    assert i[:, 0].tolist() == np.argmax(x, axis=1).tolist()          # k=1: argmax
    v, i = oracle_lib.topk_sort(x, oracle_lib.FP32, 500)
    for r in range(3):                                                 # k=N: full sort
        assert i[r].tolist() == np.argsort(-x[r].astype(np.float64), kind="stable").tolist()


def test_topk_sort_padded_rows(oracle_lib):
    w = synth.indexer_bf16(rows=3, N=1000, stride=1024)
    assert w.x.shape == (3, 1024)
    v, i = oracle_lib.topk_sort(w.x, oracle_lib.BF16, 16, N=1000)
    assert i.max() < 1000
    v2, i2 = oracle_lib.topk_sort(np.ascontiguousarray(w.x[:, :1000]), oracle_lib.BF16, 16)
    assert np.array_equal(v, v2) and np.array_equal(i, i2)


# --------------------------------------------------------- transcription -----------

def _check_topk(x_bits, dtype, k, vals, idx, oracle_lib):
    """Accept exactly the results a top-k may return: the value multiset of the stable
    sort, distinct indices that point at their values, and every index whose key is
    strictly above the k-th key."""
    ref_v, ref_i = oracle_lib.topk_sort(x_bits, dtype, k)
    for r in range(x_bits.shape[0]):
        assert sorted(vals[r].tolist()) == sorted(ref_v[r].tolist())
        assert len(set(idx[r].tolist())) == k
        assert np.array_equal(x_bits[r][idx[r]], vals[r])
        kth = oracle_lib.key(int(ref_v[r][-1]), dtype)
        must = {int(j) for j, v in zip(ref_i[r], ref_v[r]) if oracle_lib.key(int(v), dtype) > kth}
        assert must <= set(idx[r].tolist())


def test_deepselect_every_order_tiny(oracle_lib):
    """For tiny rows, every block order gives the sort's multiset (random order changes
    the cost, never the result)."""
    rng = np.random.default_rng(3)
    for trial in range(40):
        n = int(rng.integers(2, 13))
        x = (rng.integers(-3, 4, size=(1, n)).astype(np.float32) / 2)
        x[0, rng.integers(0, n)] = -0.0
        bits = x.view(np.uint32)
        B = int(rng.integers(-(-n // 6), 5))       # at most 6 blocks: 720 orders
        B2 = int(rng.integers(1, 4))
        k = int(rng.integers(1, n + 1))
        m = -(-n // B)
        assert m <= 6
        for perm in itertools.permutations(range(m)):
            v, i, st = oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=0,
                                             perm=np.array(perm))
            assert st[0, oracle_lib.STAT_FLAGS] == 0
            _check_topk(bits, oracle_lib.FP32, k, v, i, oracle_lib)


def test_deepselect_random_shapes(oracle_lib):
    rng = np.random.default_rng(4)
    for trial in range(60):
        rows = int(rng.integers(1, 4))
        n = int(rng.integers(1, 3000))
        k = int(rng.integers(1, min(n, 300) + 1))
        B = int(rng.integers(1, 700))
        B2 = int(rng.integers(1, 700))
        dtype = oracle_lib.BF16 if trial % 2 else oracle_lib.FP32
        if dtype == oracle_lib.BF16:
            x = synth.f32_to_bf16_bits(rng.standard_normal((rows, n)).astype(np.float32))
            bits = x
        else:
            x = rng.standard_normal((rows, n)).astype(np.float32)
            if trial % 3 == 0:
                x = np.round(x * 2) / 2          # heavy ties
            bits = x.view(np.uint32)
        v, i, st = oracle_lib.deepselect(x, dtype, k, B, B2, seed=trial)
        assert (st[:, oracle_lib.STAT_FLAGS] == 0).all()
        A, R, W = st[:, 0], st[:, 1], st[:, 2]
        assert (W == A + k * R).all() and (R * B2 <= A).all()
        assert (st[:, oracle_lib.STAT_MAXC] <= k + B + B2).all()
        _check_topk(bits, dtype, k, v, i, oracle_lib)


@pytest.mark.parametrize("order", ["ascending", "descending", "staircase"])
def test_block_order_table_sequential(oracle_lib, order):
    rows = {(r[0], r[1]): tuple(int(v) for v in r[2:]) for r in golden_rows("block_order_experiment.txt")}
    N, k, B, B2 = 262144, 512, 1024, 1024
    x = synth.block_ordered(N, B, order)
    v, i, st = oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=0, perm=np.arange(N // B))
    assert tuple(st[0, :3]) == rows[(order, "sequential")]
    assert st[0, oracle_lib.STAT_FLAGS] == 0
    _check_topk(x.reshape(1, -1).view(np.uint32), oracle_lib.FP32, k, v, i, oracle_lib)


def _records_after_two(values_in_order):
    """Left-to-right maxima at positions 3..m."""
    best = max(values_in_order[0], values_in_order[1])
    rho = 0
    for v in values_in_order[2:]:
        if v > best:
            rho += 1
            best = v
    return rho


@pytest.mark.parametrize("order", ["ascending", "descending", "staircase"])
def test_block_ordered_closed_form(oracle_lib, order):
    """With k <= B, B2 <= B and B < k+B2 <= 2B, a block-ordered row is accepted block by
    block, whole or not at all: A = B(2+rho), R = 1+rho, rho = records of the visiting
    order after the first two blocks."""
    N, k, B, B2 = 262144, 512, 1024, 1024
    m = N // B
    x = synth.block_ordered(N, B, order)
    for seed in range(25):
        perm = oracle_lib.block_permutation(seed, 0, m)
        value = perm if order != "descending" else -perm
        rho = _records_after_two(list(value))
        v, i, st = oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=seed)
        assert (st[0, 0], st[0, 1]) == (B * (2 + rho), 1 + rho)


def test_block_order_table_random_rows_reachable(oracle_lib):
    """The table's random-order rows for block-ordered inputs are points of the closed
    form (A = B(2+rho), R = 1+rho, W = A+kR); the oracle reaches each one for some seed."""
    table = {(r[0], r[1]): tuple(int(v) for v in r[2:]) for r in golden_rows("block_order_experiment.txt")}
    N, k, B, B2 = 262144, 512, 1024, 1024
    for order in ["ascending", "descending", "staircase"]:
        A, R, W = table[(order, "random")]
        assert A == B * (2 + (R - 1)) and W == A + k * R
        x = synth.block_ordered(N, B, order)
        found = False
        for seed in range(400):
            v, i, st = oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=seed)
            if tuple(st[0, :3]) == (A, R, W):
                found = True
                break
        assert found, order


def test_block_order_table_iid_row(oracle_lib):
    """The table's i.i.d. row is one draw; A, R and W depend only on ranks, so any
    continuous i.i.d. law gives the same distribution.  The mean over many rows must sit
    within a few standard deviations of a single draw of about 61 elements."""
    table = {(r[0], r[1]): tuple(int(v) for v in r[2:]) for r in golden_rows("block_order_experiment.txt")}
    N, k, B, B2 = 262144, 512, 1024, 1024
    rng = np.random.default_rng(11)
    x = rng.standard_normal((96, N)).astype(np.float32)
    for mode in ["sequential", "random"]:
        perm = np.arange(N // B) if mode == "sequential" else None
        v, i, st = oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=5, perm=perm,
                                         threads=oracle_lib.max_threads())
        A, R, W = table[("random", mode)]
        assert abs(st[:, 0].mean() - A) < 250
        assert np.mean(st[:, 1] == R) > 0.9
        assert abs(st[:, 2].mean() - W) < 250
        assert (st[:, 2] <= oracle_lib.work_bound(N, k, B, B2)).all()


def test_expected_appends_block_ordered(oracle_lib):
    """E[A] = B (H_m + 1/2) for block-ordered rows under a uniform block order."""
    k, B, B2, m = 4, 8, 8, 256
    N = m * B
    x = synth.block_ordered(N, B, "ascending")
    trials = 2000
    As = np.zeros(trials)
    for s in range(trials):
        v, i, st = oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=1000 + s)
        As[s] = st[0, 0]
    H = sum(1.0 / i for i in range(1, m + 1))
    H2 = sum(1.0 / i ** 2 for i in range(1, m + 1))
    sd_rho = math.sqrt(H - 1.5 - (H2 - 1.25))
    assert abs(As.mean() / B - (H + 0.5)) < 4 * sd_rho / math.sqrt(trials)


# ------------------------------------------------------------------ bound ----------

def test_complexity_tables(oracle_lib):
    for r in golden_rows("complexity_tables.txt"):
        if r[0] == "table2":
            N, bound, asym, klog = (int(v) for v in r[1:])
            k, B, B2 = 512, 1024, 1024
            assert round(oracle_lib.work_bound(N, k, B, B2)) == bound
            assert round((1 + k / B2) * (k + B + B2) * math.log(N / B)) == asym
            assert round(k * math.log(N / k)) == klog
        elif r[0] == "sec63":
            N, k, B, B2, approx = (int(v) for v in r[1:])
            assert abs(oracle_lib.work_bound(N, k, B, B2) - approx) / approx < 0.01
        elif r[0] == "table4":
            N, k, model = (int(v) for v in r[1:])
            assert N * math.log2(k) == model
        elif r[0] == "sec37":
            N, k, approx = (int(v) for v in r[1:])
            assert abs(k * math.log(N / k) - approx) / approx < 0.01


@pytest.mark.parametrize("N,k,B,B2,dtype", [
    (65536, 512, 1024, 1024, 1),     # single fp32 row shape
    (131072, 512, 4096, 4096, 0),    # indexer shape
    (129280, 512, 8192, 4096, 1),    # sampler shape
    (129280, 64, 8192, 4096, 1),
    (262144, 512, 4096, 4096, 0),
])
def test_expected_work_below_bound(oracle_lib, N, k, B, B2, dtype):
    rows = 48
    rng = np.random.default_rng(N + k)
    x = rng.standard_normal((rows, N)).astype(np.float32)
    if dtype == 0:
        x = synth.f32_to_bf16_bits(x)
    Ws = []
    for s in range(4):
        v, i, st = oracle_lib.deepselect(x, dtype, k, B, B2, seed=77 + s, threads=oracle_lib.max_threads())
        assert (st[:, oracle_lib.STAT_FLAGS] == 0).all()
        Ws.append(st[:, 2])
    assert np.concatenate(Ws).mean() <= oracle_lib.work_bound(N, k, B, B2)


def test_adversarial_orders_below_bound(oracle_lib):
    """Sorted inputs are the worst case for an in-order scan; with the random order the
    mean work stays below the bound (the block-order experiment's point)."""
    N, k, B, B2 = 65536, 256, 512, 512
    bound = oracle_lib.work_bound(N, k, B, B2)
    for order in ["ascending", "descending", "staircase"]:
        x = synth.block_ordered(N, B, order)
        Ws = [oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=s)[2][0, 2] for s in range(300)]
        assert np.mean(Ws) <= bound
    x = synth.block_ordered(N, B, "ascending")
    v, i, st = oracle_lib.deepselect(x, oracle_lib.FP32, k, B, B2, seed=0, perm=np.arange(N // B))
    assert st[0, 2] > bound          # the in-order scan is far above it


def test_synth_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 3,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 65504.0], dtype=np.float32)])
    ours = synth.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- top-k sampling ----
# Pins of oracle.topk_sample by cases whose answer is fixed without its formula: one
# candidate, equal logits (uniform choice), two candidates (a logistic in the logit gap),
# a vanishing temperature (the arg max), and the candidate order among equal values.

def test_sample_k1_is_argmax(oracle_lib):
    rng = np.random.default_rng(41)
    x = rng.standard_normal((5, 300)).astype(np.float32)
    x[2, 7] = x[2, 200] = 9.0            # a tie at the maximum: the smaller column
    for u in (0.0, 0.3, 0.999999):
        tok, prob, _ = oracle_lib.topk_sample(x, synth.FP32, 1, 0.8, [u] * 5)
        assert tok.tolist() == [int(np.argmax(r)) for r in x]
        assert np.all(prob == 1.0)


def test_sample_equal_logits_is_uniform(oracle_lib):
    k = 37
    x = np.full((1, k), 1.25, dtype=np.float32)
    for m in range(k):
        u = (m + 0.5) / k
        tok, prob, cdf = oracle_lib.topk_sample(x, synth.FP32, k, 1.7, [u])
        assert tok[0] == m                      # equal values come by column
        assert abs(prob[0] - 1.0 / k) < 1e-15
        assert abs(cdf[0, m] - (m + 1) / k) < 1e-12


def test_sample_two_candidates_logistic(oracle_lib):
    for a, b, T in ((2.0, 0.5, 1.0), (0.0, -3.0, 0.5), (10.0, 9.0, 4.0)):
        x = np.array([[b, a]], dtype=np.float32)      # the larger value sits in column 1
        p_hi = 1.0 / (1.0 + math.exp((np.float32(b) - np.float32(a)) / T))
        tok, prob, _ = oracle_lib.topk_sample(x, synth.FP32, 2, T, [p_hi - 1e-9])
        assert tok[0] == 1 and abs(prob[0] - p_hi) < 1e-12
        tok, prob, _ = oracle_lib.topk_sample(x, synth.FP32, 2, T, [p_hi + 1e-9])
        assert tok[0] == 0 and abs(prob[0] - (1.0 - p_hi)) < 1e-12


def test_sample_cold_temperature_and_bf16(oracle_lib):
    rng = np.random.default_rng(42)
    x = rng.standard_normal((4, 1000)).astype(np.float32)
    xb = synth.f32_to_bf16_bits(x)
    xf = synth.bf16_bits_to_f32(xb)
    for u in (0.0, 0.5, 0.99):
        tok, _, _ = oracle_lib.topk_sample(xb, synth.BF16, 64, 1e-6, [u] * 4)
        assert tok.tolist() == [int(np.argmax(r)) for r in xf]


def test_sample_candidate_order_with_ties(oracle_lib):
    x = np.array([[5.0, 7.0, 7.0, 1.0]], dtype=np.float32)
    # candidates: columns 1, 2 (weight 1 each), then 0 (weight e^-2); total 2 + e^-2
    tot = 2.0 + math.exp(-2.0)
    for u, want in ((0.4 / tot, 1), (1.4 / tot, 2), (2.05 / tot, 0)):
        tok, _, _ = oracle_lib.topk_sample(x, synth.FP32, 3, 1.0, [u])
        assert tok[0] == want


def test_block_permutation_every_cell_uniform(oracle_lib):
    """Chi-square over every (block, position) cell: with m = 32 blocks and 3,200 seeds,
    each block lands in each position 100 times on average.  For a uniform permutation
    the statistic has (m - 1)^2 = 961 degrees of freedom (mean 961, sd ~44); a bias at
    any position, early or late, adds to it.  The bound is the mean + 6 sd."""
    m, seeds = 32, 3200
    counts = np.zeros((m, m), dtype=np.int64)
    for s in range(seeds):
        p = oracle_lib.block_permutation(0xC0FFEE + s, s % 7, m)
        counts[p, np.arange(m)] += 1
    assert np.all(counts.sum(axis=0) == seeds) and np.all(counts.sum(axis=1) == seeds)
    e = seeds / m
    chi2 = float(((counts - e) ** 2 / e).sum())
    dof = (m - 1) ** 2
    assert chi2 < dof + 6 * math.sqrt(2 * dof), chi2
