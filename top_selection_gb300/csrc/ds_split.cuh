// ds_split.cuh -- DeepSelect on rows split over several CTAs (a thread-block cluster per
// group of G parts, and optionally C clusters per row), and on rows that have a CTA to
// themselves but many neighbours (G = 1).
//
// DeepSelect-deep-dive.md, "Implementation", has the CTAs of a cluster scan parts of one
// row, share the threshold T through distributed shared memory and merge their
// candidates.  This kernel keeps that structure and arranges the work for short critical
// paths on sm_103a:
//
//   * Parts and copies: part p of a row takes blocks p, p + P, p + 2P, ... in the order
//     the row's Philox draws give them.  8 warps, no producer: stage s of an 8- or
//     16-stage ring of 1-D bulk copies belongs to warp s mod 8, which filters every chunk
//     landing there and issues the stage's next copy itself.  The warm-up's chunks are
//     requested first, the rest once chunk 0 landed.  When every CTA can have an SM to
//     itself, a part of up to 16 chunks of 8 KB is held whole in the SM's shared memory.
//   * Warm-up (init window): the first ww chunks of every CTA are reduced to group
//     maxima (the largest key of each group of consecutive vectors) and exchanged with
//     bulk copies into each other's shared memory; every CTA derives the same edge from
//     the union.  At least k groups have a maximum at or above the edge, so at least k
//     elements of the row are kept above T = edge - 1: every element at or below T is
//     outside the top k (the threshold invariant of the deep dive's proof).  Rows held
//     whole take the edge from the 2048-bin top-digit bucket of the k-th largest maximum
//     and may start from a speculative edge instead (the spec_k-th largest maximum,
//     checked by the final select and redone from the proven edge when it fails); rows
//     streamed through the ring bin the maxima below the union's largest.
//   * Filter: each warp compares its chunk's packed values against T with one
//     instruction per word, reserves its survivors' slots with one shared atomic and
//     appends them -- sparse passes in two steps (columns per lane, then keys and columns
//     for the warp's slots in order), dense passes position by position, shared out in
//     slices with idle warps on rows held whole -- counting each key into the final
//     select's first histogram.  On streamed rows a warp raises T from that histogram
//     each time the buffer passes a mark.  A reservation that does not fit makes every
//     warp join a compaction: a cut at the histogram bin of the k-th largest key where
//     that frees enough room, else a RadixSelectTopK to exactly k; either raises T.
//   * Final: the cluster selects the k largest keys of the union of its buffers by
//     most-significant-digit radix passes over 512 bins.  Each pass, every CTA pushes
//     its histogram to every other CTA and the whole CTA finds the same pivot bin and
//     every CTA's count above it, so each CTA writes its share of the output at offsets
//     it computes itself, in one pass with two shared slot cursors.  A bin holding just
//     the keys still needed is taken whole; on rows of one CTA a bin of at most 32 keys
//     is ranked in one warp.
//
// The packed compare is "greater or unordered" against a float threshold chosen so that
// every element whose key exceeds T passes (NaNs always pass, and -0 passes a -0
// threshold); elements that pass without exceeding T are extra candidates that the
// key-based selections never pick, since at least k keys above T exist.
#pragma once

namespace dsk {

constexpr int kXBits = 9;               // final-select digit width
constexpr int kXBins = 1 << kXBits;     // final-select bins per pass (exchanged as uint16)
static_assert(kXBins == 32 * 16, "warp_pivot_x gives each lane 16 bins");
constexpr int kWarmMaxBytes = 16384;    // group maxima exchanged by the warm-up, all CTAs
constexpr int kSplitThreads = kNCW * 32;  // consumer warps only: each issues its own copies

struct SplitLayout {
    size_t ring, ckey, cidx, scratch, wx, xf, perm, ctrl, total;
};

// Scratch: the warm-up's 2048-bin histogram, the final select's histogram, and the
// compaction's hole and fill lists (k uint16 each).
__host__ __device__ inline size_t split_scratch_bytes(int k) {
    const size_t lists = static_cast<size_t>(4) * k;
    return align_up(lists > kBins * 4 ? lists : static_cast<size_t>(kBins) * 4, 16);
}

// wm: group maxima per CTA in the warm-up (a multiple of 256).  Regions that other CTAs
// write into (wx: the warm-up's maxima and each CTA's largest, xf: two rounds of the final
// select's uint16 histograms) are separate from the copy ring and from each other, so a CTA that runs
// ahead never writes over memory a slower CTA still uses.
__host__ __device__ inline SplitLayout split_layout(int es, int chunk, int stages, int cap, int G, int wm, int k,
                                                   int perm_cap) {
    SplitLayout L;
    size_t off = 0;
    L.ring = off;
    off += align_up(static_cast<size_t>(stages) * chunk * es, 128);
    L.ckey = off;
    off += align_up(static_cast<size_t>(cap) * es, 16);
    L.cidx = off;
    off += align_up(static_cast<size_t>(cap) * 4, 16);
    L.scratch = off;
    off += split_scratch_bytes(k);
    L.wx = off;  // G rows of wm maxima, each followed by a 16-byte slot for its largest
    off += static_cast<size_t>(G) * (static_cast<size_t>(wm) * es + 16);
    L.xf = off;
    off += align_up(static_cast<size_t>(4) * kXBins * G, 16);
    L.perm = off;
    off += align_up(static_cast<size_t>(perm_cap) * 4, 16);
    L.ctrl = off;
    off += align_up(sizeof(Ctrl), 16);
    L.total = off;
    return L;
}

// Bits of the float compare threshold for key T (see the file comment).  No threshold:
// a NaN, against which every value compares unordered.
template <typename KeyT>
__device__ __forceinline__ uint32_t compare_bits(bool has, uint32_t T) {
    if (sizeof(KeyT) == 2) {
        uint32_t t = 0x7FC0u;
        if (has) {
            const uint32_t b = unkey_bf16(T);
            if ((b & 0x7F80u) == 0x7F80u && (b & 0x7Fu)) t = (b & 0x8000u) ? 0x7FC0u : 0x7F80u;
            else if (b == 0x8000u) t = 0x8001u;
            else t = b;
        }
        return t | (t << 16);
    } else {
        if (!has) return 0x7FC00000u;
        const uint32_t b = unkey_f32(T);
        if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x7FFFFFu)) return (b & 0x80000000u) ? 0x7FC00000u : 0x7F800000u;
        if (b == 0x80000000u) return 0x80000001u;
        return b;
    }
}

// Bounded wait with cluster-scope acquire (data other CTAs pushed is visible after it).
__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity, Ctrl* ctrl) {
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<volatile int*>(&ctrl->abort)) return false;
        if (clock64() - t0 > kSpinLimit) {
            set_status(kErrTimeout);
            *reinterpret_cast<volatile int*>(&ctrl->abort) = 1;
            return false;
        }
    }
}

// bf16x2 / f32 maximum that ignores NaN operands (a NaN only when both are NaN).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Key of the largest non-NaN value of a packed word set reduced with max_bf16x2 (both
// halves) or fmaxf, or 0 when only NaNs were seen.  Never above the largest key of the
// values it came from (it is one of them, or a NaN mapped to 0).
template <typename KeyT>
__device__ __forceinline__ uint32_t max_word_key(uint32_t m) {
    if (sizeof(KeyT) == 2) {
        const uint32_t lo = m & 0xFFFFu, hi = m >> 16;
        const uint32_t klo = (lo & 0x7FFFu) > 0x7F80u ? 0u : key_bf16(lo);
        const uint32_t khi = (hi & 0x7FFFu) > 0x7F80u ? 0u : key_bf16(hi);
        return max(klo, khi);
    } else {
        return (m & 0x7FFFFFFFu) > 0x7F800000u ? 0u : key_f32(m);
    }
}

// Warm-up group maxima of one thread: its vectors t, t + NC, ... (VT <= NV of them) of
// the ww sampled chunks (cvec vectors each; nvw[q] whole vectors in chunk q), in groups
// of 2^gsh vectors; gk[g] is the key of group g's largest value (0: none).  NV is 4 or 8
// so that small samples run the short loop.
template <typename KeyT, int NV>
__device__ __forceinline__ void warm_maxima(const uint4* v0, int tid, int cvec, int ww, int VT, int gsh, bool gotw,
                                            const int (&nvw)[8], uint32_t (&gk)[4]) {
    constexpr int ES = sizeof(KeyT);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int v = tid + j * kSplitThreads;
        int q = 0;
#pragma unroll
        for (int t = 1; t < NV; ++t) q += v >= t * cvec ? 1 : 0;
        int nv = nvw[0];
#pragma unroll
        for (int t = 1; t < NV; ++t)
            if (q == t) nv = nvw[t];
        if (gotw && j < VT && q < ww && v - q * cvec < nv) {
            const uint4 x = v0[v];
            uint32_t m;
            if (ES == 2) {
                m = max_bf16x2(max_bf16x2(x.x, x.y), max_bf16x2(x.z, x.w));
            } else {
                m = __float_as_uint(fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)),
                                          fmaxf(__uint_as_float(x.z), __uint_as_float(x.w))));
            }
            const uint32_t kk = max_word_key<KeyT>(m);  // keys keep the value order
            const int g = j >> gsh;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (g == r) gk[r] = max(gk[r], kk);
        }
    }
}

// The same for samples of 9..16 vectors per thread (rows streamed through the ring): up
// to 8 chunks, groups of 2^gsh consecutive vectors of the thread, each group's key stored
// straight to out[g] for g < R (no register array of groups).  Returns the largest key
// stored.
template <typename KeyT>
__device__ __forceinline__ uint32_t warm_maxima16(const uint4* v0, int tid, int cvec, int ww, int VT, int gsh, int R,
                                              bool gotw, const int (&nvw)[8], KeyT* out) {
    constexpr int ES = sizeof(KeyT);
    uint32_t cur = 0u, top = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int v = tid + j * kSplitThreads;
        int q = 0;
#pragma unroll
        for (int t = 1; t < 8; ++t) q += v >= t * cvec ? 1 : 0;
        int nv = nvw[0];
#pragma unroll
        for (int t = 1; t < 8; ++t)
            if (q == t) nv = nvw[t];
        if (gotw && j < VT && q < ww && v - q * cvec < nv) {
            const uint4 x = v0[v];
            uint32_t m;
            if (ES == 2) {
                m = max_bf16x2(max_bf16x2(x.x, x.y), max_bf16x2(x.z, x.w));
            } else {
                m = __float_as_uint(fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)),
                                          fmaxf(__uint_as_float(x.z), __uint_as_float(x.w))));
            }
            cur = max(cur, max_word_key<KeyT>(m));
        }
        if (((j + 1) & ((1 << gsh) - 1)) == 0) {
            const int g = j >> gsh;
            if (g < R) {
                out[g] = static_cast<KeyT>(cur);
                top = max(top, cur);
            }
            cur = 0u;
        }
    }
    return top;
}

// The warm-up maxima when every sampled chunk is whole and the sample a multiple of the
// CTA's threads (the usual case): no per-vector chunk bookkeeping, and each group's
// values are reduced packed (NaNs ignored) and keyed once.  Same results as warm_maxima
// and warm_maxima16.
template <typename KeyT>
__device__ __forceinline__ uint32_t packed_max(uint32_t a, uint32_t b) {
    if (sizeof(KeyT) == 2) return max_bf16x2(a, b);
    return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
}
template <typename KeyT>
__device__ __forceinline__ uint32_t vec_max(const uint4& x) {
    return packed_max<KeyT>(packed_max<KeyT>(x.x, x.y), packed_max<KeyT>(x.z, x.w));
}
template <typename KeyT, int NV>
__device__ __forceinline__ void warm_maxima_whole(const uint4* v0, int tid, int VT, int gsh, uint32_t (&gk)[4]) {
    constexpr uint32_t kNaN = sizeof(KeyT) == 2 ? 0x7FC07FC0u : 0x7FC00000u;  // (ignored by the max)
    uint32_t acc[4] = {kNaN, kNaN, kNaN, kNaN};
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        if (j < VT) {
            const uint32_t m = vec_max<KeyT>(v0[tid + j * kSplitThreads]);
            const int g = j >> gsh;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (g == r) acc[r] = packed_max<KeyT>(acc[r], m);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) gk[r] = max_word_key<KeyT>(acc[r]);
}
template <typename KeyT>
__device__ __forceinline__ uint32_t warm_maxima16_whole(const uint4* v0, int tid, int stride, int VT, int gsh, int R,
                                                        KeyT* out) {
    constexpr uint32_t kNaN = sizeof(KeyT) == 2 ? 0x7FC07FC0u : 0x7FC00000u;
    uint32_t acc = kNaN, top = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (j < VT) acc = packed_max<KeyT>(acc, vec_max<KeyT>(v0[tid + j * stride]));
        if (((j + 1) & ((1 << gsh) - 1)) == 0) {
            const int g = j >> gsh;
            if (g < R) {
                const uint32_t kk = max_word_key<KeyT>(acc);
                out[g] = static_cast<KeyT>(kk);
                top = max(top, kk);
            }
            acc = kNaN;
        }
    }
    return top;
}

// The pivot of a final-select pass, found by every warp on its own (no barrier).  The
// cluster's histogram is G rows of kXBins 16-bit counts (pairs in 32-bit words), row c
// from the CTA of rank c; lane l owns bins [16l, 16l + 16), higher bins holding larger
// keys.  For the bin bstar holding the krem-th largest key (-1 when all bins together
// hold fewer): the keys in the bins above it (above), those held by CTAs of rank below
// crank (low_above), and the bin's keys held by CTAs of rank below crank (eq_lower).
// With bstar = -1, above and low_above count every key.
struct XPivot {
    int bstar;
    uint32_t above, low_above, eq_lower;
};
__device__ __forceinline__ XPivot warp_pivot_x(const uint32_t* rows, int G, int crank, uint32_t krem, int lane) {
    uint32_t ca[16], cl[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) ca[j] = cl[j] = 0u;
#pragma unroll 4
    for (int c = 0; c < G; ++c) {
        if (c == crank) {
#pragma unroll
            for (int j = 0; j < 16; ++j) cl[j] = ca[j];
        }
        const uint4* r4 = reinterpret_cast<const uint4*>(rows + static_cast<size_t>(c) * (kXBins / 2)) + 2 * lane;
        const uint4 a = r4[0], b = r4[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            ca[2 * j] += w[j] & 0xFFFFu;
            ca[2 * j + 1] += w[j] >> 16;
        }
    }
    uint32_t t = 0u, tl = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        t += ca[j];
        tl += cl[j];
    }
    uint32_t sf = t, sl = tl;  // inclusive suffix sums over lanes >= lane
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_down_sync(0xFFFFFFFFu, sf, d);
        const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, sl, d);
        if (lane + d < 32) {
            sf += u;
            sl += v;
        }
    }
    XPivot r;
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, sf >= krem);
    if (hit == 0u) {
        r.bstar = -1;
        r.above = __shfl_sync(0xFFFFFFFFu, sf, 0);
        r.low_above = __shfl_sync(0xFFFFFFFFu, sl, 0);
        r.eq_lower = 0u;
        return r;
    }
    const int L = 31 - __clz(hit);
    uint32_t acc = sf - t, lacc = sl - tl, eql = 0u;  // keys in the lanes above
    int jb = 0;
    bool found = false;
#pragma unroll
    for (int j = 15; j >= 0; --j) {
        if (!found) {
            if (acc + ca[j] >= krem) {
                found = true;
                jb = j;
                eql = cl[j];
            } else {
                acc += ca[j];
                lacc += cl[j];
            }
        }
    }
    r.bstar = 16 * L + __shfl_sync(0xFFFFFFFFu, jb, L);
    r.above = __shfl_sync(0xFFFFFFFFu, acc, L);
    r.low_above = __shfl_sync(0xFFFFFFFFu, lacc, L);
    r.eq_lower = __shfl_sync(0xFFFFFFFFu, eql, L);
    return r;
}

// Calls f(key) for each key of G rows of wm keys, each row followed by one 16-byte vector
// that is skipped (wm / keys-per-vector a power of two, `keys` 16-byte aligned), the CTA's
// threads taking one 16-byte vector each at a time: the loads of a thread's keys do not
// wait on one another.
template <typename KeyT, typename F>
__device__ __forceinline__ void each_key(const KeyT* keys, int G, int wm, int tid, F&& f) {
    constexpr int KPV = 16 / static_cast<int>(sizeof(KeyT));
    const int W = wm / KPV, wl = 31 - __clz(W);  // vectors per row
    const uint4* v4 = reinterpret_cast<const uint4*>(keys);
    for (int j = tid; j < G * W; j += kSplitThreads) {
        const uint4 v = v4[(j >> wl) * (W + 1) + (j & (W - 1))];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (sizeof(KeyT) == 2) {
                f(w[i] & 0xFFFFu);
                f(w[i] >> 16);
            } else {
                f(w[i]);
            }
        }
    }
}

// The bucket of the kk-th largest count among 2048, found by the whole CTA (kSplitThreads
// threads): thread t sums buckets [8t, 8t + 8), suffix sums over the threads (a shuffle
// scan in each warp, then the warps' totals through `wt`) pick the thread whose buckets
// hold it, and that thread walks its eight.  Sets ctrl->bstar (-1 when all buckets
// together hold fewer than kk), ctrl->above (the count in buckets above it; all of them
// when none) and ctrl->bcount (the total); for a second rank k2 > 0, ctrl->spec_b,
// spec_above and spec_c (the bucket's own count) the same way.  Every thread calls it; it
// ends with a barrier.
__device__ __forceinline__ void cta_bucket_2048(const uint32_t* hist, uint32_t kk, uint32_t k2, int tid, uint32_t* wt,
                                                Ctrl* ctrl) {
    static_assert(kBins == 8 * kSplitThreads, "eight buckets per thread");
    const int lane = tid & 31, warp = tid >> 5;
    const uint4 a = reinterpret_cast<const uint4*>(hist)[2 * tid];
    const uint4 b = reinterpret_cast<const uint4*>(hist)[2 * tid + 1];
    const uint32_t c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t t = c[0] + c[1] + c[2] + c[3] + c[4] + c[5] + c[6] + c[7];
    uint32_t sf = t;  // buckets of this warp's threads >= tid
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_down_sync(0xFFFFFFFFu, sf, d);
        if (lane + d < 32) sf += u;
    }
    if (lane == 0) wt[warp] = sf;
    __syncthreads();
    uint32_t tot = 0u, up = 0u;
#pragma unroll
    for (int w = 0; w < kSplitThreads / 32; ++w) {
        const uint32_t x = wt[w];
        tot += x;
        up += w > warp ? x : 0u;
    }
    const uint32_t incl = sf + up;  // buckets of threads >= tid
    // the bucket of rank r when this thread holds it: index, count above, own count
    const auto locate = [&](uint32_t r, int& bs, uint32_t& ab, uint32_t& cnt) -> bool {
        if (!(incl >= r && incl - t < r)) return false;
        uint32_t acc = incl - t;
        bs = 8 * tid;
        cnt = 0u;
        bool found = false;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
            if (!found) {
                if (acc + c[j] >= r) {
                    found = true;
                    bs = 8 * tid + j;
                    cnt = c[j];
                } else {
                    acc += c[j];
                }
            }
        }
        ab = acc;
        return true;
    };
    int bs;
    uint32_t ab, cnt;
    if (locate(kk, bs, ab, cnt)) {
        ctrl->bstar = bs;
        ctrl->above = ab;
    }
    if (k2 && locate(k2, bs, ab, cnt)) {
        ctrl->spec_b = bs;
        ctrl->spec_above = ab;
        ctrl->spec_c = cnt;
    }
    if (tid == 0) {
        if (tot < kk) {
            ctrl->bstar = -1;
            ctrl->above = tot;
        }
        if (k2 && tot < k2) ctrl->spec_b = -1;
        ctrl->bcount = tot;
    }
    __syncthreads();
}

// warp_pivot_x's result found by the whole CTA: thread t owns bins 2t and 2t + 1 (word t
// of every CTA's row), suffix sums go through `wt` as in cta_bucket_2048, and the thread
// holding the krem-th largest key writes the pivot to ctrl->fp_tot[0..3] (bstar, above,
// low_above, eq_lower).  Every thread calls it; it ends with a barrier.
__device__ __forceinline__ void cta_pivot_x(const uint32_t* rows, int G, int crank, uint32_t krem, int tid,
                                            uint32_t* wt, Ctrl* ctrl) {
    static_assert(kXBins == 2 * kSplitThreads, "two bins per thread");
    constexpr int XW = kXBins / 2;
    constexpr int NW = kSplitThreads / 32;
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t a0 = 0u, a1 = 0u, l0 = 0u, l1 = 0u;  // bins 2t, 2t + 1: all CTAs, CTAs of rank below crank
#pragma unroll 4
    for (int c = 0; c < G; ++c) {
        if (c == crank) {
            l0 = a0;
            l1 = a1;
        }
        const uint32_t w = rows[static_cast<size_t>(c) * XW + tid];
        a0 += w & 0xFFFFu;
        a1 += w >> 16;
    }
    const uint32_t t = a0 + a1, tl = l0 + l1;
    uint32_t sf = t, sl = tl;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_down_sync(0xFFFFFFFFu, sf, d);
        const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, sl, d);
        if (lane + d < 32) {
            sf += u;
            sl += v;
        }
    }
    if (lane == 0) {
        wt[warp] = sf;
        wt[NW + warp] = sl;
    }
    __syncthreads();
    uint32_t tot = 0u, totl = 0u, up = 0u, upl = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t x = wt[w], y = wt[NW + w];
        tot += x;
        totl += y;
        up += w > warp ? x : 0u;
        upl += w > warp ? y : 0u;
    }
    const uint32_t incl = sf + up, incll = sl + upl;  // keys in bins >= 2t
    if (incl >= krem && incl - t < krem) {
        uint32_t acc = incl - t, lacc = incll - tl;
        int bs = 2 * tid + 1;
        uint32_t eql = l1;
        if (acc + a1 < krem) {
            acc += a1;
            lacc += l1;
            bs = 2 * tid;
            eql = l0;
        }
        ctrl->fp_tot[0] = static_cast<uint32_t>(bs);
        ctrl->fp_tot[1] = acc;
        ctrl->fp_tot[2] = lacc;
        ctrl->fp_tot[3] = eql;
    }
    if (tid == 0 && tot < krem) {
        ctrl->fp_tot[0] = static_cast<uint32_t>(-1);
        ctrl->fp_tot[1] = tot;
        ctrl->fp_tot[2] = totl;
        ctrl->fp_tot[3] = 0u;
    }
    __syncthreads();
}

// Counts a key in the final select's first histogram (kXBins 16-bit counts in pairs):
// keys from `edge` up, in bins of 2^s keys, the last bin open-ended.
__device__ __forceinline__ void xhist_add(uint32_t* xh, uint32_t key, uint32_t edge, int s) {
    if (key >= edge) {
        uint32_t d = (key - edge) >> s;
        d = d < kXBins - 1 ? d : kXBins - 1;
        atomicAdd(&xh[d >> 1], 1u << ((d & 1u) * 16u));
    }
}

// A dense pass of a row held whole may be shared out: slice s holds vectors 2s and 2s + 1 of
// each lane (kDenseSlices slices cover a pass of 512 vectors).  Whoever claims a slice
// compares it again, reserves its hits' slots from the pass's reservation and appends them
// position by position; a lane's elements are neighbours in the row, so it counts runs of
// one histogram bin (sorted or clustered rows) with one atomic per run.
constexpr int kDenseSlices = 8;
constexpr int kJobOpen = 1 << 16;  // added to Ctrl::done_warps while a dense pass is shared out

template <typename KeyT>
__device__ __forceinline__ void dense_slice(const uint8_t* stage, int p0, int nvec, int s, uint32_t tb, uint32_t col0,
                                            KeyT* ckey, uint32_t* cidx, Ctrl* ctrl, int lane, uint32_t& tmax,
                                            uint32_t* xh, uint32_t hedge, int hs) {
    constexpr int ES = sizeof(KeyT);
    constexpr int EPV = 16 / ES;
    const uint4* vec = reinterpret_cast<const uint4*>(stage);
    uint4 xv[2];
    uint32_t mk[2], c = 0u;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int v = p0 + lane + 32 * (2 * s + t);
        xv[t] = make_uint4(0u, 0u, 0u, 0u);
        mk[t] = 0u;
        if (v < nvec) {
            xv[t] = vec[v];
            if (ES == 2)  // element 2q at bit q, element 2q + 1 at bit 16 + q
                mk[t] = (set_gtu_bf16x2(xv[t].x, tb) & 0x10001u) | (set_gtu_bf16x2(xv[t].y, tb) & 0x20002u) |
                        (set_gtu_bf16x2(xv[t].z, tb) & 0x40004u) | (set_gtu_bf16x2(xv[t].w, tb) & 0x80008u);
            else  // element q at bit q
                mk[t] = (set_gtu_f32(xv[t].x, tb) & 1u) | (set_gtu_f32(xv[t].y, tb) & 2u) |
                        (set_gtu_f32(xv[t].z, tb) & 4u) | (set_gtu_f32(xv[t].w, tb) & 8u);
        }
        c += static_cast<uint32_t>(__popc(mk[t]));
    }
    const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, c);
    if (tot == 0u) return;
    uint32_t run = 0u;
    if (lane == 0) run = atomicAdd(reinterpret_cast<unsigned int*>(&ctrl->job_cursor), tot);
    run = __shfl_sync(0xFFFFFFFFu, run, 0);
    const uint32_t ltm = lanemask_lt();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int v = p0 + lane + 32 * (2 * s + t);
        const uint32_t xw[4] = {xv[t].x, xv[t].y, xv[t].z, xv[t].w};
        const uint32_t cb = col0 + static_cast<uint32_t>(v * EPV);  // row column of the vector's first element
        uint32_t rb = 0u, rc = 0u;  // the current run's histogram bin and length
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int bit = ES == 2 ? (e & 1) * 16 + (e >> 1) : e;
            const uint32_t raw = ES == 2 ? ((e & 1) ? (xw[e >> 1] >> 16) : (xw[e >> 1] & 0xFFFFu)) : xw[e];
            const bool hit = (mk[t] >> bit) & 1u;
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, hit);
            if (hit) {
                const uint32_t slot = run + static_cast<uint32_t>(__popc(bal & ltm));
                const uint32_t key = ES == 2 ? key_bf16(raw) : key_f32(raw);
                ckey[slot] = static_cast<KeyT>(key);
                cidx[slot] = cb + static_cast<uint32_t>(e);
                tmax = max(tmax, key);
                if (key >= hedge) {
                    uint32_t b = (key - hedge) >> hs;
                    b = b < kXBins - 1 ? b : kXBins - 1;
                    if (rc != 0u && b != rb) {
                        atomicAdd(&xh[rb >> 1], rc << ((rb & 1u) * 16u));
                        rc = 0u;
                    }
                    rb = b;
                    ++rc;
                }
            }
            run += static_cast<uint32_t>(__popc(bal));
        }
        if (rc != 0u) atomicAdd(&xh[rb >> 1], rc << ((rb & 1u) * 16u));
    }
}

// Claims and appends slices of the open dense pass until none is left; returns the largest
// key this lane appended (0: none).  Never waits: a slice, once claimed, is finished by its
// claimant.  Out of line: it runs rarely, and the chunk loop keeps its registers.
template <typename KeyT>
__device__ __noinline__ uint32_t dense_claim(KeyT* ckey, uint32_t* cidx, Ctrl* ctrl, int lane, uint32_t* xh,
                                             uint32_t hedge, int hs) {
    uint32_t mx = 0u;
    while (true) {
        int s = 0;
        if (lane == 0) s = atomicAdd(&ctrl->job_next, 1);
        s = __shfl_sync(0xFFFFFFFFu, s, 0);
        if (s >= kDenseSlices) return mx;
        __threadfence_block();
        const volatile Ctrl* vc = ctrl;
        dense_slice<KeyT>(vc->job_stage, vc->job_p0, vc->job_nvec, s, vc->job_tb, vc->job_col0, ckey, cidx, ctrl,
                          lane, mx, xh, hedge, hs);
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            atomicSub(&ctrl->job_left, 1);
        }
    }
}

// The owner's side of a shared dense pass (slots [base, base + nbits) already reserved):
// takes the job if no other is open, claims slices with the helpers and waits for theirs.
// Returns 1 + the largest key this lane appended, or 0 when another job was open (the
// caller then appends the pass alone).  Out of line, like dense_claim.
template <typename KeyT>
__device__ __noinline__ uint64_t dense_share(const uint8_t* stage, int p0, int nvec, uint32_t tb, uint32_t col0,
                                             uint32_t base, KeyT* ckey, uint32_t* cidx, Ctrl* ctrl, int lane,
                                             uint32_t* xh, uint32_t hedge, int hs) {
    int own = 0;
    if (lane == 0) own = atomicCAS(&ctrl->job_on, 0, 1) == 0;
    if (!__shfl_sync(0xFFFFFFFFu, own, 0)) return 0u;
    if (lane == 0) {
        ctrl->job_stage = stage;
        ctrl->job_p0 = p0;
        ctrl->job_nvec = nvec;
        ctrl->job_tb = tb;
        ctrl->job_col0 = col0;
        ctrl->job_cursor = static_cast<int>(base);
        ctrl->job_left = kDenseSlices;
        __threadfence_block();
        atomicExch(&ctrl->job_next, 0);          // open
        atomicAdd(&ctrl->done_warps, kJobOpen);  // (waiting warps look here)
    }
    __syncwarp();
    const uint32_t mx = dense_claim<KeyT>(ckey, cidx, ctrl, lane, xh, hedge, hs);
    const long long t0 = clock64();
    while (true) {  // the slices other warps claimed
        int left = 0;
        if (lane == 0) left = *reinterpret_cast<volatile int*>(&ctrl->job_left);
        if (__shfl_sync(0xFFFFFFFFu, left, 0) <= 0) break;
        if (clock64() - t0 > kSpinLimit) {  // cannot happen: a claimed slice never waits
            if (lane == 0) {
                set_status(kErrTimeout);
                *reinterpret_cast<volatile int*>(&ctrl->abort) = 1;
            }
            break;
        }
    }
    __threadfence_block();
    if (lane == 0) {
        atomicSub(&ctrl->done_warps, kJobOpen);
        *reinterpret_cast<volatile int*>(&ctrl->job_on) = 0;
    }
    __syncwarp();
    return 1ull + mx;
}

// One warp filters vectors [0, nvec) of a staged chunk (plus, when tail_n > 0, the row's
// last tail_n elements from global memory) against the compare bits tb and appends the
// survivors.  Work goes in passes of 512 vectors (16 per lane, lane l taking l, l + 32,
// ...); `pass` is the first pass to run and, when a reservation does not fit the buffer,
// the pass to resume after the compaction (the function then returns false and has
// written nothing of that pass).
//
// Hit masks: a compare leaves all-ones or zero per element (per 16-bit half for bf16), and
// one and-or per compared word keeps one bit of it, so a vector costs four compares and
// four logic ops.  bf16: word w holds vectors 4w..4w+3; bit h*16 + 4*(i%4) + q is element
// 2q+h of vector i.  fp32: word w holds vectors 8w..8w+7; bit 4*(i%8) + q is element q.
// Sparse passes append in two steps: each lane writes the chunk columns of its hits into
// its run of the reserved index slots, then the warp walks the reserved slots together
// (contiguous accesses) to store each hit's key and its row column.  Dense passes (a third
// or more of the elements pass) skip the per-lane bit loop: the warp walks the pass's
// element positions, one ballot each, and its lanes' hits take consecutive slots; on rows
// held whole (SHARE) the pass is shared out in slices with warps that have nothing to
// filter (dense_share).  The row's tail elements take the last slots.
template <typename KeyT, bool SHARE>
__device__ __forceinline__ bool warp_chunk(const uint8_t* stage, int nvec, uint32_t col0, const char* xrow,
                                           int64_t tail_first, int tail_n, uint32_t tb, KeyT* ckey, uint32_t* cidx,
                                           Ctrl* ctrl, uint32_t cap, int lane, int& pass, uint32_t& tmax,
                                           uint32_t* xh, uint32_t hedge, int hs) {
    constexpr int ES = sizeof(KeyT);
    constexpr int EPV = 16 / ES;          // elements per vector
    constexpr int MW = 16 * EPV / 32;     // mask words per pass and lane
    constexpr int VPW = 16 / MW;          // vectors per mask word
    const uint4* vec = reinterpret_cast<const uint4*>(stage);
    const int npass = nvec > 0 ? (nvec + 511) / 512 : (tail_n > 0 ? 1 : 0);
    for (; pass < npass; ++pass) {
        const int p0 = pass * 512;
        uint32_t m[MW];
#pragma unroll
        for (int w = 0; w < MW; ++w) m[w] = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int v = p0 + lane + 32 * i;
            if (v < nvec) {
                const uint4 x = vec[v];
                uint32_t& mw = m[i / VPW];
                const int sh = 4 * (i % VPW);
                if (ES == 2) {
                    const uint32_t c = 0x10001u << sh;
                    mw |= set_gtu_bf16x2(x.x, tb) & c;
                    mw |= set_gtu_bf16x2(x.y, tb) & (c << 1);
                    mw |= set_gtu_bf16x2(x.z, tb) & (c << 2);
                    mw |= set_gtu_bf16x2(x.w, tb) & (c << 3);
                } else {
                    const uint32_t c = 1u << sh;
                    mw |= set_gtu_f32(x.x, tb) & c;
                    mw |= set_gtu_f32(x.y, tb) & (c << 1);
                    mw |= set_gtu_f32(x.z, tb) & (c << 2);
                    mw |= set_gtu_f32(x.w, tb) & (c << 3);
                }
            }
        }
        // the row's last elements (fewer than 16 bytes), one per lane, in the first pass
        uint32_t tkey = 0u;
        bool thit = false;
        if (pass == 0 && lane < tail_n) {
            if (ES == 2) {
                const uint32_t h = reinterpret_cast<const uint16_t*>(xrow)[tail_first + lane];
                thit = (set_gtu_bf16x2(h | (h << 16), tb) & 1u) != 0u;
                tkey = key_bf16(h);
            } else {
                const uint32_t h = reinterpret_cast<const uint32_t*>(xrow)[tail_first + lane];
                thit = set_gtu_f32(h, tb) != 0u;
                tkey = key_f32(h);
            }
        }
        uint32_t c = 0u;
#pragma unroll
        for (int w = 0; w < MW; ++w) c += __popc(m[w]);
        const uint32_t incl = warp_incl_scan(c, lane);
        const uint32_t nbits = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const uint32_t tmask = __ballot_sync(0xFFFFFFFFu, thit);
        const uint32_t tot = nbits + static_cast<uint32_t>(__popc(tmask));
        if (tot == 0u) continue;
        uint32_t base = 0u;
        int fits = 1;
        if (lane == 0) {
            base = atomicAdd(reinterpret_cast<unsigned int*>(&ctrl->cnt), tot);
            if (base + tot > cap) {
                fits = 0;
                atomicMin(&ctrl->fail_base, static_cast<int>(base));
                *reinterpret_cast<volatile int*>(&ctrl->compact_req) = 1;
            }
        }
        if (!__shfl_sync(0xFFFFFFFFu, fits, 0)) return false;
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        uint64_t shared = 0u;  // a dense pass of a row held whole, shared out when no other is
        if (SHARE && nbits * 3u >= 512u * EPV)
            shared = dense_share<KeyT>(stage, p0, nvec, tb, col0, base, ckey, cidx, ctrl, lane, xh, hedge, hs);
        if (shared) {
            tmax = max(tmax, static_cast<uint32_t>(shared - 1u));
        } else if (nbits * 3u >= 512u * EPV) {
            // dense pass (a third or more of its elements pass): the warp writes its hits
            // position by position, lanes in order, to consecutive slots -- no per-lane bit
            // loop, no bank conflicts
            const uint32_t ltm = lanemask_lt();
            uint32_t run = base;
#pragma unroll 1
            for (int i = 0; i < 16; ++i) {
                const int v = p0 + lane + 32 * i;
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                if (v < nvec) x = vec[v];
                const int wsel = i / VPW;
                uint32_t mw = m[0];
#pragma unroll
                for (int w = 1; w < MW; ++w)
                    if (wsel == w) mw = m[w];
                const int sh = 4 * (i % VPW);
                const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
                const uint32_t cb = static_cast<uint32_t>(v * EPV);  // column of the vector's first element
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    int bit;
                    uint32_t raw;
                    if (ES == 2) {
                        bit = (e & 1) * 16 + sh + (e >> 1);
                        raw = (e & 1) ? (xw[e >> 1] >> 16) : (xw[e >> 1] & 0xFFFFu);
                    } else {
                        bit = sh + e;
                        raw = xw[e];
                    }
                    const bool hit = (mw >> bit) & 1u;
                    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, hit);
                    if (hit) {
                        const uint32_t slot = run + static_cast<uint32_t>(__popc(bal & ltm));
                        const uint32_t key = ES == 2 ? key_bf16(raw) : key_f32(raw);
                        ckey[slot] = static_cast<KeyT>(key);
                        cidx[slot] = col0 + cb + static_cast<uint32_t>(e);
                        tmax = max(tmax, key);
                        xhist_add(xh, key, hedge, hs);
                    }
                    run += static_cast<uint32_t>(__popc(bal));
                }
            }
        } else {  // sparse pass
            // step 1: the chunk columns of this lane's hits
            uint32_t pos = base + incl - c;
            const int cl = (p0 + lane) * EPV;  // column of the lane's first element in the pass
#pragma unroll
            for (int w = 0; w < MW; ++w) {
                uint32_t mm = m[w];
                while (mm) {
                    const int bb = __ffs(mm) - 1;
                    mm &= mm - 1u;
                    int col;
                    if (ES == 2) col = cl + 32 * EPV * (w * VPW + ((bb & 15) >> 2)) + 2 * (bb & 3) + (bb >> 4);
                    else col = cl + 32 * EPV * (w * VPW + (bb >> 2)) + (bb & 3);
                    cidx[pos++] = static_cast<uint32_t>(col);
                }
            }
            __syncwarp();
            // step 2: keys and row columns, the warp's slots in order
            for (uint32_t j = static_cast<uint32_t>(lane); j < nbits; j += 32u) {
                const uint32_t col = cidx[base + j];
                const uint32_t raw = ES == 2 ? reinterpret_cast<const uint16_t*>(stage)[col]
                                             : reinterpret_cast<const uint32_t*>(stage)[col];
                const uint32_t key = ES == 2 ? key_bf16(raw) : key_f32(raw);
                ckey[base + j] = static_cast<KeyT>(key);
                cidx[base + j] = col0 + col;
                tmax = max(tmax, key);
                xhist_add(xh, key, hedge, hs);
            }
        }
        if (thit) {
            const uint32_t slot = base + nbits + static_cast<uint32_t>(__popc(tmask & lanemask_lt()));
            ckey[slot] = static_cast<KeyT>(tkey);
            cidx[slot] = static_cast<uint32_t>(tail_first + lane);
            tmax = max(tmax, tkey);
            xhist_add(xh, tkey, hedge, hs);
        }
    }
    return true;
}

// A compaction that every consumer thread of a split-row CTA joins.  The buffer's slots
// [0, min(first failed reservation, count)) are cut down, the threshold rises and is pushed
// to every CTA of the cluster (and to the row's global word gT, tagged with the call's
// epoch, when the row spans clusters).  Returns the new threshold.
//   The first final histogram counts every key of those slots (bins of 2^hs0 keys from
// hedge up).  Its bin b* holding the k-th largest key gives a cut: the keys of bins b*
// and above, at least k of them, stay (in slot order, moved down one tile at a time) and
// the threshold becomes the bin's smallest key less one.  When that keeps too many keys
// (a wide or crowded bin) or b* is the lowest bin, the buffer is cut to exactly the k
// largest keys instead (a radix select) and the histogram is counted anew.  Either way at
// least `room` slots (one chunk, the most one pass reserves) are free afterwards, so the
// pass that failed to reserve, retried, fits unless other warps' passes took the room
// first: every compaction is followed by at least one appended pass.  Out of line: it
// runs rarely, and its code then stays out of the chunk loop's instruction stream.
template <typename KeyT>
__device__ __noinline__ uint32_t split_compaction(KeyT* ckey, uint32_t* cidx, uint32_t* hist, Ctrl* ctrl, int cap,
                                                  int room, int k, uint32_t tmax, int tid, bool hasT, uint32_t T,
                                                  uint32_t* xh0,
                                                  uint32_t hedge, int hs0, int G, uint32_t* shT,
                                                  unsigned long long* gT, uint32_t epoch) {
    constexpr int NC = kSplitThreads;
    const int lane = tid & 31;
    named_bar_sync(2, NC);
    const int fb = *reinterpret_cast<volatile int*>(&ctrl->fail_base);
    const int cn = *reinterpret_cast<volatile int*>(&ctrl->cnt);
    int n = fb < cn ? fb : cn;
    n = n < cap ? n : cap;  // (a bound only: reservations never pass cap)
    // No pass appended since the last compaction: another would change nothing.  This
    // cannot happen (see above); if it did, the CTA reports it and stops instead of looping.
    const bool stuck = n == ctrl->last_kept;
    if (tid < 32 && !stuck) {
        const XPivot r = warp_pivot_x(xh0, 1, 0, static_cast<uint32_t>(k), lane);
        if (lane == 0) {
            int cb = -1;
            uint32_t keep = 0u;
            if (r.bstar > 0) {
                const uint64_t lo = static_cast<uint64_t>(hedge) + (static_cast<uint64_t>(r.bstar) << hs0);
                if (lo - 1u <= (sizeof(KeyT) == 2 ? 0xFFFFull : 0xFFFFFFFFull)) {
                    cb = r.bstar;
                    keep = r.above + reinterpret_cast<const uint16_t*>(xh0)[r.bstar];
                }
            }
            ctrl->cut_bin = cb;
            ctrl->cut_keep = keep;
        }
    }
    named_bar_sync(2, NC);
    if (tid == 0) {
        ctrl->compact_req = 0;
        ctrl->fail_base = 0x7FFFFFFF;
        ctrl->raise_mark = 0u;
    }
    if (stuck) {
        if (tid == 0) {
            set_status(kErrInternal);
            *reinterpret_cast<volatile int*>(&ctrl->abort) = 1;
        }
        named_bar_sync(2, NC);
        return T;
    }
    const int cb = ctrl->cut_bin;
    const uint32_t keep = ctrl->cut_keep;
    uint32_t nt;
    if (cb > 0 && keep <= static_cast<uint32_t>(k + (cap - k) / 2) &&
        keep + static_cast<uint32_t>(room) <= static_cast<uint32_t>(cap)) {
        const uint32_t lo = hedge + (static_cast<uint32_t>(cb) << hs0);
        constexpr int PER = 8;  // (4: 2.2 us more per call on sampler rows at k = 4096; 16: slower on sorted rows)
        uint32_t off = 0u;
        for (int t0 = 0, it = 0; t0 < n; t0 += NC * PER, ++it) {
            KeyT kk[PER];
            uint32_t ii[PER];
            uint32_t c = 0u, f = 0u;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int i = t0 + tid + NC * j;
                kk[j] = 0;
                ii[j] = 0u;
                if (i < n) {
                    kk[j] = ckey[i];
                    ii[j] = cidx[i];
                    if (static_cast<uint32_t>(kk[j]) >= lo) {
                        f |= 1u << j;
                        ++c;
                    }
                }
            }
            uint32_t total;
            // the scan's barrier also orders every read of this tile before its writes
            uint32_t d = off + team_excl_scan<NC, 2>(c, ctrl, it & 1, total, tid);
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                if (f & (1u << j)) {
                    ckey[d] = kk[j];
                    cidx[d] = ii[j];
                    ++d;
                }
            }
            off += total;
        }
        if (off != keep) set_status(kErrInternal);
        // the bins below the cut are empty now
        for (int i = tid; i < (cb >> 1); i += NC) xh0[i] = 0u;
        if ((cb & 1) && tid == 0) xh0[cb >> 1] &= 0xFFFF0000u;
        if (tid == 0) ctrl->cnt = static_cast<int>(off);
        nt = hasT && T > lo - 1u ? T : lo - 1u;
    } else {
        // The threshold bounds the cluster's union, not this buffer alone, so the
        // compaction ranks every key of the buffer.
        const uint32_t piv = compact<KeyT, NC, 1>(ckey, cidx, hist, ctrl, n, k, 0u, tmax, tid, true);
        nt = hasT && T > piv ? T : piv;
        // the first final histogram, counted anew over the k keys kept
        for (int i = tid; i < kXBins / 2; i += NC) xh0[i] = 0u;
        named_bar_sync(2, NC);
        for (int i = tid; i < k; i += NC) xhist_add(xh0, static_cast<uint32_t>(ckey[i]), hedge, hs0);
    }
    if (tid == 0) {
        for (int r = 0; r < G; ++r) red_cluster_max_u32(map_rank(shT, r), nt);
        if (gT) atomicMax(gT, (static_cast<unsigned long long>(epoch) << 32) | nt);
        ctrl->last_kept = ctrl->cnt;
    }
    named_bar_sync(2, NC);  // the buffer, its count and the histogram are settled
    return nt;
}

// A threshold raise by one warp, from the first final histogram of the keys appended so
// far (bins of 2^hs keys from `edge` up): the smallest key of the bin that holds the k-th
// largest appended key, less one, is at most the row's k-th largest key.  Returns it, or 0
// when the histogram holds fewer than k keys or the bin is the lowest.  Counts read while
// other warps append are never above the final ones, so the bound holds.  Out of line, as
// it runs a few times per call.
template <typename KeyT>
__device__ __noinline__ uint32_t split_raise(const uint32_t* xh0, int k, uint32_t edge, int hs, int lane) {
    const XPivot r = warp_pivot_x(xh0, 1, 0, static_cast<uint32_t>(k), lane);
    if (r.bstar <= 0) return 0u;
    const uint64_t lo = static_cast<uint64_t>(edge) + (static_cast<uint64_t>(r.bstar) << hs);
    return lo - 1u <= (sizeof(KeyT) == 2 ? 0xFFFFull : 0xFFFFFFFFull) ? static_cast<uint32_t>(lo - 1u) : 0u;
}

// The final select's output: one pass over this CTA's n candidates, four per thread at
// a time.  Each warp takes slots for its keys above the pivot and its pivot-equal keys
// from two shared cursors (one atomic each per batch), so slots are this CTA's range in
// any order; pivot-equal keys past the quota are dropped.  TK: write keys (partial
// results of rows over several clusters) instead of values.  Returns nonzero when a slot
// fell outside the row's k.
template <typename KeyT, bool TK>
__device__ __forceinline__ uint32_t split_output(const KeyT* ckey, const uint32_t* cidx, int n, Ctrl* ctrl,
                                                 uint32_t edge, uint32_t pivot, bool take_all, uint32_t gt_lower,
                                                 uint32_t eq_first, uint32_t eq_take, const OutTarget& out,
                                                 uint32_t kslots, bool write_ok, int lane, int tid) {
    constexpr int ES = sizeof(KeyT);
    constexpr int NT = kSplitThreads;
    const uint32_t ltm = lanemask_lt();
    uint32_t bad = 0u;
#pragma unroll 1
    for (int i0 = 0; i0 < n; i0 += 4 * NT) {
        uint32_t kb[4], ib[4], bg[4], be[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + tid + j * NT;
            kb[j] = i < n ? static_cast<uint32_t>(ckey[i]) : 0u;
            ib[j] = i < n ? cidx[i] : 0u;
        }
        uint32_t sg = 0u, se = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool ok = i0 + tid + j * NT < n && kb[j] >= edge;
            const bool isg = ok && (take_all || kb[j] > pivot);
            const bool ise = ok && !take_all && kb[j] == pivot;
            bg[j] = __ballot_sync(0xFFFFFFFFu, isg);
            be[j] = __ballot_sync(0xFFFFFFFFu, ise);
            sg += static_cast<uint32_t>(__popc(bg[j]));
            se += static_cast<uint32_t>(__popc(be[j]));
        }
        if ((sg | se) == 0u) continue;
        uint32_t gb = 0u, eb = 0u;
        if (lane == 0) {
            if (sg) gb = atomicAdd(reinterpret_cast<unsigned int*>(&ctrl->out_g), sg);
            if (se) eb = atomicAdd(reinterpret_cast<unsigned int*>(&ctrl->out_e), se);
        }
        gb = __shfl_sync(0xFFFFFFFFu, gb, 0);
        eb = __shfl_sync(0xFFFFFFFFu, eb, 0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool isg = (bg[j] >> lane) & 1u, ise = (be[j] >> lane) & 1u;
            const uint32_t te = eb + static_cast<uint32_t>(__popc(be[j] & ltm));
            const uint32_t slot = isg ? gt_lower + gb + static_cast<uint32_t>(__popc(bg[j] & ltm)) : eq_first + te;
            const bool put = isg || (ise && te < eq_take);
            if (put && slot < kslots && write_ok) {
                const int64_t o = out.base + slot;
                if (TK) static_cast<uint32_t*>(out.vals)[o] = kb[j];
                else if (ES == 2) static_cast<uint16_t*>(out.vals)[o] = static_cast<uint16_t>(unkey_bf16(kb[j]));
                else static_cast<uint32_t*>(out.vals)[o] = unkey_f32(kb[j]);
                out.idx[o] = static_cast<int32_t>(ib[j]);
            }
            bad |= (put && slot >= kslots) ? 1u : 0u;
            gb += static_cast<uint32_t>(__popc(bg[j]));
            eb += static_cast<uint32_t>(__popc(be[j]));
        }
    }
    return bad;
}

// HELD: every CTA's chunks fit its ring at once (no refills, no streamed-row threshold
// raises or refined warm-up, a sample of at most 4 vectors per thread); MCT: rows span
// several clusters.  The launch picks the instance for its plan, so each call runs only
// its own class's code.
template <typename KeyT, bool HELD, bool MCT>
__global__ void __launch_bounds__(kSplitThreads, 2) ds_split_kernel(const ScanParams p) {
    constexpr int NC = kSplitThreads;
    constexpr int NT = kSplitThreads;
    constexpr int ES = sizeof(KeyT);
    constexpr int KW = 8 * ES;  // key width in bits
    extern __shared__ __align__(1024) uint8_t smem[];
    const int G = p.G;
    const int wm = p.wm;
    const SplitLayout L = split_layout(ES, p.chunk, p.stages, p.cap, G, wm, p.k, p.perm_cap);
    uint8_t* ring = smem + L.ring;
    KeyT* ckey = reinterpret_cast<KeyT*>(smem + L.ckey);
    uint32_t* cidx = reinterpret_cast<uint32_t*>(smem + L.cidx);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L.scratch);
    KeyT* wx = reinterpret_cast<KeyT*>(smem + L.wx);
    int32_t* perm = reinterpret_cast<int32_t*>(smem + L.perm);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + L.ctrl);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = static_cast<int>(blockIdx.x);
    const int rowi = cta / p.parts;
    const int64_t row = rowi;
    const int part = cta - rowi * p.parts;
    const int cl = part / G;
    const uint32_t crank = G > 1 ? cluster_ctarank() : 0u;
    // this part's blocks: every parts-th block of the row from block `part` (parts [0, mr)
    // take mq + 1 blocks, the others mq), so that rows whose large values sit in one
    // region spread them over the CTAs
    const int mp = static_cast<int>(p.mq) + (part < p.mr ? 1 : 0);
    const char* xrow = p.x + row * p.stride_bytes;
    const int chunk_bytes = p.chunk * ES;
    const int cpb = p.cpb;  // chunk slots per block
    // q / cpb and q % cpb for small q, through the reciprocal and one correction
    const auto qdiv = [&](int q, int& bi, int& sub) {
        bi = __float2int_rz(static_cast<float>(q) * p.cpb_rcp);
        sub = q - bi * cpb;
        if (sub < 0) {
            --bi;
            sub += cpb;
        } else if (sub >= cpb) {
            ++bi;
            sub -= cpb;
        }
    };
    const int nq = mp * cpb;
    constexpr bool MC = MCT;
    const uint32_t cap = static_cast<uint32_t>(p.cap);
    // Rows held whole in one cluster may start from a speculative edge (spec_k > 0): every
    // chunk stays in its CTA's ring, so a second attempt can filter them all again.
    const bool spec_ok = HELD && !MC && p.spec_k > 0;

    // The next kernel on the stream may start as this one's CTAs leave.  This kernel may
    // have started before the previous one completed: it waits for it before reading x
    // (unless the caller stated that x was complete earlier) and before any global write
    // (at once when rows span several clusters, which share a global threshold word and a
    // workspace between calls).
    pdl_launch_dependents();
    if (MC) pdl_wait();
    {
        int* z = reinterpret_cast<int*>(ctrl);
        for (int i = tid; i < static_cast<int>(sizeof(Ctrl) / sizeof(int)); i += NT) z[i] = 0;
    }
    __syncthreads();
    if (tid < p.stages) {
        mbar_init(&ctrl->full[tid], 1);
        fence_mbar_init();
    } else if (tid == 32) {
        mbar_init(&ctrl->wbar, 1);
        mbar_init(&ctrl->xbar[0], 1);
        mbar_init(&ctrl->xbar[1], 1);
        ctrl->fail_base = 0x7FFFFFFF;
        ctrl->job_next = kDenseSlices;  // no dense pass open
        fence_mbar_init();
    }
    {  // this CTA's slot of the final select's first exchange round
        uint32_t* x0 = reinterpret_cast<uint32_t*>(smem + L.xf) + static_cast<size_t>(crank) * (kXBins / 2);
        for (int i = tid; i < kXBins / 2; i += NT) x0[i] = 0u;
    }
    block_order<NT>(p.seed, row, part, p.parts, mp, hist, perm, tid);

    // chunk slot q: block perm[bi] with bi = q / cpb, sub-chunk q % cpb (empty past the
    // row's end); the chunk loop steps (bi, sub) without dividing
    const auto chunk_of = [&](int bi, int sub, int64_t& c0, int64_t& ce) {
        const int64_t lo = static_cast<int64_t>(perm[bi]) * p.B;
        const int64_t hi = lo + p.B < p.N ? lo + p.B : p.N;
        c0 = lo + static_cast<int64_t>(sub) * p.chunk;
        ce = c0 < hi ? ((hi - c0) < p.chunk ? (hi - c0) : p.chunk) : 0;
    };
    const auto chunk_at = [&](int q, int64_t& c0, int64_t& ce) {
        int bi, sub;
        qdiv(q, bi, sub);
        chunk_of(bi, sub, c0, ce);
    };
    const auto publish_T = [&](uint32_t t) {
        for (int r = 0; r < G; ++r) red_cluster_max_u32(map_rank(&ctrl->sharedT[0], r), t);
        if (MC) atomicMax(p.gT + row, (static_cast<unsigned long long>(p.epoch) << 32) | t);
    };

    // Copies: stage s belongs to warp s % 8 (the ring depth is a multiple of 8), which
    // consumes every chunk that lands there and refills the stage itself once it is done
    // with it, so no warp ever waits on another warp's stage.
    const uint64_t pol = policy_evict_first();
    const auto issue_to = [&](int s, int use, int bi, int sub) {
        int64_t c0, ce;
        chunk_of(bi, sub, c0, ce);
        const uint32_t bytes = static_cast<uint32_t>(ce * ES) & ~15u;
        if (bytes) {
            mbar_arrive_expect_tx(&ctrl->full[s], bytes);
            bulk_g2s(ring + static_cast<size_t>(s) * chunk_bytes, xrow + c0 * ES, bytes, &ctrl->full[s], pol);
        } else {
            mbar_arrive(&ctrl->full[s]);
        }
        ctrl->issued[s] = use + 1;
    };
    const auto issue = [&](int q) {
        int bi, sub;
        qdiv(q, bi, sub);
        issue_to(q & (p.stages - 1), q >> p.slog, bi, sub);
    };
    if (!MC && !p.early) pdl_wait();
    // The warm-up's chunks go first; the rest of the ring follows once chunk 0 has landed,
    // so that the sample reaches every CTA early.
    const int ww = min(min(p.ww, nq), 8);  // the warm-up tracks at most 8 chunks
    if (tid == 0)
        for (int q = 0; q < ww; ++q) issue(q);
    // Cluster-wide start: every thread arrives now (its CTA's barriers are initialised)
    // and waits only before its CTA's first access to another CTA's memory, so the
    // cluster's CTAs meet while the first copies are in flight.
    if (G > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // the final select's outcome (set by the last attempt)
    int n = 0;
    uint32_t edge = 0u, pivot = 0u;
    uint32_t gt_all = 0u, gt_lower = 0u;   // keys above the pivot: all CTAs, CTAs of lower rank
    uint32_t eq_lower = 0u, eq_mine = 0u;  // pivot-equal keys: CTAs of lower rank, this CTA
    bool take_all = false;
    // two rounds of G histograms of kXBins uint16 counts, as pairs in 32-bit words
    constexpr int XW = kXBins / 2;
    uint32_t* const xr = reinterpret_cast<uint32_t*>(smem + L.xf);
    {
        bool hasT = false;
        uint32_t T = 0u;
        uint32_t tmax = 0u;
        uint32_t gnext = 0u;  // other clusters' threshold, loaded one chunk ahead
        // The final select's first histogram (this CTA's slot of its first exchange round)
        // is counted as keys are appended: keys from the warm-up's edge up, in bins of
        // 2^hs0 keys (set once the edge is known).
        int att = 0;  // attempt: 1 after a speculative edge failed (rows held whole only)
        // attempt a counts its first histogram into this CTA's slot of round a
        const auto xh0 = [&]() { return xr + (static_cast<size_t>(att) * G + crank) * XW; };
        uint32_t hedge = 0u;
        int hs0 = KW - kXBits;
        // every consumer warp calls this together (from its chunk loop or the drain); the
        // work is out of line, away from the chunk loop's code
        const auto join_compaction = [&]() {
            T = split_compaction<KeyT>(ckey, cidx, hist, ctrl, p.cap, p.chunk, p.k, tmax, tid, hasT, T, xh0(), hedge,
                                       hs0, G, ctrl->sharedT + att, MC ? p.gT + row : nullptr, p.epoch);
            hasT = true;
        };
        // A warp waiting for its next chunk joins any compaction requested meanwhile, so
        // the requesting warp does not wait for this chunk to land.  Decisions are
        // warp-uniform.
        const auto wait_data = [&](uint64_t* bar, uint32_t parity) -> bool {
            if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
            const long long t0 = clock64();
            while (true) {
                if (__all_sync(0xFFFFFFFFu, mbar_try_wait_sleep(bar, parity, 2000u))) return true;
                int f = 0, a = 0, d = 0;
                if (lane == 0) {
                    f = *reinterpret_cast<volatile int*>(&ctrl->compact_req);
                    a = *reinterpret_cast<volatile int*>(&ctrl->abort);
                    if (HELD) d = *reinterpret_cast<volatile int*>(&ctrl->done_warps);
                }
                if (HELD && __shfl_sync(0xFFFFFFFFu, d, 0) >= kJobOpen)  // help with a shared dense pass
                    tmax = max(tmax, dense_claim<KeyT>(ckey, cidx, ctrl, lane, xh0(), hedge, hs0));
                if (__shfl_sync(0xFFFFFFFFu, a, 0)) return false;
                if (__shfl_sync(0xFFFFFFFFu, f, 0)) join_compaction();
                if (clock64() - t0 > kSpinLimit) {
                    if (lane == 0) {
                        set_status(kErrTimeout);
                        *reinterpret_cast<volatile int*>(&ctrl->abort) = 1;
                    }
                    return false;
                }
            }
        };

        // the chunk loop's stepping (block and sub-chunk of this warp's first chunk, of
        // kNCW chunks ahead and of one ring ahead), set up before the warm-up's waits
        int bi0, sub0, d8, r8, dS, rS;
        qdiv(warp, bi0, sub0);
        qdiv(kNCW, d8, r8);
        qdiv(p.stages, dS, rS);
        // ---- warm-up on the first ww chunks (all consumer warps) ----
        for (int b = tid; b < kBins; b += NC) hist[b] = 0u;  // the warm-up's histogram, while the sample lands
        const int cvec = chunk_bytes / 16;  // vectors per full chunk
        int nvw[8];                         // whole vectors in each sampled chunk
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            nvw[q] = 0;
            if (q < ww) {
                int64_t c0, ce;
                chunk_at(q, c0, ce);
                nvw[q] = static_cast<int>(ce * ES / 16);
            }
        }
        // With one sampled chunk per warp (streamed rows sampling kNCW whole chunks) each warp
        // takes the group maxima of its own chunk as soon as that chunk lands.
        const int R = wm / 256;
        const int VT = (ww * cvec + NC - 1) / NC;  // at most 16
        // log2 of vectors per group
        const int gsh = VT >= 16 * R ? 4 : (VT >= 8 * R ? 3 : (VT >= 4 * R ? 2 : (VT >= 2 * R ? 1 : 0)));
        const int WS = wm + 16 / ES;  // row stride of the union in wx: the maxima, then a slot
        bool whole = (ww * cvec) % NC == 0;  // every sampled chunk whole
#pragma unroll
        for (int q = 0; q < 8; ++q) whole = whole && (q >= ww || nvw[q] == cvec);
        const bool perwarp = !HELD && ww == kNCW && whole;
        uint32_t lm = 0u;  // the largest of this thread's group maxima
        bool gotw;
        if (perwarp) {
            gotw = wait_bounded(&ctrl->full[warp], 0, ctrl);
            if (lane == 0 && gotw) ctrl->observed[warp] = 1;
            if (lane == 0)
                for (int q = warp + kNCW; q < nq && q < p.stages; q += kNCW) issue(q);
            if (gotw) {
                const uint4* own = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(warp) * chunk_bytes);
                lm = warm_maxima16_whole<KeyT>(own, lane, 32, VT, gsh, R, wx + crank * WS + tid * R);
            }
        } else {
            const bool got0 = wait_bounded(&ctrl->full[0], 0, ctrl);
            if (tid == 0 && got0) ctrl->observed[0] = 1;
            if (lane == 0)
                for (int q = warp < ww ? warp + kNCW : warp; q < nq && q < p.stages; q += kNCW) issue(q);
            gotw = got0;
            for (int q = 1; q < ww; ++q) {
                const bool g = wait_bounded(&ctrl->full[q], 0, ctrl);
                if (tid == 0 && g) ctrl->observed[q] = 1;
                gotw = gotw && g;
            }
        }
        {
            // group maxima: thread t owns vectors t, t + NC, ... of the sample (VT of them)
            // and splits them into R groups; a group's maximum is taken on the packed values
            // (NaNs ignored) and keyed once
            const uint4* v0 = reinterpret_cast<const uint4*>(ring);
            if (perwarp) {
                // (done above)
            } else if (HELD || VT <= 8) {
                uint32_t gk[4] = {0u, 0u, 0u, 0u};  // key of each group's maximum (0: none)
                if (whole) {
                    if (HELD || VT <= 4) warm_maxima_whole<KeyT, 4>(v0, tid, VT, gsh, gk);
                    else warm_maxima_whole<KeyT, 8>(v0, tid, VT, gsh, gk);
                } else if (HELD || VT <= 4) {
                    warm_maxima<KeyT, 4>(v0, tid, cvec, ww, VT, gsh, gotw, nvw, gk);
                } else {
                    warm_maxima<KeyT, 8>(v0, tid, cvec, ww, VT, gsh, gotw, nvw, gk);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r < R) {
                        wx[crank * WS + tid * R + r] = static_cast<KeyT>(gk[r]);
                        lm = max(lm, gk[r]);
                    }
                }
            } else {
                lm = whole ? warm_maxima16_whole<KeyT>(v0, tid, NC, VT, gsh, R, wx + crank * WS + tid * R)
                           : warm_maxima16<KeyT>(v0, tid, cvec, ww, VT, gsh, R, gotw, nvw, wx + crank * WS + tid * R);
            }
            if (!HELD) {  // (streamed rows bin the union below its largest maximum)
                lm = __reduce_max_sync(0xFFFFFFFFu, lm);
                if (lane == 0) atomicMax(&ctrl->lmax, lm);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, NC);
            if (G > 1) {
                asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
                if (tid == 0) {  // the row (and its largest, in the slot after it) to every peer
                    if (!HELD) {
                        *reinterpret_cast<uint32_t*>(wx + crank * WS + wm) = ctrl->lmax;
                        fence_proxy_async_smem();
                    }
                    const uint32_t bytes = static_cast<uint32_t>(HELD ? wm : WS) * ES;
                    mbar_arrive_expect_tx(&ctrl->wbar, bytes * static_cast<uint32_t>(G - 1));
                    for (int r = 0; r < G; ++r)
                        if (r != static_cast<int>(crank))
                            bulk_s2s_cluster(map_rank(wx + crank * WS, r), wx + crank * WS, bytes,
                                             map_rank(&ctrl->wbar, r));
                }
                wait_bounded_cluster(&ctrl->wbar, 0, ctrl);
            }
            // The edge: the smallest key of the bin of a histogram of the union's maxima that
            // holds the k-th largest.  At least k maxima, each an element of the row, lie at or
            // above it.  Streamed rows bin the maxima in kBins bins of 2^FS keys below M, the
            // union's largest maximum (one key each for bf16, 1/1024 of an octave for fp32);
            // rows held whole, and rows with fewer than k maxima in that range, by the top
            // kDigitBits key bits, streamed rows then narrowing the bucket to its 32nd part
            // that holds the k-th largest (refine).  (On rows held whole the narrower edge
            // saves fewer appends than finding it costs.)
            uint32_t wedge0 = 0u;
            bool coarse = HELD;
            uint32_t Mw = 0u;  // the union's largest maximum (streamed rows)
            if (!HELD) {
                uint32_t M = ctrl->lmax;
                for (int r = 0; r < G; ++r)
                    if (r != static_cast<int>(crank)) M = max(M, *reinterpret_cast<const uint32_t*>(wx + r * WS + wm));
                Mw = M;
                constexpr int FS = ES == 2 ? 0 : 13;
                each_key<KeyT>(wx, G, wm, tid, [&](uint32_t kk) {
                    const uint32_t d = (M - kk) >> FS;
                    if (kk && d < static_cast<uint32_t>(kBins)) atomicAdd(&hist[kBins - 1 - d], 1u);
                });
                __syncthreads();
                cta_bucket_2048(hist, static_cast<uint32_t>(p.k), 0u, tid, ctrl->warp_tot[0], ctrl);
                if (ctrl->bcount >= static_cast<uint32_t>(p.k) && ctrl->bstar >= 0) {
                    const int64_t lo =
                        static_cast<int64_t>(M) - (static_cast<int64_t>(kBins - ctrl->bstar) << FS) + 1;
                    wedge0 = lo > 0 ? static_cast<uint32_t>(lo) : 0u;
                    if (tid == 0) ctrl->wedge = wedge0;
                } else {
                    coarse = true;
                    __syncthreads();  // (every thread has read the bin above)
                    for (int b = tid; b < kBins; b += NC) hist[b] = 0u;
                    __syncthreads();
                }
            }
            if (coarse) {
                each_key<KeyT>(wx, G, wm, tid, [&](uint32_t kk) {
                    if (kk) atomicAdd(&hist[(kk << (32 - KW)) >> (32 - kDigitBits)], 1u);
                });
                __syncthreads();
                cta_bucket_2048(hist, static_cast<uint32_t>(p.k), spec_ok ? static_cast<uint32_t>(p.spec_k) : 0u, tid,
                                ctrl->warp_tot[0], ctrl);
                const int bstar = ctrl->bstar;
                const uint32_t above = ctrl->above, total = ctrl->bcount;
                if (HELD || !p.refine) {
                    if (total >= static_cast<uint32_t>(p.k) && bstar > 0) {
                        wedge0 = static_cast<uint32_t>(bstar) << (KW - kDigitBits);
                        if (!HELD && tid == 0) ctrl->wedge = wedge0;
                    }
                } else if (total >= static_cast<uint32_t>(p.k) && bstar >= 0) {
                    constexpr int SB = KW - kDigitBits - 5;  // shift of the 5 bits below the bucket's
                    uint32_t* sub = ctrl->block_cnt[0];     // zero since start-up
                    each_key<KeyT>(wx, G, wm, tid, [&](uint32_t kk) {
                        if (kk && (kk >> (KW - kDigitBits)) == static_cast<uint32_t>(bstar))
                            atomicAdd(&sub[(kk >> SB) & 31u], 1u);
                    });
                    __syncthreads();
                    if (warp == 0) {
                        uint32_t sfx = sub[lane];  // maxima in parts >= lane of the bucket
#pragma unroll
                        for (int d = 1; d < 32; d <<= 1) {
                            const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, sfx, d);
                            if (lane + d < 32) sfx += t;
                        }
                        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, above + sfx >= static_cast<uint32_t>(p.k));
                        const uint32_t l = hit ? 31u - __clz(hit) : 0u;
                        if (lane == 0)
                            ctrl->wedge = (static_cast<uint32_t>(bstar) << (KW - kDigitBits)) | (l << SB);
                    }
                    __syncthreads();
                    wedge0 = ctrl->wedge;
                }
            }
            // Rows held whole may start from a speculative edge: the spec_k-th largest
            // maximum (spec_k about twice the sample's expected share of the row's k largest),
            // placed in its bucket as if the bucket's maxima were spread evenly over its keys.
            // Nothing proves that k keys of the row reach it; the final select's first pass
            // counts every key at or above it over the cluster and, when there are fewer than
            // k, the chunks (all still in the ring) are filtered again from the proven edge.
            uint32_t sedge = wedge0;
            if (HELD) {
                if (spec_ok && wedge0 > 0u && ctrl->spec_b >= 0) {
                    constexpr uint32_t BW = 1u << (KW - kDigitBits);  // keys per bucket
                    const uint32_t bc = ctrl->spec_c;
                    const uint32_t r = static_cast<uint32_t>(p.spec_k) - ctrl->spec_above;  // 1 <= r <= bc
                    const uint64_t top = (static_cast<uint64_t>(ctrl->spec_b) + 1u) * BW;  // one past the bucket
                    // about r * BW / bc keys below the top, rounded up, within [1, BW]: an estimate
                    // needs no exact quotient (a 64-bit integer division here cost every thread
                    // several hundred cycles)
                    const float q = __fdividef(static_cast<float>(r), static_cast<float>(bc)) * static_cast<float>(BW);
                    const uint32_t down = min(BW, max(1u, static_cast<uint32_t>(ceilf(q))));
                    sedge = max(wedge0, static_cast<uint32_t>(top - down));
                }
                if (tid == 0) {
                    ctrl->wedge = sedge;
                    ctrl->wedge_p = wedge0;
                }
            }
            if (sedge > 0u) {
                hasT = true;
                T = sedge - 1u;
                hedge = sedge;
                // (fp32: bins of 2^14 keys span an octave above the edge; a speculative edge
                // lies close below the k-th key, so bins four times narrower usually leave
                // the pivot's bin holding just the keys still needed: one pass)
                hs0 = ES == 2 ? 0 : (sedge > wedge0 ? 23 - kXBits - 2 : 23 - kXBits);
            }
            // A window below M: kXBins bins of one key (bf16) or 2^16 keys (fp32, 4 octaves in
            // all), M in the next-to-last.  Streamed rows with no warm-up edge, or with one so
            // far below M that M lies past the edge's bins and the edge below the window (k
            // beyond what the sample can bound tightly), bin their first final histogram there
            // instead, so that threshold raises and compaction cuts see fine bins.  Nothing
            // proves the k-th key lies in the window; the final select's first pass checks it
            // and counts the whole range from the edge otherwise.
            if (!HELD && Mw > 0u) {
                constexpr int WSH = ES == 2 ? 0 : 16;
                const uint32_t span = static_cast<uint32_t>(kXBins - 2) << WSH;
                const uint64_t reach =  // where the edge's bins end (the last is open-ended)
                    sedge ? static_cast<uint64_t>(sedge) + (static_cast<uint64_t>(kXBins - 1) << hs0) : 0u;
                const uint32_t wb = Mw > span ? Mw - span : 0u;
                if (Mw >= reach && (sedge == 0u || wb > sedge)) {  // (the edge lies below the window)
                    hedge = wb;
                    hs0 = WSH;
                }
            }
            if (tid == 0) {
                ctrl->hshift = hs0;
                ctrl->hbase = hedge;
            }
            // (every CTA of the cluster derived this same threshold: only the row's other
            // clusters need it)
            if (tid == 0 && hasT && MC) publish_T(T);
        }

        // The chunks, the drain and the final select, once, or twice when a speculative edge
        // failed (rows held whole only).
        for (;; ++att) {
            // ---- the chunks, one warp each (warp 0 takes chunk 0 too) ----
            // this warp's chunk q: ring stage s = q % stages and use q / stages, block index bi
            // and sub-chunk sub, stepped by kNCW chunks per round
            int st = warp, use = 0, bi = bi0, sub = sub0;
            for (int q = warp; q < nq; q += kNCW) {
                int req = 0;
                if (lane == 0) req = *reinterpret_cast<volatile int*>(&ctrl->compact_req);
                if (__shfl_sync(0xFFFFFFFFu, req, 0)) join_compaction();
                // the threshold: this CTA's, the cluster's and the other clusters'
                uint32_t tk = T;
                bool have = hasT;
                {
                    uint32_t sh = gnext;
                    if ((G > 1 || (!HELD && p.rstep)) && lane == 0)
                        sh = max(sh, *reinterpret_cast<volatile uint32_t*>(ctrl->sharedT + att));
                    sh = __shfl_sync(0xFFFFFFFFu, sh, 0);
                    if (sh != 0u && (!have || sh > tk)) {
                        tk = sh;
                        have = true;
                    }
                    if (MC && lane == 0) {
                        const unsigned long long g = ld_relaxed_gpu_u64(p.gT + row);
                        gnext = static_cast<uint32_t>(g >> 32) == p.epoch ? static_cast<uint32_t>(g) : 0u;
                    }
                }
                int64_t c0, ce;
                chunk_of(bi, sub, c0, ce);
                const uint32_t bytes = static_cast<uint32_t>(ce * ES) & ~15u;
                const int s = st;
                const bool got = wait_data(&ctrl->full[s], use & 1);
                if (lane == 0 && got) ctrl->observed[s] = use + 1;
                if (hasT && (!have || T > tk)) {  // a compaction ran while the warp waited
                    tk = T;
                    have = true;
                }
                if (got && ce > 0) {
                    const int nvec = static_cast<int>(bytes / 16);
                    const int tail = static_cast<int>(ce - bytes / ES);
                    int pass = 0;
                    while (!warp_chunk<KeyT, HELD>(ring + static_cast<size_t>(s) * chunk_bytes, nvec,
                                                   static_cast<uint32_t>(c0), xrow, c0 + bytes / ES, tail,
                                                   compare_bits<KeyT>(have, tk), ckey, cidx, ctrl, cap, lane, pass,
                                                   tmax, xh0(), hedge, hs0)) {
                        join_compaction();
                        if (!have || T > tk) {
                            tk = T;
                            have = true;
                        }
                        int ab = 0;
                        if (lane == 0) ab = *reinterpret_cast<volatile int*>(&ctrl->abort);
                        if (__shfl_sync(0xFFFFFFFFu, ab, 0)) break;
                    }
                }
                __syncwarp();  // every lane is done with the stage: refill it with this warp's next chunk there
                if (!HELD && lane == 0 && got && q + p.stages < nq &&
                    !*reinterpret_cast<volatile int*>(&ctrl->abort)) {
                    int bj = bi + dS, sj = sub + rS;
                    if (sj >= cpb) {
                        sj -= cpb;
                        ++bj;
                    }
                    issue_to(s, use + 1, bj, sj);
                }
                if (!HELD && p.rstep) {  // one warp raises the threshold each time the buffer passes the mark
                    int due = 0;
                    if (lane == 0) {
                        const uint32_t c = static_cast<uint32_t>(*reinterpret_cast<volatile int*>(&ctrl->cnt));
                        const uint32_t mk = *reinterpret_cast<volatile uint32_t*>(&ctrl->raise_mark);
                        if (c >= (mk ? mk : static_cast<uint32_t>(p.rmark)))
                            due = atomicCAS(&ctrl->raise_mark, mk, c + static_cast<uint32_t>(p.rstep)) == mk;
                    }
                    if (__shfl_sync(0xFFFFFFFFu, due, 0)) {
                        const uint32_t t = split_raise<KeyT>(xh0(), p.k, hedge, hs0, lane);
                        if (lane == 0 && t != 0u) {
                            if (G > 1 || MC) publish_T(t);
                            else atomicMax(&ctrl->sharedT[0], t);
                        }
                    }
                }
                bi += d8;
                sub += r8;
                if (sub >= cpb) {
                    sub -= cpb;
                    ++bi;
                }
                st += kNCW;
                if (st >= p.stages) {
                    st -= p.stages;
                    ++use;
                }
            }
            // A warp out of chunks still joins compactions other warps request: it reads the
            // count of finished warps before the request flag, so a request raised by the
            // last warp before it finished is always seen.
            __threadfence_block();
            if (lane == 0) atomicAdd(&ctrl->done_warps, 1);
            {
                const long long t0 = clock64();
                while (true) {
                    int d = 0, f = 0;
                    if (lane == 0) {
                        d = *reinterpret_cast<volatile int*>(&ctrl->done_warps);
                        __threadfence_block();
                        f = *reinterpret_cast<volatile int*>(&ctrl->compact_req);
                    }
                    d = __shfl_sync(0xFFFFFFFFu, d, 0);
                    f = __shfl_sync(0xFFFFFFFFu, f, 0);
                    if (HELD && d >= kJobOpen) {  // help with a shared dense pass
                        tmax = max(tmax, dense_claim<KeyT>(ckey, cidx, ctrl, lane, xh0(), hedge, hs0));
                        d -= kJobOpen;
                    }
                    if (f) {
                        join_compaction();
                        continue;
                    }
                    if (d >= kNCW) break;
                    if (clock64() - t0 > kSpinLimit) {  // cannot happen; keep the CTA alive
                        set_status(kErrTimeout);
                        break;
                    }
                }
            }
            // every warp is done: the buffer, its count and the first histogram are final
            // (the histogram leaves by bulk copy: the async proxy must see the appends)
            fence_proxy_async_smem();
            named_bar_sync(1, NC);
            if (ctrl->abort) {
                if (tid == 0)
                    for (int s = 0; s < p.stages; ++s)
                        if (ctrl->issued[s] > ctrl->observed[s])
                            drain_wait(&ctrl->full[s], (ctrl->issued[s] - 1) & 1);
                __syncthreads();
            }

            // ---------------------------- final selection over the cluster ------------
            n = ctrl->cnt < p.cap ? ctrl->cnt : p.cap;
            // Keys below the edge are out of play: at least k keys of the cluster's union lie
            // at or above it (on a speculative edge, the first pass checks that they do).
            edge = ctrl->wedge;  // the same in every CTA of the cluster
            const uint32_t kmax = KW == 16 ? 0xFFFFu : 0xFFFFFFFFu;
            const auto in_play = [&](uint32_t kk) { return kk >= edge; };
            // pass state (identical in every CTA): keys in [lbase, lhi] binned by
            // (key - lbase) >> s, the last bin open-ended
            uint32_t lbase = ctrl->hbase, lhi = kmax;  // the first pass: the appends' bins
            int s = ctrl->hshift;
            uint32_t krem = static_cast<uint32_t>(p.k);
            gt_all = gt_lower = eq_lower = eq_mine = pivot = 0u;
            take_all = false;
            bool retry = false;
            // Pass lvl exchanges its histograms through round lvl % 2; attempt a starts with
            // pass a, whose counts this CTA made as keys were appended.
            for (int lvl = att;; ++lvl) {
                uint32_t* mine = xr + (static_cast<size_t>(lvl & 1) * G + crank) * XW;
                if (lvl > att) {  // (the slot was cleared before the previous pass's last barrier)
#pragma unroll 4
                    for (int i = tid; i < n; i += NT) {
                        const uint32_t kk = ckey[i];
                        if (in_play(kk) && kk >= lbase && kk <= lhi) {
                            uint32_t d = (kk - lbase) >> s;
                            d = d < kXBins - 1 ? d : kXBins - 1;
                            atomicAdd(&mine[d >> 1], 1u << ((d & 1u) * 16u));
                        }
                    }
                }
                if (lvl > att) {  // (the attempt's first pass was ordered after the drain)
                    fence_proxy_async_smem();
                    __syncthreads();
                }
                uint64_t* xb = &ctrl->xbar[lvl & 1];
                if (G > 1) {
                    if (tid == 0) {
                        const uint32_t bytes = XW * 4u;
                        mbar_arrive_expect_tx(xb, bytes * static_cast<uint32_t>(G - 1));
                        for (int r = 0; r < G; ++r)
                            if (r != static_cast<int>(crank))
                                bulk_s2s_cluster(map_rank(mine, r), mine, bytes, map_rank(xb, r));
                    }
                    wait_bounded_cluster(xb, (lvl >> 1) & 1, ctrl);
                }
                // this CTA's slot of the other round is free again (what it held was pushed a round
                // ago and every peer has used it since): clear it for the next pass
                uint32_t* next_mine = xr + (static_cast<size_t>((lvl + 1) & 1) * G + crank) * XW;
                for (int i = tid; i < XW; i += NT) next_mine[i] = 0u;
                // the cluster's histogram: the CTA finds the pivot bin
                const uint32_t* rows = xr + static_cast<size_t>(lvl & 1) * G * XW;
                cta_pivot_x(rows, G, static_cast<int>(crank), krem, tid, ctrl->warp_tot[0], ctrl);
                XPivot pv;
                pv.bstar = static_cast<int>(ctrl->fp_tot[0]);
                pv.above = ctrl->fp_tot[1];
                pv.low_above = ctrl->fp_tot[2];
                pv.eq_lower = ctrl->fp_tot[3];
                const int bstar = pv.bstar;
                gt_lower += pv.low_above;
                gt_all += pv.above;
                if (bstar < 0) {  // fewer than krem keys in play (only possible in the first pass)
                    if (spec_ok && att == 0 && edge > ctrl->wedge_p) {  // the speculative edge failed
                        retry = true;
                        break;
                    }
                    if (lbase > edge && lvl == att) {  // the keys below the first pass's bins:
                        lbase = edge;                  // count the whole range from the edge
                        lhi = kmax;
                        s = edge ? (ES == 2 ? 0 : 23 - kXBits) : (KW - kXBits);
                        krem = static_cast<uint32_t>(p.k);
                        gt_all = gt_lower = 0u;
                        continue;
                    }
                    take_all = true;  // keep them all
                    break;
                }
                krem -= pv.above;
                if (s > 0 || bstar == kXBins - 1) {
                    // The bin holds exactly the keys still needed: take it whole, with every key
                    // above it, and stop (no further pass to find the pivot key inside it).
                    uint32_t binc = 0u;
                    for (int c = 0; c < G; ++c) binc += reinterpret_cast<const uint16_t*>(rows)[c * kXBins + bstar];
                    const uint32_t lo_bin = lbase + (static_cast<uint32_t>(bstar) << s);
                    if (binc == krem && lo_bin > 0u) {
                        pivot = lo_bin - 1u;  // keys above it are taken; none equal to it is
                        gt_lower += pv.eq_lower;
                        gt_all += binc;
                        krem = 0u;
                        break;
                    }
                }
                if (s == 0 && bstar < kXBins - 1) {
                    pivot = lbase + static_cast<uint32_t>(bstar);
                    eq_lower = pv.eq_lower;
                    eq_mine = reinterpret_cast<const uint16_t*>(rows)[crank * kXBins + bstar];
                    break;
                }
                if (G == 1 && bstar < kXBins - 1 && reinterpret_cast<const uint16_t*>(rows)[bstar] <= 32u) {
                    // one CTA and few keys in the bin: collect them and rank them in one warp
                    // instead of counting further passes over the buffer
                    const uint32_t blo = lbase + (static_cast<uint32_t>(bstar) << s);
                    const uint64_t top = static_cast<uint64_t>(blo) + ((uint64_t(1) << s) - 1u);
                    const uint32_t bhi = top < lhi ? static_cast<uint32_t>(top) : lhi;
                    if (tid == 0) ctrl->fp_tot[8] = 0u;
                    __syncthreads();
                    for (int i = tid; i < n; i += NT) {
                        const uint32_t kk = ckey[i];
                        if (in_play(kk) && kk >= blo && kk <= bhi) {
                            const uint32_t q = atomicAdd(&ctrl->fp_tot[8], 1u);
                            if (q < 32u) hist[q] = kk;
                        }
                    }
                    __syncthreads();
                    if (warp == 0) {
                        const uint32_t cnt = min(ctrl->fp_tot[8], 32u);
                        const uint32_t mk = static_cast<uint32_t>(lane) < cnt ? hist[lane] : 0u;
                        uint32_t gt = 0u, eq = 0u;  // keys of the bin above and equal to this lane's
                        for (uint32_t j = 0; j < cnt; ++j) {
                            const uint32_t o = __shfl_sync(0xFFFFFFFFu, mk, static_cast<int>(j));
                            gt += o > mk ? 1u : 0u;
                            eq += o == mk ? 1u : 0u;
                        }
                        const bool hold = static_cast<uint32_t>(lane) < cnt && gt < krem && krem <= gt + eq;
                        const uint32_t hb = __ballot_sync(0xFFFFFFFFu, hold);
                        if (hb == 0u && lane == 0) set_status(kErrInternal);  // (the bin holds the krem-th key)
                        if (hb != 0u && lane == __ffs(hb) - 1) {
                            ctrl->fp_tot[9] = mk;
                            ctrl->fp_tot[10] = gt;
                            ctrl->fp_tot[11] = eq;
                        }
                    }
                    __syncthreads();
                    pivot = ctrl->fp_tot[9];
                    gt_all += ctrl->fp_tot[10];
                    eq_lower = 0u;
                    eq_mine = ctrl->fp_tot[11];
                    break;
                }
                if (bstar < kXBins - 1) {
                    lbase += static_cast<uint32_t>(bstar) << s;
                    const uint64_t top = static_cast<uint64_t>(lbase) + ((uint64_t(1) << s) - 1u);
                    lhi = top < lhi ? static_cast<uint32_t>(top) : lhi;
                    s = s > kXBits ? s - kXBits : 0;
                } else {  // the open top bin: its keys all lie in [lbase + (kXBins - 1) << s, lhi]
                    lbase += static_cast<uint32_t>(kXBins - 1) << s;
                    const int sb = bit_length(lhi - lbase) - kXBits;
                    s = sb > 0 ? sb : 0;
                }
            }
            if (!retry) break;
            // Fewer than k keys of the row reach the speculative edge.  Every chunk is still in
            // the ring: filter them all again from the proven edge, counting the first
            // histogram into this CTA's slot of the next round (cleared by the pass above).
            const uint32_t pe = ctrl->wedge_p;
            __syncthreads();  // every thread has read the pass's results
            if (tid == 0) {
                ctrl->cnt = 0;
                ctrl->fail_base = 0x7FFFFFFF;
                ctrl->done_warps = 0;
                ctrl->compact_req = 0;
                ctrl->last_kept = 0;
                ctrl->raise_mark = 0u;
                ctrl->wedge = pe;
            }
            hasT = true;
            T = pe - 1u;
            hedge = pe;
            hs0 = ES == 2 ? 0 : 23 - kXBits;
            if (tid == 0) {
                ctrl->hshift = hs0;
                ctrl->hbase = pe;
            }
            tmax = 0u;
            gnext = 0u;
            __syncthreads();
        }
    }
    // Every CTA has read and pushed all it will: the cluster barrier's arrival goes now and
    // its wait at the very end, so no CTA leaves while another may still use its memory.
    if (G > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // this CTA's output slots: keys above the pivot after those of lower ranks, then the
    // pivot-equal keys by rank until the quota k - (keys above) is used up
    const uint32_t quota = take_all ? 0u : static_cast<uint32_t>(p.k) - gt_all;
    const uint32_t eq_take = take_all ? 0u : (quota > eq_lower ? min(quota - eq_lower, eq_mine) : 0u);
    const uint32_t eq_first = gt_all + min(eq_lower, quota);
    OutTarget out;
    if (MC) {
        out.vals = p.ws_key;
        out.idx = p.ws_idx;
        out.base = (row * p.C + cl) * static_cast<int64_t>(p.k);
        out.to_keys = true;
    } else {
        out.vals = p.out_vals;
        out.idx = p.out_idx;
        out.base = row * static_cast<int64_t>(p.k);
        out.to_keys = false;
    }
    const bool write_ok = !ctrl->abort;
    pdl_wait();  // the previous call's outputs are complete before this call writes its own
    // One pass over the candidates (split_output); partial results of rows over several
    // clusters go out as keys
    const uint32_t bad =
        out.to_keys ? split_output<KeyT, true>(ckey, cidx, n, ctrl, edge, pivot, take_all, gt_lower, eq_first, eq_take,
                                               out, static_cast<uint32_t>(p.k), write_ok, lane, tid)
                    : split_output<KeyT, false>(ckey, cidx, n, ctrl, edge, pivot, take_all, gt_lower, eq_first,
                                                eq_take, out, static_cast<uint32_t>(p.k), write_ok, lane, tid);
    if (bad) set_status(kErrInternal);
    if (take_all && !MC && tid == 0) set_status(kErrInternal);  // a whole row held fewer than k keys in play
    if (MC && crank == 0 && tid == 0)
        p.ws_cnt[row * p.C + cl] = static_cast<int32_t>(take_all ? gt_all : static_cast<uint32_t>(p.k));
    if (G > 1) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace dsk
