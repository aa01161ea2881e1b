// ds_select.cuh -- the candidate buffer of DeepSelectTopk in shared memory.
//
// The candidate buffer (topk_candidate in DeepSelect-deep-dive.md, "Algorithm") holds
// (key, column) pairs: keys are the order-preserving integer keys of the values
// (uint16_t for bf16, uint32_t for fp32), columns are uint32.  Three operations:
//   - warp appends of elements that pass the threshold filter ("Filter" step);
//   - compact(): RadixSelectTopK back to exactly k entries ("Compact" step), returning
//     the k-th largest key, which becomes the threshold T;
//   - the final selection, which may span the CTAs of a thread-block cluster (the
//     deep-dive's "Implementation" section: each CTA holds candidates of one part of the
//     row and the cluster selects the k largest of their union).
//
// RadixSelectTopK is a most-significant-digit radix select over the keys, with an
// adaptive digit: all keys of the buffer lie in [lo, hi] (lo = the current T, hi = the
// largest key appended), and each pass histograms (key - lo) >> s into at most 2048
// bins, s chosen so the range fits.  The bin holding the k-th largest key becomes the
// next range; when s reaches 0 the pivot key is known exactly.  Ties at the pivot are
// resolved by a quota: exactly k - (number of keys above the pivot) pivot-equal entries
// are kept (the tutorial's eq_quota, section 4.6).
#pragma once

#include "ds_common.cuh"

namespace dsk {

__device__ unsigned int g_ds_status;  // per-device status word (OR of kErr* bits)

__device__ __forceinline__ void set_status(uint32_t bits) { atomicOr(&g_ds_status, bits); }

// shared-memory control block
struct Ctrl {
    uint64_t full[kMaxStages];   // ring stage filled (one arrival + bytes)
    uint64_t empty[kMaxStages];  // ring stage drained (one-CTA rows: one arrival per consumer warp)
    int issued[kMaxStages];      // copies issued per stage
    int observed[kMaxStages];    // copies seen complete per stage
    int cnt;                     // append cursor of the candidate buffer
    uint32_t maxkey;             // largest key appended (reduced from the threads at each select)
    uint32_t sharedT[2];         // split rows: the cluster's threshold key (each CTA's copy), 0 = none;
                                 //   one word per attempt of a row held whole (see wedge_p)
    int abort;                   // a bounded wait ran out: skip the remaining waits
    int bstar;                   // pivot search results
    uint32_t above;
    uint32_t bcount;             // keys in the pivot bin (or a second count above it)
    uint32_t fp_tot[32];         // pivot-search scratch
    uint32_t warp_tot[2][32];    // team-scan scratch, two rows used alternately (2 x 16 words)
    uint32_t block_cnt[2][32];   // per-warp appends of the current block, by block parity
    int compact_req;             // split rows: a reservation did not fit the buffer
    int done_warps;              // split rows: warps that have filtered all their chunks, plus
                                 //   kJobOpen while a dense pass is shared out (rows held whole)
    int fail_base;               // split rows: first slot of a reservation that did not fit
    uint64_t wbar;               // split rows: warm-up exchange of group maxima
    uint64_t xbar[2];            // split rows: final-select histogram exchange, by pass parity
    uint32_t wedge;              // split rows: the edge the final select starts from (the warm-up's;
                                 //   speculative while the first attempt runs on one)
    uint32_t wedge_p;            // split rows held whole: the proven edge (k keys of the row at or above)
    int spec_b;                  // split rows held whole: the warm-up bucket of the speculative rank,
    uint32_t spec_above;         //   the maxima above it and in it
    uint32_t spec_c;
    int fin_n;                   // consumer state handed to the whole CTA after the scan
    int fin_hasT;
    uint32_t fin_T;
    int out_g;                   // split rows: output cursors of the final select (keys above
    int out_e;                   // the pivot, pivot-equal keys)
    uint32_t raise_mark;         // split rows: buffer count at which a warp next raises T from
                                 //   the appended keys' histogram (0 = the first mark)
    int cut_bin;                 // split rows: a compaction's cut from that histogram (bin,
    uint32_t cut_keep;           //   keys kept)
    int last_kept;               // split rows: the buffer's count after the last compaction
    uint32_t lmax;               // split rows: the largest of this CTA's warm-up group maxima
    int hshift;                  // split rows: the first final histogram's bins are 2^hshift keys wide,
    uint32_t hbase;              //   from key hbase up
    const uint8_t* job_stage;    // split rows held whole, the shared dense pass: its chunk,
    int job_on;                  //   the owner's lock,
    int job_next;                //   the next slice to claim (kDenseSlices or more: none open),
    int job_left;                //   slices not yet finished,
    int job_cursor;              //   the next free slot of the pass's reservation,
    int job_p0;                  //   the pass's first vector and the chunk's vectors,
    int job_nvec;
    uint32_t job_tb;             //   the compare bits and the chunk's first row column
    uint32_t job_col0;
};

// Bounded wait on an mbarrier phase.  On expiry it records a timeout in the status word,
// raises the CTA's abort flag and returns false; it also returns false at once when the
// abort flag is already up.
// Each try_wait suspends the thread in hardware for up to 20 us, so a waiting warp costs
// no issue slots and no shared-memory bandwidth.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, Ctrl* ctrl) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<volatile int*>(&ctrl->abort)) return false;
        if (clock64() - t0 > kSpinLimit) {
            set_status(kErrTimeout);
            *reinterpret_cast<volatile int*>(&ctrl->abort) = 1;
            return false;
        }
    }
}

// Barrier over the first NTH threads: named barrier BAR (0 is the CTA barrier).
template <int NTH, int BAR>
__device__ __forceinline__ void team_sync() {
    named_bar_sync(BAR, NTH);
}

// Exclusive prefix sum of v over the team's threads in thread order, plus the team total.
// Two back-to-back scans must use different rows.
template <int NTH, int BAR>
__device__ __forceinline__ uint32_t team_excl_scan(uint32_t v, Ctrl* ctrl, int row, uint32_t& total, int tid) {
    constexpr int NW = NTH / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t incl = warp_incl_scan(v, lane);
    if (lane == 31) ctrl->warp_tot[row][warp] = incl;
    team_sync<NTH, BAR>();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t t = ctrl->warp_tot[row][w];
        all += t;
        before += (w < warp) ? t : 0u;
    }
    total = all;
    return before + incl - v;
}

// Reserves `tot` consecutive candidate slots for the warp; returns the first one.
__device__ __forceinline__ uint32_t warp_reserve(Ctrl* ctrl, uint32_t tot, int lane) {
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(reinterpret_cast<unsigned int*>(&ctrl->cnt), tot);
    return __shfl_sync(0xFFFFFFFFu, base, 0);
}

// Finds the bin holding the krem-th largest key counted in h[0..nbins).  Every thread
// of the team returns total (all counted keys); when total >= krem, bstar is the bin and
// above the number of keys in higher bins.
template <int NTH, int BAR>
__device__ __forceinline__ void find_pivot_bin(const uint32_t* h, int nbins, uint32_t krem, Ctrl* ctrl, int tid,
                                               int& bstar, uint32_t& above, uint32_t& total) {
    constexpr int PER = (kBins + NTH - 1) / NTH;
    constexpr int NW = NTH / 32;
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t c[PER];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int b = tid * PER + j;
        c[j] = (b < nbins) ? h[b] : 0u;
        sum += c[j];
    }
    // inclusive suffix sum within the warp (lane l: bins of lanes >= l)
    uint32_t suf = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suf, d);
        if (lane + d < 32) suf += t;
    }
    if (lane == 0) ctrl->fp_tot[warp] = suf;
    team_sync<NTH, BAR>();
    uint32_t higher = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t t = ctrl->fp_tot[w];
        all += t;
        if (w > warp) higher += t;
    }
    const uint32_t excl = higher + suf - sum;  // keys in bins owned by higher threads
    if (excl < krem && krem <= excl + sum) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = PER - 1; j >= 0; --j) {
            if (acc < krem && acc + c[j] >= krem) {
                ctrl->bstar = tid * PER + j;
                ctrl->above = acc;
                ctrl->bcount = c[j];
            }
            acc += c[j];
        }
    }
    team_sync<NTH, BAR>();
    total = all;
    bstar = ctrl->bstar;
    above = ctrl->above;
}

__device__ __forceinline__ uint32_t group_key(const uint4& g, int e, int es) {
    const uint32_t w = (es == 2) ? ((e >> 1) == 0 ? g.x : (e >> 1) == 1 ? g.y : (e >> 1) == 2 ? g.z : g.w)
                                 : (e == 0 ? g.x : e == 1 ? g.y : e == 2 ? g.z : g.w);
    return (es == 2) ? ((e & 1) ? (w >> 16) : (w & 0xFFFFu)) : w;
}

// Digit shift for the key range [lo, hi].
__device__ __forceinline__ int range_shift(uint32_t lo, uint32_t hi) {
    const int s = bit_length(hi - lo) - kDigitBits;
    return s > 0 ? s : 0;
}

// Histogram of (key - lo) >> s for the keys of [0, n) inside [lo, hi].
// Calls f(i, key) for every key of [0, n) owned by thread `tid`: thread t takes the
// 16-byte groups t, t + NTH, ... (16 / sizeof(KeyT) keys each, in index order), so a warp
// reads contiguous 512-byte rows.  Only the last group pays for bounds checks; the
// candidate buffer is padded to whole groups.
template <typename KeyT, int NTH, typename F>
__device__ __forceinline__ void for_each_key(const KeyT* ckey, int n, int tid, F&& f) {
    constexpr int ES = sizeof(KeyT), GK = 16 / ES;
    const int full = n / GK;
    const uint4* g4 = reinterpret_cast<const uint4*>(ckey);
    int g = tid;
#pragma unroll 2
    for (; g < full; g += NTH) {
        const uint4 v = g4[g];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (ES == 2) {
                f(g * GK + 2 * q, w[q] & 0xFFFFu);
                f(g * GK + 2 * q + 1, w[q] >> 16);
            } else {
                f(g * GK + q, w[q]);
            }
        }
    }
    if (g == full && full * GK < n) {
        const uint4 v = g4[g];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (ES == 2) {
                if (g * GK + 2 * q < n) f(g * GK + 2 * q, w[q] & 0xFFFFu);
                if (g * GK + 2 * q + 1 < n) f(g * GK + 2 * q + 1, w[q] >> 16);
            } else {
                if (g * GK + q < n) f(g * GK + q, w[q]);
            }
        }
    }
}

// Calls f(i0, keys, valid) for each 16-byte group of keys owned by thread `tid` (groups
// t, t + NTH, ...): i0 is the index of the group's first key, keys[] its GK keys and
// valid a bit mask of the keys below n.
template <typename KeyT, int NTH, typename F>
__device__ __forceinline__ void for_each_group(const KeyT* ckey, int n, int tid, F&& f) {
    constexpr int ES = sizeof(KeyT), GK = 16 / ES;
    const int ng = (n + GK - 1) / GK;
    const uint4* g4 = reinterpret_cast<const uint4*>(ckey);
#pragma unroll 2
    for (int g = tid; g < ng; g += NTH) {
        const uint4 v = g4[g];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t keys[GK];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (ES == 2) {
                keys[2 * q] = w[q] & 0xFFFFu;
                keys[2 * q + 1] = w[q] >> 16;
            } else {
                keys[q] = w[q];
            }
        }
        const int left = n - g * GK;
        const uint32_t valid = left >= GK ? ((1u << GK) - 1u) : ((1u << left) - 1u);
        f(g * GK, keys, valid);
    }
}

template <typename KeyT, int NTH>
__device__ __forceinline__ void build_hist(const KeyT* ckey, int n, uint32_t lo, uint32_t hi, int s, uint32_t* hist,
                                           int tid, bool all_in_range) {
    if (all_in_range) {
        for_each_key<KeyT, NTH>(ckey, n, tid, [&](int, uint32_t kk) { atomicAdd(&hist[(kk - lo) >> s], 1u); });
    } else {
        for_each_key<KeyT, NTH>(ckey, n, tid, [&](int, uint32_t kk) {
            if (kk - lo <= hi - lo) atomicAdd(&hist[(kk - lo) >> s], 1u);
        });
    }
}

// The key of rank krem (1 = largest) among the keys in [lo, hi] of the team's buffer, by
// radix passes over adaptive digits.  On return krem is the number of pivot-equal keys
// to keep.  take_all is set when the range holds fewer than krem keys (then every key in
// range is kept).  hist must be zero on entry; it is left dirty.
template <typename KeyT, int NTH, int BAR>
__device__ uint32_t radix_pivot(const KeyT* ckey, int n, uint32_t lo, uint32_t hi, uint32_t& krem, bool& take_all,
                                uint32_t* hist, Ctrl* ctrl, int tid, uint32_t* eq_count = nullptr,
                                bool all_in_range = false) {
    take_all = false;
    for (int pass = 0;; ++pass) {
        const int s = range_shift(lo, hi);
        const int nbins = static_cast<int>((hi - lo) >> s) + 1;
        build_hist<KeyT, NTH>(ckey, n, lo, hi, s, hist, tid, pass == 0 && all_in_range);
        team_sync<NTH, BAR>();
        int bstar;
        uint32_t above, total;
        find_pivot_bin<NTH, BAR>(hist, nbins, krem, ctrl, tid, bstar, above, total);
        if (total < krem) {
            take_all = true;
            return lo;
        }
        krem -= above;
        lo += static_cast<uint32_t>(bstar) << s;
        if (s == 0) {
            if (eq_count) *eq_count = ctrl->bcount;
            return lo;
        }
        const uint32_t top = lo + ((1u << s) - 1u);
        hi = top < hi ? top : hi;
        for (int b = tid; b < ((nbins + 3) & ~3); b += NTH) hist[b] = 0u;
        team_sync<NTH, BAR>();
    }
}

// Team-wide largest key: reduces every thread's running maximum into ctrl->maxkey and
// clears the histogram.  Ends with a team barrier.
template <int NTH, int BAR>
__device__ __forceinline__ uint32_t reduce_max_and_clear(uint32_t tmax, uint32_t* hist, Ctrl* ctrl, int tid) {
    const uint32_t wm = warp_max(tmax);
    if ((tid & 31) == 0) atomicMax(&ctrl->maxkey, wm);
    for (int b = tid; b < kBins; b += NTH) hist[b] = 0u;
    team_sync<NTH, BAR>();
    return ctrl->maxkey;
}

// Exclusive prefix sums of two values at once (one pair of barriers).
template <int NTH, int BAR>
__device__ __forceinline__ void team_excl_scan2(uint32_t a, uint32_t b, Ctrl* ctrl, int row, uint32_t& pa,
                                                uint32_t& pb, uint32_t& ta, uint32_t& tb, int tid) {
    constexpr int NW = NTH / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t ia = warp_incl_scan(a, lane), ib = warp_incl_scan(b, lane);
    if (lane == 31) {
        ctrl->warp_tot[row][warp] = ia;
        ctrl->warp_tot[row][16 + warp] = ib;
    }
    team_sync<NTH, BAR>();
    uint32_t ba = 0, bb = 0, sa = 0, sb = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t x = ctrl->warp_tot[row][w], y = ctrl->warp_tot[row][16 + w];
        sa += x;
        sb += y;
        ba += (w < warp) ? x : 0u;
        bb += (w < warp) ? y : 0u;
    }
    pa = ba + ia - a;
    pb = bb + ib - b;
    ta = sa;
    tb = sb;
}

// RadixSelectTopK on the team's own buffer: keeps exactly k of the n entries (n > k), the
// k largest keys, in positions [0, k).  Keys lie in [lo, ...]; tmax is the thread's
// largest appended key.  Returns the k-th key.  Entries that stay are not moved; entries
// from [k, n) fill the holes in [0, k).
//   One counting pass gives, per thread, the sure holes (key < pivot, i < k), the sure
// fills (key > pivot, i >= k) and the pivot-equal keys on each side of k.  Pivot-equal
// keys draw tickets in thread order (a thread's keys below k come before its keys at or
// above k); the first `quota` are kept.  A listing pass writes the hole positions and
// fill sources, and the moves then run from the two lists, so no load waits on a store
// to the array it reads.
template <typename KeyT, int NTH, int BAR>
__device__ __noinline__ uint32_t compact(KeyT* ckey, uint32_t* cidx, uint32_t* hist, Ctrl* ctrl, int n, int k, uint32_t lo,
                            uint32_t tmax, int tid, bool all_in_range = true) {
    const uint32_t hi = reduce_max_and_clear<NTH, BAR>(tmax, hist, ctrl, tid);
    uint32_t krem = static_cast<uint32_t>(k);
    bool take_all;
    uint32_t eqn = 0;
    const uint32_t pivot =
        radix_pivot<KeyT, NTH, BAR>(ckey, n, lo, hi, krem, take_all, hist, ctrl, tid, &eqn, all_in_range);
    if (take_all) set_status(kErrInternal);  // n > k keys all lie in [lo, hi]
    const uint32_t quota = krem;
    constexpr int GK = 16 / sizeof(KeyT);
    // Per group of GK keys: bit masks of the keys above, equal to and below the pivot,
    // and of the keys below position k; counts are popcounts of their combinations.
    const auto masks = [&](int i0, const uint32_t (&kk)[GK], uint32_t valid, uint32_t& gt, uint32_t& eq,
                           uint32_t& lt, uint32_t& low) {
        gt = 0u;
        eq = 0u;
#pragma unroll
        for (int e = 0; e < GK; ++e) {
            gt |= (kk[e] > pivot ? 1u : 0u) << e;
            eq |= (kk[e] == pivot ? 1u : 0u) << e;
        }
        gt &= valid;
        eq &= valid;
        lt = valid & ~(gt | eq);
        const int below = k - i0;  // keys of the group below position k
        low = below >= GK ? ((1u << GK) - 1u) : (below <= 0 ? 0u : ((1u << below) - 1u));
    };
    // The first MASKED groups of each thread keep their masks in registers for the listing
    // pass (GK bits each, 32 bits of "greater" and 32 of "equal"); later groups recompute.
    constexpr int MASKED = 32 / GK;
    uint32_t gt_keep = 0u, eq_keep_m = 0u;
    uint32_t hdef = 0, fdef = 0, eqlo = 0, eqhi = 0;
    {
        int slot = 0;
        for_each_group<KeyT, NTH>(ckey, n, tid, [&](int i0, const uint32_t (&kk)[GK], uint32_t valid) {
            uint32_t gt, eq, lt, low;
            masks(i0, kk, valid, gt, eq, lt, low);
            hdef += __popc(lt & low);
            fdef += __popc(gt & ~low);
            eqlo += __popc(eq & low);
            eqhi += __popc(eq & ~low);
            if (slot < MASKED) {
                gt_keep |= gt << (slot * GK);
                eq_keep_m |= eq << (slot * GK);
            }
            ++slot;
        });
    }
    // tickets: pivot-equal keys before this thread
    uint32_t e0, junk, te, tj;
    team_excl_scan2<NTH, BAR>(eqlo + eqhi, 0u, ctrl, 0, e0, junk, te, tj, tid);
    const uint32_t keep_lo = quota > e0 ? min(quota - e0, eqlo) : 0u;
    const uint32_t keep_hi = quota > e0 + eqlo ? min(quota - e0 - eqlo, eqhi) : 0u;
    uint32_t h0, f0, th, tf;
    team_excl_scan2<NTH, BAR>(hdef + eqlo - keep_lo, fdef + keep_hi, ctrl, 1, h0, f0, th, tf, tid);
    uint16_t* holes = reinterpret_cast<uint16_t*>(hist);  // at most k positions
    uint16_t* srcs = holes + k;                          // at most k sources
    uint32_t h = h0, f = f0, e = e0;
    const auto list_group = [&](int i0, uint32_t valid, uint32_t gt, uint32_t eq) {
        const int below = k - i0;
        const uint32_t low = below >= GK ? ((1u << GK) - 1u) : (below <= 0 ? 0u : ((1u << below) - 1u));
        uint32_t eq_keep = 0u;
        uint32_t m = eq;
        while (m) {  // pivot-equal keys kept by ticket, in index order
            const int b = __ffs(m) - 1;
            m &= m - 1u;
            if (e++ < quota) eq_keep |= 1u << b;
        }
        const uint32_t keep = gt | eq_keep;
        uint32_t hm = valid & low & ~keep;
        uint32_t fm = keep & ~low;
        while (hm) {
            const int b = __ffs(hm) - 1;
            hm &= hm - 1u;
            if (h < static_cast<uint32_t>(k)) holes[h] = static_cast<uint16_t>(i0 + b);
            ++h;
        }
        while (fm) {
            const int b = __ffs(fm) - 1;
            fm &= fm - 1u;
            if (f < static_cast<uint32_t>(k)) srcs[f] = static_cast<uint16_t>(i0 + b);
            ++f;
        }
    };
    {
        const int ng = (n + GK - 1) / GK;
        int slot = 0;
        int g = tid;
        for (; g < ng && slot < MASKED; g += NTH, ++slot) {
            const int left = n - g * GK;
            const uint32_t valid = left >= GK ? ((1u << GK) - 1u) : ((1u << left) - 1u);
            const uint32_t gm = (gt_keep >> (slot * GK)) & ((1u << GK) - 1u);
            const uint32_t em = (eq_keep_m >> (slot * GK)) & ((1u << GK) - 1u);
            const int below = k - g * GK;
            // groups entirely at or above k with nothing kept, and groups entirely below k
            // with everything kept, contribute no hole and no fill
            if (em == 0u && ((below <= 0 && gm == 0u) || (below >= GK && gm == valid))) continue;
            list_group(g * GK, valid, gm, em);
        }
        const uint4* g4 = reinterpret_cast<const uint4*>(ckey);
        for (; g < ng; g += NTH) {
            const uint4 v = g4[g];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t kk[GK];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (GK == 8) {
                    kk[2 * q] = w[q] & 0xFFFFu;
                    kk[2 * q + 1] = w[q] >> 16;
                } else {
                    kk[q] = w[q];
                }
            }
            const int left = n - g * GK;
            const uint32_t valid = left >= GK ? ((1u << GK) - 1u) : ((1u << left) - 1u);
            uint32_t gt, eq, lt, low;
            masks(g * GK, kk, valid, gt, eq, lt, low);
            list_group(g * GK, valid, gt, eq);
        }
    }
    team_sync<NTH, BAR>();
    if (th != tf || th > static_cast<uint32_t>(k)) set_status(kErrInternal);  // every hole has one fill
    const uint32_t moves = min(min(th, tf), static_cast<uint32_t>(k));
    for (uint32_t m = tid; m < moves; m += NTH) {
        const int j = holes[m], i = srcs[m];
        if (j < k && i < n) {
            ckey[j] = ckey[i];
            cidx[j] = cidx[i];
        }
    }
    if (tid == 0) ctrl->cnt = k;
    team_sync<NTH, BAR>();
    return pivot;
}

// Where the final selection writes.
struct OutTarget {
    void* vals;          // raw values (dtype) -- or keys (uint32) when to_keys
    int32_t* idx;        // columns
    int64_t base;        // first slot of this row (or row-cluster) in vals/idx
    bool to_keys;        // write uint32 keys instead of raw values (cluster partials)
    int esize;           // bytes per raw value
};

// Final RadixSelectTopK over this CTA's candidates.  All NT threads call it.  lo0 bounds
// every key that may belong to the answer from below (keys below it are ignored) and hi0
// every key from above.  Writes min(k, kept) entries and returns that count.
template <typename KeyT, int NT>
__device__ uint32_t final_select(const KeyT* ckey, const uint32_t* cidx, uint32_t* hist, Ctrl* ctrl, int n, int k,
                                 uint32_t lo0, uint32_t hi0, OutTarget out, bool write_ok, int tid) {
    for (int b = tid; b < kBins; b += NT) hist[b] = 0u;
    __syncthreads();
    uint32_t krem = static_cast<uint32_t>(k);
    bool take_all = true;
    uint32_t pivot = 0;
    if (hi0 >= lo0) pivot = radix_pivot<KeyT, NT, 0>(ckey, n, lo0, hi0, krem, take_all, hist, ctrl, tid);
    const uint32_t quota = krem;
    uint32_t gc = 0, ec = 0;
    for (int i = tid; i < n; i += NT) {
        const uint32_t kk = ckey[i];
        const bool inr = kk >= lo0 && kk <= hi0;
        gc += (take_all ? inr : (inr && kk > pivot)) ? 1u : 0u;
        ec += (!take_all && inr && kk == pivot) ? 1u : 0u;
    }
    uint32_t tot;
    const uint32_t pre = team_excl_scan<NT, 0>(gc | (ec << 16), ctrl, 0, tot, tid);
    uint32_t g = pre & 0xFFFFu;
    uint32_t e = pre >> 16;
    for (int i = tid; i < n; i += NT) {
        const uint32_t kk = ckey[i];
        const bool inr = kk >= lo0 && kk <= hi0;
        int64_t slot = -1;
        if (take_all ? inr : (inr && kk > pivot)) {
            slot = g++;
        } else if (!take_all && inr && kk == pivot) {
            const uint32_t t = e++;
            if (t < quota) slot = static_cast<int64_t>(k - quota) + t;
        }
        if (slot >= 0 && write_ok) {
            if (slot < k) {
                const int64_t o = out.base + slot;
                if (out.to_keys) {
                    static_cast<uint32_t*>(out.vals)[o] = kk;
                } else if (out.esize == 2) {
                    static_cast<uint16_t*>(out.vals)[o] = static_cast<uint16_t>(unkey_bf16(kk));
                } else {
                    static_cast<uint32_t*>(out.vals)[o] = unkey_f32(kk);
                }
                out.idx[o] = static_cast<int32_t>(cidx[i]);
            } else {
                set_status(kErrInternal);
            }
        }
    }
    __syncthreads();
    return take_all ? (tot & 0xFFFFu) : static_cast<uint32_t>(k);
}

}  // namespace dsk
