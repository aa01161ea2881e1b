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
    uint64_t full[kMaxStages];   // ring stage filled (one producer arrival + bytes)
    uint64_t empty[kMaxStages];  // ring stage drained (one arrival per consumer warp)
    int issued[kMaxStages];      // copies issued per stage (producer)
    int observed[kMaxStages];    // copies seen complete per stage (consumers)
    int cnt;                     // append cursor of the candidate buffer
    uint32_t maxkey;             // largest key appended so far
    uint32_t sharedT;            // cluster-shared threshold key (authoritative in rank 0), 0 = none
    uint32_t gmax;               // cluster-wide largest key (rank 0)
    int abort;                   // a bounded wait ran out: skip the remaining waits
    int bstar;                   // pivot search results
    uint32_t above;
    uint32_t eq_taken, holes, fills;
    uint32_t out_gt, out_eq;     // output cursors (rank 0 of the cluster)
    uint32_t warp_tot[32];
    uint32_t block_cnt[2][32];   // per-warp appends of the current block, by block parity
    int fin_n;                   // consumer state handed to the whole CTA after the scan
    int fin_hasT;
    uint32_t fin_T;
};

// Bounded wait on an mbarrier phase.  On expiry it records a timeout in the status word,
// raises the CTA's abort flag and returns false; it also returns false at once when the
// abort flag is already up.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, Ctrl* ctrl) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (*reinterpret_cast<volatile int*>(&ctrl->abort)) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > kSpinLimit) {
            set_status(kErrTimeout);
            *reinterpret_cast<volatile int*>(&ctrl->abort) = 1;
            return false;
        }
    }
}

template <int NTH, int BAR>
__device__ __forceinline__ void team_sync() {
    if (BAR == 0 && NTH == 0) {
        __syncthreads();
    } else {
        named_bar_sync(BAR, NTH);
    }
}

// Warp append of up to VEC elements per lane.  `mask` selects the lane's elements,
// keys[e] / cols[e] describe element e.  Returns the number the whole warp appended.
template <typename KeyT, int VEC>
__device__ __forceinline__ uint32_t warp_append(uint32_t mask, const uint32_t (&keys)[VEC], uint32_t col0,
                                                KeyT* ckey, uint32_t* cidx, Ctrl* ctrl, int cap, int lane) {
    const uint32_t c = __popc(mask);
    const uint32_t incl = warp_incl_scan(c, lane);
    const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(reinterpret_cast<unsigned int*>(&ctrl->cnt), tot);
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    uint32_t pos = base + incl - c;
    uint32_t mk = 0;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        if (mask & (1u << e)) {
            if (pos < static_cast<uint32_t>(cap)) {
                ckey[pos] = static_cast<KeyT>(keys[e]);
                cidx[pos] = col0 + e;
            } else {
                set_status(kErrOverflow);
            }
            ++pos;
            mk = max(mk, keys[e]);
        }
    }
    mk = warp_max(mk);
    if (lane == 0 && tot) atomicMax(&ctrl->maxkey, mk);
    return tot;
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
    if (lane == 0) ctrl->warp_tot[warp] = suf;
    team_sync<NTH, BAR>();
    uint32_t higher = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t t = ctrl->warp_tot[w];
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
            }
            acc += c[j];
        }
    }
    team_sync<NTH, BAR>();
    total = all;
    bstar = ctrl->bstar;
    above = ctrl->above;
}

// Digit shift for the key range [lo, hi].
__device__ __forceinline__ int range_shift(uint32_t lo, uint32_t hi) {
    const int s = bit_length(hi - lo) - kDigitBits;
    return s > 0 ? s : 0;
}

// RadixSelectTopK on the team's own buffer: keeps exactly k of the n entries (n > k), the
// k largest keys, in positions [0, k).  lo/hi bound every key.  Returns the k-th key.
// Entries that stay are not moved; entries from [k, n) fill the holes in [0, k).
template <typename KeyT, int NTH, int BAR>
__device__ uint32_t compact(KeyT* ckey, uint32_t* cidx, uint32_t* hist, Ctrl* ctrl, int n, int k, uint32_t lo,
                            uint32_t hi, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t krem = static_cast<uint32_t>(k);
    uint32_t pivot;
    while (true) {
        const int s = range_shift(lo, hi);
        const int nbins = static_cast<int>((hi - lo) >> s) + 1;
        for (int b = tid; b < nbins; b += NTH) hist[b] = 0u;
        team_sync<NTH, BAR>();
        for (int i = tid; i < n; i += NTH) {
            const uint32_t kk = ckey[i];
            if (kk >= lo && kk <= hi) atomicAdd(&hist[(kk - lo) >> s], 1u);
        }
        team_sync<NTH, BAR>();
        int bstar;
        uint32_t above, total;
        find_pivot_bin<NTH, BAR>(hist, nbins, krem, ctrl, tid, bstar, above, total);
        if (total < krem) {  // cannot happen for n > k; keep the team consistent anyway
            set_status(kErrInternal);
            bstar = 0;
            above = 0;
        }
        krem -= above;
        lo = lo + (static_cast<uint32_t>(bstar) << s);
        if (s == 0) {
            pivot = lo;
            break;
        }
        const uint32_t top = lo + ((1u << s) - 1u);
        hi = top < hi ? top : hi;
        // the next pass rewrites hist and bstar only after two more team barriers
    }
    // keep: key > pivot, or key == pivot with a ticket below the quota
    const uint32_t quota = krem;
    if (tid == 0) {
        ctrl->eq_taken = 0;
        ctrl->holes = 0;
        ctrl->fills = 0;
    }
    team_sync<NTH, BAR>();
    uint16_t* holes = reinterpret_cast<uint16_t*>(hist);  // k <= 4096 positions fit
    for (int base = warp * 32; base < k; base += NTH) {
        const int i = base + lane;
        const bool valid = i < k;
        const uint32_t kk = valid ? static_cast<uint32_t>(ckey[i]) : 0u;
        const bool gt = valid && kk > pivot;
        const bool eq = valid && kk == pivot;
        const uint32_t emask = __ballot_sync(0xFFFFFFFFu, eq);
        uint32_t tb = 0;
        if (emask) {
            if (lane == 0) tb = atomicAdd(&ctrl->eq_taken, __popc(emask));
            tb = __shfl_sync(0xFFFFFFFFu, tb, 0);
        }
        const bool keep = gt || (eq && tb + __popc(emask & lanemask_lt()) < quota);
        const bool hole = valid && !keep;
        const uint32_t hmask = __ballot_sync(0xFFFFFFFFu, hole);
        if (hmask) {
            uint32_t hb = 0;
            if (lane == 0) hb = atomicAdd(&ctrl->holes, __popc(hmask));
            hb = __shfl_sync(0xFFFFFFFFu, hb, 0);
            if (hole) holes[hb + __popc(hmask & lanemask_lt())] = static_cast<uint16_t>(i);
        }
    }
    team_sync<NTH, BAR>();
    for (int base = k + warp * 32; base < n; base += NTH) {
        const int i = base + lane;
        const bool valid = i < n;
        const uint32_t kk = valid ? static_cast<uint32_t>(ckey[i]) : 0u;
        const bool gt = valid && kk > pivot;
        const bool eq = valid && kk == pivot;
        const uint32_t emask = __ballot_sync(0xFFFFFFFFu, eq);
        uint32_t tb = 0;
        if (emask) {
            if (lane == 0) tb = atomicAdd(&ctrl->eq_taken, __popc(emask));
            tb = __shfl_sync(0xFFFFFFFFu, tb, 0);
        }
        const bool keep = gt || (eq && tb + __popc(emask & lanemask_lt()) < quota);
        const uint32_t kmask = __ballot_sync(0xFFFFFFFFu, keep);
        if (kmask) {
            uint32_t fb = 0;
            if (lane == 0) fb = atomicAdd(&ctrl->fills, __popc(kmask));
            fb = __shfl_sync(0xFFFFFFFFu, fb, 0);
            if (keep) {
                const uint32_t slot = fb + __popc(kmask & lanemask_lt());
                if (slot < static_cast<uint32_t>(k)) {
                    const int j = holes[slot];
                    ckey[j] = static_cast<KeyT>(kk);
                    cidx[j] = cidx[i];
                } else {
                    set_status(kErrInternal);
                }
            }
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

// Final RadixSelectTopK over the union of the candidates of the cluster's CTAs (CL) or of
// this CTA alone.  All NT threads of every CTA call it.  lo0 bounds every key that may
// belong to the answer from below; keys below it are ignored.  Writes min(k, kept) entries
// and returns that count (meaningful in rank 0; identical everywhere).
template <typename KeyT, int NT, bool CL>
__device__ uint32_t final_select(const KeyT* ckey, const uint32_t* cidx, uint32_t* hist, uint32_t* ghist, Ctrl* ctrl,
                                 int n, int k, uint32_t lo0, uint32_t hi0, int G, OutTarget out, bool write_ok,
                                 int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t lo = lo0, hi = hi0;
    uint32_t krem = static_cast<uint32_t>(k);
    bool take_all = false;
    uint32_t pivot = 0, total0 = 0;
    if (hi0 < lo0) {
        take_all = true;  // nothing in range
    } else {
        for (int pass = 0;; ++pass) {
            const int s = range_shift(lo, hi);
            const int nbins = static_cast<int>((hi - lo) >> s) + 1;
            for (int b = tid; b < nbins; b += NT) hist[b] = 0u;
            __syncthreads();
            for (int i = tid; i < n; i += NT) {
                const uint32_t kk = ckey[i];
                if (kk >= lo && kk <= hi) atomicAdd(&hist[(kk - lo) >> s], 1u);
            }
            const uint32_t* hsum = hist;
            if (CL) {
                cluster_sync_all();
                for (int b = tid; b < nbins; b += NT) {
                    uint32_t g = 0;
                    for (int r = 0; r < G; ++r) g += ld_cluster_u32(map_rank(hist + b, r));
                    ghist[b] = g;
                }
                hsum = ghist;
            }
            __syncthreads();
            int bstar;
            uint32_t above, total;
            find_pivot_bin<NT, 0>(hsum, nbins, krem, ctrl, tid, bstar, above, total);
            if (CL) cluster_sync_all();  // all remote reads of hist done before it is cleared
            if (pass == 0) total0 = total;
            if (total < krem) {  // fewer than k keys in range: keep them all
                take_all = true;
                break;
            }
            krem -= above;
            lo = lo + (static_cast<uint32_t>(bstar) << s);
            if (s == 0) {
                pivot = lo;
                break;
            }
            const uint32_t top = lo + ((1u << s) - 1u);
            hi = top < hi ? top : hi;
            __syncthreads();
        }
    }
    const uint32_t quota = krem;
    const uint32_t kept = take_all ? total0 : static_cast<uint32_t>(k);
    const uint32_t a_gt = CL ? map_rank(&ctrl->out_gt, 0) : 0u;
    const uint32_t a_eq = CL ? map_rank(&ctrl->out_eq, 0) : 0u;
    for (int base = warp * 32; base < n; base += NT) {
        const int i = base + lane;
        const bool valid = i < n;
        const uint32_t kk = valid ? static_cast<uint32_t>(ckey[i]) : 0u;
        const bool inr = valid && kk >= lo0 && kk <= hi0;
        const bool gt = take_all ? inr : (inr && kk > pivot);
        const bool eq = !take_all && inr && kk == pivot;
        const uint32_t gmask = __ballot_sync(0xFFFFFFFFu, gt);
        const uint32_t emask = __ballot_sync(0xFFFFFFFFu, eq);
        uint32_t gb = 0, eb = 0;
        if (lane == 0) {
            if (gmask) gb = CL ? atom_cluster_add_u32(a_gt, __popc(gmask)) : atomicAdd(&ctrl->out_gt, __popc(gmask));
            if (emask) eb = CL ? atom_cluster_add_u32(a_eq, __popc(emask)) : atomicAdd(&ctrl->out_eq, __popc(emask));
        }
        gb = __shfl_sync(0xFFFFFFFFu, gb, 0);
        eb = __shfl_sync(0xFFFFFFFFu, eb, 0);
        int64_t slot = -1;
        if (gt) slot = gb + __popc(gmask & lanemask_lt());
        if (eq) {
            const uint32_t t = eb + __popc(emask & lanemask_lt());
            if (t < quota) slot = static_cast<int64_t>(k - quota) + t;
        }
        if (slot >= 0 && write_ok) {
            if (slot < kept) {
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
    if (CL) cluster_sync_all();
    else __syncthreads();
    return kept;
}

}  // namespace dsk
