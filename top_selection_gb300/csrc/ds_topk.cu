// ds_topk.cu -- GB300 (sm_103a) DeepSelect row-wise top-k: kernels and the C ABI.
//
// DeepSelectTopk (DeepSelect-deep-dive.md, "Algorithm") per row: T = -inf; visit blocks
// of B elements in a random order independent of x; append every element with key > T
// to the candidate buffer; after a block, if the buffer holds >= k + B2 entries, run
// RadixSelectTopK back to k and set T to the smallest kept key; finish with a final
// RadixSelectTopK.
//
// GB300 mapping
//   * Rows processed one CTA each (ds_scan_kernel, the algorithm as written): a producer
//     warp streams the row's blocks, in the row's Philox order, into a ring of shared-
//     memory stages with 1-D bulk copies (cp.async.bulk, completion on mbarriers; the
//     input is read from HBM exactly once, with an L2 evict-first hint).  Consumer warps
//     filter each staged chunk against T with integer compares on the raw bits and
//     append survivors in warp order after one named barrier.  After each block, at
//     >= k + B2 entries, RadixSelectTopK runs in shared memory (ds_select.cuh).
//   * Rows split over several CTAs (ds_split_kernel in ds_split.cuh; the deep dive's
//     "Implementation" section has the CTAs of a thread-block cluster share T through
//     distributed shared memory and select over the union of their candidates).  Rows
//     split over more than one cluster also share T through a global per-row word,
//     write per-cluster results to a workspace, and ds_merge_kernel finishes the row.
//   * No tensor cores: nothing on this path is a dense contraction.
//
// Every wait on an mbarrier is bounded (about one second of SM clock); on expiry the
// CTA records DS_ERR_TIMEOUT in the device status word, stops waiting, keeps its barrier
// sequence so that no other thread is left waiting, and drains its own copies in flight
// before exiting.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <thread>
#include <unordered_map>
#include <vector>

#include "ds_common.cuh"
#include "ds_select.cuh"
#include "ds_topk.h"

namespace dsk {

constexpr int kNCW = 8;                        // consumer warps per CTA
constexpr int kScanThreads = (kNCW + 1) * 32;
constexpr int kMergeThreads = 512;              // one CTA per row over several clusters
constexpr int kChunkBytesMax = 16384;          // one bulk copy
constexpr int kLiteralStages = 8;              // deepest ring of one-CTA rows
constexpr int kSpecMargin = 2;                 // speculative rank: this many times the sample's
constexpr int kSpecMin = 64;                   //   expected share of the top k, at least kSpecMin

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared memory of the one-CTA-per-row kernel.
struct ScanLayout {
    size_t ring, ckey, cidx, hist, perm, ctrl, total;
};

__host__ __device__ inline ScanLayout scan_layout(int es, int chunk, int stages, int cap, int perm_cap) {
    ScanLayout L;
    size_t off = 0;
    L.ring = off;
    off += align_up(static_cast<size_t>(stages) * chunk * es, 128);
    L.ckey = off;
    off += align_up(static_cast<size_t>(cap) * es, 16);
    L.cidx = off;
    off += align_up(static_cast<size_t>(cap) * 4, 16);
    L.hist = off;
    off += kScratchWords * 4;
    L.perm = off;
    off += align_up(static_cast<size_t>(perm_cap) * 4, 16);
    L.ctrl = off;
    off += align_up(sizeof(Ctrl), 16);
    L.total = off;
    return L;
}

struct ScanParams {
    const char* x;
    int64_t rows, N, stride_bytes, m;
    int32_t k, B, B2;
    uint64_t seed;
    void* out_vals;
    int32_t* out_idx;
    long long* stats;
    int32_t parts, G, C;          // CTAs per row, CTAs per cluster, clusters per row
    int32_t chunk, stages, cap, perm_cap;
    int32_t wm;                   // split rows: warm-up group maxima per CTA
    int32_t ww;                   // split rows: chunks sampled by the warm-up (1, 2 or 4)
    int32_t refine;               // split rows: the warm-up refines its pivot bucket (same for all CTAs)
    int32_t cpb;                  // split rows: chunk slots per block, ceil(B / chunk)
    float cpb_rcp;                //   1 / cpb (with a correction step: exact quotients of small ints)
    int32_t slog;                 //   log2 of the ring depth (8 or 16 stages)
    int32_t mr;                   //   m % parts: parts [0, mr) get mq + 1 blocks, the rest mq
    int64_t mq;                   //   m / parts
    int32_t early;                // start reading x before the previous kernel completes
    int32_t rmark, rstep;         // split rows: raise T from the appended keys' histogram when the
                                  //   buffer holds rmark keys, then every rstep more (0 = never)
    int32_t spec_k;               // split rows held whole: the first attempt filters from the
                                  //   spec_k-th largest sampled maximum (0 = never)
    uint32_t epoch;
    unsigned long long* gT;       // per-row shared threshold (C > 1)
    uint32_t* ws_key;             // per (row, cluster) partial results (C > 1)
    int32_t* ws_idx;
    int32_t* ws_cnt;
};

struct MergeParams {
    const uint32_t* ws_key;
    const int32_t* ws_idx;
    const int32_t* ws_cnt;
    int32_t C, k, B2, cap;
    uint32_t epoch;
    const unsigned long long* gT;
    void* out_vals;
    int32_t* out_idx;
};

// ---------------------------------------------------------------- filter ----------
// MODE 0: T = -inf, every element passes.  MODE 1: T >= +0, pass iff (int)bits > thr.
// MODE 2: T <= -0, pass iff (unsigned)bits < thr.  For bf16 each 32-bit word holds two
// values; the low one is shifted up, and thr is the threshold's bits << 16 (| 0xFFFF in
// MODE 1), so one 32-bit compare decides each value.
template <int MODE>
__device__ __forceinline__ uint32_t pass_bits(uint32_t a, uint32_t thr) {
    if (MODE == 1) return static_cast<int32_t>(a) > static_cast<int32_t>(thr) ? 1u : 0u;
    return a < thr ? 1u : 0u;
}

// Warp exclusive prefix of per-lane counts c < 64 and the warp total, from six
// independent ballots of the count's bit planes (no serial shuffle chain).
__device__ __forceinline__ uint32_t warp_prefix_small(uint32_t c, uint32_t& total) {
    const uint32_t lt = lanemask_lt();
    uint32_t pre = 0u, tot = 0u;
#pragma unroll
    for (int b = 0; b < 6; ++b) {
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, (c >> b) & 1u);
        pre += static_cast<uint32_t>(__popc(m & lt)) << b;
        tot += static_cast<uint32_t>(__popc(m)) << b;
    }
    total = tot;
    return pre;
}

// Filters one staged chunk and appends its survivors without atomics.  Each consumer
// thread loads its vectors (t, t + NC, ... up to 4) into registers and the warp releases
// the ring stage at once; survivors are marked in a bit mask (a max/min tree first
// decides whether anything passes at all); each warp publishes its count, and after one
// consumer barrier every warp knows its offset from the counts of the warps before it.
// Warp 0 also takes the row's last < 16 bytes (one element per lane, from global memory).
// Returns the chunk's survivor count, identical in every consumer thread; survivors go to
// positions [n, n + count) in warp order.
template <typename KeyT, int MODE>
__device__ __forceinline__ uint32_t filter_chunk_sync(const uint4* src, int nvec, uint32_t col0, uint32_t thr,
                                                      const char* xrow, int64_t tail_first, int tail_n, bool have,
                                                      uint32_t tk, uint64_t* empty_bar, KeyT* ckey, uint32_t* cidx,
                                                      Ctrl* ctrl, int cap, int tid, int n, int parity,
                                                      uint32_t& tmax) {
    constexpr int NC = kNCW * 32;
    constexpr int ES = sizeof(KeyT);
    constexpr int VEC = 16 / ES;
    constexpr int V = 4;
    const int lane = tid & 31, warp = tid >> 5;
    uint4 v[V];
    int nv = 0;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int vi = tid + j * NC;
        v[j] = make_uint4(0u, 0u, 0u, 0u);
        if (vi < nvec) {
            v[j] = src[vi];
            ++nv;
        }
    }
    uint32_t tkey = 0u;
    bool thit = false;
    if (warp == 0 && lane < tail_n) {
        tkey = ES == 2 ? key_bf16(reinterpret_cast<const uint16_t*>(xrow)[tail_first + lane])
                       : key_f32(reinterpret_cast<const uint32_t*>(xrow)[tail_first + lane]);
        thit = !have || tkey > tk;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);  // the stage is free: everything is in registers
    bool any = true;
    if (MODE != 0) {
        uint32_t r[2 * V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const uint32_t e0 = v[j].x, e1 = v[j].y, e2 = v[j].z, e3 = v[j].w;
            uint32_t a, b;
            if (MODE == 1) {
                a = static_cast<uint32_t>(max(static_cast<int32_t>(e0), static_cast<int32_t>(e1)));
                b = static_cast<uint32_t>(max(static_cast<int32_t>(e2), static_cast<int32_t>(e3)));
                if (ES == 2) {
                    a = static_cast<uint32_t>(max(static_cast<int32_t>(a),
                                                  max(static_cast<int32_t>(e0 << 16), static_cast<int32_t>(e1 << 16))));
                    b = static_cast<uint32_t>(max(static_cast<int32_t>(b),
                                                  max(static_cast<int32_t>(e2 << 16), static_cast<int32_t>(e3 << 16))));
                }
                if (j >= nv) a = b = 0x80000000u;
            } else {
                a = min(e0, e1);
                b = min(e2, e3);
                if (ES == 2) {
                    a = min(a, min(e0 << 16, e1 << 16));
                    b = min(b, min(e2 << 16, e3 << 16));
                }
                if (j >= nv) a = b = 0xFFFFFFFFu;
            }
            r[2 * j] = a;
            r[2 * j + 1] = b;
        }
#pragma unroll
        for (int w = 1; w < 2 * V; w *= 2) {
#pragma unroll
            for (int i = 0; i + w < 2 * V; i += 2 * w) {
                r[i] = (MODE == 1) ? static_cast<uint32_t>(max(static_cast<int32_t>(r[i]), static_cast<int32_t>(r[i + w])))
                                   : min(r[i], r[i + w]);
            }
        }
        any = __any_sync(0xFFFFFFFFu, pass_bits<MODE>(r[0], thr) != 0u);
    }
    uint32_t mask = 0u;
    if (any) {
#pragma unroll
        for (int j = 0; j < V; ++j) {
            if (j < nv) {
                const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                uint32_t bits;
                if (MODE == 0) {
                    bits = (1u << VEC) - 1u;
                } else {
                    uint32_t b0 = 0u, b1 = 0u;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (ES == 4) {
                            b0 |= pass_bits<MODE>(w[q], thr) << q;
                        } else {
                            b0 |= pass_bits<MODE>(w[q] << 16, thr) << (2 * q);
                            b1 |= pass_bits<MODE>(w[q], thr) << (2 * q + 1);
                        }
                    }
                    bits = b0 | b1;
                }
                mask |= bits << (j * VEC);
            }
        }
    }
    const uint32_t c = __popc(mask);
    uint32_t wtot = 0u, pre = 0u;
    if (__any_sync(0xFFFFFFFFu, c != 0u)) pre = warp_prefix_small(c, wtot);
    const uint32_t tmask = __ballot_sync(0xFFFFFFFFu, thit);
    const uint32_t ttot = __popc(tmask);
    if (lane == 0) ctrl->block_cnt[parity][warp] = wtot + ttot;
    named_bar_sync(1, NC);
    uint32_t base = static_cast<uint32_t>(n), total = 0u;
#pragma unroll
    for (int w = 0; w < kNCW; ++w) {
        const uint32_t cw = ctrl->block_cnt[parity][w];
        base += (w < warp) ? cw : 0u;
        total += cw;
    }
    if (static_cast<uint32_t>(n) + total > static_cast<uint32_t>(cap)) {
        set_status(kErrOverflow);
        return 0u;  // nothing written; the buffer keeps its entries (a consistency failure)
    }
    if (wtot) {
        bool done = false;
        if (MODE == 0) {
            // whole warp full: lane-interleaved slots (bank-conflict free stores)
            const int warp_first = tid - lane;
            int full_v = 0;
#pragma unroll
            for (int j = 0; j < V; ++j) full_v += (warp_first + j * NC + 31 < nvec) ? 1 : 0;
            if (full_v > 0 && wtot == 32u * full_v * VEC && c == static_cast<uint32_t>(full_v * VEC)) {
                done = true;
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    if (j < full_v) {
                        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                        const uint32_t col = col0 + static_cast<uint32_t>(tid + j * NC) * VEC;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (ES == 4) {
                                const uint32_t key = key_f32(w[q]);
                                const uint32_t pos = base + (j * 4 + q) * 32 + lane;
                                ckey[pos] = static_cast<KeyT>(key);
                                cidx[pos] = col + q;
                                tmax = max(tmax, key);
                            } else {
                                // two bf16 keys at once: each half inverted if its sign is set,
                                // else its sign bit set
                                const uint32_t kk = w[q] ^ ((((w[q] >> 15) & 0x00010001u) * 0x7FFFu) | 0x80008000u);
                                const uint32_t pos = base + ((j * 4 + q) * 32 + lane) * 2;
                                if ((base & 1u) == 0u) {
                                    *reinterpret_cast<uint32_t*>(ckey + pos) = kk;
                                    *reinterpret_cast<uint2*>(cidx + pos) = make_uint2(col + 2 * q, col + 2 * q + 1);
                                } else {
                                    ckey[pos] = static_cast<KeyT>(kk & 0xFFFFu);
                                    ckey[pos + 1] = static_cast<KeyT>(kk >> 16);
                                    cidx[pos] = col + 2 * q;
                                    cidx[pos + 1] = col + 2 * q + 1;
                                }
                                tmax = max(tmax, max(kk & 0xFFFFu, kk >> 16));
                            }
                        }
                    }
                }
            }
        }
        if (!done) {
            uint32_t pos = base + pre;
            while (mask) {
                const int b = __ffs(mask) - 1;
                mask &= mask - 1u;
                const int j = b / VEC, e = b % VEC;
                uint4 vv = v[0];
                if (j == 1) vv = v[1];
                if (j == 2) vv = v[2];
                if (j == 3) vv = v[3];
                const int q = (e * ES) >> 2;
                uint32_t w = vv.x;
                if (q == 1) w = vv.y;
                if (q == 2) w = vv.z;
                if (q == 3) w = vv.w;
                const uint32_t key = (ES == 4) ? key_f32(w) : key_bf16((e & 1) ? (w >> 16) : (w & 0xFFFFu));
                ckey[pos] = static_cast<KeyT>(key);
                cidx[pos] = col0 + static_cast<uint32_t>(tid + j * NC) * VEC + e;
                ++pos;
                tmax = max(tmax, key);
            }
        }
    }
    if (thit) {
        const uint32_t pos = base + wtot + __popc(tmask & lanemask_lt());
        ckey[pos] = static_cast<KeyT>(tkey);
        cidx[pos] = static_cast<uint32_t>(tail_first + lane);
        tmax = max(tmax, tkey);
    }
    return total;
}

__device__ __forceinline__ void threshold_mode(int es, bool have, uint32_t tk, int& mode, uint32_t& thr) {
    if (!have) {
        mode = 0;
        thr = 0u;
        return;
    }
    if (es == 4) {
        const uint32_t raw = unkey_f32(tk);
        mode = (raw & 0x80000000u) ? 2 : 1;
        thr = raw;
    } else {
        const uint32_t raw = unkey_bf16(tk);
        mode = (raw & 0x8000u) ? 2 : 1;
        thr = (mode == 1) ? ((raw << 16) | 0xFFFFu) : (raw << 16);
    }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kSpinLimit) {
            set_status(kErrTimeout);
            return;
        }
    }
}

// Visiting order of the mp blocks b0, b0 + stride, ..., b0 + (mp - 1) * stride of `row`:
// draw u_b = Philox(seed; b, row) for each block, and place each block at its rank in
// (u_b, b) order -- the row's own order restricted to these blocks.  `draws` is scratch
// of mp words.  Ends with a CTA barrier.
template <int NT>
__device__ void block_order(uint64_t seed, int64_t row, int64_t b0, int64_t stride, int mp, uint32_t* draws,
                            int32_t* perm, int tid) {
    for (int j = tid; j < mp; j += NT) draws[j] = block_draw(seed, row, b0 + j * stride);
    __syncthreads();
    for (int j = tid; j < mp; j += NT) {
        const uint32_t u = draws[j];
        int r = 0;
        for (int j2 = 0; j2 < mp; ++j2) {
            const uint32_t v = draws[j2];
            r += (v < u || (v == u && j2 < j)) ? 1 : 0;
        }
        perm[r] = static_cast<int32_t>(b0 + j * stride);
    }
    __syncthreads();
}

// Exposes block_order for parity checks: one CTA, mp <= kPermMax.
__global__ void __launch_bounds__(256) ds_block_order_kernel(uint64_t seed, int64_t row, int64_t b0, int mp,
                                                              int32_t* out) {
    __shared__ uint32_t draws[kPermMax];
    __shared__ int32_t perm[kPermMax];
    block_order<256>(seed, row, b0, 1, mp, draws, perm, threadIdx.x);
    for (int j = threadIdx.x; j < mp; j += 256) out[j] = perm[j];
}

// Waits on an mbarrier phase that never completes, with the given cycle limit: the same
// bounded wait as the scan kernel, used to check that a wait that runs out is reported
// through the status word and leaves the context usable.
__global__ void ds_wait_probe_kernel(long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        const long long t0 = clock64();
        while (!mbar_try_wait(&bar, 0)) {
            if (clock64() - t0 > limit) {
                set_status(kErrTimeout);
                break;
            }
        }
    }
}

// ---------------------------------------------------------------- scan kernel -----
// One CTA per row, the deep dive's algorithm as written: a producer warp streams the
// row's blocks in Philox order through the copy ring; after each block the consumers
// compact the candidate buffer with RadixSelectTopK once it holds k + B2 entries or more
// (T becomes the k-th key), and a final RadixSelectTopK writes the k results.
template <typename KeyT>
__global__ void __launch_bounds__(kScanThreads, 2) ds_scan_kernel(const ScanParams p) {
    constexpr int NC = kNCW * 32;
    constexpr int NT = kScanThreads;
    constexpr int ES = sizeof(KeyT);
    extern __shared__ __align__(1024) uint8_t smem[];
    const ScanLayout L = scan_layout(ES, p.chunk, p.stages, p.cap, p.perm_cap);
    uint8_t* ring = smem + L.ring;
    KeyT* ckey = reinterpret_cast<KeyT*>(smem + L.ckey);
    uint32_t* cidx = reinterpret_cast<uint32_t*>(smem + L.cidx);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L.hist);
    int32_t* perm = reinterpret_cast<int32_t*>(smem + L.perm);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + L.ctrl);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const int mp = static_cast<int>(p.m);
    const char* xrow = p.x + row * p.stride_bytes;
    const int chunk_bytes = p.chunk * ES;

    // The next kernel on the stream may start as this one's CTAs leave.  This kernel may
    // have started before the previous one completed: it waits for it before reading x
    // (unless the caller stated that x was complete earlier) and before writing anything.
    pdl_launch_dependents();
    {
        int* z = reinterpret_cast<int*>(ctrl);
        for (int i = tid; i < static_cast<int>(sizeof(Ctrl) / sizeof(int)); i += NT) z[i] = 0;
    }
    __syncthreads();
    if (tid < p.stages) {
        mbar_init(&ctrl->full[tid], 1);
        mbar_init(&ctrl->empty[tid], kNCW);
        fence_mbar_init();
    }
    block_order<NT>(p.seed, row, 0, 1, mp, hist, perm, tid);
    if (!p.early) pdl_wait();

    if (warp == kNCW) {
        // ------------------------------ producer: bulk copies in block order ------
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int seq = 0;
            bool stop = false;
            for (int i = 0; i < mp && !stop; ++i) {
                const int64_t lo = static_cast<int64_t>(perm[i]) * p.B;
                const int64_t hi = lo + p.B < p.N ? lo + p.B : p.N;
                for (int64_t c0 = lo; c0 < hi; c0 += p.chunk) {
                    const int64_t ce = (hi - c0) < p.chunk ? (hi - c0) : p.chunk;
                    const uint32_t bytes = static_cast<uint32_t>(ce * ES) & ~15u;
                    const int s = seq % p.stages, use = seq / p.stages;
                    if (use > 0 && !wait_bounded(&ctrl->empty[s], (use - 1) & 1, ctrl)) {
                        stop = true;
                        break;
                    }
                    if (bytes) {
                        mbar_arrive_expect_tx(&ctrl->full[s], bytes);
                        bulk_g2s(ring + static_cast<size_t>(s) * chunk_bytes, xrow + c0 * ES, bytes, &ctrl->full[s],
                                 pol);
                    } else {
                        mbar_arrive(&ctrl->full[s]);
                    }
                    ctrl->issued[s] = use + 1;
                    ++seq;
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------ consumers: filter, append, compact ---------
        int seq = 0;
        int n = 0;
        bool hasT = false;
        uint32_t T = 0u;
        uint32_t badd = 0u;  // appends of the current block
        uint32_t tmax = 0u;
        long long sA = 0, sR = 0, sW = 0, sMax = 0;
        for (int i = 0; i < mp; ++i) {
            const int64_t lo = static_cast<int64_t>(perm[i]) * p.B;
            const int64_t hi = lo + p.B < p.N ? lo + p.B : p.N;
            int mode;
            uint32_t thr;
            threshold_mode(ES, hasT, T, mode, thr);
            for (int64_t c0 = lo; c0 < hi; c0 += p.chunk) {
                const int64_t ce = (hi - c0) < p.chunk ? (hi - c0) : p.chunk;
                const uint32_t bytes = static_cast<uint32_t>(ce * ES) & ~15u;
                const int s = seq % p.stages, use = seq / p.stages;
                const bool got = wait_bounded(&ctrl->full[s], use & 1, ctrl);
                if (got && tid == 0) ctrl->observed[s] = use + 1;
                const uint4* src = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(s) * chunk_bytes);
                const int nvec = got ? static_cast<int>(bytes / 16) : 0;
                const int tail = got ? static_cast<int>(ce - bytes / ES) : 0;
                const uint32_t col0 = static_cast<uint32_t>(c0);
                const int64_t tfirst = c0 + bytes / ES;
                uint32_t add;
                if (mode == 0)
                    add = filter_chunk_sync<KeyT, 0>(src, nvec, col0, thr, xrow, tfirst, tail, hasT, T, &ctrl->empty[s],
                                                     ckey, cidx, ctrl, p.cap, tid, n, seq & 1, tmax);
                else if (mode == 1)
                    add = filter_chunk_sync<KeyT, 1>(src, nvec, col0, thr, xrow, tfirst, tail, hasT, T, &ctrl->empty[s],
                                                     ckey, cidx, ctrl, p.cap, tid, n, seq & 1, tmax);
                else
                    add = filter_chunk_sync<KeyT, 2>(src, nvec, col0, thr, xrow, tfirst, tail, hasT, T, &ctrl->empty[s],
                                                     ckey, cidx, ctrl, p.cap, tid, n, seq & 1, tmax);
                n += static_cast<int>(add);
                badd += add;
                ++seq;
            }
            // end of block: |C| is known in every thread; compact at >= k + B2
            if (tid == 0) {
                sA += badd;
                sMax = n > sMax ? n : sMax;
            }
            badd = 0u;
            if (n >= p.k + p.B2) {
                const uint32_t lo_k = hasT ? T : 0u;
                if (tid == 0) {
                    sW += n;
                    sR += 1;
                }
                T = compact<KeyT, NC, 1>(ckey, cidx, hist, ctrl, n, p.k, lo_k, tmax, tid);
                hasT = true;
                n = p.k;
            }
        }
        const uint32_t wm = warp_max(tmax);
        if (lane == 0) atomicMax(&ctrl->maxkey, wm);
        if (tid == 0) {
            ctrl->fin_n = n;
            ctrl->fin_hasT = hasT ? 1 : 0;
            ctrl->fin_T = T;
            pdl_wait();  // the previous call has completed before this call writes
            if (p.stats) {
                long long* st = p.stats + row * DS_NSTAT;
                st[0] = sA;
                st[1] = sR;
                st[2] = sW + n;
                st[3] = sMax;
                st[4] = mp;
                st[5] = 0;
                st[6] = sR;
                st[7] = 0;
            }
        }
    }
    __syncthreads();
    if (ctrl->abort && tid == 0) {
        for (int s = 0; s < p.stages; ++s)
            if (ctrl->issued[s] > ctrl->observed[s]) drain_wait(&ctrl->full[s], (ctrl->issued[s] - 1) & 1);
    }
    const int n = ctrl->fin_n;

    // ------------------------------ final selection --------------------------------
    OutTarget out;
    out.vals = p.out_vals;
    out.idx = p.out_idx;
    out.base = row * static_cast<int64_t>(p.k);
    out.to_keys = false;
    out.esize = ES;
    const uint32_t lo0 = ctrl->fin_hasT ? ctrl->fin_T : 0u;
    pdl_wait();  // the previous call's outputs are complete before this call writes its own
    final_select<KeyT, NT>(ckey, cidx, hist, ctrl, n, p.k, lo0, ctrl->maxkey, out, !ctrl->abort, tid);
}

}  // namespace dsk

#include "ds_split.cuh"

namespace dsk {

// ---------------------------------------------------------------- merge kernel ----
// The bucket of the kk-th largest count among 2048 (one warp): lane l sums buckets
// [64l, 64l + 64), a suffix scan over the lanes picks the lane, then the lanes split its
// buckets in pairs.  bstar = -1 when all buckets together hold fewer than kk; above =
// the count in buckets above bstar (all of them when bstar = -1), total = all.
__device__ __forceinline__ void warp_bucket_2048(const uint32_t* hist, uint32_t kk, int lane, int& bstar,
                                                 uint32_t& above, uint32_t& total) {
    const uint4* h4 = reinterpret_cast<const uint4*>(hist) + 16 * lane;
    uint32_t t = 0u;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        const uint4 x = h4[(j + lane) & 15];  // rotated: fewer bank conflicts
        t += x.x + x.y + x.z + x.w;
    }
    uint32_t sf = t;  // buckets of lanes >= lane
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_down_sync(0xFFFFFFFFu, sf, d);
        if (lane + d < 32) sf += u;
    }
    total = __shfl_sync(0xFFFFFFFFu, sf, 0);
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, sf >= kk);
    bstar = -1;
    above = total;
    if (!hit) return;
    const int L = 31 - __clz(hit);
    const uint32_t aboveL = __shfl_sync(0xFFFFFFFFu, sf - t, L);
    const uint2 c2 = reinterpret_cast<const uint2*>(hist)[32 * L + lane];
    const uint32_t c = c2.x + c2.y;
    uint32_t s2 = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_down_sync(0xFFFFFFFFu, s2, d);
        if (lane + d < 32) s2 += u;
    }
    const uint32_t hit2 = __ballot_sync(0xFFFFFFFFu, aboveL + s2 >= kk);
    const int J = 31 - __clz(hit2);
    const uint32_t aJ = __shfl_sync(0xFFFFFFFFu, aboveL + s2 - c, J);
    const uint32_t hiJ = __shfl_sync(0xFFFFFFFFu, c2.y, J);
    const bool top = aJ + hiJ >= kk;
    bstar = 64 * L + 2 * J + (top ? 1 : 0);
    above = top ? aJ : aJ + hiJ;
}

// Finishes rows split over C clusters.  Each cluster left its share of its union's top k
// (at most k (key, column) pairs) in the workspace; the row's top k are the k largest of
// these.  They stay in global memory (L2): radix passes of 2048 buckets over the key
// range still in play, [lo, hi], narrow it to the k-th largest key, starting from the
// row's shared threshold (the largest the clusters published: one cluster alone holds k
// pairs at or above it); then one output pass takes the keys above the pivot and the
// quota of pivot-equal keys, slots from two shared cursors.
template <typename KeyT>
__global__ void __launch_bounds__(kMergeThreads, 1) ds_merge_kernel(const MergeParams p) {
    constexpr int NT = kMergeThreads;
    constexpr int ES = sizeof(KeyT);
    __shared__ __align__(16) uint32_t hist[kBins];
    __shared__ int sh_b;
    __shared__ uint32_t sh_above, sh_total;
    __shared__ unsigned int cur_g, cur_e;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const int64_t seg0 = row * p.C;
    uint32_t lo = 0u;
    {
        const unsigned long long g = ld_relaxed_gpu_u64(p.gT + row);
        if (static_cast<uint32_t>(g >> 32) == p.epoch) lo = static_cast<uint32_t>(g);
    }
    const uint32_t lo0 = lo;
    uint32_t hi = ES == 2 ? 0xFFFFu : 0xFFFFFFFFu;
    uint32_t krem = static_cast<uint32_t>(p.k), pivot = 0u, total0 = 0u;
    bool take_all = false;
    if (tid == 0) {
        cur_g = 0u;
        cur_e = 0u;
    }
    for (int pass = 0;; ++pass) {
        const int sb = bit_length(hi - lo) - kDigitBits;
        const int s = sb > 0 ? sb : 0;
        for (int b = tid; b < kBins; b += NT) hist[b] = 0u;
        __syncthreads();
        for (int c = 0; c < p.C; ++c) {
            const int cnt = p.ws_cnt[seg0 + c];
            const uint32_t* sk = p.ws_key + (seg0 + c) * p.k;
            for (int j = tid; j < cnt; j += NT) {
                const uint32_t key = sk[j];
                if (key >= lo && key <= hi) atomicAdd(&hist[(key - lo) >> s], 1u);
            }
        }
        __syncthreads();
        if (warp == 0) {
            int b;
            uint32_t above, total;
            warp_bucket_2048(hist, krem, lane, b, above, total);
            if (lane == 0) {
                sh_b = b;
                sh_above = above;
                sh_total = total;
            }
        }
        __syncthreads();
        const int b = sh_b;
        const uint32_t above = sh_above;
        if (pass == 0) total0 = sh_total;
        __syncthreads();  // sh_* are read before the next pass writes them
        if (b < 0) {  // fewer than krem keys in play: keep them all
            take_all = true;
            break;
        }
        krem -= above;
        lo += static_cast<uint32_t>(b) << s;
        if (s == 0) {
            pivot = lo;
            break;
        }
        hi = lo + ((1u << s) - 1u);
    }
    if (take_all && tid == 0 && total0 < static_cast<uint32_t>(p.k)) set_status(kErrInternal);
    // keys above the pivot take slots [0, k - krem), pivot-equal keys the next krem
    const uint32_t ngt = static_cast<uint32_t>(p.k) - krem;
    const uint32_t ltm = lanemask_lt();
    const int64_t obase = row * static_cast<int64_t>(p.k);
    for (int c = 0; c < p.C; ++c) {
        const int cnt = p.ws_cnt[seg0 + c];
        const uint32_t* sk = p.ws_key + (seg0 + c) * p.k;
        const int32_t* si = p.ws_idx + (seg0 + c) * p.k;
        for (int j0 = 0; j0 < cnt; j0 += NT) {
            const int j = j0 + tid;
            const uint32_t key = j < cnt ? sk[j] : 0u;
            const bool ok = j < cnt && key >= lo0;
            const bool isg = ok && (take_all || key > pivot);
            const bool ise = ok && !take_all && key == pivot;
            const uint32_t bg = __ballot_sync(0xFFFFFFFFu, isg);
            const uint32_t be = __ballot_sync(0xFFFFFFFFu, ise);
            if ((bg | be) == 0u) continue;
            uint32_t gb = 0u, eb = 0u;
            if (lane == 0) {
                if (bg) gb = atomicAdd(&cur_g, static_cast<unsigned int>(__popc(bg)));
                if (be) eb = atomicAdd(&cur_e, static_cast<unsigned int>(__popc(be)));
            }
            gb = __shfl_sync(0xFFFFFFFFu, gb, 0) + static_cast<uint32_t>(__popc(bg & ltm));
            eb = __shfl_sync(0xFFFFFFFFu, eb, 0) + static_cast<uint32_t>(__popc(be & ltm));
            const uint32_t slot = isg ? gb : ngt + eb;
            const bool put = isg || (ise && eb < krem);
            if (put && slot < static_cast<uint32_t>(p.k)) {
                if (ES == 2) static_cast<uint16_t*>(p.out_vals)[obase + slot] = static_cast<uint16_t>(unkey_bf16(key));
                else static_cast<uint32_t*>(p.out_vals)[obase + slot] = unkey_f32(key);
                p.out_idx[obase + slot] = si[j];
            } else if (put) {
                set_status(kErrInternal);
            }
        }
    }
}

// ---------------------------------------------------------------- sorted output ---
// The optional last step of the operation (the pages' sorted_value flag; the DeepSelect
// TopK tutorial notes that sorting happens only at the end, on the k survivors): each
// row's k results, already exact, are put in order of key descending, column ascending.
// One CTA per row sorts (key << 32 | ~column) descending with a bitonic network in
// shared memory over the next power of two >= k (padding 0 sorts last: a real entry's
// low word ~column is never 0, as columns are below 2^31).
constexpr int kSortThreads = 512;

// Loads row `row`'s k results into sv as (key << 32 | ~column), sorts them descending
// (bitonic network over n2, the next power of two >= k) and writes them back in order.
// All kSortThreads threads of the CTA call it; ends with a CTA barrier.
template <typename KeyT>
__device__ __forceinline__ void sort_row_desc(void* vals, int32_t* idx, int64_t base, int k, int n2,
                                              unsigned long long* sv, int tid) {
    constexpr int ES = sizeof(KeyT);
    for (int i = tid; i < n2; i += kSortThreads) {
        unsigned long long c = 0ull;
        if (i < k) {
            const uint32_t raw = ES == 2 ? static_cast<const uint16_t*>(vals)[base + i]
                                         : static_cast<const uint32_t*>(vals)[base + i];
            const uint32_t key = ES == 2 ? key_bf16(raw) : key_f32(raw);
            c = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx[base + i]));
        }
        sv[i] = c;
    }
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < (n2 >> 1); t += kSortThreads) {
                const int lo = 2 * t - (t & (stride - 1));  // first of the pair (lo, lo + stride)
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;        // this run sorts descending
                const unsigned long long a = sv[lo], b = sv[hi];
                if ((a < b) == desc) {
                    sv[lo] = b;
                    sv[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < k; i += kSortThreads) {
        const unsigned long long c = sv[i];
        const uint32_t key = static_cast<uint32_t>(c >> 32);
        if (ES == 2) static_cast<uint16_t*>(vals)[base + i] = static_cast<uint16_t>(unkey_bf16(key));
        else static_cast<uint32_t*>(vals)[base + i] = unkey_f32(key);
        idx[base + i] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(c));
    }
    __syncthreads();
}

// Runs after the top-k kernel(s) on the stream (see launch_row_kernel).
template <typename KeyT>
__global__ void __launch_bounds__(kSortThreads) ds_sort_kernel(void* vals, int32_t* idx, int k, int n2) {
    extern __shared__ __align__(16) unsigned long long sv[];
    pdl_launch_dependents();
    pdl_wait();
    sort_row_desc<KeyT>(vals, idx, static_cast<int64_t>(blockIdx.x) * k, k, n2, sv, threadIdx.x);
}

// ---------------------------------------------------------------- sampling ------
// Top-k sampling, the second place the pages put top-k (the DeepSelect TopK tutorial,
// section 1.1: the sampler picks candidate tokens from the vocabulary's logits with
// top-k).  After the sorted top-k of a row (value descending, equal values by column
// ascending), candidate i gets weight e_i = exp((v_i - v_0) / temperature) and the token
// is the candidate at the first i whose running sum of weights exceeds u * (sum of all
// weights), u being the row's uniform draw in [0, 1) (supplied by the caller).  One CTA
// per row: it sorts the row's k results in shared memory (and writes them back sorted),
// then each thread sums a run of consecutive candidates, a CTA scan gives each run's
// offset, and the count of running sums <= u * total is the chosen position.  fp32
// throughout (expf, sums in this fixed order).
constexpr int kSampleThreads = kSortThreads;

template <typename KeyT>
__global__ void __launch_bounds__(kSampleThreads) ds_sample_kernel(void* vals, int32_t* idx, int k, int n2,
                                                                   float inv_temp, const float* uniforms,
                                                                   int32_t* out_token, float* out_prob) {
    constexpr int ES = sizeof(KeyT);
    extern __shared__ __align__(16) unsigned long long sv[];
    __shared__ float wsum[kSampleThreads / 32];
    __shared__ int wcnt[kSampleThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * k;
    pdl_launch_dependents();
    pdl_wait();  // the top-k results are complete
    sort_row_desc<KeyT>(vals, idx, base, k, n2, sv, tid);  // sorted, also in sv
    const auto value = [&](int i) -> float {
        const uint32_t key = static_cast<uint32_t>(sv[i] >> 32);
        return ES == 2 ? __uint_as_float(unkey_bf16(key) << 16) : __uint_as_float(unkey_f32(key));
    };
    const float v0 = value(0);
    const int per = (k + kSampleThreads - 1) / kSampleThreads;
    const int i0 = tid * per, i1 = min(i0 + per, k);
    float run = 0.f;
    for (int i = i0; i < i1; ++i) run += expf((value(i) - v0) * inv_temp);
    // exclusive scan of the runs over the CTA (warp scan, then the warp totals)
    float incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    float before = 0.f, total = 0.f;
    for (int w = 0; w < kSampleThreads / 32; ++w) {
        const float t = wsum[w];
        before += w < warp ? t : 0.f;
        total += t;
    }
    before += incl - run;
    const float target = uniforms[blockIdx.x] * total;
    // positions whose running sum is <= target: the token is the next one
    int cnt = 0;
    float acc = before;
    for (int i = i0; i < i1; ++i) {
        acc += expf((value(i) - v0) * inv_temp);
        cnt += acc <= target ? 1 : 0;
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, d);
    if (lane == 0) wcnt[warp] = cnt;
    __syncthreads();
    if (tid == 0) {
        int c = 0;
        for (int w = 0; w < kSampleThreads / 32; ++w) c += wcnt[w];
        const int pos = c < k ? c : k - 1;
        out_token[blockIdx.x] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(sv[pos]));
        if (out_prob) out_prob[blockIdx.x] = expf((value(pos) - v0) * inv_temp) / total;
    }
}

// Launches a per-row kernel of the sorted-output family (one CTA per row).  A plain
// launch: it starts once the top-k results are complete.  (Letting these CTAs start early
// under programmatic dependent launch was slower: 54.0 against 49.9 us per sampling call
// on the sampler shape.)  The kernels still let a following programmatic launch start
// early, and wait for their predecessor, which is a no-op here.
template <typename Kern, typename... Args>
static ds_status launch_row_kernel(Kern kern, int64_t rows, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
    cfg.blockDim = dim3(kSortThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

// ================================================================ host ============

struct DevInfo {
    int sms = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    bool ok = false;
};

static std::mutex g_mu;
static DevInfo g_dev[64];
static std::atomic<uint32_t> g_epoch{0};

// Library-owned workspaces (rows split over several clusters), one per (device, stream):
// calls on one stream are ordered, so they may share a workspace; calls on different
// streams never do.  The per-thread default stream is a different stream in every thread,
// so it is keyed by thread as well.  A workspace that is outgrown is retired, not freed:
// a launch already enqueued (on this or an earlier call) may still use it, and freeing it
// safely would need a device-wide synchronisation.  Growth is geometric, so the retired
// buffers hold less than the live one.
struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
struct WsKey {
    int dev;
    cudaStream_t stream;
    std::thread::id thread;
    bool operator==(const WsKey& o) const { return dev == o.dev && stream == o.stream && thread == o.thread; }
};
struct WsKeyHash {
    size_t operator()(const WsKey& k) const {
        return std::hash<const void*>()(k.stream) ^ (std::hash<std::thread::id>()(k.thread) << 1) ^
               static_cast<size_t>(k.dev) * 0x9E3779B97F4A7C15ull;
    }
};
static std::unordered_map<WsKey, Workspace, WsKeyHash> g_ws;
static std::vector<void*> g_ws_retired;

// Scratch for ds_topk_noalloc: a fixed array in the library's device image.  Every device
// that loads the library holds it until the process exits; calls share it.
constexpr size_t kStaticWorkspaceBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];
static void* g_static_ws_addr[64];  // device address of g_static_ws, per device

static bool dev_info(int dev, DevInfo& out) {
    if (dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev];
    if (!d.ok) {
        bool ok = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess;
        if (!ok) {
            // Planning queries without a device (host tests): DS_PLAN_DEVICE="sms,smem_optin,smem_per_sm"
            // describes one.  Launches still need the real device.
            const char* e = std::getenv("DS_PLAN_DEVICE");
            if (!e || std::sscanf(e, "%d,%d,%d", &d.sms, &d.smem_optin, &d.smem_per_sm) != 3 || d.sms < 1)
                return false;
            cudaGetLastError();
        }
        d.ok = true;
    }
    out = d;
    return true;
}

struct Plan {
    int dev, es, parts, G, C, chunk, stages, cap, perm_cap, ctas_per_sm, wm, ww, refine;
    int B, B2;  // block size and compaction slack in effect (the library's choice when given as 0)
    bool split;  // the split-row kernel (also for one part per row), else the one-CTA-per-row kernel
    bool held;   // split rows: every CTA's chunks fit its ring at once
    int spec_k;  // split rows held whole in one cluster: the speculative rank (0 = none)
    int64_t m;
    size_t smem, merge_smem, ws_bytes;
    int merge_cap;
    size_t off_gT, off_key, off_idx, off_cnt;
};

// B = 0 or B2 = 0 asks the library to choose them.  The choice follows the shipped CUDA
// configuration the DeepSelect TopK tutorial describes (section 4.7, the wave rule of
// api.cpp): with num_waves = ceil(rows / SMs) equal to 1 the block is 8192 elements,
// otherwise 4096; the compaction slack (reconstruct threshold) is 4096.  Both are Theta(k)
// for the supported k <= 4096, which the expected-work bound needs (tutorial section 3.7).
static ds_status resolve_blocks(int dev, int64_t rows, int32_t& B, int32_t& B2) {
    if (B < 0 || B2 < 0) return DS_ERR_INVALID_ARG;
    if (B == 0) {
        DevInfo di;
        if (!dev_info(dev, di)) return DS_ERR_CUDA;
        const int64_t waves = (rows + di.sms - 1) / di.sms;
        B = waves <= 1 ? 8192 : 4096;
    }
    if (B2 == 0) B2 = 4096;
    return DS_OK;
}

static ds_status validate(const void* x, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride, int32_t k,
                          int32_t B, int32_t B2, const void* out_vals, const int32_t* out_idx) {
    if (dtype != DS_BF16 && dtype != DS_FP32) return DS_ERR_INVALID_ARG;
    if (rows < 0 || N < 1 || k < 1 || k > N || B < 1 || B2 < 1 || row_stride < N) return DS_ERR_INVALID_ARG;
    if (rows > 0 && (!x || !out_vals || !out_idx)) return DS_ERR_INVALID_ARG;
    const int es = dtype == DS_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out_vals) |
         reinterpret_cast<uintptr_t>(out_idx)) & 15u)
        return DS_ERR_ALIGNMENT;
    if (rows > 1 && (row_stride * es) % 16 != 0) return DS_ERR_ALIGNMENT;
    if (k > kMaxK || N >= (int64_t(1) << 31)) return DS_ERR_UNSUPPORTED;
    if ((static_cast<int64_t>(B) * es) % 16 != 0) return DS_ERR_UNSUPPORTED;
    return DS_OK;
}

static ds_status make_plan(int dev, int32_t dtype, int64_t rows, int64_t N, int32_t k, int32_t B, int32_t B2,
                           const ds_options* opt, Plan& P) {
    DevInfo di;
    if (!dev_info(dev, di)) return DS_ERR_CUDA;
    P.dev = dev;
    P.B = B;
    P.B2 = B2;
    P.es = dtype == DS_BF16 ? 2 : 4;
    P.m = (N + B - 1) / B;
    P.chunk = B < kChunkBytesMax / P.es ? B : kChunkBytesMax / P.es;
    int64_t cap64 = static_cast<int64_t>(k) + B + B2;
    if (cap64 > (int64_t(1) << 20)) return DS_ERR_UNSUPPORTED;
    int parts = opt ? opt->parts : 0;
    if (parts < 0) return DS_ERR_INVALID_ARG;
    if (parts == 0 && opt && opt->stats) parts = 1;  // the statistics describe the one-CTA schedule
    const bool spread = N * P.es >= (int64_t(16) << 20);
    bool split1 = false;
    if (parts == 0) {
        // Enough CTAs to cover the SMs: rows split in parts of at least 4 blocks.  Rows under
        // 16 MB stay in one cluster (at most 16 CTAs: no merge pass) and are not split so
        // finely that a warp would get no chunk; larger rows spread over several clusters
        // and a merge kernel.
        parts = 1;
        const int64_t maxp = P.m / 4 > 1 ? P.m / 4 : 1;
        const int64_t fillp = N / (static_cast<int64_t>(P.chunk) * kNCW);
        const int64_t capp = spread ? 256 : 16;
        while (rows * parts < di.sms && parts * 2 <= maxp && parts * 2 <= capp && (spread || parts * 2 <= fillp))
            parts *= 2;
        // Rows that already cover the SMs run one per CTA in the split-row kernel (its
        // warm-up threshold, k + at least one chunk of candidates, two CTAs per SM where
        // they fit); the one-CTA-per-row kernel of the pages' schedule keeps the
        // statistics, explicit parts = 1 and rows of fewer than 8 blocks.
        split1 = parts == 1 && maxp >= 2;
        while ((P.m + parts - 1) / parts > kPermMax) parts *= 2;
        if (parts > P.m) return DS_ERR_UNSUPPORTED;
    } else {
        if (parts > P.m || (P.m + parts - 1) / parts > kPermMax) return DS_ERR_UNSUPPORTED;
    }
    P.parts = parts;
    // (split rows keep k entries plus one chunk's survivors: a warp reserves a chunk's
    // slots at once and a reservation that does not fit triggers a compaction; their
    // capacity is set with the chunk below)
    P.cap = static_cast<int>(cap64);
    P.perm_cap = static_cast<int>((P.m + parts - 1) / parts);
    int G = opt ? opt->cluster : 0;
    if (G < 0 || G > 16) return DS_ERR_INVALID_ARG;
    if (G == 0) {
        // one cluster per row when a row has at most 16 parts and no more than 16 MB
        G = 1;
        const int gmax = (!spread && parts <= 16) ? 16 : 8;
        while (G * 2 <= gmax && parts % (G * 2) == 0) G *= 2;
    }
    if (parts % G != 0) return DS_ERR_INVALID_ARG;
    P.G = G;
    P.C = parts / G;
    if (opt && opt->stats && parts != 1) return DS_ERR_INVALID_ARG;
    P.wm = 0;
    P.ww = 1;
    P.refine = 0;
    P.held = false;
    P.spec_k = 0;
    P.split = parts > 1 || split1;
    if (P.split) {
        // Split rows: each consumer warp owns whole chunks, so the ring depth is a multiple
        // of the consumer warps (every stage is then used by one warp only, and a warp
        // never waits on a stage whose previous fill belongs to another warp).  Take the
        // largest chunk (halving from 16 KB, at least 1 KB) whose layout lets two CTAs
        // share an SM, 16 stages before 8; else the largest that fits one CTA.
        // The warm-up samples the first ww chunks of each CTA (up to 16 vectors per thread,
        // never more chunks than the CTA with the fewest has).
        const auto warm_chunks = [&](int chunk, int stages) {
            const int64_t per = (static_cast<int64_t>(B) + chunk - 1) / chunk;
            const int64_t nq_min = (P.m / parts) * per;
            const int cvec = chunk * P.es / 16;
            int w = 1;
            // rows streamed through the ring sample up to 8 chunks when a CTA has the row to
            // itself, 4 in a cluster (whose union of maxima is larger already); rows held
            // whole 2: their filter waits for the sample's threshold
            const int wmax = nq_min > stages ? (G == 1 ? 8 : 4) : 2;
            while (w * 2 <= wmax && w * 2 <= stages && w * 2 * cvec <= 16 * kNCW * 32 && w * 2 <= nq_min) w *= 2;
            return w;
        };
        int ww_try = 1;
        const auto warm_groups = [&](int chunk) {
            // R group maxima per consumer thread (groups of whole vectors), enough for
            // about 4k in the cluster's union when they fit the exchange
            const int vt = (ww_try * chunk * P.es / 16 + kNCW * 32 - 1) / (kNCW * 32);
            int R = 1;
            // (up to 4 groups per thread for samples of up to 8 vectors, 8 for larger ones;
            // a CTA without a cluster exchanges nothing and takes twice as many)
            const int rmax = vt > 8 ? 8 : 4;
            const int64_t umax = (G == 1 ? 8 : 4) * static_cast<int64_t>(k);
            while (R * 2 <= vt && R * 2 <= rmax && static_cast<int64_t>(G) * 256 * R * 2 * P.es <= kWarmMaxBytes &&
                   static_cast<int64_t>(G) * 256 * R < umax)
                R *= 2;
            return 256 * R;
        };
        const auto fit = [&](int chunk, int stages, size_t limit) -> bool {
            int cap = static_cast<int>(align_up(static_cast<size_t>(k) + chunk, 16 / P.es));
            ww_try = warm_chunks(chunk, stages);
            const int wm = warm_groups(chunk);
            size_t need = split_layout(P.es, chunk, stages, cap, G, wm, k, P.perm_cap).total;
            if (need > limit) return false;
            // the shared memory left over widens the candidate buffer (fewer compactions)
            const int unit_c = 16 / P.es * 16;  // keeps the buffer's arrays 16-byte aligned
            const int extra = static_cast<int>((limit - need) / (P.es + 4)) / unit_c * unit_c;
            if (extra > 0 && static_cast<int64_t>(cap) + extra <= (int64_t(1) << 20)) {
                const size_t need2 = split_layout(P.es, chunk, stages, cap + extra, G, wm, k, P.perm_cap).total;
                if (need2 <= limit) {
                    cap += extra;
                    need = need2;
                }
            }
            P.chunk = chunk;
            P.stages = stages;
            P.cap = cap;
            P.wm = wm;
            P.ww = ww_try;
            // Rows streamed through the ring (more chunks per CTA than stages) gain more from
            // a tighter warm-up threshold than its extra pass costs; rows held whole do not.
            P.refine = (P.m / parts) * ((static_cast<int64_t>(B) + chunk - 1) / chunk) > stages ? 1 : 0;
            P.smem = need;
            return true;
        };
        const int unit = 16 / P.es;
        const int first = B < kChunkBytesMax / P.es ? B : kChunkBytesMax / P.es;
        const size_t two = static_cast<size_t>(di.smem_per_sm) / 2 - 1024;
        bool ok = false;
        // Rows whose CTAs each get an SM of their own (rows x parts <= SMs) keep each part's
        // chunks in the ring at once where a ring of at most 16 stages of at most 8 KB fits
        // an SM's whole shared memory: every copy issues at start-up and the rows run the
        // held instance, instead of streaming through a ring sized for two CTAs per SM.
        if (rows * parts <= di.sms) {
            const int c = first * P.es <= 8192 ? first : 8192 / P.es;
            const int64_t chunks = (P.m + parts - 1) / parts * ((static_cast<int64_t>(B) + c - 1) / c);
            if (chunks <= 2 * kNCW) ok = fit(c, chunks <= kNCW ? kNCW : 2 * kNCW, static_cast<size_t>(di.smem_optin));
        }
        for (int c = first; !ok && c * P.es >= 1024; c = (c / 2) / unit * unit)
            ok = fit(c, 2 * kNCW, two) || fit(c, kNCW, two);
        for (int c = first; !ok && c * P.es >= 1024; c = (c / 2) / unit * unit)
            ok = fit(c, kNCW, static_cast<size_t>(di.smem_optin));
        if (!ok && first * P.es < 1024) ok = fit(first, kNCW, static_cast<size_t>(di.smem_optin));
        if (!ok) return DS_ERR_UNSUPPORTED;
        // (held rows also keep chunks of at most 8 KB: their warm-up samples at most two
        // chunks, so a thread's sample is at most 4 vectors)
        P.held = (P.m + parts - 1) / parts * ((static_cast<int64_t>(B) + P.chunk - 1) / P.chunk) <= P.stages &&
                 P.chunk * P.es <= 8192;
        // Rows held whole in one cluster speculate: the cluster's sample of S elements holds
        // about k * S / N of the row's k largest, so its spec_k-th largest maximum, spec_k
        // twice that, likely lies below the row's k-th largest and well above the proven
        // edge.  The final select checks it, and a failure filters the resident chunks once
        // more.  Too small a spec_k (a noisy estimate) or one not below k turns it off.
        if (P.held && G == parts) {
            const int64_t S = static_cast<int64_t>(G) * P.ww * P.chunk;
            const int64_t sk = (kSpecMargin * static_cast<int64_t>(k) * S + N - 1) / N;
            if (sk >= kSpecMin && sk < k) P.spec_k = static_cast<int>(sk);
        }
    } else {
        const auto layout_bytes = [&](int s) -> size_t {
            return scan_layout(P.es, P.chunk, s, P.cap, P.perm_cap).total;
        };
        // Ring depth: the deepest ring (3..8) that still lets two CTAs share an SM;
        // otherwise the deepest ring that fits one CTA (at least 2 stages).
        P.stages = 0;
        for (int s = kLiteralStages; s >= 3; --s) {
            if (2 * (layout_bytes(s) + 1024) <= static_cast<size_t>(di.smem_per_sm)) {
                P.stages = s;
                break;
            }
        }
        if (P.stages == 0) {
            for (int s = kLiteralStages; s >= 2; --s) {
                if (layout_bytes(s) <= static_cast<size_t>(di.smem_optin)) {
                    P.stages = s;
                    break;
                }
            }
        }
        if (P.stages == 0) return DS_ERR_UNSUPPORTED;
        P.smem = layout_bytes(P.stages);
    }
    P.ctas_per_sm = static_cast<int>(di.smem_per_sm / (P.smem + 1024));
    if (P.ctas_per_sm < 1) P.ctas_per_sm = 1;
    P.ws_bytes = 0;
    P.merge_smem = 0;
    P.merge_cap = 0;
    if (P.C > 1) {
        P.merge_cap = k;
        P.merge_smem = 0;  // the merge kernel's shared memory is static
        size_t off = 0;
        P.off_gT = off;
        off = align_up(off + rows * 8, 256);
        P.off_key = off;
        off = align_up(off + static_cast<size_t>(rows) * P.C * k * 4, 256);
        P.off_idx = off;
        off = align_up(off + static_cast<size_t>(rows) * P.C * k * 4, 256);
        P.off_cnt = off;
        off = align_up(off + static_cast<size_t>(rows) * P.C * 4, 256);
        P.ws_bytes = off;
    }
    return DS_OK;
}

// Raises a kernel's dynamic shared-memory limit (and allows 16-CTA clusters) once per
// device; later calls that need no more than what was set make no runtime call, so a
// call under stream capture only launches.
template <typename Kern>
static cudaError_t set_smem(Kern kern, int slot, int dev, size_t bytes, bool nonportable) {
    static size_t done[16][64];
    static bool np_done[16][64];
    std::lock_guard<std::mutex> lk(g_mu);
    if (done[slot][dev] < bytes) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
        if (e != cudaSuccess) return e;
        done[slot][dev] = bytes;
    }
    if (nonportable && !np_done[slot][dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        np_done[slot][dev] = true;
    }
    return cudaSuccess;
}

template <typename KeyT>
static ds_status launch(const Plan& P, const void* x, int64_t rows, int64_t N, int64_t row_stride, int32_t k,
                        int32_t B, int32_t B2, uint64_t seed, void* out_vals, int32_t* out_idx, long long* stats,
                        char* ws, bool early, bool sorted, cudaStream_t stream) {
    ScanParams sp;
    sp.x = static_cast<const char*>(x);
    sp.rows = rows;
    sp.N = N;
    sp.stride_bytes = row_stride * P.es;
    sp.m = P.m;
    sp.k = k;
    sp.B = B;
    sp.B2 = B2;
    sp.seed = seed;
    sp.out_vals = out_vals;
    sp.out_idx = out_idx;
    sp.stats = stats;
    sp.parts = P.parts;
    sp.G = P.G;
    sp.C = P.C;
    sp.chunk = P.chunk;
    sp.stages = P.stages;
    sp.cap = P.cap;
    sp.perm_cap = P.perm_cap;
    sp.wm = P.wm;
    sp.ww = P.ww;
    sp.refine = P.refine;
    sp.cpb = static_cast<int32_t>((B + P.chunk - 1) / P.chunk);
    sp.cpb_rcp = 1.0f / static_cast<float>(sp.cpb);
    sp.slog = P.stages >= 16 ? 4 : 3;
    sp.mq = P.m / P.parts;
    sp.mr = static_cast<int32_t>(P.m % P.parts);
    sp.early = early ? 1 : 0;
    // Streamed rows raise their threshold from the appended keys' histogram: first when
    // the buffer holds k keys plus a step (or half of its room past k), then every step.
    sp.rstep = P.split && P.refine ? (k > 256 ? k : 256) : 0;
    sp.rmark = sp.rstep ? k + (sp.rstep < (P.cap - k) / 2 ? sp.rstep : (P.cap - k) / 2) : 0;
    sp.spec_k = P.spec_k;
    sp.epoch = 0;
    sp.gT = nullptr;
    sp.ws_key = nullptr;
    sp.ws_idx = nullptr;
    sp.ws_cnt = nullptr;
    if (P.C > 1) {
        uint32_t e = g_epoch.fetch_add(1) + 1;
        if (e == 0) e = g_epoch.fetch_add(1) + 1;
        sp.epoch = e;
        sp.gT = reinterpret_cast<unsigned long long*>(ws + P.off_gT);
        sp.ws_key = reinterpret_cast<uint32_t*>(ws + P.off_key);
        sp.ws_idx = reinterpret_cast<int32_t*>(ws + P.off_idx);
        sp.ws_cnt = reinterpret_cast<int32_t*>(ws + P.off_cnt);
    }
    void (*kern)(ScanParams);
    int slot = sizeof(KeyT) == 2 ? 0 : 1;
    if (!P.split) {
        kern = ds_scan_kernel<KeyT>;
    } else {
        // one instance per plan class: held whole or streamed, one cluster or several
        kern = P.held ? (P.C > 1 ? ds_split_kernel<KeyT, true, true> : ds_split_kernel<KeyT, true, false>)
                      : (P.C > 1 ? ds_split_kernel<KeyT, false, true> : ds_split_kernel<KeyT, false, false>);
        slot += 8 + 2 * (P.held ? 1 : 0) + 4 * (P.C > 1 ? 1 : 0);
    }
    if (set_smem(kern, slot, P.dev, P.smem, P.G > 8) != cudaSuccess) return DS_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows * P.parts), 1, 1);
    cfg.blockDim = dim3(P.split ? kSplitThreads : kScanThreads, 1, 1);
    cfg.dynamicSmemBytes = P.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    // programmatic dependent launch: consecutive calls on a stream overlap their edges
    // (each kernel waits for its predecessor before its first global write)
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (P.G > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = P.G;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kern, sp) != cudaSuccess) return DS_ERR_CUDA;
    if (P.C > 1) {
        MergeParams mp;
        mp.ws_key = sp.ws_key;
        mp.ws_idx = sp.ws_idx;
        mp.ws_cnt = sp.ws_cnt;
        mp.C = P.C;
        mp.k = k;
        mp.B2 = B2;
        mp.cap = P.merge_cap;
        mp.epoch = sp.epoch;
        mp.gT = sp.gT;
        mp.out_vals = out_vals;
        mp.out_idx = out_idx;
        auto mk = ds_merge_kernel<KeyT>;
        if (set_smem(mk, 6 + (sizeof(KeyT) == 2 ? 0 : 1), P.dev, P.merge_smem, false) != cudaSuccess)
            return DS_ERR_CUDA;
        mk<<<static_cast<unsigned>(rows), kMergeThreads, P.merge_smem, stream>>>(mp);
        if (cudaGetLastError() != cudaSuccess) return DS_ERR_CUDA;
    }
    if (sorted && k > 1) {  // after the results above are complete
        int n2 = 1;
        while (n2 < k) n2 <<= 1;
        return launch_row_kernel(ds_sort_kernel<KeyT>, rows, n2 * sizeof(unsigned long long), stream, out_vals,
                                 out_idx, static_cast<int>(k), n2);
    }
    return DS_OK;
}

static ds_status library_workspace(int dev, size_t bytes, cudaStream_t stream, void** out) {
    const bool per_thread = stream == cudaStreamPerThread;
    const WsKey key{dev, stream, per_thread ? std::this_thread::get_id() : std::thread::id()};
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_ws[key];
    if (w.bytes >= bytes) {
        *out = w.ptr;
        return DS_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return DS_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return DS_ERR_WORKSPACE;
    void* p = nullptr;
    const size_t grow = bytes + bytes / 4;
    if (cudaMalloc(&p, grow) != cudaSuccess) return DS_ERR_CUDA;
    // zeroed on the caller's stream, so the clear is ordered before this call's launches
    // (the per-row threshold words carry a call number; zero is never a live one)
    if (cudaMemsetAsync(p, 0, grow, stream) != cudaSuccess) {
        cudaFree(p);
        return DS_ERR_CUDA;
    }
    if (w.ptr) g_ws_retired.push_back(w.ptr);
    w.ptr = p;
    w.bytes = grow;
    *out = p;
    return DS_OK;
}

}  // namespace dsk

using namespace dsk;

extern "C" {

ds_status ds_get_plan(int32_t dtype, int64_t rows, int64_t N, int32_t k, int32_t B, int32_t B2,
                      const ds_options* options, ds_plan* plan) {
    if (!plan) return DS_ERR_INVALID_ARG;
    if (dtype != DS_BF16 && dtype != DS_FP32) return DS_ERR_INVALID_ARG;
    if (rows < 0 || N < 1 || k < 1 || k > N || B < 0 || B2 < 0) return DS_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {  // no device: only a described one (DS_PLAN_DEVICE) plans
        cudaGetLastError();
        if (!std::getenv("DS_PLAN_DEVICE")) return DS_ERR_CUDA;
        dev = 0;
    }
    ds_status rs = resolve_blocks(dev, rows, B, B2);
    if (rs != DS_OK) return rs;
    const int es = dtype == DS_BF16 ? 2 : 4;
    if (k > kMaxK || N >= (int64_t(1) << 31) || (static_cast<int64_t>(B) * es) % 16 != 0) return DS_ERR_UNSUPPORTED;
    Plan P;
    const ds_status st = make_plan(dev, dtype, rows, N, k, B, B2, options, P);
    if (st != DS_OK) return st;
    plan->parts = P.parts;
    plan->cluster = P.G;
    plan->threads = P.split ? kSplitThreads : kScanThreads;
    plan->chunk_elems = P.chunk;
    plan->stages = P.stages;
    plan->capacity = P.cap;
    plan->smem_bytes = static_cast<int64_t>(P.smem);
    plan->workspace_bytes = static_cast<int64_t>(P.ws_bytes);
    plan->ctas_per_sm = P.ctas_per_sm;
    plan->merge_launch = P.C > 1 ? 1 : 0;
    plan->B = P.B;
    plan->B2 = P.B2;
    plan->spec_k = P.spec_k;
    return DS_OK;
}

ds_status ds_workspace_bytes(int32_t dtype, int64_t rows, int64_t N, int32_t k, int32_t B, int32_t B2,
                             const ds_options* options, size_t* bytes) {
    if (!bytes) return DS_ERR_INVALID_ARG;
    ds_plan pl;
    const ds_status st = ds_get_plan(dtype, rows, N, k, B, B2, options, &pl);
    if (st != DS_OK) return st;
    *bytes = static_cast<size_t>(pl.workspace_bytes);
    return DS_OK;
}

ds_status ds_topk_ex(const void* x, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride, int32_t k,
                     int32_t B, int32_t B2, uint64_t seed, void* out_vals, int32_t* out_idx,
                     const ds_options* options, cudaStream_t stream) {
    if (B < 0 || B2 < 0) return DS_ERR_INVALID_ARG;
    if (rows > 0 && (B == 0 || B2 == 0)) {  // the library's choice (resolve_blocks)
        int d = 0;
        if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return DS_ERR_CUDA;
        const ds_status rs = resolve_blocks(d, rows, B, B2);
        if (rs != DS_OK) return rs;
    }
    ds_status st = validate(x, dtype, rows, N, row_stride, k, B ? B : 4096, B2 ? B2 : 4096, out_vals, out_idx);
    if (st != DS_OK) return st;
    if (rows == 0) return DS_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DS_ERR_CUDA;
    if (dev < 0 || dev >= 64) return DS_ERR_CUDA;
    Plan P;
    st = make_plan(dev, dtype, rows, N, k, B, B2, options, P);
    if (st != DS_OK) return st;
    if (rows * P.parts > 0x7FFFFFFFLL) return DS_ERR_UNSUPPORTED;
    char* ws = nullptr;
    if (P.ws_bytes > 0) {
        if (options && options->workspace) {
            if (options->workspace_bytes < P.ws_bytes) return DS_ERR_WORKSPACE;
            if (reinterpret_cast<uintptr_t>(options->workspace) & 255u) return DS_ERR_ALIGNMENT;
            ws = static_cast<char*>(options->workspace);
        } else {
            void* p = nullptr;
            st = library_workspace(dev, P.ws_bytes, stream, &p);
            if (st != DS_OK) return st;
            ws = static_cast<char*>(p);
        }
    }
    long long* stats = options ? reinterpret_cast<long long*>(options->stats) : nullptr;
    const bool early = options && options->input_ready;
    const bool sorted = options && options->sorted;
    if (dtype == DS_BF16)
        return launch<uint16_t>(P, x, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, stats, ws, early,
                                sorted, stream);
    return launch<uint32_t>(P, x, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, stats, ws, early, sorted,
                            stream);
}

ds_status ds_topk(const void* x, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride, int32_t k, int32_t B,
                  int32_t B2, uint64_t seed, void* out_vals, int32_t* out_idx, cudaStream_t stream) {
    return ds_topk_ex(x, dtype, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, nullptr, stream);
}

// The same launch as ds_topk_ex, for callers that must not allocate: when the launch
// needs scratch (rows split over several clusters) it uses g_static_ws instead of a
// cudaMalloc'ed workspace.  Host code cannot use the array's name as a device address,
// so the first call on each device (with that device current) looks the address up
// with cudaGetSymbolAddress and keeps it.  Nothing in the scratch has to start at zero:
// the per-row shared thresholds carry a call number and stale ones are ignored, and the
// partial results and their counts are written before they are read in the same call.
ds_status ds_topk_noalloc(const void* x, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride, int32_t k,
                          int32_t B, int32_t B2, uint64_t seed, void* out_vals, int32_t* out_idx, int32_t parts,
                          int32_t cluster, cudaStream_t stream) {
    if (B < 0 || B2 < 0) return DS_ERR_INVALID_ARG;
    if (rows > 0 && (B == 0 || B2 == 0)) {  // the library's choice (resolve_blocks)
        int d = 0;
        if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return DS_ERR_CUDA;
        const ds_status rs = resolve_blocks(d, rows, B, B2);
        if (rs != DS_OK) return rs;
    }
    ds_status st = validate(x, dtype, rows, N, row_stride, k, B ? B : 4096, B2 ? B2 : 4096, out_vals, out_idx);
    if (st != DS_OK) return st;
    if (rows == 0) return DS_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DS_ERR_CUDA;
    if (dev < 0 || dev >= 64) return DS_ERR_CUDA;
    ds_options opt = {};
    opt.parts = parts;
    opt.cluster = cluster;
    Plan P;
    st = make_plan(dev, dtype, rows, N, k, B, B2, &opt, P);
    if (st != DS_OK) return st;
    if (rows * P.parts > 0x7FFFFFFFLL) return DS_ERR_UNSUPPORTED;
    if (P.ws_bytes > kStaticWorkspaceBytes) return DS_ERR_WORKSPACE;
    char* ws = nullptr;
    if (P.ws_bytes > 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_static_ws_addr[dev]) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_static_ws) != cudaSuccess || !addr) return DS_ERR_CUDA;
            g_static_ws_addr[dev] = addr;
        }
        ws = static_cast<char*>(g_static_ws_addr[dev]);
    }
    if (dtype == DS_BF16)
        return launch<uint16_t>(P, x, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, nullptr, ws, false,
                                false, stream);
    return launch<uint32_t>(P, x, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, nullptr, ws, false,
                            false, stream);
}

size_t ds_noalloc_scratch_bytes(void) { return kStaticWorkspaceBytes; }

// Top-k sampling: the top-k of each row (ds_topk_ex), then ds_sample_kernel sorts each
// row's k results in place and draws one token per row from the softmax of the k values.
ds_status ds_topk_sample(const void* logits, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride, int32_t k,
                         int32_t B, int32_t B2, uint64_t seed, float temperature, const float* uniforms,
                         void* out_vals, int32_t* out_idx, int32_t* out_token, float* out_prob,
                         cudaStream_t stream) {
    if (!(temperature > 0.f) || !(temperature < INFINITY)) return DS_ERR_INVALID_ARG;
    if (rows > 0 && (!uniforms || !out_token)) return DS_ERR_INVALID_ARG;
    const ds_status st = ds_topk_ex(logits, dtype, rows, N, row_stride, k, B, B2, seed, out_vals, out_idx, nullptr,
                                    stream);
    if (st != DS_OK || rows == 0) return st;
    const float inv = 1.0f / temperature;
    int n2 = 1;
    while (n2 < k) n2 <<= 1;
    const size_t smem = n2 * sizeof(unsigned long long);
    if (dtype == DS_BF16)
        return launch_row_kernel(ds_sample_kernel<uint16_t>, rows, smem, stream, out_vals, out_idx,
                                 static_cast<int>(k), n2, inv, uniforms, out_token, out_prob);
    return launch_row_kernel(ds_sample_kernel<uint32_t>, rows, smem, stream, out_vals, out_idx, static_cast<int>(k),
                             n2, inv, uniforms, out_token, out_prob);
}

ds_status ds_get_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DS_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, dsk::g_ds_status, sizeof(v)) != cudaSuccess) return DS_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(dsk::g_ds_status, &zero, sizeof(zero)) != cudaSuccess) return DS_ERR_CUDA;
    if (v & kErrTimeout) return DS_ERR_TIMEOUT;
    if (v & (kErrOverflow | kErrInternal)) return DS_ERR_INTERNAL;
    return DS_OK;
}

const char* ds_status_string(ds_status s) {
    switch (s) {
        case DS_OK: return "ok";
        case DS_ERR_INVALID_ARG: return "invalid argument";
        case DS_ERR_ALIGNMENT: return "misaligned pointer or row stride";
        case DS_ERR_UNSUPPORTED: return "unsupported size or parameter";
        case DS_ERR_CUDA: return "CUDA runtime error";
        case DS_ERR_TIMEOUT: return "device-side wait timed out";
        case DS_ERR_INTERNAL: return "device-side consistency check failed";
        case DS_ERR_WORKSPACE: return "workspace too small or unavailable";
    }
    return "unknown status";
}

const char* ds_version(void) { return "ds_topk 0.1 sm_103a"; }

ds_status ds_block_order(uint64_t seed, int64_t row, int64_t first_block, int32_t nblocks, int32_t* out_perm,
                         cudaStream_t stream) {
    if (!out_perm || nblocks < 1 || nblocks > kPermMax || row < 0 || first_block < 0) return DS_ERR_INVALID_ARG;
    ds_block_order_kernel<<<1, 256, 0, stream>>>(seed, row, first_block, nblocks, out_perm);
    return cudaGetLastError() == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

ds_status ds_wait_probe(int64_t cycles, cudaStream_t stream) {
    if (cycles < 0 || cycles > kSpinLimit) return DS_ERR_INVALID_ARG;
    ds_wait_probe_kernel<<<1, 32, 0, stream>>>(cycles);
    return cudaGetLastError() == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

}  // extern "C"
