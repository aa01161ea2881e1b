// ds_common.cuh -- device helpers for the DeepSelect top-k kernels (sm_103a).
//
// Inline PTX for mbarriers, 1-D bulk copies (cp.async.bulk), thread-block-cluster
// shared memory, and the order-preserving key of IEEE values used everywhere in the
// library (DeepSelect TopK tutorial, section 4.6: floats are "distorted" to unsigned
// integers whose order is the value order).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dsk {

// ------------------------------------------------------------------ limits --------
constexpr int kDigitBits = 11;                 // radix-select digit width
constexpr int kBins = 1 << kDigitBits;         // 2048 histogram bins
constexpr int kScratchWords = 4096;            // histogram, or the hole and fill lists (2 x 4096 u16)
constexpr int kMaxK = 4096;                    // largest k the pages support
constexpr int kPermMax = 1024;                 // blocks one CTA may visit
constexpr int kMaxStages = 16;                 // deepest copy ring
constexpr long long kSpinLimit = 2000000000LL; // ~1 s of SM clock for any single wait

// device status bits (OR-ed into the per-device status word)
enum : uint32_t { kErrTimeout = 1u, kErrOverflow = 2u, kErrInternal = 4u };

// ------------------------------------------------------------------ keys ----------
// key(bits): sign set -> ~bits, sign clear -> bits | sign.  Unsigned order of keys is
// the value order, with -0 < +0 and NaNs at the two ends by sign.
__device__ __forceinline__ uint32_t key_f32(uint32_t b) {
    return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}
__device__ __forceinline__ uint32_t unkey_f32(uint32_t k) {
    return (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
}
// 16-bit value h in the low half of a register
__device__ __forceinline__ uint32_t key_bf16(uint32_t h) {
    const uint32_t s = static_cast<uint32_t>(static_cast<int32_t>(h << 16) >> 31);
    return (h ^ (s | 0x8000u)) & 0xFFFFu;
}
__device__ __forceinline__ uint32_t unkey_bf16(uint32_t k) {
    return ((k & 0x8000u) ? (k ^ 0x8000u) : ~k) & 0xFFFFu;
}

// ------------------------------------------------------------------ Philox --------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11), first output word.
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

__device__ __forceinline__ uint32_t block_draw(uint64_t seed, int64_t row, int64_t b) {
    return philox_word0(static_cast<uint32_t>(b), static_cast<uint32_t>(row),
                        static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32), 0u,
                        static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

// ------------------------------------------------------------------ PTX -----------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread until the phase completes or
// `hint_ns` nanoseconds pass, so that waiting warps do not occupy issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Arrive on an mbarrier of any CTA of the cluster (a shared::cluster address from mapa),
// releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// try_wait with cluster-scope acquire: after it succeeds, writes that other CTAs released
// with their arrivals are visible.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// 1-D bulk copy global -> this CTA's shared memory, completion counted in bytes on bar.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 1-D bulk copy from this CTA's shared memory into another CTA of the cluster: dst and
// bar are shared::cluster addresses (from mapa) in the receiving CTA, whose mbarrier
// counts the bytes.  Addresses and size are multiples of 16 bytes.
__device__ __forceinline__ void bulk_s2s_cluster(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "r"(smem_u32(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Makes this thread's generic-proxy writes to shared memory visible to bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Packed threshold compares.  Each result lane is all ones where a > b or the two are
// unordered (either is NaN), else zero: 16-bit lanes for two bf16 values per word.
__device__ __forceinline__ uint32_t set_gtu_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("set.gtu.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t set_gtu_f32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("set.gtu.u32.f32 %0, %1, %2;" : "=r"(d) : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)));
    return d;
}

// Programmatic dependent launch: let the stream's next kernel start launching its CTAs
// as this one's leave, and wait until the stream's previous kernel has completed and its
// memory operations are visible.  Both are no-ops for kernels launched without it.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- thread-block cluster ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// address of the same shared variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.relaxed.cluster.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.relaxed.cluster.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void red_cluster_max_u32(uint32_t addr, uint32_t v) {
    asm volatile("red.relaxed.cluster.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_cluster_add_u32(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// inclusive warp prefix sum
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v += t;
    }
    return v;
}

__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    return v;
}

__device__ __forceinline__ int bit_length(uint32_t v) { return v ? 32 - __clz(v) : 0; }

}  // namespace dsk
