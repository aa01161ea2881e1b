/*
 * ds_topk.h -- C ABI of the GB300 DeepSelect row-wise top-k library (libds_topk.so).
 *
 * The operation is DeepSelectTopk as defined in DeepSelect-deep-dive.md ("Algorithm"):
 * for every row of N scores, keep a threshold T (initially -inf), visit the row in
 * blocks of B elements in a random block order that does not depend on the data,
 * append every element greater than T to an on-chip candidate buffer, and when the
 * buffer holds at least k + B2 entries after a block, shrink it back to its k largest
 * entries (RadixSelectTopK) and set T to the smallest of them.  A final RadixSelectTopK
 * returns k values and their int32 column indices.  The split-row mode that spreads one
 * row over several CTAs and merges their candidates follows the same page's
 * "Implementation" section (thread-block cluster paragraph).
 *
 * Order of values.  Values are compared by their IEEE bit patterns mapped to an
 * order-preserving unsigned key (sign set: invert all bits; sign clear: set the sign
 * bit), the mapping the DeepSelect TopK tutorial (section 4.6) uses for radix
 * selection.  This is a total order: -NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN.
 *
 * Block order.  Block b of row r is visited in the order of
 *   u_b = Philox4x32-10(key = (seed & 0xffffffff, seed >> 32), counter = (b, r, 0, 0))[0]
 * ascending, ties by b (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
 * SC'11).  When a row is split into P parts, part p takes every P-th block from block p
 * (blocks p, p + P, p + 2P, ...) and visits them in the order of the same draws.
 *
 * Results.  out_vals[r*k + j] / out_idx[r*k + j], j < k, hold the k largest values of
 * row r (bit copies of the input) and their columns, in no particular order (in order of
 * value descending, equal values by column ascending, with ds_options.sorted).  Among
 * values equal to the k-th largest, which columns are returned is unspecified; the
 * value multiset is always exact.
 *
 * All calls are asynchronous on `stream` and return once the work is enqueued.  Errors
 * found on the host are returned before anything is launched.  Errors found on the
 * device (a bounded wait that ran out) are recorded in a per-device status word that
 * ds_get_device_status() reads.  Nothing here allocates memory except ds_topk() when a
 * row is split over more than one cluster (see ds_topk_ex).
 */
#ifndef DS_TOPK_H
#define DS_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same declaration as the CUDA runtime's; a cudaStream_t may be passed directly. */
typedef struct CUstream_st* cudaStream_t;

typedef enum {
    DS_BF16 = 0, /* 16-bit bfloat16, passed as raw 16-bit patterns */
    DS_FP32 = 1  /* 32-bit IEEE float */
} ds_dtype;

typedef enum {
    DS_OK = 0,
    DS_ERR_INVALID_ARG = 1, /* null pointer, rows < 0, N < 1, k < 1, k > N, B < 0, B2 < 0,
                               row_stride < N, unknown dtype                          */
    DS_ERR_ALIGNMENT = 2,   /* x, out_vals or out_idx not 16-byte aligned, or (rows > 1)
                               row_stride * sizeof(element) not a multiple of 16       */
    DS_ERR_UNSUPPORTED = 3, /* k > 4096, N >= 2^31, B * sizeof(element) not a multiple of
                               16, or the candidate buffer (k + B + B2 entries) and the
                               copy ring do not fit in one SM's shared memory         */
    DS_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute, alloc)    */
    DS_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (ds_get_device_status) */
    DS_ERR_INTERNAL = 6,    /* a device-side consistency check failed                   */
    DS_ERR_WORKSPACE = 7    /* caller workspace too small, or would allocate while the
                               stream is being captured                               */
} ds_status;

/* Number of int64 statistics per row written by ds_topk_ex (options.stats). */
#define DS_NSTAT 8
/* statistics layout, per row: A (elements appended), R (in-loop compactions),
   W (total input size of all compactions, the final one included), max |C|,
   m = ceil(N/B), 0, R, 0 -- the quantities of the expected-work analysis of
   DeepSelect-deep-dive.md ("Expected Upper Bound"). */

/*
 * ds_topk -- row-wise top-k of `rows` rows.
 *   x           device pointer; row r starts at element r*row_stride.  16-byte aligned.
 *   dtype       DS_BF16 or DS_FP32.
 *   rows        number of rows (0: nothing is done, DS_OK).
 *   N           elements per row, 1 <= N < 2^31.
 *   row_stride  elements between row starts, >= N; when rows > 1, row_stride*sizeof(element)
 *               must be a multiple of 16 bytes (1024 recommended).
 *   k           1 <= k <= min(N, 4096).
 *   B, B2       block size and compaction slack of the method (>= 1), or 0 for the
 *               library's choice: B = 8192 when the rows fit one wave of CTAs
 *               (ceil(rows / SMs) == 1) and 4096 otherwise, B2 = 4096 -- the shipped
 *               CUDA configuration the DeepSelect TopK tutorial describes (section 4.7);
 *               ds_get_plan reports the values in effect.  B*sizeof(element) must be a
 *               multiple of 16 bytes, k + B + B2 <= 2^20, and one CTA visits at most 1024
 *               blocks (with one CTA per row: ceil(N/B) <= 1024).
 *   seed        selects the block order (see above).
 *   out_vals    device, rows*k elements of dtype; 16-byte aligned.  Caller-owned.
 *   out_idx     device, rows*k int32; 16-byte aligned.  Caller-owned.
 *   stream      CUDA stream (0 = legacy default stream).
 * The library chooses how many CTAs share a row: rows split over a cluster, or rows
 * that already fill the GPU one per CTA, run the split-row kernel (warm-up threshold
 * from a sample of the row, compaction when a chunk's survivors do not fit; rows held
 * whole in one cluster start from a speculative threshold, checked and redone when it
 * was too high -- ds_plan.spec_k); only ds_topk_ex with parts = 1 runs the pages'
 * one-CTA schedule exactly.  Results are exact on every path.  When a row is
 * split over more than one thread-block cluster it uses a library-owned workspace, one
 * per (device, stream) -- per thread as well for cudaStreamPerThread -- so calls on
 * different streams may run concurrently.  It is grown with cudaMalloc (and cleared with
 * cudaMemsetAsync on `stream`) on a call that is not being stream-captured; a call under
 * capture that would need to grow it returns DS_ERR_WORKSPACE.  An outgrown workspace is
 * kept, not freed, until the process exits (launches already enqueued may still use it),
 * so growing never synchronises the device.  Launches let the
 * next kernel on the stream start as this one's CTAs leave (programmatic dependent
 * launch); a call reads x only once the kernel before it has completed (see
 * ds_options.input_ready).
 */
ds_status ds_topk(const void* x, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride,
                  int32_t k, int32_t B, int32_t B2, uint64_t seed, void* out_vals,
                  int32_t* out_idx, cudaStream_t stream);

typedef struct {
    int32_t parts;          /* CTAs per row: 0 = library choice; 1 = one CTA per row (the
                               pages' schedule, required for stats); P > 1 splits each
                               row's blocks into P interleaved sets (block b to part
                               b mod P)                                               */
    int32_t cluster;        /* CTAs per thread-block cluster (divides parts, <= 16);
                               0 = library choice                                     */
    int64_t* stats;         /* optional device array rows*DS_NSTAT, parts == 1 only    */
    void* workspace;        /* optional caller-owned device workspace; NULL = library  */
    size_t workspace_bytes; /* its size; see ds_workspace_bytes                        */
    int32_t input_ready;    /* 0 (default): the call reads x only after every earlier
                               kernel on the stream has completed, so x may be written
                               by the kernel just before it.  Nonzero: the caller states
                               that x was complete before that kernel started, and the
                               call starts reading x while that kernel is still running
                               (consecutive calls on static inputs overlap their edges) */
    int32_t sorted;         /* nonzero: each row's k results in order of value descending
                               (the key order above), equal values by column ascending
                               -- the pages' sorted_value flag; a second kernel sorts the
                               k results of each row in shared memory at the end      */
} ds_options;

/* ds_topk with explicit options (NULL = defaults, identical to ds_topk). */
ds_status ds_topk_ex(const void* x, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride,
                     int32_t k, int32_t B, int32_t B2, uint64_t seed, void* out_vals,
                     int32_t* out_idx, const ds_options* options, cudaStream_t stream);

/* The launch the library would use for these arguments (host only, no launch). */
typedef struct {
    int32_t parts;          /* CTAs per row                                            */
    int32_t cluster;        /* CTAs per cluster                                        */
    int32_t threads;        /* threads per CTA                                         */
    int32_t chunk_elems;    /* elements per bulk copy                                  */
    int32_t stages;         /* depth of the copy ring                                  */
    int32_t capacity;       /* candidate-buffer entries: k + B + B2 for rows of one CTA;
                               at least k + one chunk for split rows, widened into the
                               shared memory the layout leaves over                    */
    int64_t smem_bytes;     /* dynamic shared memory per CTA                           */
    int64_t workspace_bytes;/* device workspace needed (0 unless split over clusters)  */
    int32_t ctas_per_sm;    /* resident CTAs per SM for this configuration             */
    int32_t merge_launch;   /* 1 when a second (merge) kernel runs                      */
    int32_t B;              /* block size in effect (the library's choice when 0 was passed) */
    int32_t B2;             /* compaction slack in effect (likewise)                   */
    int32_t spec_k;         /* rows held whole in one cluster: the first attempt filters
                               from an estimate of the spec_k-th largest sampled group
                               maximum, a threshold nothing proves; the final select
                               checks that k keys reach it and otherwise filters the
                               row's chunks, still in shared memory, from the proven
                               threshold (0 = no speculation)                          */
} ds_plan;

/* Errors as ds_topk's host checks (DS_ERR_INVALID_ARG, DS_ERR_UNSUPPORTED), and
   DS_ERR_CUDA when no device can be queried.  Without a device, the environment variable
   DS_PLAN_DEVICE="sms,smem_optin,smem_per_sm" (SM count and the two shared-memory limits
   in bytes) describes one, for planning only; launches still need the real device. */
ds_status ds_get_plan(int32_t dtype, int64_t rows, int64_t N, int32_t k, int32_t B, int32_t B2,
                      const ds_options* options, ds_plan* plan);

/* Workspace bytes ds_topk_ex needs for these arguments (0 when none). */
ds_status ds_workspace_bytes(int32_t dtype, int64_t rows, int64_t N, int32_t k, int32_t B,
                             int32_t B2, const ds_options* options, size_t* bytes);

/*
 * ds_topk_sample -- top-k sampling, the sampler use of top-k (DeepSelect TopK tutorial,
 * section 1.1: at sampling time top-k picks the candidate tokens out of the vocabulary's
 * logits).  Per row: the k largest logits, sorted as with ds_options.sorted (value
 * descending, equal values by column ascending), are written to out_vals / out_idx as by
 * ds_topk_ex; candidate i gets weight w_i = exp((v_i - v_0) / temperature); the row's
 * token is out_idx[row*k + j] for the first j whose running sum w_0 + ... + w_j exceeds
 * uniforms[row] * (w_0 + ... + w_{k-1}) (the last candidate if rounding leaves none), and
 * out_prob[row] = w_j / (sum of all w).  Weights and sums are fp32, summed in candidate
 * order.
 *   logits, dtype .. seed, out_vals, out_idx   as ds_topk (B = 0 / B2 = 0 allowed)
 *   temperature  > 0 and finite, else DS_ERR_INVALID_ARG
 *   uniforms     device, rows floats in [0, 1): the caller's random draws (one per row)
 *   out_token    device, rows int32: the sampled column of each row
 *   out_prob     device, rows floats, or NULL: the sampled candidate's probability
 * Logits are expected finite (an infinite or NaN logit makes the weights undefined; the
 * top-k part is exact for any values).  Asynchronous on `stream`.
 */
ds_status ds_topk_sample(const void* logits, int32_t dtype, int64_t rows, int64_t N, int64_t row_stride,
                         int32_t k, int32_t B, int32_t B2, uint64_t seed, float temperature,
                         const float* uniforms, void* out_vals, int32_t* out_idx, int32_t* out_token,
                         float* out_prob, cudaStream_t stream);

/* Synchronizes `stream`, then reads and clears the calling device's status word:
   DS_OK, DS_ERR_TIMEOUT or DS_ERR_INTERNAL. */
ds_status ds_get_device_status(cudaStream_t stream);

/* Static description of a status code. */
const char* ds_status_string(ds_status status);

/* Library version, e.g. "ds_topk 0.1 sm_103a". */
const char* ds_version(void);

/* The block visiting order the scan kernel uses (see "Block order" above), computed on
 * the device by the same code: out_perm[i] (device, nblocks int32) = the i-th block
 * visited among blocks first_block .. first_block+nblocks-1 of `row`.
 * 1 <= nblocks <= 1024.  For parity checks of the block order; asynchronous on stream. */
ds_status ds_block_order(uint64_t seed, int64_t row, int64_t first_block, int32_t nblocks,
                         int32_t* out_perm, cudaStream_t stream);

/* Runs one bounded wait on an mbarrier phase that never completes, with a limit of
 * `cycles` SM clock cycles (0 .. 2e9).  The wait runs out, the kernel records
 * DS_ERR_TIMEOUT in the device status word and returns; ds_get_device_status() then
 * reports it.  Checks the failure path of the device-side waits without a GPU fault. */
ds_status ds_wait_probe(int64_t cycles, cudaStream_t stream);

/*
 * ds_topk_noalloc -- ds_topk_ex for callers that cannot allocate device memory.
 *
 * This entry point has no counterpart in the pages; it exists for callers that may not
 * call cudaMalloc: code that runs while a CUDA graph is being captured (where an
 * allocation would break or escape the capture), serving loops that forbid allocator
 * calls because cudaMalloc/cudaFree can synchronise the device and stall other work,
 * and processes whose caching allocator has already reserved nearly all device memory.
 *
 * Arguments are those of ds_topk_ex, with `parts` and `cluster` as in ds_options
 * (0 = library choice).  When the launch needs scratch memory (a row split over more
 * than one thread-block cluster) it uses a fixed array compiled into the library's
 * device image instead of a workspace: at most ds_noalloc_scratch_bytes() bytes
 * (4 MiB; about rows * clusters_per_row * k * 8 bytes are needed); a launch that would
 * need more returns DS_ERR_WORKSPACE.  The array exists on every device that loads the
 * library until the process exits.  It calls no cudaMalloc, cudaFree or allocating
 * library routine.
 *
 * The first call on a device that needs the scratch looks up its device address (with
 * that device current); make that first call before any stream capture.  The address is
 * kept per device index for the life of the process: after cudaDeviceReset (or with a
 * different primary context for that device) the kept address is stale, so such a
 * process must not call this entry point again on that device.  All calls
 * share the one array: calls whose work overlaps on the GPU (for instance on different
 * streams) race on it and must be ordered by the caller.
 */
ds_status ds_topk_noalloc(const void* x, int32_t dtype, int64_t rows, int64_t N,
                          int64_t row_stride, int32_t k, int32_t B, int32_t B2, uint64_t seed,
                          void* out_vals, int32_t* out_idx, int32_t parts, int32_t cluster,
                          cudaStream_t stream);

/* Size of the fixed scratch array ds_topk_noalloc uses, in bytes. */
size_t ds_noalloc_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* DS_TOPK_H */
