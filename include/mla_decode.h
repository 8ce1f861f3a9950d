/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) paged MLA decode library.
 *
 * Operation (absorbed multi-head latent attention, decode, one query token):
 * every token of the paged cache holds ONE latent KV head, a ckv row of width
 * head_dim_ckv = kv_lora_rank = 512 and a kpe row of width head_dim_kpe =
 * qk_rope_head_dim = 64.  For request b, head h:
 *
 *   s_i        = sm_scale * (q_nope[b,h] . ckv_i + q_pe[b,h] . kpe_i)
 *   out[b,h,:] = sum_i softmax(s)_i * ckv_i          (width 512)
 *   lse[b,h]   = ln sum_i exp(s_i)                    (natural log)
 *
 * over the kv_len[b] tokens of the request, with no causal mask.
 *
 * The plan/run split and the plan arguments (head_dim_ckv, head_dim_kpe,
 * page_size, causal=False, sm_scale), the single KV head of MLA and the
 * host-side paging arrays come from "[WIP] support flashinfer_mla"
 * (vLLM-metax PR #113), code-review comments on the decode_wrapper.plan(...)
 * call and on the paged_kv_indptr_cpu / paged_kv_len_arr_cpu slices.
 * CUDA-graph capture of the run step is the concern raised in "[WIP][Kernel]
 * Flashinfer MLA support" (vLLM PR #13630): mla_decode_run allocates nothing,
 * never synchronises and reads no host memory, so it can be captured.
 * A KV cache whose dtype differs from the query dtype (fp8 cache, bf16
 * queries) is the limitation noted in "[V1][Core] FlashInfer attention backend
 * for V1" (vLLM PR #14061), "Current limitations".
 *
 * Errors: every call returns a status code.  No call throws, exits or traps,
 * and there is no silent fallback: an unsupported request is an error.
 * The text of the last error of a plan is kept by mla_plan_last_error().
 *
 * Threading: a plan is not thread-safe; use one plan per host thread.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mla_plan_s* mla_plan_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,    /* inconsistent or malformed arguments */
  MLA_ERR_UNSUPPORTED = 2,    /* well-formed but not supported (dims, page size, dtype) */
  MLA_ERR_CAPACITY = 3,       /* exceeds what the plan was created for */
  MLA_ERR_CUDA = 4,           /* a CUDA runtime call failed; see mla_plan_last_error */
  MLA_ERR_DEVICE_TIMEOUT = 5, /* a bounded wait inside a kernel ran out */
  MLA_ERR_DEVICE_BOUNDS = 6,  /* a kernel saw a page id outside [0, num_pages) */
  MLA_ERR_NOT_PLANNED = 7     /* mla_decode_run before a successful mla_decode_plan */
} mla_status_t;

typedef enum {
  MLA_DTYPE_BF16 = 0,
  MLA_DTYPE_FP8_E4M3 = 1,     /* OCP E4M3 ("e4m3fn"), value = code * kv_scale */
  MLA_DTYPE_FP32 = 2
} mla_dtype_t;

typedef enum {
  MLA_KERNEL_DEFAULT = 0,     /* MLA_KERNEL_PAIR (an fp8 cache with 16-token pages runs on
                                 the tcgen05 kernel over the same plan, which rejects it) */
  MLA_KERNEL_TCGEN05 = 1,     /* one-CTA tcgen05 / TMEM kernel (bf16 and fp8 caches) */
  MLA_KERNEL_MMA_SYNC = 2,    /* warp-level mma.sync kernel (legacy tensor path, for comparison) */
  MLA_KERNEL_PAIR = 3         /* tcgen05 kernel whose MMAs span a CTA pair (cta_group::2); bf16
                                 caches, and fp8 caches with page_size >= 32 (e4m3 MMAs) */
} mla_kernel_t;

/* Plan statistics, filled by mla_plan_info. */
typedef struct {
  int32_t num_sms;            /* SMs of the plan's device */
  int32_t num_workers;        /* persistent workers (CTA pairs for tcgen05, CTAs for mma.sync) */
  int32_t num_units;          /* work units (contiguous tile ranges of one request) */
  int32_t num_partial_slots;  /* split partial results written to the workspace */
  int32_t num_merge;          /* split and empty requests (merged / zero-filled) */
  int32_t total_tiles;        /* KV tiles (of tile_tokens tokens) over the batch */
  int32_t batch;
  int32_t num_heads;
  int32_t page_size;
  int32_t kernel;             /* mla_kernel_t the partition is made for (DEFAULT: PAIR) */
  int32_t tile_tokens;        /* token granularity of the split (128 tcgen05, 64 mma.sync) */
  int64_t workspace_bytes;    /* device bytes owned by the plan */
} mla_plan_info_t;

/*
 * Create a plan on the CURRENT CUDA device.  Allocates (once, here) the
 * work-unit buffers, the merge map, the split-request counters and the
 * split-KV partial workspace sized
 * for up to max_batch requests of num_heads heads, so later plans and runs
 * never allocate.  num_heads in 1..128.  kernel: an mla_kernel_t.
 * On success *out receives the plan; the caller releases it with
 * mla_plan_destroy.  Returns MLA_ERR_INVALID_ARG for bad sizes,
 * MLA_ERR_CUDA when there is no device or an allocation fails.
 */
mla_status_t mla_plan_create(int max_batch, int num_heads, int kernel, mla_plan_t* out);

/*
 * Plan one decode batch (host work + one async upload on `stream`).
 *   kv_indptr_host [batch+1] int32, HOST: CSR offsets into kv_indices, in pages;
 *                  kv_indptr[0] = 0, non-decreasing.
 *   kv_indices_dev [kv_indptr[batch]] int32, DEVICE: page ids.  Borrowed, not
 *                  copied: it must stay allocated, at the same address, until the
 *                  last run of this plan.  Its contents may change between runs.
 *   kv_len_host    [batch] int32, HOST: tokens per request, >= 0, with
 *                  kv_indptr[b+1]-kv_indptr[b] == ceil(kv_len[b]/page_size).
 *                  A request with kv_len 0 gets out = 0, lse = -inf.
 *   num_heads      must equal the plan's num_heads.
 *   head_dim_ckv   must be 512, head_dim_kpe must be 64 (else MLA_ERR_UNSUPPORTED;
 *                  this rejects e.g. passing the KV-head count as head_dim_ckv).
 *   page_size      16, 32 or 64 tokens.
 *   sm_scale       finite softmax scale applied to q.k.
 *   stream         cudaStream_t (may be NULL = legacy default stream).
 * The host arrays are read before the call returns.  Re-planning reuses the
 * plan's buffers; a run already queued on `stream` sees the old plan.
 */
mla_status_t mla_decode_plan(mla_plan_t plan, const int32_t* kv_indptr_host,
                             const int32_t* kv_indices_dev, const int32_t* kv_len_host,
                             int batch, int num_heads, int head_dim_ckv, int head_dim_kpe,
                             int page_size, float sm_scale, void* stream);

/*
 * Plan a decode step of q_len query tokens per request (speculative or
 * multi-token decode: decode with short query lengths, which "[V1][Core]
 * FlashInfer attention backend for V1" (vLLM PR #14061) finds the prefill
 * wrapper serves poorly).
 *   The q_len new tokens of request b are the last q_len of its kv_len cached
 *   tokens; query j (0-based) sees the tokens at positions
 *   0 .. kv_len[b] - q_len + j.  This is a causal mask inside the query block
 *   and none before it.
 *   Arguments as for mla_decode_plan.  In addition:
 *   - q_len >= 1;
 *   - every kv_len[b] >= q_len (else MLA_ERR_INVALID_ARG);
 *   - batch * q_len <= the plan's max_batch (else MLA_ERR_CAPACITY).
 *   mla_decode_run then takes
 *     q_nope [batch, q_len, num_heads, 512],  q_pe [batch, q_len, num_heads, 64],
 *     out    [batch, q_len, num_heads, 512],  lse  [batch, q_len, num_heads].
 *   With the CTA-pair kernel (MLA_KERNEL_DEFAULT or MLA_KERNEL_PAIR) and
 *   q_len * num_heads <= 128, the q_len query tokens of a request share
 *   the rows of one request (row j * num_heads + h of the [batch, q_len *
 *   num_heads] view of the query and output arrays, each row masked to its
 *   own prefix), so a step reads each request's cache once;
 *   mla_plan_info then reports batch requests.  Otherwise each query token
 *   is planned as its own request over a prefix of its request's pages
 *   (mla_plan_info reports batch * q_len), so a step reads each request's
 *   cache q_len times; consecutive queries of a request sit next to each
 *   other in the work list, so those reads are mostly served by L2.
 *   q_len = 1 plans exactly what mla_decode_plan plans.  A graph captured
 *   from a run of such a plan replays re-plans with the same q_len.
 */
mla_status_t mla_decode_plan_multi(mla_plan_t plan, const int32_t* kv_indptr_host,
                                   const int32_t* kv_indices_dev, const int32_t* kv_len_host,
                                   int batch, int q_len, int num_heads, int head_dim_ckv,
                                   int head_dim_kpe, int page_size, float sm_scale,
                                   void* stream);

/*
 * Run the planned batch on `stream`.  All tensor arguments are DEVICE pointers
 * to contiguous row-major arrays owned by the caller:
 *   q_nope    [batch, num_heads, 512]   q_dtype (MLA_DTYPE_BF16 only)
 *   q_pe      [batch, num_heads, 64]    q_dtype
 *   ckv_cache [num_pages, page_size, 512]  kv_dtype (BF16 or FP8_E4M3), 16-byte aligned
 *   kpe_cache [num_pages, page_size, 64]   kv_dtype, 16-byte aligned
 *   kv_scale  per-tensor dequantisation scale of an FP8_E4M3 cache (value =
 *             code * kv_scale), finite and > 0; ignored for a BF16 cache
 * An FP8_E4M3 cache runs on the tcgen05 kernel with page_size 32 or 64 (each
 * copied tile is expanded to bf16 in shared memory; every e4m3 value is exact
 * in bf16), and on the mma.sync kernel with any page size; with the tcgen05
 * kernel and 16-token pages the call returns MLA_ERR_UNSUPPORTED.  The
 * CTA-pair kernel (and so MLA_KERNEL_DEFAULT) takes fp8 caches with 32- or
 * 64-token pages: e4m3 MMAs (kind::f8f6f4) read the copied codes as they
 * are, against the query and the probabilities P each split into two e4m3
 * terms (hi = e4m3(x), lo = e4m3(x - hi)); each query row is first scaled
 * by a power of two so that its largest magnitude lies in [2^7, 2^8), which
 * makes hi + lo the bf16 query exactly for magnitudes from 2^-2 up (after
 * the scaling) and within 2^-10 below.  With 16-token pages it returns
 * MLA_ERR_UNSUPPORTED.
 *   out       [batch, num_heads, 512]   out_dtype (BF16 or FP32)
 *   lse       [batch, num_heads]        fp32, natural log
 * Launches the decode kernel; with the tcgen05 kernel that is the only launch
 * (a request split across workers is combined by log-sum-exp in the epilogue
 * of its last-finishing unit, requests with kv_len 0 are filled by the same
 * kernel), with the CTA-pair and mma.sync kernels a merge kernel follows.  The combination
 * order is fixed, so repeated runs give bit-identical results.
 * The decode and merge kernels (like the projection and state-merge kernels
 * below) are programmatic dependent launches: each may be scheduled while the kernel
 * before it on the stream drains, and waits for that kernel to complete
 * before it reads anything; each lets the next kernel on the stream be
 * scheduled early.  A caller kernel launched after them with programmatic
 * stream serialization must therefore wait on its dependency
 * (griddepcontrol.wait) before it reads their outputs; plain launches and
 * copies are ordered as usual.
 * No allocation, no synchronisation, no host reads: capturable in a
 * CUDA graph.  The graph keeps the pointers and the extent of the query and
 * output arrays of the captured call (the batch planned then, times its
 * heads): re-planning with the same plan between replays is allowed (new
 * lengths, page table and split) for a batch no larger than the captured
 * one; a replay after a re-plan to a larger batch would read the query rows
 * past the captured extent as zeros.  A page id outside [0, num_pages) found by the
 * kernel is recorded and reported by mla_plan_check_status; that page is read
 * as zeros.
 */
mla_status_t mla_decode_run(mla_plan_t plan, const void* q_nope, const void* q_pe,
                            int q_dtype, const void* ckv_cache, const void* kpe_cache,
                            int kv_dtype, float kv_scale, int num_pages, void* out,
                            int out_dtype, float* lse, void* stream);

/*
 * One whole decode step from HOST buffers: copies q_nope / q_pe from host to
 * plan-owned device staging buffers, runs, copies out / lse back to host and
 * synchronises `stream`.  The KV cache stays device-resident (device
 * pointers, as for mla_decode_run).  Pinned host memory gives the fastest
 * copies.  The staging buffers are allocated on the first call (so this call
 * is not graph-capturable) and kept by the plan.  Sizes and dtypes as for
 * mla_decode_run.
 */
mla_status_t mla_decode_run_host(mla_plan_t plan, const void* q_nope_host,
                                 const void* q_pe_host, int q_dtype, const void* ckv_cache,
                                 const void* kpe_cache, int kv_dtype, float kv_scale,
                                 int num_pages, void* out_host, int out_dtype,
                                 float* lse_host, void* stream);

/*
 * Plan + run one batch without any allocation, for callers that may not
 * allocate device memory after start-up (e.g. a serving process whose
 * allocator owns all memory).  The pages have no counterpart to this call; it
 * is an engineering variant of mla_decode_plan + mla_decode_run on the
 * tcgen05 kernel.
 *   Everything besides the caller's tensors -- work units, split partials,
 *   split-request counters, the device status word -- lives in one fixed
 *   48 MiB scratch array inside the library; the work-unit list is built in
 *   static host memory.  Nothing is allocated (no cudaMalloc, no pinned host
 *   memory, no heap allocation on success).
 *   The array is a __device__ variable of the library image: its 48 MiB are
 *   taken on every device where the library's module is loaded, whether or
 *   not this call is ever used (plan / run callers pay it too), until the
 *   process exits.
 *   Limits: batch <= 4096 (else MLA_ERR_CAPACITY, before any device work); the
 *   batch's partials and work units must fit the scratch (else
 *   MLA_ERR_CAPACITY; with 128 heads they take about 38 MiB at most on a
 *   152-SM GPU).  bf16 q and caches only (the call has no dtype argument: an
 *   fp8 cache passed here is read as bf16 and gives wrong results);
 *   kv_scale must be 1 (another value is MLA_ERR_UNSUPPORTED); head dims
 *   512 / 64.
 *   Arguments as for mla_decode_plan / mla_decode_run (kv_indptr_host and
 *   kv_len_host on the host, everything else on the device; kv_indices_dev is
 *   only read by this call's kernel).
 *   The first call on a device does the setup (looks up the scratch address,
 *   queries the SM count and kernel residency); make it before any work that
 *   must not see those calls.
 *   Each call zeroes, on `stream`, the split counters the kernel expects at
 *   zero, uploads its work units and launches one kernel; it returns without
 *   waiting unless check_status is nonzero.  The device status word is
 *   sticky: it keeps the first error (a page id out of range, an expired
 *   device wait) that any call recorded, until a call with check_status != 0
 *   synchronises `stream`, reads it, clears it and returns it
 *   (MLA_ERR_DEVICE_BOUNDS / MLA_ERR_DEVICE_TIMEOUT).  So a caller that
 *   checks only every few steps still learns of an error in a step it did
 *   not check; that step's out / lse are not to be trusted.
 *   The scratch and the host staging are shared by all calls in the process:
 *   calls that overlap (other streams, other host threads) race and corrupt
 *   each other.  Issue them one after another on one stream.
 */
mla_status_t mla_decode_noalloc(const int32_t* kv_indptr_host, const int32_t* kv_indices_dev,
                                const int32_t* kv_len_host, int batch, int num_heads,
                                int page_size, float sm_scale, const void* q_nope,
                                const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                                float kv_scale, int num_pages, void* out, int out_dtype,
                                float* lse, int check_status, void* stream);

/*
 * Combine two attention states of the same query rows over disjoint sets of
 * tokens.  This is the log-sum-exp combination cascade (multi-level)
 * attention relies on ("[V1][Core] FlashInfer attention backend for V1",
 * vLLM PR #14061, "Outstanding items").  Decode a shared prefix and each
 * request's own suffix as two batches, then merge: the result is the decode
 * over the concatenated pages.
 * For every row r (a request and head):
 *   M = max(lse_a[r], lse_b[r]),  w_x = exp(lse_x[r] - M),
 *   out[r] = (w_a o_a[r] + w_b o_b[r]) / (w_a + w_b),
 *   lse_out[r] = M + ln(w_a + w_b).
 *   A state with lse = -inf carries no weight, whatever its o holds.  Both
 *   -inf give out = 0, lse = -inf.
 *   o_a, o_b  DEVICE fp32 [rows, 512], 16-byte aligned;
 *   lse_a, lse_b  DEVICE fp32 [rows] (natural log);
 *   out       DEVICE [rows, 512] of out_dtype (MLA_DTYPE_BF16 or FP32), 16-byte
 *             aligned; it may be o_a or o_b (fp32);
 *   lse_out   DEVICE fp32 [rows]; it may be lse_a or lse_b.
 * No allocation and no synchronisation; the work is queued on `stream`.
 * Returns MLA_ERR_INVALID_ARG for rows < 0, a NULL pointer or a misaligned
 * tensor, MLA_ERR_UNSUPPORTED for another out_dtype, MLA_ERR_CUDA when the
 * launch fails.
 */
mla_status_t mla_merge_states(const float* o_a, const float* lse_a, const float* o_b,
                              const float* lse_b, void* out, int out_dtype, float* lse_out,
                              int rows, void* stream);

/*
 * The per-head projections on either side of the latent decode (absorbed MLA:
 * the decode runs in the kv_lora_rank-wide latent space of the compressed
 * cache, head_dim_ckv = kv_lora_rank -- "[WIP] support flashinfer_mla",
 * vLLM-metax PR #113, review of the decode_wrapper.plan parameters).
 *
 * mla_absorb_q: q_nope[b,h,:] = W_UK[h] . q_raw[b,h,:]
 *   q_raw  DEVICE bf16 [batch, num_heads, head_dim_nope]  (a head's no-rope query)
 *   w_uk   DEVICE bf16 [num_heads, 512, head_dim_nope]    (key up-projection)
 *   q_nope DEVICE bf16 [batch, num_heads, 512]            (the decode's q_nope)
 * mla_project_out: o[b,h,:] = out[b,h,:] . W_UV[h]
 *   out    DEVICE bf16 [batch, num_heads, 512]            (the decode's out)
 *   w_uv   DEVICE bf16 [num_heads, 512, head_dim_v]       (value up-projection)
 *   o      DEVICE bf16 [batch, num_heads, head_dim_v]
 * head_dim_nope, head_dim_v: 64 or 128 (else MLA_ERR_UNSUPPORTED).  All
 * pointers 16-byte aligned (else MLA_ERR_INVALID_ARG).  The products
 * accumulate in fp32 on the tensor cores and are rounded to bf16 once.  No
 * allocation.  The work is queued on `stream`.  check_status != 0 waits for
 * it and returns MLA_ERR_DEVICE_TIMEOUT if a device wait gave up (the error
 * is then cleared); otherwise the call returns at once.  Calls on different
 * streams may overlap.
 */
mla_status_t mla_absorb_q(const void* q_raw, const void* w_uk, void* q_nope, int batch,
                          int num_heads, int head_dim_nope, int check_status, void* stream);
mla_status_t mla_project_out(const void* out, const void* w_uv, void* o, int batch,
                             int num_heads, int head_dim_v, int check_status, void* stream);

/*
 * Synchronise the device, then read and clear the plan's device error word.
 * Returns MLA_OK, MLA_ERR_DEVICE_TIMEOUT or MLA_ERR_DEVICE_BOUNDS (the first
 * error a kernel recorded since the last check), or MLA_ERR_CUDA.
 */
mla_status_t mla_plan_check_status(mla_plan_t plan);

/*
 * Profiling hook: when set (non-NULL cudaEvent_t handles created by the
 * caller on the plan's device), every mla_decode_run records start_event on
 * its stream immediately before the decode kernel and stop_event immediately
 * after it (before the merge kernel of the CTA-pair and mma.sync paths), so
 * the caller can time the decode kernel alone with cudaEventElapsedTime.
 * Pass NULLs to stop recording.
 * The events are borrowed; they must outlive the runs that record them.
 */
mla_status_t mla_plan_set_profile_events(mla_plan_t plan, void* start_event, void* stop_event);

/* Fill *info with the current plan's statistics. */
mla_status_t mla_plan_info(mla_plan_t plan, mla_plan_info_t* info);

/* Release every buffer of the plan (synchronises the device first). NULL is a no-op. */
mla_status_t mla_plan_destroy(mla_plan_t plan);

/* Static text for a status code. */
const char* mla_status_string(mla_status_t status);

/* Text of the plan's last error ("" if none).  Valid until the next call on the plan. */
const char* mla_plan_last_error(mla_plan_t plan);

/*
 * Host-only planner, exposed for inspection and testing (no CUDA call).
 * Validates the batch exactly as mla_decode_plan does and splits the
 * tile_tokens-token tiles of the batch (tile_tokens 64 or 128, else
 * MLA_ERR_UNSUPPORTED) into num_workers contiguous, balanced ranges.
 * Outputs (caller-allocated host arrays; pass capacities):
 *   units  [units_cap * 6] int32: per unit {req, tok_begin, tok_end,
 *          out_slot (-1 = final output), page_base (= kv_indptr[req]), kv_len};
 *          tok_begin is a multiple of tile_tokens, tok_end <= kv_len
 *   worker_ptr [num_workers + 1] int32: units of worker w are
 *          units[worker_ptr[w] .. worker_ptr[w+1])
 *   merge  [merge_cap * 3] int32: per merged request {req, first_slot, n_slots}
 *          (n_slots = 0 for an empty request: out = 0, lse = -inf)
 *   counts [3] int32: {num_units, num_partial_slots, num_merge}
 * Returns MLA_ERR_CAPACITY when units_cap or merge_cap is too small.
 * This is the default-cost partition.  A CTA-pair plan may instead keep a
 * partition with fewer split requests when its estimated step (slowest
 * worker plus the merge pass over the split shares) is shorter.
 */
mla_status_t mla_plan_partition_host(const int32_t* kv_indptr_host, const int32_t* kv_len_host,
                                     int batch, int head_dim_ckv, int head_dim_kpe,
                                     int page_size, float sm_scale, int num_workers,
                                     int tile_tokens, int32_t* units, int units_cap,
                                     int32_t* worker_ptr,
                                     int32_t* merge, int merge_cap, int32_t* counts);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
