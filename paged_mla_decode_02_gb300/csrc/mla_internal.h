// Internal structures shared by the host planner, the C ABI layer and the
// kernels of the paged MLA decode library.  Not part of the public ABI.
#pragma once
#include <cstdint>

namespace mla {

constexpr int kDCkv = 512;          // kv_lora_rank: latent (ckv) width, also the value width
constexpr int kDKpe = 64;           // qk_rope_head_dim: rope key (kpe) width
constexpr int kD = kDCkv + kDKpe;   // 576: contraction width of the scores
constexpr int kMaxHeads = 128;

// Token granularity of the split-KV partition for each kernel: a work unit
// starts on a multiple of it.  Every supported page size (16, 32, 64)
// divides both, so a tile is a whole number of pages (the last page of a
// request may be partially filled).
constexpr int kTileMma = 64;        // mma.sync kernel: 64-token tiles
constexpr int kTileTc = 128;        // tcgen05 kernel: 128-token tiles
constexpr int kTilePair = 256;      // CTA-pair tcgen05 kernel: 256-token tiles

// One contiguous token range of one request, processed by one worker.
struct WorkUnit {
  int32_t req;
  int32_t tok_begin;   // multiple of the kernel's tile size
  int32_t tok_end;     // <= kv_len
  int32_t out_slot;    // -1: the unit covers the whole request -> final out/lse
  int32_t page_base;   // kv_indptr[req]: first entry of the request in kv_indices
  int32_t kv_len;      // tokens of the request
  int32_t slot0;       // split request: its first partial slot (its units use
  int32_t n_slots;     //   slot0 .. slot0 + n_slots - 1); 0, 0 otherwise
};
static_assert(sizeof(WorkUnit) == 32, "WorkUnit layout");

// A request whose partial results (slots first_slot .. first_slot+n_slots-1)
// the merge kernel combines; n_slots == 0 marks an empty request.
struct MergeEntry {
  int32_t req;
  int32_t first_slot;
  int32_t n_slots;
};
static_assert(sizeof(MergeEntry) == 12, "MergeEntry layout");

// Plan parameters the kernels read from device memory, so a captured CUDA
// graph keeps working after a re-plan with the same plan object.
struct PlanDev {
  int32_t n_units;
  int32_t n_merge;
  int32_t n_workers;
  int32_t batch;
  int32_t num_heads;
  int32_t page_size;
  float sm_scale;
  int32_t n_slots;
  // Several query tokens of a request packed into the rows of one request
  // (CTA-pair kernel, q_len * heads_per_token <= 128): row h is query token
  // h / heads_per_token of its request and sees the request's first
  // kv_len - (q_len - 1 - h / heads_per_token) tokens.  q_len <= 1: one
  // query token per request (every row sees kv_len tokens).
  int32_t q_len;
  int32_t heads_per_token;
};
static_assert(sizeof(PlanDev) == 40, "PlanDev layout");

// Device error codes (same values as mla_status_t).
constexpr int kErrTimeout = 5;
constexpr int kErrBounds = 6;

}  // namespace mla
