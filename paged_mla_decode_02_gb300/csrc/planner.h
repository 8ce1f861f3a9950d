// Host-side planner: validation of a decode batch and its split into
// balanced split-KV work units.  Pure C++ (no CUDA calls).
#pragma once
#include <string>
#include <vector>

#include "mla_decode.h"
#include "mla_internal.h"

namespace mla {

struct Partition {
  std::vector<WorkUnit> units;
  std::vector<int32_t> worker_ptr;   // n_workers + 1
  std::vector<MergeEntry> merge;
  int n_slots = 0;
  int total_tiles = 0;
};

// Checks the arguments of one batch; on failure returns the status and sets *why.
mla_status_t validate_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                            int head_dim_ckv, int head_dim_kpe, int page_size,
                            float sm_scale, std::string* why);

// Splits the batch's tile_tokens-token tiles into n_workers contiguous ranges
// of (nearly) equal tile count; each range is cut at request boundaries into
// work units.
void partition_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                     int n_workers, int tile_tokens, Partition* out);

// Upper bounds of the partition sizes, used to size plan buffers at creation:
// each worker range adds at most one unit beyond the requests it starts.
inline int max_units(int n_workers, int max_batch) { return n_workers + max_batch; }
inline int max_slots(int n_workers, int max_batch) { return n_workers + max_batch; }

}  // namespace mla
