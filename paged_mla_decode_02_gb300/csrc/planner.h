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

// Cost model of the split, in quarter tiles: one tile costs `tile`, a work
// unit `unit` on top (pipeline fill and epilogue), a unit of a split request
// `split` more (its share is stored and merged).  Requests are cut only into
// pieces of at least `min_piece` tiles.  The constants were picked by A/B on
// the GPU for each kernel's tile: 128-token tiles (the one-CTA tcgen05
// kernel) and 256-token tiles (the CTA-pair kernel, whose tile takes about as
// long as a unit's fill).
struct PlanCosts {
  int tile, unit, split, min_piece;
};
constexpr PlanCosts plan_costs(int tile_tokens) {
  return tile_tokens >= 256 ? PlanCosts{4, 4, 2, 2} : PlanCosts{4, 8, 4, 4};
}

// Deals the requests' tile_tokens-token tiles to n_workers workers (each a
// contiguous run of requests, cut into work units at request boundaries) so
// that the largest worker cost is as small as the greedy fill allows.  Writes
// units[0 .. return value) (out_slot -1, no slots yet) and worker_ptr[0 ..
// n_workers]; units needs max_units(n_workers, batch) entries.  Allocates
// nothing.
int partition_units(const int32_t* kv_indptr, const int32_t* kv_len, int batch, int n_workers,
                    int tile_tokens, WorkUnit* units, int32_t* worker_ptr);
// The same under explicit costs.
int partition_units(const int32_t* kv_indptr, const int32_t* kv_len, int batch, int n_workers,
                    int tile_tokens, const PlanCosts& c, WorkUnit* units, int32_t* worker_ptr);

// Gives the units of every split request consecutive partial slots and
// writes one merge entry per split request and per empty request (at most
// batch entries).  Returns the number of slots.  Allocates nothing.
int assign_slots(WorkUnit* units, int n_units, const int32_t* kv_len, int batch, int tile_tokens,
                 MergeEntry* merge, int* n_merge);

// Both steps into growable arrays (default or explicit costs).
void partition_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                     int n_workers, int tile_tokens, Partition* out);
void partition_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                     int n_workers, int tile_tokens, const PlanCosts& c, Partition* out);

// The largest worker cost of a partition under the default costs.
long long partition_makespan(const Partition& p, int tile_tokens);

// The CTA-pair kernel's partition (256-token tiles, `rows` query rows per
// request).  A split request costs its workers the stores of its shares (the
// `split` cost), and the whole step one merge pass over all the shares,
// which no per-worker cost expresses.  So when the default partition splits
// requests, a second one that splits only where a worker cannot hold a
// request whole (a split unit costs kFewSplitsCost quarter tiles) is built
// as well, and the one with the smaller estimated step kept: the makespan at
// ~3.9 us per tile, plus, with shares, ~2.5 us and their bytes (rows x 2 KB
// each) at ~2.75 TB/s.  (Measured on 128-head batches: two query tokens per
// request of 64 x 4096 tokens, 156.7 -> 148.6 us per step without splits;
// ragged and fp8 batches keep their splits.)
constexpr int kFewSplitsCost = 12;
double pair_step_estimate_us(const Partition& p, int rows);
void partition_batch_pair(const int32_t* kv_indptr, const int32_t* kv_len, int batch, int n_workers,
                          int rows, Partition* out);

// Upper bounds of the partition sizes, used to size plan buffers at creation:
// a request is cut only where a worker ends, so each worker adds at most one
// unit beyond the requests.
inline int max_units(int n_workers, int max_batch) { return n_workers + max_batch; }
inline int max_slots(int n_workers, int max_batch) { return n_workers + max_batch; }

}  // namespace mla
