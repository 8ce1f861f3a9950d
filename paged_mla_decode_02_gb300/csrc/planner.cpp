// Host planner for paged MLA decode.
//
// The plan step takes the host-side paging arrays of the decode requests
// (a page-count CSR and per-request token counts, the arrays sliced on the
// host in "[WIP] support flashinfer_mla", vLLM-metax PR #113, review comment
// on paged_kv_indptr_cpu / paged_kv_len_arr_cpu) and the plan parameters of
// the same PR's decode_wrapper.plan review (head_dim_ckv = kv_lora_rank,
// head_dim_kpe = qk_rope_head_dim, page_size, causal=False, sm_scale).
//
// Split policy: requests are laid end to end and dealt to the n_workers
// workers in order, each worker taking a contiguous run of them.  The plan
// minimises the largest worker cost under a simple model (quarter tiles, see
// plan_costs): a tile costs `tile`, every work unit `unit` more (the pipeline
// refills and an epilogue runs), and a unit of a split request `split` more
// again (its share goes out to memory and is merged).  A request is cut only
// where a worker fills up, and only into pieces of at least `min_piece`
// tiles.  A request covered by one unit
// writes its final output directly; a request cut into several units writes
// one partial (O, lse) per unit, combined by log-sum-exp, the combination
// that cascade attention relies on ("[V1][Core] FlashInfer attention backend
// for V1", vLLM PR #14061, "Outstanding items").
#include "planner.h"

#include <algorithm>
#include <cmath>
#include <cstdio>

namespace mla {

static std::string fmt(const char* f, long long a, long long b = 0, long long c = 0) {
  char buf[256];
  std::snprintf(buf, sizeof(buf), f, a, b, c);
  return buf;
}

mla_status_t validate_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                            int head_dim_ckv, int head_dim_kpe, int page_size,
                            float sm_scale, std::string* why) {
  if (head_dim_ckv != kDCkv || head_dim_kpe != kDKpe) {
    *why = fmt("head_dim_ckv=%lld head_dim_kpe=%lld: only 512 / 64 (kv_lora_rank / "
               "qk_rope_head_dim) are supported", head_dim_ckv, head_dim_kpe);
    return MLA_ERR_UNSUPPORTED;
  }
  if (page_size != 16 && page_size != 32 && page_size != 64) {
    *why = fmt("page_size=%lld: supported page sizes are 16, 32, 64", page_size);
    return MLA_ERR_UNSUPPORTED;
  }
  if (!std::isfinite(sm_scale)) {
    *why = "sm_scale is not finite";
    return MLA_ERR_INVALID_ARG;
  }
  if (batch < 1) {
    *why = fmt("batch=%lld must be >= 1", batch);
    return MLA_ERR_INVALID_ARG;
  }
  if (kv_indptr == nullptr || kv_len == nullptr) {
    *why = "kv_indptr_host / kv_len_host must not be NULL";
    return MLA_ERR_INVALID_ARG;
  }
  if (kv_indptr[0] != 0) {
    *why = fmt("kv_indptr[0]=%lld must be 0", kv_indptr[0]);
    return MLA_ERR_INVALID_ARG;
  }
  for (int b = 0; b < batch; ++b) {
    if (kv_len[b] < 0) {
      *why = fmt("kv_len[%lld]=%lld is negative", b, kv_len[b]);
      return MLA_ERR_INVALID_ARG;
    }
    const long long pages = (static_cast<long long>(kv_len[b]) + page_size - 1) / page_size;
    const long long have = static_cast<long long>(kv_indptr[b + 1]) - kv_indptr[b];
    if (have != pages) {
      *why = fmt("request %lld: kv_indptr gives %lld pages, kv_len needs %lld", b, have, pages);
      return MLA_ERR_INVALID_ARG;
    }
  }
  return MLA_OK;
}

namespace {

constexpr int tiles_of(int32_t len, int tile_tokens) { return (len + tile_tokens - 1) / tile_tokens; }

// Greedy fill at makespan `budget` (cost units).  Requests are taken in
// order; a worker takes whole requests while they fit, and the first one that
// does not is cut so that the worker is full, when both pieces keep at least
// min_piece tiles (else the next worker starts with it).  Writes the
// units (req, token range, page base, length) and the worker offsets when
// `units` is non-null.  Returns the number of units, or -1 when the batch
// needs more than n_workers workers at this budget.
int fill_workers(const int32_t* kv_indptr, const int32_t* kv_len, int batch, int n_workers,
                 int tile_tokens, const PlanCosts& c, long long budget, WorkUnit* units,
                 int32_t* worker_ptr) {
  int w = 0, nu = 0;
  long long used = 0;   // cost taken by worker w
  if (worker_ptr) worker_ptr[0] = 0;
  auto emit = [&](int b, int t0, int t1) {
    if (units) {
      WorkUnit& u = units[nu];
      u.req = b;
      u.tok_begin = t0 * tile_tokens;
      u.tok_end = std::min(t1 * tile_tokens, kv_len[b]);
      u.out_slot = -1;
      u.page_base = kv_indptr[b];
      u.kv_len = kv_len[b];
      u.slot0 = 0;
      u.n_slots = 0;
    }
    ++nu;
  };
  auto next_worker = [&]() {
    ++w;
    used = 0;
    if (worker_ptr && w <= n_workers) worker_ptr[w] = nu;
  };
  for (int b = 0; b < batch; ++b) {
    const int n = tiles_of(kv_len[b], tile_tokens);
    int t = 0;
    bool split = false;
    while (t < n) {
      if (w >= n_workers) return -1;
      const int rest = n - t;
      const long long whole = c.unit + static_cast<long long>(c.tile) * rest + (split ? c.split : 0);
      if (used + whole <= budget) {
        emit(b, t, n);
        used += whole;
        break;
      }
      // tiles that fit as a piece of a split request; both pieces keep at
      // least min_piece tiles
      const long long room = (budget - used - c.unit - c.split) / c.tile;
      const long long take = std::min<long long>(room, rest - c.min_piece);
      if (take < c.min_piece) {
        if (used == 0) return -1;   // not even an empty worker takes a piece
        next_worker();              // the next worker starts with this request
        continue;
      }
      emit(b, t, t + static_cast<int>(take));
      t += static_cast<int>(take);
      split = true;
      next_worker();
    }
  }
  if (worker_ptr)
    for (int v = w + 1; v <= n_workers; ++v) worker_ptr[v] = nu;
  return nu;
}

}  // namespace

int partition_units(const int32_t* kv_indptr, const int32_t* kv_len, int batch, int n_workers,
                    int tile_tokens, WorkUnit* units, int32_t* worker_ptr) {
  return partition_units(kv_indptr, kv_len, batch, n_workers, tile_tokens, plan_costs(tile_tokens),
                         units, worker_ptr);
}

int partition_units(const int32_t* kv_indptr, const int32_t* kv_len, int batch, int n_workers,
                    int tile_tokens, const PlanCosts& c, WorkUnit* units, int32_t* worker_ptr) {
  // Smallest budget the greedy fill meets.  Whether the fill succeeds is not
  // monotone in the budget (where a request is cut depends on it), so a
  // bisection finds a feasible budget `hi` only; the smallest one is then
  // looked for upward from the lower bound every partition obeys (the work
  // spread evenly), at most kMaxScan budgets.  One worker holding everything
  // always fits.
  long long total = 0, nonempty = 0;
  for (int b = 0; b < batch; ++b) {
    total += tiles_of(kv_len[b], tile_tokens);
    nonempty += kv_len[b] > 0;
  }
  long long lo = 0;
  long long hi = c.tile * total + static_cast<long long>(c.unit + c.split) * (batch + n_workers);
  while (lo + 1 < hi) {
    const long long mid = lo + (hi - lo) / 2;
    if (fill_workers(kv_indptr, kv_len, batch, n_workers, tile_tokens, c, mid, nullptr, nullptr) >= 0)
      hi = mid;
    else
      lo = mid;
  }
  constexpr long long kMaxScan = 4096;
  const long long bound = (c.tile * total + c.unit * nonempty + n_workers - 1) / n_workers;
  for (long long b = std::max(bound, hi - kMaxScan); b < hi; ++b)
    if (fill_workers(kv_indptr, kv_len, batch, n_workers, tile_tokens, c, b, nullptr, nullptr) >= 0) {
      hi = b;
      break;
    }
  return fill_workers(kv_indptr, kv_len, batch, n_workers, tile_tokens, c, hi, units, worker_ptr);
}

int assign_slots(WorkUnit* units, int n_units, const int32_t* kv_len, int batch, int tile_tokens,
                 MergeEntry* merge, int* n_merge) {
  // Units of one request are consecutive (the fill walks requests in order):
  // a run of two or more is a split request, whose k-th unit takes slot
  // first + k.  Empty requests get a merge entry without slots.
  int slot = 0, nm = 0, i = 0;
  for (int b = 0; b < batch; ++b) {
    if (tiles_of(kv_len[b], tile_tokens) == 0) {
      merge[nm++] = MergeEntry{b, 0, 0};
      continue;
    }
    int j = i;
    while (j < n_units && units[j].req == b) ++j;
    if (j - i >= 2) {
      for (int k = i; k < j; ++k) {
        units[k].out_slot = slot + (k - i);
        units[k].slot0 = slot;
        units[k].n_slots = j - i;
      }
      merge[nm++] = MergeEntry{b, slot, j - i};
      slot += j - i;
    }
    i = j;
  }
  *n_merge = nm;
  return slot;
}

void partition_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                     int n_workers, int tile_tokens, Partition* out) {
  partition_batch(kv_indptr, kv_len, batch, n_workers, tile_tokens, plan_costs(tile_tokens), out);
}

void partition_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                     int n_workers, int tile_tokens, const PlanCosts& c, Partition* out) {
  out->units.resize(max_units(n_workers, batch));
  out->worker_ptr.assign(n_workers + 1, 0);
  out->merge.resize(batch);
  long long total = 0;
  for (int b = 0; b < batch; ++b) total += tiles_of(kv_len[b], tile_tokens);
  out->total_tiles = static_cast<int>(total);
  const int nu = partition_units(kv_indptr, kv_len, batch, n_workers, tile_tokens, c,
                                 out->units.data(), out->worker_ptr.data());
  out->units.resize(nu);
  int nm = 0;
  out->n_slots = assign_slots(out->units.data(), nu, kv_len, batch, tile_tokens, out->merge.data(), &nm);
  out->merge.resize(nm);
}

long long partition_makespan(const Partition& p, int tile_tokens) {
  const PlanCosts c = plan_costs(tile_tokens);
  long long worst = 0;
  for (size_t w = 0; w + 1 < p.worker_ptr.size(); ++w) {
    long long used = 0;
    for (int i = p.worker_ptr[w]; i < p.worker_ptr[w + 1]; ++i) {
      const WorkUnit& u = p.units[i];
      used += c.unit + static_cast<long long>(c.tile) * tiles_of(u.tok_end - u.tok_begin, tile_tokens) +
              (u.n_slots > 0 ? c.split : 0);
    }
    worst = std::max(worst, used);
  }
  return worst;
}

double pair_step_estimate_us(const Partition& p, int rows) {
  constexpr double kTileUs = 3.9;            // one 256-token tile of a CTA pair
  constexpr double kMergeFixedUs = 2.5;      // a merge pass that combines something
  constexpr double kMergeBytesPerUs = 2.75e6;
  double us = partition_makespan(p, kTilePair) * (kTileUs / 4.0);
  if (p.n_slots > 0)
    us += kMergeFixedUs + static_cast<double>(p.n_slots) * rows * kDCkv * sizeof(float) / kMergeBytesPerUs;
  return us;
}

void partition_batch_pair(const int32_t* kv_indptr, const int32_t* kv_len, int batch, int n_workers,
                          int rows, Partition* out) {
  partition_batch(kv_indptr, kv_len, batch, n_workers, kTilePair, out);
  if (out->n_slots == 0) return;
  Partition whole;
  PlanCosts few = plan_costs(kTilePair);
  few.split = kFewSplitsCost;
  partition_batch(kv_indptr, kv_len, batch, n_workers, kTilePair, few, &whole);
  if (pair_step_estimate_us(whole, rows) < pair_step_estimate_us(*out, rows)) *out = std::move(whole);
}

}  // namespace mla

extern "C" mla_status_t mla_plan_partition_host(
    const int32_t* kv_indptr_host, const int32_t* kv_len_host, int batch, int head_dim_ckv,
    int head_dim_kpe, int page_size, float sm_scale, int num_workers, int tile_tokens,
    int32_t* units, int units_cap, int32_t* worker_ptr, int32_t* merge, int merge_cap,
    int32_t* counts) {
  std::string why;
  mla_status_t st = mla::validate_batch(kv_indptr_host, kv_len_host, batch, head_dim_ckv,
                                        head_dim_kpe, page_size, sm_scale, &why);
  if (st != MLA_OK) return st;
  if (num_workers < 1 || !units || !worker_ptr || !merge || !counts) return MLA_ERR_INVALID_ARG;
  if (tile_tokens != mla::kTileMma && tile_tokens != mla::kTileTc && tile_tokens != mla::kTilePair)
    return MLA_ERR_UNSUPPORTED;
  mla::Partition p;
  mla::partition_batch(kv_indptr_host, kv_len_host, batch, num_workers, tile_tokens, &p);
  if (static_cast<int>(p.units.size()) > units_cap || static_cast<int>(p.merge.size()) > merge_cap)
    return MLA_ERR_CAPACITY;
  for (size_t i = 0; i < p.units.size(); ++i) {
    const mla::WorkUnit& u = p.units[i];
    int32_t* d = units + 6 * i;
    d[0] = u.req; d[1] = u.tok_begin; d[2] = u.tok_end;
    d[3] = u.out_slot; d[4] = u.page_base; d[5] = u.kv_len;
  }
  for (int w = 0; w <= num_workers; ++w) worker_ptr[w] = p.worker_ptr[w];
  for (size_t i = 0; i < p.merge.size(); ++i) {
    merge[3 * i] = p.merge[i].req;
    merge[3 * i + 1] = p.merge[i].first_slot;
    merge[3 * i + 2] = p.merge[i].n_slots;
  }
  counts[0] = static_cast<int32_t>(p.units.size());
  counts[1] = p.n_slots;
  counts[2] = static_cast<int32_t>(p.merge.size());
  return MLA_OK;
}
