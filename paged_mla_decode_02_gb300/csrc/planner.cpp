// Host planner for paged MLA decode.
//
// The plan step takes the host-side paging arrays of the decode requests
// (a page-count CSR and per-request token counts, the arrays sliced on the
// host in "[WIP] support flashinfer_mla", vLLM-metax PR #113, review comment
// on paged_kv_indptr_cpu / paged_kv_len_arr_cpu) and the plan parameters of
// the same PR's decode_wrapper.plan review (head_dim_ckv = kv_lora_rank,
// head_dim_kpe = qk_rope_head_dim, page_size, causal=False, sm_scale).
//
// Split policy: the batch's tiles are laid end to end, request after request,
// and cut into n_workers contiguous ranges of equal tile count (the first
// total % n_workers ranges take one tile more).  A range that crosses a
// request boundary becomes several work units.  A request covered by a single
// unit writes its final output directly; a request cut into several units
// writes one partial (O, lse) per unit and is combined by the merge kernel by
// log-sum-exp, the combination that cascade attention relies on ("[V1][Core]
// FlashInfer attention backend for V1", vLLM PR #14061, "Outstanding items").
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

void partition_batch(const int32_t* kv_indptr, const int32_t* kv_len, int batch,
                     int n_workers, int tile_tokens, Partition* out) {
  out->units.clear();
  out->merge.clear();
  out->worker_ptr.assign(n_workers + 1, 0);
  std::vector<int> tiles(batch);
  long long total = 0;
  for (int b = 0; b < batch; ++b) {
    tiles[b] = (kv_len[b] + tile_tokens - 1) / tile_tokens;
    total += tiles[b];
  }
  out->total_tiles = static_cast<int>(total);

  // Equal shares: the first (total % n_workers) workers take one tile more.
  const long long base = total / n_workers;
  const long long extra = total % n_workers;
  int req = 0, tile = 0;  // cursor over the flattened tile sequence
  while (req < batch && tiles[req] == 0) ++req;
  for (int w = 0; w < n_workers; ++w) {
    out->worker_ptr[w] = static_cast<int32_t>(out->units.size());
    long long quota = base + (w < extra ? 1 : 0);
    while (quota > 0 && req < batch) {
      const int take = static_cast<int>(std::min<long long>(quota, tiles[req] - tile));
      WorkUnit u;
      u.req = req;
      u.tok_begin = tile * tile_tokens;
      u.tok_end = std::min((tile + take) * tile_tokens, kv_len[req]);
      u.out_slot = -1;
      u.page_base = kv_indptr[req];
      u.kv_len = kv_len[req];
      u.slot0 = 0;
      u.n_slots = 0;
      out->units.push_back(u);
      quota -= take;
      tile += take;
      if (tile == tiles[req]) {
        tile = 0;
        ++req;
        while (req < batch && tiles[req] == 0) ++req;
      }
    }
  }
  out->worker_ptr[n_workers] = static_cast<int32_t>(out->units.size());

  // Slots for split requests, merge entries for split and empty requests.
  std::vector<int> n_units(batch, 0);
  for (const WorkUnit& u : out->units) ++n_units[u.req];
  int slot = 0;
  for (int b = 0; b < batch; ++b) {
    if (tiles[b] == 0) {
      out->merge.push_back(MergeEntry{b, 0, 0});
      continue;
    }
    if (n_units[b] < 2) continue;
    out->merge.push_back(MergeEntry{b, slot, n_units[b]});
    slot += n_units[b];
  }
  // Units of one request are consecutive in the unit list (the walk above is
  // in tile order), so the k-th unit of request b takes slot first_slot + k.
  std::vector<int> first(batch, 0), next(batch, 0);
  for (const MergeEntry& m : out->merge) first[m.req] = next[m.req] = m.first_slot;
  for (WorkUnit& u : out->units)
    if (n_units[u.req] >= 2) {
      u.out_slot = next[u.req]++;
      u.slot0 = first[u.req];
      u.n_slots = n_units[u.req];
    }
  out->n_slots = slot;
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
  if (tile_tokens != mla::kTileMma && tile_tokens != mla::kTileTc) return MLA_ERR_UNSUPPORTED;
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
