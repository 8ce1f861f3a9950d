// C ABI of the paged MLA decode library: plan objects, the plan / run entry
// points and status reporting.  The plan/run split and the plan arguments
// follow the decode_wrapper.plan(...) call reviewed in "[WIP] support
// flashinfer_mla" (vLLM-metax PR #113); run never allocates or synchronises,
// so it can be captured in a CUDA graph (the concern of "[WIP][Kernel]
// Flashinfer MLA support", vLLM PR #13630).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "kernels.h"
#include "merge.h"
#include "tmap.h"
#include "mla_decode.h"
#include "planner.h"

using namespace mla;

struct mla_plan_s {
  int device = 0;
  int num_sms = 0;
  int max_batch = 0;
  int num_heads = 0;
  int kernel = MLA_KERNEL_TCGEN05;   // the kernel the plan's partition is made for
  int kernel_requested = MLA_KERNEL_DEFAULT;
  int tile_tokens = kTileTc;
  int n_workers = 0;
  int units_cap = 0;
  int slots_cap = 0;
  int merge_cap = 0;
  size_t part_rows_cap = 0;          // rows (head x share) of the partial-share buffers

  // One device blob: PlanDev | units | worker_ptr | merge (16-byte aligned parts).
  void* d_blob = nullptr;
  size_t blob_bytes = 0;
  size_t off_units = 0, off_wptr = 0, off_merge = 0;
  void* h_blob = nullptr;            // pinned staging of the blob
  cudaEvent_t upload_done = nullptr; // the pinned blob may be rewritten once this fired

  float* d_o_part = nullptr;         // [slots_cap, H, 512]
  float* d_lse_part = nullptr;       // [slots_cap, 4, H]
  int32_t* d_counters = nullptr;     // [max_batch, 8]: split-request counts (tcgen05)
  int32_t* d_err = nullptr;

  // Staging of mla_decode_run_host (allocated on first use).
  void* d_q = nullptr;
  size_t d_q_bytes = 0;
  void* d_res = nullptr;
  size_t d_res_bytes = 0;

  cudaEvent_t prof_start = nullptr;  // recorded around the decode kernel when set
  cudaEvent_t prof_stop = nullptr;

  bool planned = false;
  PlanDev params{};
  const int32_t* kv_indices = nullptr;
  int total_tiles = 0;
  std::string last_error;
};

namespace {

size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

mla_status_t fail(mla_plan_t p, mla_status_t st, const std::string& why) {
  if (p) p->last_error = why;
  return st;
}

mla_status_t cuda_fail(mla_plan_t p, cudaError_t e, const char* what) {
  cudaGetLastError();  // clear a non-sticky error so later calls start clean
  return fail(p, MLA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

int workers_for(int kernel, int num_sms, int num_heads) {
  if (kernel == MLA_KERNEL_MMA_SYNC) {
    const int head_groups = (num_heads + 15) / 16;
    const int w = 2 * num_sms / head_groups;
    return w < 1 ? 1 : w;
  }
  return num_sms / 2 < 1 ? 1 : num_sms / 2;   // one 2-CTA cluster per worker
}

void release(mla_plan_t p) {
  if (p->d_blob) cudaFree(p->d_blob);
  if (p->h_blob) cudaFreeHost(p->h_blob);
  if (p->upload_done) cudaEventDestroy(p->upload_done);
  if (p->d_o_part) cudaFree(p->d_o_part);
  if (p->d_lse_part) cudaFree(p->d_lse_part);
  if (p->d_counters) cudaFree(p->d_counters);
  if (p->d_err) cudaFree(p->d_err);
  if (p->d_q) cudaFree(p->d_q);
  if (p->d_res) cudaFree(p->d_res);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (the library
// does not link libcuda directly, so it loads on machines without a driver).
EncodeTiledFn get_encode_fn() { return tensor_map_encoder(); }

}  // namespace

EncodeTiledFn mla::tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

namespace {

// 2-D row-major map [rows, cols] of elements of elem_bytes, box [box_rows, box_cols]
// (box_cols * elem_bytes = 128 bytes with the 128-byte swizzle, 64 with the
// 64-byte one).
bool encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
               uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view of a row-major [rows, 512] bf16 matrix as 64-element panels:
// (element within panel, row, panel) with strides (2 B, 1024 B, 128 B); a box
// (64, box_rows, box_panels) lands in shared memory panel by panel, each
// panel box_rows x 128 bytes with the 128-byte swizzle -- the layout the MMA
// reads -- in one copy instead of one per panel.
// An e4m3 cache (one byte per element) is mapped with either 64-element
// panels and the 64-byte swizzle (16-byte chunk c of row r lands at chunk
// c ^ ((r >> 1) & 3), so a kernel's row-per-lane reads are free of bank
// conflicts) or, wide = true, 128-element panels of 128-byte rows and the
// 128-byte swizzle, the MN-major layout an e4m3 MMA reads.
bool encode_panels_3d(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows,
                      uint32_t box_panels, bool fp8 = false, bool wide = false) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const uint64_t eb = fp8 ? 1 : 2;
  const uint64_t pw = fp8 && wide ? 128 : 64;   // elements per panel row
  cuuint64_t dims[3] = {pw, rows, kDCkv / pw};
  cuuint64_t strides[2] = {kDCkv * eb, pw * eb};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(pw), box_rows, box_panels};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fp8 && !wide ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// The tcgen05 kernel's tensor maps for one batch (also used by the entry point
// that works from static scratch memory).
bool mla::encode_tc_maps(TcMaps* maps, const void* q_nope, const void* ckv_cache, const void* kpe_cache,
                    int batch, int num_heads, int page_size, int num_pages, bool kv_fp8) {
  const uint64_t qrows = static_cast<uint64_t>(batch) * num_heads;
  const uint64_t kvrows = static_cast<uint64_t>(num_pages) * page_size;
  const CUtensorMapDataType kt = kv_fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle ks = kv_fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const int eb = kv_fp8 ? 1 : 2;
  return encode_2d(&maps->q_nope, q_nope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, qrows, kDCkv,
                   num_heads, 64) &&
         encode_2d(&maps->ckv_k, ckv_cache, kt, eb, kvrows, kDCkv, page_size, 64, ks) &&
         encode_2d(&maps->kpe_k, kpe_cache, kt, eb, kvrows, kDKpe, page_size, 64, ks) &&
         encode_panels_3d(&maps->ckv_v, ckv_cache, kvrows, page_size >= kTcVChunkTok ? kTcVChunkTok : 16,
                          8 / kTcCluster, kv_fp8);
}

// The CTA-pair kernel's tensor maps: the query of 64 heads per box (one per
// CTA of the pair), K panels of one page, V chunks of four 64-dim panels (an
// fp8 cache: byte maps; K panels of 64-byte rows with the 64-byte swizzle, V
// chunks of two 128-dim panels with the 128-byte swizzle).
bool mla::encode_pair_maps(PairMaps* maps, const void* q_nope, const void* q_pe, const void* ckv_cache,
                           const void* kpe_cache, int batch, int num_heads, int page_size, int num_pages,
                           bool kv_fp8) {
  const uint64_t qrows = static_cast<uint64_t>(batch) * num_heads;
  const uint64_t kvrows = static_cast<uint64_t>(num_pages) * page_size;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType kt = kv_fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : bf;
  const CUtensorMapSwizzle ks = kv_fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const int eb = kv_fp8 ? 1 : 2;
  return encode_2d(&maps->q_nope, q_nope, bf, 2, qrows, kDCkv, 64, 64) &&
         encode_2d(&maps->q_pe, q_pe, bf, 2, qrows, kDKpe, 64, 64) &&
         encode_2d(&maps->ckv_k, ckv_cache, kt, eb, kvrows, kDCkv, page_size, 64, ks) &&
         encode_2d(&maps->kpe_k, kpe_cache, kt, eb, kvrows, kDKpe, page_size, 64, ks) &&
         encode_panels_3d(&maps->ckv_v, ckv_cache, kvrows, page_size >= kTcVChunkTok ? kTcVChunkTok : 16,
                          kv_fp8 ? 2 : 4, kv_fp8, true);
}

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported";
    case MLA_ERR_CAPACITY: return "exceeds plan capacity";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MLA_ERR_DEVICE_BOUNDS: return "page id out of range";
    case MLA_ERR_NOT_PLANNED: return "run before a successful plan";
  }
  return "unknown status";
}

const char* mla_plan_last_error(mla_plan_t plan) {
  return plan ? plan->last_error.c_str() : "";
}

mla_status_t mla_plan_create(int max_batch, int num_heads, int kernel, mla_plan_t* out) {
  if (!out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_batch < 1 || num_heads < 1 || num_heads > kMaxHeads) return MLA_ERR_INVALID_ARG;
  if (kernel != MLA_KERNEL_DEFAULT && kernel != MLA_KERNEL_TCGEN05 &&
      kernel != MLA_KERNEL_MMA_SYNC && kernel != MLA_KERNEL_PAIR)
    return MLA_ERR_INVALID_ARG;
  mla_plan_t p = new (std::nothrow) mla_plan_s();
  if (!p) return MLA_ERR_CUDA;
  p->max_batch = max_batch;
  p->num_heads = num_heads;
  // DEFAULT: the CTA-pair kernel for bf16 caches and for fp8 caches with
  // pages of 32 or 64 tokens; an fp8 cache with 16-token pages goes to the
  // one-CTA tcgen05 kernel over the same partition (its 256-token unit
  // boundaries are also 128-token tile boundaries), which rejects it
  p->kernel_requested = kernel;
  p->kernel = kernel == MLA_KERNEL_DEFAULT ? MLA_KERNEL_PAIR : kernel;
  p->tile_tokens = p->kernel == MLA_KERNEL_MMA_SYNC ? kTileMma : p->kernel == MLA_KERNEL_PAIR ? kTilePair : kTileTc;
  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) {
    delete p;
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  p->n_workers = workers_for(p->kernel, p->num_sms, num_heads);
  if (p->kernel == MLA_KERNEL_TCGEN05 || p->kernel == MLA_KERNEL_PAIR) {
    int resident = 0;
    if ((e = p->kernel == MLA_KERNEL_PAIR ? decode_pair_max_workers(&resident) : decode_tc_max_workers(&resident)) !=
            cudaSuccess ||
        resident < 1) {
      delete p;
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    if (resident < p->n_workers) p->n_workers = resident;
    // the tcgen05 kernel merges split requests in place, waiting on the
    // other workers: all of them must be resident at once
    if (kernel == MLA_KERNEL_DEFAULT) {
      if ((e = decode_tc_max_workers(&resident)) != cudaSuccess || resident < 1) {
        delete p;
        cudaGetLastError();
        return MLA_ERR_CUDA;
      }
      if (resident < p->n_workers) p->n_workers = resident;
    }
  }
  p->units_cap = max_units(p->n_workers, max_batch);
  p->slots_cap = max_slots(p->n_workers, max_batch);
  p->merge_cap = max_batch;

  p->off_units = align16(sizeof(PlanDev));
  p->off_wptr = align16(p->off_units + sizeof(WorkUnit) * p->units_cap);
  p->off_merge = align16(p->off_wptr + sizeof(int32_t) * (p->n_workers + 1));
  p->blob_bytes = align16(p->off_merge + sizeof(MergeEntry) * p->merge_cap);
  // Partial shares: a row per (share, head).  A CTA-pair plan may pack up
  // to 128 rows per request (several query tokens), whose split units take
  // at most n_workers x 128 + max_batch x num_heads rows in all.
  p->part_rows_cap = static_cast<size_t>(p->slots_cap) * num_heads;
  if (p->kernel == MLA_KERNEL_PAIR)
    p->part_rows_cap = static_cast<size_t>(p->n_workers) * kMaxHeads + static_cast<size_t>(max_batch) * num_heads;
  const size_t o_bytes = sizeof(float) * p->part_rows_cap * kDCkv;
  const size_t l_bytes = sizeof(float) * p->part_rows_cap * kLsePartCopies;
  const size_t c_bytes = sizeof(int32_t) * static_cast<size_t>(max_batch) * 8;
  if ((e = cudaMalloc(&p->d_blob, p->blob_bytes)) != cudaSuccess ||
      (e = cudaMallocHost(&p->h_blob, p->blob_bytes)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&p->upload_done, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaMalloc(reinterpret_cast<void**>(&p->d_o_part), o_bytes)) != cudaSuccess ||
      (e = cudaMalloc(reinterpret_cast<void**>(&p->d_lse_part), l_bytes)) != cudaSuccess ||
      (e = cudaMalloc(reinterpret_cast<void**>(&p->d_counters), c_bytes)) != cudaSuccess ||
      (e = cudaMemset(p->d_counters, 0, c_bytes)) != cudaSuccess ||
      (e = cudaMalloc(reinterpret_cast<void**>(&p->d_err), sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMemset(p->d_err, 0, sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMemset(p->d_blob, 0, p->blob_bytes)) != cudaSuccess) {
    release(p);
    delete p;
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  std::memset(p->h_blob, 0, p->blob_bytes);
  *out = p;
  return MLA_OK;
}

mla_status_t mla_plan_destroy(mla_plan_t plan) {
  if (!plan) return MLA_OK;
  cudaDeviceSynchronize();
  release(plan);
  delete plan;
  return MLA_OK;
}

namespace {

// Partition and upload for n_req requests given by the position of their
// first page id in kv_indices (page_base) and their token counts (the
// caller validated both).  num_heads is the rows per request the kernels
// see: the plan's heads, or q_len x heads when q_len > 1 query tokens of a
// request share its rows (heads_per_token = the plan's heads); each partial
// share of a request takes that many rows of the share buffers.
mla_status_t plan_requests(mla_plan_t plan, const int32_t* page_base, const int32_t* len, int n_req,
                           const int32_t* kv_indices_dev, int num_heads, int page_size,
                           float sm_scale, void* stream, int q_len = 1, int heads_per_token = 0) {
  Partition part;
  if (plan->kernel == MLA_KERNEL_PAIR)
    partition_batch_pair(page_base, len, n_req, plan->n_workers, num_heads, &part);
  else
    partition_batch(page_base, len, n_req, plan->n_workers, plan->tile_tokens, &part);
  if (static_cast<int>(part.units.size()) > plan->units_cap || part.n_slots > plan->slots_cap ||
      static_cast<size_t>(part.n_slots) * num_heads > plan->part_rows_cap ||
      static_cast<int>(part.merge.size()) > plan->merge_cap)
    return fail(plan, MLA_ERR_CAPACITY, "partition exceeds plan buffers");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The pinned blob may still be the source of the previous upload.
  cudaError_t e = cudaEventSynchronize(plan->upload_done);
  if (e != cudaSuccess) return cuda_fail(plan, e, "cudaEventSynchronize");

  PlanDev prm{};
  prm.n_units = static_cast<int32_t>(part.units.size());
  prm.n_merge = static_cast<int32_t>(part.merge.size());
  prm.n_workers = plan->n_workers;
  prm.batch = n_req;
  prm.num_heads = num_heads;
  prm.page_size = page_size;
  prm.sm_scale = sm_scale;
  prm.n_slots = part.n_slots;
  prm.q_len = q_len;
  prm.heads_per_token = heads_per_token > 0 ? heads_per_token : num_heads;
  char* h = static_cast<char*>(plan->h_blob);
  std::memcpy(h, &prm, sizeof(prm));
  if (!part.units.empty())
    std::memcpy(h + plan->off_units, part.units.data(), sizeof(WorkUnit) * part.units.size());
  std::memcpy(h + plan->off_wptr, part.worker_ptr.data(), sizeof(int32_t) * part.worker_ptr.size());
  if (!part.merge.empty())
    std::memcpy(h + plan->off_merge, part.merge.data(), sizeof(MergeEntry) * part.merge.size());
  if ((e = cudaMemcpyAsync(plan->d_blob, plan->h_blob, plan->blob_bytes, cudaMemcpyHostToDevice,
                           s)) != cudaSuccess)
    return cuda_fail(plan, e, "plan upload");
  // The tcgen05 kernel leaves its arrival counters at zero; a launch that
  // stopped on a device error may not have, so every plan starts from zero.
  if ((e = cudaMemsetAsync(plan->d_counters, 0, sizeof(int32_t) * 8 * plan->max_batch, s)) !=
      cudaSuccess)
    return cuda_fail(plan, e, "counter reset");
  if ((e = cudaEventRecord(plan->upload_done, s)) != cudaSuccess)
    return cuda_fail(plan, e, "cudaEventRecord");

  plan->params = prm;
  plan->kv_indices = kv_indices_dev;
  plan->total_tiles = part.total_tiles;
  plan->planned = true;
  plan->last_error.clear();
  return MLA_OK;
}

// Checks shared by both plan entry points.
mla_status_t check_plan_args(mla_plan_t plan, const int32_t* kv_indptr_host,
                             const int32_t* kv_indices_dev, const int32_t* kv_len_host, int batch,
                             int num_heads, int head_dim_ckv, int head_dim_kpe, int page_size,
                             float sm_scale) {
  std::string why;
  mla_status_t st = validate_batch(kv_indptr_host, kv_len_host, batch, head_dim_ckv,
                                   head_dim_kpe, page_size, sm_scale, &why);
  if (st != MLA_OK) return fail(plan, st, why);
  if (num_heads != plan->num_heads)
    return fail(plan, MLA_ERR_INVALID_ARG, "num_heads differs from the plan's num_heads");
  if (kv_indptr_host[batch] > 0 && kv_indices_dev == nullptr)
    return fail(plan, MLA_ERR_INVALID_ARG, "kv_indices_dev is NULL");
  return MLA_OK;
}

}  // namespace

mla_status_t mla_decode_plan(mla_plan_t plan, const int32_t* kv_indptr_host,
                             const int32_t* kv_indices_dev, const int32_t* kv_len_host,
                             int batch, int num_heads, int head_dim_ckv, int head_dim_kpe,
                             int page_size, float sm_scale, void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  mla_status_t st = check_plan_args(plan, kv_indptr_host, kv_indices_dev, kv_len_host, batch,
                                    num_heads, head_dim_ckv, head_dim_kpe, page_size, sm_scale);
  if (st != MLA_OK) return st;
  if (batch > plan->max_batch)
    return fail(plan, MLA_ERR_CAPACITY, "batch exceeds the plan's max_batch");
  return plan_requests(plan, kv_indptr_host, kv_len_host, batch, kv_indices_dev, num_heads,
                       page_size, sm_scale, stream);
}

mla_status_t mla_decode_plan_multi(mla_plan_t plan, const int32_t* kv_indptr_host,
                                   const int32_t* kv_indices_dev, const int32_t* kv_len_host,
                                   int batch, int q_len, int num_heads, int head_dim_ckv,
                                   int head_dim_kpe, int page_size, float sm_scale,
                                   void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  mla_status_t st = check_plan_args(plan, kv_indptr_host, kv_indices_dev, kv_len_host, batch,
                                    num_heads, head_dim_ckv, head_dim_kpe, page_size, sm_scale);
  if (st != MLA_OK) return st;
  if (q_len < 1) return fail(plan, MLA_ERR_INVALID_ARG, "q_len must be >= 1");
  if (static_cast<long long>(batch) * q_len > plan->max_batch)
    return fail(plan, MLA_ERR_CAPACITY, "batch * q_len exceeds the plan's max_batch");
  for (int b = 0; b < batch; ++b)
    if (kv_len_host[b] < q_len)
      return fail(plan, MLA_ERR_INVALID_ARG,
                  "every request must hold its q_len query tokens in the cache (kv_len >= q_len)");
  // Query j of request b sees the first kv_len - q_len + 1 + j tokens.  On
  // the CTA-pair kernel, when q_len x heads <= 128, the q_len query tokens of
  // a request share its MMA rows (row j * heads + h of the [batch, q_len *
  // heads] view of the query and output arrays, each row masked to its own
  // prefix), so its pages are read once (the plan's share buffers hold any
  // such partition; should one not fit, the form below is used).
  if (plan->kernel == MLA_KERNEL_PAIR && q_len > 1 && q_len * num_heads <= kMaxHeads) {
    st = plan_requests(plan, kv_indptr_host, kv_len_host, batch, kv_indices_dev, q_len * num_heads,
                       page_size, sm_scale, stream, q_len, num_heads);
    if (st != MLA_ERR_CAPACITY) return st;
    plan->last_error.clear();
  }
  // Otherwise query j of request b is planned as its own request over a
  // prefix of b's pages, at row b * q_len + j of the [batch * q_len, heads]
  // query and output arrays.
  std::vector<int32_t> base(static_cast<size_t>(batch) * q_len), len(base.size());
  for (int b = 0; b < batch; ++b)
    for (int j = 0; j < q_len; ++j) {
      base[static_cast<size_t>(b) * q_len + j] = kv_indptr_host[b];
      len[static_cast<size_t>(b) * q_len + j] = kv_len_host[b] - q_len + 1 + j;
    }
  return plan_requests(plan, base.data(), len.data(), batch * q_len, kv_indices_dev, num_heads,
                       page_size, sm_scale, stream);
}

mla_status_t mla_decode_run(mla_plan_t plan, const void* q_nope, const void* q_pe, int q_dtype,
                            const void* ckv_cache, const void* kpe_cache, int kv_dtype,
                            float kv_scale, int num_pages, void* out, int out_dtype, float* lse,
                            void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  if (!plan->planned) return fail(plan, MLA_ERR_NOT_PLANNED, "mla_decode_run before mla_decode_plan");
  if (q_dtype != MLA_DTYPE_BF16)
    return fail(plan, MLA_ERR_UNSUPPORTED, "q_dtype must be MLA_DTYPE_BF16");
  if (kv_dtype != MLA_DTYPE_BF16 && kv_dtype != MLA_DTYPE_FP8_E4M3)
    return fail(plan, MLA_ERR_UNSUPPORTED, "kv_dtype must be BF16 or FP8_E4M3");
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_FP32)
    return fail(plan, MLA_ERR_UNSUPPORTED, "out_dtype must be BF16 or FP32");
  if (!q_nope || !q_pe || !ckv_cache || !kpe_cache || !out || !lse)
    return fail(plan, MLA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (num_pages < 1) return fail(plan, MLA_ERR_INVALID_ARG, "num_pages must be >= 1");
  if ((reinterpret_cast<uintptr_t>(ckv_cache) | reinterpret_cast<uintptr_t>(kpe_cache) |
       reinterpret_cast<uintptr_t>(q_nope) | reinterpret_cast<uintptr_t>(q_pe) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(plan, MLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(kv_scale) || kv_scale <= 0.f)
    return fail(plan, MLA_ERR_INVALID_ARG, "kv_scale must be finite and positive");
  const bool fp8 = kv_dtype == MLA_DTYPE_FP8_E4M3;
  const bool out_f32 = out_dtype == MLA_DTYPE_FP32;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const char* blob = static_cast<const char*>(plan->d_blob);
  DecodeArgs a{};
  a.q_nope = q_nope;
  a.q_pe = q_pe;
  a.ckv = ckv_cache;
  a.kpe = kpe_cache;
  a.kv_indices = plan->kv_indices;
  a.units = reinterpret_cast<const WorkUnit*>(blob + plan->off_units);
  a.worker_ptr = reinterpret_cast<const int32_t*>(blob + plan->off_wptr);
  a.params = reinterpret_cast<const PlanDev*>(blob);
  a.out = out;
  a.lse = lse;
  a.o_part = plan->d_o_part;
  a.lse_part = plan->d_lse_part;
  a.merge = reinterpret_cast<const MergeEntry*>(blob + plan->off_merge);
  a.counters = plan->d_counters;
  a.err = plan->d_err;
  a.num_pages = num_pages;
  a.num_heads = plan->params.num_heads;   // rows per request (q_len x heads when packed)
  a.kv_scale = fp8 ? kv_scale : 1.f;   // the dequantisation scale of fp8 codes only
  a.units_cap = plan->units_cap;
  a.n_workers = plan->n_workers;

  cudaError_t e;
  if (plan->prof_start && (e = cudaEventRecord(plan->prof_start, s)) != cudaSuccess)
    return cuda_fail(plan, e, "cudaEventRecord");
  // DEFAULT: the pair kernel, for an fp8 cache with pages of 32 or more
  // tokens; 16-token fp8 pages go to the one-CTA kernel (which rejects them)
  const int kern = fp8 && plan->kernel_requested == MLA_KERNEL_DEFAULT && plan->params.page_size < kTcVChunkTok
                       ? MLA_KERNEL_TCGEN05
                       : plan->kernel;
  if (kern == MLA_KERNEL_MMA_SYNC) {
    e = launch_decode_mma(a, fp8, out_f32, s);
  } else if (kern == MLA_KERNEL_PAIR) {
    if (fp8 && plan->params.page_size < kTcVChunkTok)
      return fail(plan, MLA_ERR_UNSUPPORTED,
                  "the CTA-pair kernel takes fp8 caches with page_size >= 32; use MLA_KERNEL_MMA_SYNC");
    PairMaps maps;
    if (!encode_pair_maps(&maps, q_nope, q_pe, ckv_cache, kpe_cache, plan->params.batch, plan->params.num_heads,
                          plan->params.page_size, num_pages, fp8))
      return fail(plan, MLA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    e = launch_decode_pair(a, maps, out_f32, fp8, s);
  } else {
    if (fp8 && plan->params.page_size < kTcVChunkTok)
      return fail(plan, MLA_ERR_UNSUPPORTED,
                  "the tcgen05 kernel takes fp8 caches with page_size >= 32; use MLA_KERNEL_MMA_SYNC");
    TcMaps maps;
    if (!encode_tc_maps(&maps, q_nope, ckv_cache, kpe_cache, plan->params.batch, plan->params.num_heads,
                        plan->params.page_size, num_pages, fp8))
      return fail(plan, MLA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    e = launch_decode_tc(a, maps, out_f32, fp8, s);
  }
  if (e != cudaSuccess) return cuda_fail(plan, e, "decode kernel launch");
  if (plan->prof_stop && (e = cudaEventRecord(plan->prof_stop, s)) != cudaSuccess)
    return cuda_fail(plan, e, "cudaEventRecord");

  // The one-CTA tcgen05 kernel combines split requests and fills empty ones
  // itself; after the others a merge kernel does it.
  if (kern == MLA_KERNEL_TCGEN05) return MLA_OK;
  MergeArgs m{};
  m.merge = reinterpret_cast<const MergeEntry*>(blob + plan->off_merge);
  m.params = a.params;
  m.o_part = plan->d_o_part;
  m.lse_part = plan->d_lse_part;
  m.out = out;
  m.lse = lse;
  m.num_heads = plan->params.num_heads;
  m.merge_cap = plan->merge_cap;
  e = launch_merge(m, out_f32, s);
  if (e != cudaSuccess) return cuda_fail(plan, e, "merge kernel launch");
  return MLA_OK;
}

mla_status_t mla_decode_run_host(mla_plan_t plan, const void* q_nope_host, const void* q_pe_host,
                                 int q_dtype, const void* ckv_cache, const void* kpe_cache,
                                 int kv_dtype, float kv_scale, int num_pages, void* out_host,
                                 int out_dtype, float* lse_host, void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  if (!plan->planned) return fail(plan, MLA_ERR_NOT_PLANNED, "run before plan");
  if (!q_nope_host || !q_pe_host || !out_host || !lse_host)
    return fail(plan, MLA_ERR_INVALID_ARG, "NULL host pointer");
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_FP32)
    return fail(plan, MLA_ERR_UNSUPPORTED, "out_dtype must be BF16 or FP32");
  const size_t rows = static_cast<size_t>(plan->params.batch) * plan->params.num_heads;
  const size_t qn = rows * kDCkv * 2, qp = rows * kDKpe * 2;
  const size_t ob = rows * kDCkv * (out_dtype == MLA_DTYPE_FP32 ? 4 : 2), lb = rows * 4;
  cudaError_t e;
  const size_t q_need = align16(qn) + align16(qp);
  const size_t r_need = align16(ob) + align16(lb);
  if (plan->d_q_bytes < q_need) {
    if (plan->d_q) cudaFree(plan->d_q);
    plan->d_q = nullptr;
    plan->d_q_bytes = 0;
    if ((e = cudaMalloc(&plan->d_q, q_need)) != cudaSuccess) return cuda_fail(plan, e, "cudaMalloc");
    plan->d_q_bytes = q_need;
  }
  if (plan->d_res_bytes < r_need) {
    if (plan->d_res) cudaFree(plan->d_res);
    plan->d_res = nullptr;
    plan->d_res_bytes = 0;
    if ((e = cudaMalloc(&plan->d_res, r_need)) != cudaSuccess) return cuda_fail(plan, e, "cudaMalloc");
    plan->d_res_bytes = r_need;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* dq = static_cast<char*>(plan->d_q);
  char* dr = static_cast<char*>(plan->d_res);
  if ((e = cudaMemcpyAsync(dq, q_nope_host, qn, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dq + align16(qn), q_pe_host, qp, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(plan, e, "host to device copy");
  mla_status_t st = mla_decode_run(plan, dq, dq + align16(qn), q_dtype, ckv_cache, kpe_cache,
                                   kv_dtype, kv_scale, num_pages, dr, out_dtype,
                                   reinterpret_cast<float*>(dr + align16(ob)), stream);
  if (st != MLA_OK) return st;
  if ((e = cudaMemcpyAsync(out_host, dr, ob, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(lse_host, dr + align16(ob), lb, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(plan, e, "device to host copy");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(plan, e, "cudaStreamSynchronize");
  return MLA_OK;
}

mla_status_t mla_merge_states(const float* o_a, const float* lse_a, const float* o_b,
                              const float* lse_b, void* out, int out_dtype, float* lse_out,
                              int rows, void* stream) {
  if (rows < 0) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_FP32) return MLA_ERR_UNSUPPORTED;
  if (rows == 0) return MLA_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !out || !lse_out) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o_a) | reinterpret_cast<uintptr_t>(o_b) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return MLA_ERR_INVALID_ARG;
  cudaError_t e = launch_merge_states(o_a, lse_a, o_b, lse_b, out, out_dtype == MLA_DTYPE_FP32,
                                      lse_out, rows, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status_t mla_plan_check_status(mla_plan_t plan) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(plan, e, "cudaDeviceSynchronize");
  int32_t code = 0;
  if ((e = cudaMemcpy(&code, plan->d_err, sizeof(code), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(plan, e, "read error word");
  if ((e = cudaMemset(plan->d_err, 0, sizeof(int32_t))) != cudaSuccess)
    return cuda_fail(plan, e, "clear error word");
  // A launch that gave up on a wait may have left split-request counts
  // behind (they return to zero only when a request is combined): clear
  // them, so the next run of the same plan starts clean without a re-plan.
  if (code != 0 &&
      (e = cudaMemset(plan->d_counters, 0, sizeof(int32_t) * 8 * static_cast<size_t>(plan->max_batch))) !=
          cudaSuccess)
    return cuda_fail(plan, e, "clear split counters");
  if (code == kErrTimeout) return fail(plan, MLA_ERR_DEVICE_TIMEOUT, "a device wait timed out");
  if (code == kErrBounds) return fail(plan, MLA_ERR_DEVICE_BOUNDS, "a page id was out of range");
  return MLA_OK;
}

mla_status_t mla_plan_set_profile_events(mla_plan_t plan, void* start_event, void* stop_event) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  plan->prof_start = static_cast<cudaEvent_t>(start_event);
  plan->prof_stop = static_cast<cudaEvent_t>(stop_event);
  return MLA_OK;
}

mla_status_t mla_plan_info(mla_plan_t plan, mla_plan_info_t* info) {
  if (!plan || !info) return MLA_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->num_sms = plan->num_sms;
  info->num_workers = plan->n_workers;
  info->num_units = plan->planned ? plan->params.n_units : 0;
  info->num_partial_slots = plan->planned ? plan->params.n_slots : 0;
  info->num_merge = plan->planned ? plan->params.n_merge : 0;
  info->total_tiles = plan->total_tiles;
  info->batch = plan->planned ? plan->params.batch : 0;
  info->num_heads = plan->num_heads;
  info->page_size = plan->planned ? plan->params.page_size : 0;
  info->kernel = plan->kernel;
  info->tile_tokens = plan->tile_tokens;
  info->workspace_bytes = static_cast<int64_t>(plan->blob_bytes) +
                          static_cast<int64_t>(sizeof(float)) * static_cast<int64_t>(plan->part_rows_cap) *
                              (kDCkv + kLsePartCopies);
  return MLA_OK;
}

}  // extern "C"
