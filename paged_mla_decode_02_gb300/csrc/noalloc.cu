// Paged MLA decode from fixed scratch memory: a call that allocates nothing.
//
// Who needs it.  A serving process commonly reserves nearly all device memory
// when it starts -- the KV-cache pool plus a caching allocator that accounts
// for every byte -- and from then on a library that calls cudaMalloc on its
// own either fails (the memory is taken), escapes that accounting, or stalls
// the device (cudaFree waits for all work on it).  Such callers cannot own a
// plan object, whose buffers are allocated.  This entry point keeps everything
// the decode needs besides the caller's tensors -- the work-unit list, the
// split partials, the split-request counters and the device status word -- in
// one fixed array that is part of the library image, and assembles the
// work-unit list in static host memory.  It runs the same tcgen05 kernel as
// mla_decode_run.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <string>

#include "kernels.h"
#include "planner.h"

namespace mla {
namespace {

constexpr size_t kScratchBytes = size_t(48) << 20;   // device scratch: 48 MiB
constexpr int kMaxBatch = 4096;                       // requests per call
constexpr int kMaxWorkers = 512;
constexpr int kMaxUnits = kMaxWorkers + kMaxBatch;
constexpr int kMaxDevices = 64;

// Status word at offset 0 (its own 256 bytes), then the plan blob, the split
// partials and the counters of the current call.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];
constexpr size_t kBlobOffset = 256;

struct DeviceSetup {
  bool done;
  unsigned char* scratch;   // device address of g_scratch on that device
  int n_workers;
};
DeviceSetup g_setup[kMaxDevices];

// host staging: PlanDev | units | worker_ptr | merge entries (16-byte aligned parts)
constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
constexpr size_t kHostBlobBytes =
    align_up(sizeof(PlanDev), 16) + align_up(sizeof(WorkUnit) * kMaxUnits, 16) +
    align_up(sizeof(int32_t) * (kMaxWorkers + 1), 16) + sizeof(MergeEntry) * kMaxBatch;
alignas(16) unsigned char g_host_blob[kHostBlobBytes];

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_decode_noalloc(
    const int32_t* kv_indptr_host, const int32_t* kv_indices_dev, const int32_t* kv_len_host,
    int batch, int num_heads, int page_size, float sm_scale, const void* q_nope, const void* q_pe,
    const void* ckv_cache, const void* kpe_cache, float kv_scale, int num_pages, void* out,
    int out_dtype, float* lse, int check_status, void* stream) {
  // ---- arguments (host only; nothing touches the device before they pass) ----
  std::string why;
  if (!kv_indptr_host || !kv_len_host || batch < 0) return MLA_ERR_INVALID_ARG;
  if (batch > kMaxBatch) return MLA_ERR_CAPACITY;
  mla_status_t st = validate_batch(kv_indptr_host, kv_len_host, batch, kDCkv, kDKpe, page_size,
                                   sm_scale, &why);
  if (st != MLA_OK) return st;
  if (num_heads < 1 || num_heads > kMaxHeads) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_FP32) return MLA_ERR_UNSUPPORTED;
  if (!q_nope || !q_pe || !ckv_cache || !kpe_cache || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (kv_indptr_host[batch] > 0 && !kv_indices_dev) return MLA_ERR_INVALID_ARG;
  if (num_pages < 1 || !std::isfinite(kv_scale) || kv_scale <= 0.f) return MLA_ERR_INVALID_ARG;
  // bf16 caches only: a scale other than 1 can only mean a quantised cache
  if (kv_scale != 1.f) return MLA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(ckv_cache) | reinterpret_cast<uintptr_t>(kpe_cache) |
       reinterpret_cast<uintptr_t>(q_nope) | reinterpret_cast<uintptr_t>(q_pe) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return MLA_ERR_INVALID_ARG;

  // ---- once per device: scratch address and worker count ----
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  DeviceSetup& su = g_setup[dev];
  if (!su.done) {
    void* ptr = nullptr;
    int sms = 0, resident = 0;
    if ((e = cudaGetSymbolAddress(&ptr, g_scratch)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = decode_tc_max_workers(&resident)) != cudaSuccess || resident < 1) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    int nw = sms / 2 < 1 ? 1 : sms / 2;
    if (nw > resident) nw = resident;
    if (nw > kMaxWorkers) nw = kMaxWorkers;
    su.scratch = static_cast<unsigned char*>(ptr);
    su.n_workers = nw;
    su.done = true;
  }

  // ---- partition into static host memory ----
  // (the blob goes to scratch offset kBlobOffset; the status word stays at 0)
  const size_t off_units = align_up(sizeof(PlanDev), 16);
  WorkUnit* units = reinterpret_cast<WorkUnit*>(g_host_blob + off_units);
  // worker offsets and merge entries follow the units, whose count is known
  // only after the partition: staged separately, then placed
  int32_t wptr_tmp[kMaxWorkers + 1];
  static MergeEntry merge_stage[kMaxBatch];
  int n_merge = 0;
  const int n_units = partition_units(kv_indptr_host, kv_len_host, batch, su.n_workers, kTileTc,
                                      units, wptr_tmp);
  const int n_slots = assign_slots(units, n_units, kv_len_host, batch, kTileTc, merge_stage, &n_merge);
  const size_t off_wptr = align_up(off_units + sizeof(WorkUnit) * n_units, 16);
  const size_t off_merge = align_up(off_wptr + sizeof(int32_t) * (su.n_workers + 1), 16);
  const size_t blob_bytes = off_merge + sizeof(MergeEntry) * n_merge;
  std::memcpy(g_host_blob + off_wptr, wptr_tmp, sizeof(int32_t) * (su.n_workers + 1));
  std::memcpy(g_host_blob + off_merge, merge_stage, sizeof(MergeEntry) * n_merge);
  PlanDev prm{};
  prm.n_units = n_units;
  prm.n_merge = n_merge;
  prm.n_workers = su.n_workers;
  prm.batch = batch;
  prm.num_heads = num_heads;
  prm.page_size = page_size;
  prm.sm_scale = sm_scale;
  prm.n_slots = n_slots;
  std::memcpy(g_host_blob, &prm, sizeof(prm));

  // ---- scratch layout for this call: status word | blob | partials | counters ----
  const size_t off_opart = align_up(kBlobOffset + blob_bytes, 256);
  const size_t off_lpart =
      align_up(off_opart + sizeof(float) * static_cast<size_t>(n_slots) * num_heads * kDCkv, 256);
  const size_t off_cnt = align_up(
      off_lpart + sizeof(float) * static_cast<size_t>(n_slots) * kLsePartCopies * num_heads, 256);
  const size_t need = off_cnt + sizeof(int32_t) * 8 * static_cast<size_t>(batch);
  if (need > kScratchBytes) return MLA_ERR_CAPACITY;

  // ---- upload, zero the split counters, launch ----
  // The status word is not cleared here: it keeps the first error of any call
  // until a call with check_status != 0 reads and clears it.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* sc = su.scratch;
  if ((e = cudaMemcpyAsync(sc + kBlobOffset, g_host_blob, blob_bytes, cudaMemcpyHostToDevice, s)) !=
          cudaSuccess ||
      (e = cudaMemsetAsync(sc + off_cnt, 0, need - off_cnt, s)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  TcMaps maps;
  if (!encode_tc_maps(&maps, q_nope, ckv_cache, kpe_cache, batch, num_heads, page_size, num_pages))
    return MLA_ERR_CUDA;
  DecodeArgs a{};
  a.q_nope = q_nope;
  a.q_pe = q_pe;
  a.ckv = ckv_cache;
  a.kpe = kpe_cache;
  a.kv_indices = kv_indices_dev;
  a.units = reinterpret_cast<const WorkUnit*>(sc + kBlobOffset + off_units);
  a.worker_ptr = reinterpret_cast<const int32_t*>(sc + kBlobOffset + off_wptr);
  a.params = reinterpret_cast<const PlanDev*>(sc + kBlobOffset);
  a.out = out;
  a.lse = lse;
  a.o_part = reinterpret_cast<float*>(sc + off_opart);
  a.lse_part = reinterpret_cast<float*>(sc + off_lpart);
  a.merge = reinterpret_cast<const MergeEntry*>(sc + kBlobOffset + off_merge);
  a.counters = reinterpret_cast<int32_t*>(sc + off_cnt);
  a.err = reinterpret_cast<int32_t*>(sc);
  a.num_pages = num_pages;
  a.num_heads = num_heads;
  a.kv_scale = 1.f;   // a bf16 cache: no dequantisation scale
  a.units_cap = n_units;
  a.n_workers = su.n_workers;
  if ((e = launch_decode_tc(a, maps, out_dtype == MLA_DTYPE_FP32, false, s)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (!check_status) return MLA_OK;
  // the first error recorded since the last checking call (this one included)
  int32_t err = 0;
  if ((e = cudaMemcpyAsync(&err, a.err, sizeof(err), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess ||
      (err != 0 && (e = cudaMemsetAsync(a.err, 0, sizeof(int32_t), s)) != cudaSuccess)) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return err ? static_cast<mla_status_t>(err) : MLA_OK;
}
