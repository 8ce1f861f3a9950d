// The per-head projections on either side of the latent decode.
//
// Absorbed MLA decode attends in the 512-wide latent space of the compressed
// cache (head_dim_ckv = kv_lora_rank, with the rope part kept apart:
// "[WIP] support flashinfer_mla", vLLM-metax PR #113, review of the
// decode_wrapper.plan parameters).  A head's own no-rope query (dn wide) is
// taken into that space before the decode, and the decode's latent output
// is taken back to the head's value width (dv) after it:
//   q_nope[b,h,:] = W_UK[h] (512 x dn) . q_raw[b,h,:]      (absorb)
//   o[b,h,:]      = out[b,h,:] . W_UV[h] (512 x dv)        (project)
// Both are, per head, a GEMM with the batch as M:
//   absorb:  [B x 512] = [B x dn] . W_UK[h]^T   (W_UK[h] rows are K-major)
//   project: [B x dv]  = [B x 512] . W_UV[h]    (W_UV[h] rows are N-major)
// One persistent kernel serves both.  Work items are (head, 128 output
// columns, 128 batch rows), dealt round-robin to one CTA per SM:
// - a copy warp streams each item's operands through a three-stage ring of
//   128-byte-swizzled panels (TMA);
// - one thread issues the tcgen05 MMAs (M 128, K 16) into one of two TMEM
//   accumulators;
// - four warps drain the other accumulator (one TMEM lane quadrant each),
//   round to bf16 and store.
// Rows past the batch are zero-filled by TMA and never stored.  The weights
// dominate the traffic (128 KB per head for dn = dv = 128), so the kernels
// are bound by HBM: 2 x 16.8 MB for 128 heads.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"
#include "tc_utils.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace tc;

constexpr int kRows = 128;              // batch rows per work item (the MMA's M)
constexpr int kPanel = kRows * 128;     // one 64-element panel of 128 rows
constexpr int kKC = 128;                // K per pipeline stage (at most)
constexpr int kStages = 3;              // depth of the shared-memory ring
constexpr int kProjThreads = 192;       // warp 0 copies, warp 1 MMAs, warps 2..5 epilogue

__device__ int32_t g_proj_err;   // first device error of a projection kernel

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32]) {
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
    w[k] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) d[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// Persistent projection GEMM.  A work item is (head h, output columns
// n0 .. n0 + N - 1, batch rows m0 .. m0 + 127):
//   C[b, h, n0 + n] = sum_k A[b, h, k] . W_h(k, n)
// A is read through a 3-D map of [batch, heads, K] in boxes of a_rows rows
// (min(batch, 128)): with a smaller batch the MMA's rows past it see stale
// shared memory, which only reaches accumulator rows that are never stored.
// W is read through a 2-D map of [heads * 512, width]:
//   kWRowsN (absorb):   W_h(k, n) = W[512 h + n][k]  (rows are output columns,
//                       the K-major B operand);
//   !kWRowsN (project): W_h(k, n) = W[512 h + k][n]  (rows are the K index,
//                       the N-major B operand).
// Items go round-robin over the CTAs (one per SM).  Warp 0 streams each
// item's K in chunks of kKC through a kStages-deep ring (A: kKC / 64 panels
// of [128 rows x 64]; W: the matching panels of the slice), warp 1 issues the
// MMAs of an item into one of two TMEM accumulators, warps 2..5 drain the
// other one to global memory as bf16 rows.
template <int K, int N, bool kWRowsN, int kOutW>
__global__ void __launch_bounds__(kProjThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
                __nv_bfloat16* __restrict__ c_out, int batch, int heads, int n_items, int a_rows) {
  // launched as a programmatic dependent of the previous kernel on the
  // stream: nothing is read before that kernel has completed and its writes
  // are visible (a no-op in a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel on the stream may be scheduled now; it waits for this
  // one to complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int KC = K < kKC ? K : kKC;
  constexpr int kChunks = K / KC;                   // pipeline stages per item
  constexpr int kSlices = kOutW / N;                // column slices per head
  constexpr int kABytes = (KC / 64) * kPanel;
  constexpr int kWPanel = kWRowsN ? N * 128 : KC * 128;          // one 64-wide panel of W
  constexpr int kWBytes = kWRowsN ? (KC / 64) * kWPanel : (N / 64) * kWPanel;
  constexpr int kStage = kABytes + kWBytes;
  static_assert(kStage % 1024 == 0 && kStages * kStage <= 200 * 1024, "stage layout");
  enum { kFull = 0, kEmpty = kStages, kTFull = 2 * kStages, kTEmpty = kTFull + 2, kFinal = kTEmpty + 2,
         kNumBar };
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(sm);
  const uint32_t bars = base + kStages * kStage;
  auto bar = [&](int i) { return bars + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kStages * kStage + 8 * kNumBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kStages * kStage + 8 * kNumBar + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBar; ++i) mbar_init(bar(i), (i == kTEmpty || i == kTEmpty + 1) ? 4 : 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 2 * N);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  auto item_coords = [&](int it, int& h, int& n0, int& m0) {   // slices of one head are adjacent
    const int sl = it % kSlices, hm = it / kSlices;
    h = hm % heads;
    m0 = (hm / heads) * kRows;
    n0 = sl * N;
  };
  bool ok = true;

  if (warp == 0) {
    // ---------------- copies ----------------
    int st = 0;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      int h, n0, m0;
      item_coords(it, h, n0, m0);
      for (int kc = 0; kc < kChunks && ok; ++kc, ++st) {
        const int slot = st % kStages;
        if (!(ok = mbar_wait_warp(bar(kEmpty + slot), ((st / kStages) & 1) ^ 1, abort_flag))) break;
        if (lane == 0) {
          const uint32_t sa = base + slot * kStage, sw = sa + kABytes;
          mbar_arrive_expect_tx(bar(kFull + slot), (KC / 64) * a_rows * 128 + kWBytes);
          for (int p = 0; p < KC / 64; ++p) tma_load_3d(sa + p * kPanel, &map_a, kc * KC + 64 * p, h, m0, bar(kFull + slot));
          if (kWRowsN) {
            for (int p = 0; p < KC / 64; ++p)
              tma_load_2d(sw + p * kWPanel, &map_w, kc * KC + 64 * p, 512 * h + n0, bar(kFull + slot));
          } else {
            for (int q = 0; q < N / 64; ++q)
              tma_load_2d(sw + q * kWPanel, &map_w, n0 + 64 * q, 512 * h + kc * KC, bar(kFull + slot));
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) report_error(&g_proj_err, kErrTimeout);
    if (lane == 0)   // every copy issued has landed before the CTA leaves
      for (int k = 1; k <= kStages && k <= st; ++k)
        mbar_wait_drain(bar(kFull + (st - k) % kStages), ((st - k) / kStages) & 1);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMAs ----------------
    constexpr uint32_t idesc = idesc_bf16_f32(kRows, N, false, !kWRowsN);
    int st = 0, n = 0;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++n) {
      const int acc = n & 1;
      if (!(ok = mbar_wait_warp(bar(kTEmpty + acc), ((n >> 1) & 1) ^ 1, abort_flag))) break;
      tc_fence_after();
      for (int kc = 0; kc < kChunks && ok; ++kc, ++st) {
        const int slot = st % kStages;
        if (!(ok = mbar_wait_warp(bar(kFull + slot), (st / kStages) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t sa = base + slot * kStage, sw = sa + kABytes;
        const uint64_t a0 = smem_desc(sa, 16, 1024, kSw128);
        const uint64_t w0 = kWRowsN ? smem_desc(sw, 16, 1024, kSw128) : smem_desc(sw, kWPanel, 1024, kSw128);
#pragma unroll
        for (int kk = 0; kk < KC / 16; ++kk) {
          const uint32_t aoff = (kk / 4) * kPanel + (kk % 4) * 32;
          const uint32_t woff = kWRowsN ? (kk / 4) * kWPanel + (kk % 4) * 32 : kk * 16 * 128;
          mma_ss(tmem + acc * N, a0 + static_cast<uint64_t>(aoff >> 4), w0 + static_cast<uint64_t>(woff >> 4),
                 idesc, (kc | kk) != 0, lane == 0);
        }
        mma_commit(bar(kEmpty + slot), lane == 0);
      }
      if (!ok) break;
      mma_commit(bar(kTFull + acc), lane == 0);
    }
    if (!ok && lane == 0) report_error(&g_proj_err, kErrTimeout);
    mma_commit(bar(kFinal), lane == 0);   // every MMA issued completes before TMEM is freed
    if (lane == 0) mbar_wait_drain(bar(kFinal), 0);
    __syncwarp();
  } else {
    // ---------------- epilogue: row m0 + 32 quad + lane ----------------
    const int quad = warp & 3;
    int n = 0;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++n) {
      int h, n0, m0;
      item_coords(it, h, n0, m0);
      const int acc = n & 1;
      if (!(ok = mbar_wait_warp(bar(kTFull + acc), (n >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const int b = m0 + 32 * quad + lane;
      __nv_bfloat16* row = c_out + (static_cast<size_t>(b) * heads + h) * kOutW + n0;
#pragma unroll 1
      for (int c = 0; c < N / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + acc * N + 32 * c, v);
        tmem_ld_wait();
        if (b < batch) store_row_bf16(row + 32 * c, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kTEmpty + acc));
    }
    if (!ok && lane == 0) report_error(&g_proj_err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * N);
  }
}

template <int K, int N, bool kWRowsN, int kOutW>
constexpr int proj_smem() {
  constexpr int KC = K < kKC ? K : kKC;
  constexpr int stage = (KC / 64) * kPanel + (kWRowsN ? (KC / 64) * N * 128 : (N / 64) * KC * 128);
  return kStages * stage + 8 * (2 * kStages + 5) + 8 + 1024;
}

// 3-D map of a [batch, heads, width] bf16 array seen as (element, head, row):
// a box (64, 1, min(batch, 128)) is one 64-element panel of one head for the
// rows of one 128-row tile of the batch (rows past the batch, in the last
// tile of a larger batch, zero-filled).
bool encode_rows(CUtensorMap* m, const void* base, int batch, int heads, int width) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(width) * 2,
                           static_cast<cuuint64_t>(heads) * width * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(batch < kRows ? batch : kRows)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map of the weights [heads * 512, width] bf16, box box_rows x 64 elements.
bool encode_weights(CUtensorMap* m, const void* base, int heads, int width, uint32_t box_rows) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(heads) * 512};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(width) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int K, int N, bool kWRowsN, int kOutW>
cudaError_t launch_proj(const CUtensorMap& a, const CUtensorMap& w, __nv_bfloat16* dst, int batch,
                        int heads, cudaStream_t s) {
  auto kernel = proj_kernel<K, N, kWRowsN, kOutW>;
  constexpr int smem = proj_smem<K, N, kWRowsN, kOutW>();
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int items = heads * (kOutW / N) * ((batch + kRows - 1) / kRows);
  const int grid = items < sms ? items : sms;
  // a programmatic dependent launch: the grid is scheduled while the previous
  // kernel drains, and waits for it at its first instruction
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kProjThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, w, dst, batch, heads, items, batch < kRows ? batch : kRows);
}

mla_status_t finish(cudaError_t e, int check_status, cudaStream_t s) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (!check_status) return MLA_OK;
  int32_t err = 0;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess ||
      (e = cudaMemcpyFromSymbol(&err, g_proj_err, sizeof(err))) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (err) {
    const int32_t zero = 0;
    cudaMemcpyToSymbol(g_proj_err, &zero, sizeof(zero));
  }
  return err ? static_cast<mla_status_t>(err) : MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_absorb_q(const void* q_nope_raw, const void* w_uk, void* q_nope,
                                     int batch, int num_heads, int head_dim_nope,
                                     int check_status, void* stream) {
  if (batch < 1 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (head_dim_nope != 64 && head_dim_nope != 128) return MLA_ERR_UNSUPPORTED;
  if (!q_nope_raw || !w_uk || !q_nope) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope_raw) || !aligned16(w_uk) || !aligned16(q_nope)) return MLA_ERR_INVALID_ARG;
  CUtensorMap mq, mw;
  if (!encode_rows(&mq, q_nope_raw, batch, num_heads, head_dim_nope) ||
      !encode_weights(&mw, w_uk, num_heads, head_dim_nope, kRows))
    return MLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* dst = static_cast<__nv_bfloat16*>(q_nope);
  const cudaError_t e = head_dim_nope == 128
                            ? launch_proj<128, 128, true, kDCkv>(mq, mw, dst, batch, num_heads, s)
                            : launch_proj<64, 128, true, kDCkv>(mq, mw, dst, batch, num_heads, s);
  return finish(e, check_status, s);
}

extern "C" mla_status_t mla_project_out(const void* out, const void* w_uv, void* o, int batch,
                                        int num_heads, int head_dim_v, int check_status,
                                        void* stream) {
  if (batch < 1 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (head_dim_v != 64 && head_dim_v != 128) return MLA_ERR_UNSUPPORTED;
  if (!out || !w_uv || !o) return MLA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(w_uv) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
  CUtensorMap mo, mw;
  if (!encode_rows(&mo, out, batch, num_heads, kDCkv) ||
      !encode_weights(&mw, w_uv, num_heads, head_dim_v, kKC))
    return MLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* dst = static_cast<__nv_bfloat16*>(o);
  const cudaError_t e = head_dim_v == 128
                            ? launch_proj<kDCkv, 128, false, 128>(mo, mw, dst, batch, num_heads, s)
                            : launch_proj<kDCkv, 64, false, 64>(mo, mw, dst, batch, num_heads, s);
  return finish(e, check_status, s);
}
