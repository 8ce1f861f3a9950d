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
// Absorb runs one CTA per (head, 128 latent dims, 128 rows of the batch),
// project one per (head, 128 rows): TMA brings the head's weights and
// query / output rows into shared memory (128-byte swizzled panels), one
// thread issues tcgen05 MMAs (M 128, K 16) into TMEM, four warps read the
// fp32 accumulators back (one TMEM lane quadrant each), round to bf16 and
// store.  Rows past the batch are zero-filled by TMA and never stored.  The
// weights dominate the traffic (128 KB per head for dn = dv = 128), so the
// kernels are bound by HBM: 2 x 16.8 MB for 128 heads.
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

constexpr int kThreads = 128;   // four warps: TMEM lane quadrants 0..3
constexpr int kRows = 128;      // batch rows per CTA (the MMA's M)
constexpr int kPanel = kRows * 128;   // one 64-element panel of 128 rows

__device__ int32_t g_proj_err;   // first device error of a projection kernel

// Shared-memory tail: up to three mbarriers, the TMEM address, the abort flag.
struct Tail {
  uint64_t bar[3];
  uint32_t tmem;
  int32_t abort;
};

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

// Latent dims per absorb CTA: a quarter of the 512, so four CTAs share a
// head and each holds 64 KB of shared memory (three fit on an SM).
constexpr int kAbsorbN = 128;

// q_nope[b, h, n0 .. n0 + 127] = W_UK[h][n0 ..] . q_raw[b, h, :] for the 128
// rows of blockIdx.z, n0 = 128 blockIdx.y.  Shared memory: A = DN / 64 panels
// of [128 rows x 64] (the query rows), B = DN / 64 panels of [128 rows x 64]
// (W_UK[h] rows n0 .. n0 + 127).
template <int DN>
__global__ void __launch_bounds__(kThreads)
    absorb_q_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_w,
                    __nv_bfloat16* __restrict__ q_nope, int batch, int heads) {
  constexpr int kP = DN / 64;
  constexpr int kA = kP * kPanel;
  constexpr int kB = kP * kPanel;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(sm);
  Tail* tail = reinterpret_cast<Tail*>(sm + kA + kB);
  const uint32_t bar_full = smem_u32(&tail->bar[0]), bar_mma = smem_u32(&tail->bar[1]);
  volatile int* abort_flag = &tail->abort;
  const int h = blockIdx.x, n0 = blockIdx.y * kAbsorbN, m0 = blockIdx.z * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tail->abort = 0;
    mbar_init(bar_full, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tail->tmem), kAbsorbN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tail->tmem);

  bool issued = false;   // warp 0: the MMAs (and their commit) were issued
  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_full, kA + kB);
      for (int p = 0; p < kP; ++p) {
        tma_load_3d(base + p * kPanel, &map_q, 64 * p, h, m0, bar_full);
        tma_load_2d(base + kA + p * kPanel, &map_w, 64 * p, 512 * h + n0, bar_full);
      }
    }
    __syncwarp();
    if (mbar_wait_warp(bar_full, 0, abort_flag)) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(kRows, kAbsorbN, false, false);
      const uint64_t a0 = smem_desc(base, 16, 1024, kSw128);
      const uint64_t b0 = smem_desc(base + kA, 16, 1024, kSw128);
      for (int p = 0; p < kP; ++p)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, a0 + static_cast<uint64_t>((p * kPanel + kk * 32) >> 4),
                 b0 + static_cast<uint64_t>((p * kPanel + kk * 32) >> 4), idesc, (p | kk) != 0,
                 lane == 0);
      mma_commit(bar_mma, lane == 0);
      issued = true;
    } else if (lane == 0) {
      report_error(&g_proj_err, kErrTimeout);
    }
  }
  // epilogue: row b = m0 + 32 warp + lane, 4 chunks of 32 latent dims
  const bool ok = mbar_wait_warp(bar_mma, 0, abort_flag);
  tc_fence_after();
  if (ok) {
    const int b = m0 + 32 * warp + lane;
    __nv_bfloat16* row = q_nope + (static_cast<size_t>(b) * heads + h) * kDCkv + n0;
#pragma unroll 1
    for (int c = 0; c < kAbsorbN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32 * c, v);
      tmem_ld_wait();
      if (b < batch) store_row_bf16(row + 32 * c, v);
    }
  } else if (lane == 0) {
    report_error(&g_proj_err, kErrTimeout);
  }
  // every copy has landed and every MMA completed before TMEM is freed and
  // the CTA leaves (they have, unless a wait above gave up)
  if (warp == 0 && lane == 0) {
    mbar_wait_drain(bar_full, 0);
    if (issued) mbar_wait_drain(bar_mma, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kAbsorbN);
  }
}

// o[b, h, :] = out[b, h, :] . W_UV[h] for the 128 rows of blockIdx.y, K = 512
// in two stages of 256 (one shared buffer: A = 4 panels of [128 rows x 64],
// B = DV / 64 panels of [256 k-rows x 64 n], n contiguous).
template <int DV>
__global__ void __launch_bounds__(kThreads, 1)
    project_out_kernel(const __grid_constant__ CUtensorMap map_o, const __grid_constant__ CUtensorMap map_w,
                       __nv_bfloat16* __restrict__ o, int batch, int heads) {
  constexpr int kNP = DV / 64;
  constexpr int kA = 4 * kPanel;
  constexpr int kBPanel = 256 * 128;   // 256 k-rows of one 64-wide n panel
  constexpr int kB = kNP * kBPanel;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(sm);
  Tail* tail = reinterpret_cast<Tail*>(sm + kA + kB);
  const uint32_t bar_full = smem_u32(&tail->bar[0]);
  const uint32_t bar_mma0 = smem_u32(&tail->bar[1]), bar_mma1 = smem_u32(&tail->bar[2]);
  volatile int* abort_flag = &tail->abort;
  const int h = blockIdx.x, m0 = blockIdx.y * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tail->abort = 0;
    mbar_init(bar_full, 1);
    mbar_init(bar_mma0, 1);
    mbar_init(bar_mma1, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tail->tmem), DV);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tail->tmem);

  int staged = 0, committed = 0;   // warp 0: stages whose copies / MMAs were issued
  if (warp == 0) {
    bool ok = true;
    constexpr uint32_t idesc = idesc_bf16_f32(kRows, DV, false, true);
    const uint64_t a0 = smem_desc(base, 16, 1024, kSw128);
    const uint64_t b0 = smem_desc(base + kA, kBPanel, 1024, kSw128);
#pragma unroll 1
    for (int s = 0; s < 2 && ok; ++s) {
      // the buffer is reused: stage 1 loads once stage 0's MMAs have read it
      if (s == 1 && !(ok = mbar_wait_warp(bar_mma0, 0, abort_flag))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_full, kA + kB);
        for (int p = 0; p < 4; ++p) tma_load_3d(base + p * kPanel, &map_o, 64 * (4 * s + p), h, m0, bar_full);
        for (int q = 0; q < kNP; ++q)
          tma_load_2d(base + kA + q * kBPanel, &map_w, 64 * q, 512 * h + 256 * s, bar_full);
      }
      ++staged;
      __syncwarp();
      if (!(ok = mbar_wait_warp(bar_full, s, abort_flag))) break;
      tc_fence_after();
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, a0 + static_cast<uint64_t>((p * kPanel + kk * 32) >> 4),
                 b0 + static_cast<uint64_t>(((64 * p + 16 * kk) * 128) >> 4), idesc,
                 (s | p | kk) != 0, lane == 0);
      mma_commit(s == 0 ? bar_mma0 : bar_mma1, lane == 0);
      ++committed;
    }
    if (!ok && lane == 0) report_error(&g_proj_err, kErrTimeout);
  }
  const bool ok = mbar_wait_warp(bar_mma1, 0, abort_flag);
  tc_fence_after();
  if (ok) {
    const int b = m0 + 32 * warp + lane;
    __nv_bfloat16* row = o + (static_cast<size_t>(b) * heads + h) * DV;
#pragma unroll 1
    for (int c = 0; c < DV / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32 * c, v);
      tmem_ld_wait();
      if (b < batch) store_row_bf16(row + 32 * c, v);
    }
  } else if (lane == 0) {
    report_error(&g_proj_err, kErrTimeout);
  }
  if (warp == 0 && lane == 0) {
    if (staged > 0) mbar_wait_drain(bar_full, (staged - 1) & 1);
    if (committed > 0) mbar_wait_drain(committed == 2 ? bar_mma1 : bar_mma0, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, DV);
  }
}

// 3-D map of a [batch, heads, width] bf16 array seen as (element, head, row):
// a box (64, 1, 128) is one 64-element panel of one head for 128 rows of the
// batch, rows past the batch zero-filled.
bool encode_rows(CUtensorMap* m, const void* base, int batch, int heads, int width) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(width) * 2,
                           static_cast<cuuint64_t>(heads) * width * 2};
  cuuint32_t box[3] = {64, 1, kRows};
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

template <typename K>
cudaError_t launch(K kernel, int smem, dim3 grid, cudaStream_t s, const CUtensorMap& a,
                   const CUtensorMap& b, __nv_bfloat16* dst, int batch, int heads) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, s>>>(a, b, dst, batch, heads);
  return cudaGetLastError();
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
      !encode_weights(&mw, w_uk, num_heads, head_dim_nope, kAbsorbN))
    return MLA_ERR_CUDA;
  const dim3 grid(num_heads, kDCkv / kAbsorbN, (batch + kRows - 1) / kRows);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* dst = static_cast<__nv_bfloat16*>(q_nope);
  const cudaError_t e =
      head_dim_nope == 128
          ? launch(absorb_q_kernel<128>, 4 * kPanel + 1024 + 64, grid, s, mq, mw, dst, batch, num_heads)
          : launch(absorb_q_kernel<64>, 2 * kPanel + 1024 + 64, grid, s, mq, mw, dst, batch, num_heads);
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
      !encode_weights(&mw, w_uv, num_heads, head_dim_v, 256))
    return MLA_ERR_CUDA;
  const dim3 grid(num_heads, (batch + kRows - 1) / kRows);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* dst = static_cast<__nv_bfloat16*>(o);
  const cudaError_t e =
      head_dim_v == 128
          ? launch(project_out_kernel<128>, 4 * kPanel + 2 * 256 * 128 + 1024 + 64, grid, s, mo, mw, dst, batch, num_heads)
          : launch(project_out_kernel<64>, 4 * kPanel + 256 * 128 + 1024 + 64, grid, s, mo, mw, dst, batch, num_heads);
  return finish(e, check_status, s);
}
