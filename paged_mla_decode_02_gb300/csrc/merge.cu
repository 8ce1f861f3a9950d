// Split-KV merge: combines the partial attentions of a request, each exact
// over its own token range, by log-sum-exp.  For request b, head h with
// partials (O_i, lse_i), i = 1..n (O_i already normalised by its own sum):
//   M = max_i lse_i,  w_i = exp(lse_i - M),
//   out = sum_i w_i O_i / sum_i w_i,   lse = M + log(sum_i w_i).
// This is the combination that cascade (multi-level) attention relies on,
// whose outputs were checked against plain attention in "[V1][Core]
// FlashInfer attention backend for V1" (vLLM PR #14061, "Outstanding items").
// A request with no tokens (n = 0) gets out = 0 and lse = -inf.
#include <cuda_bf16.h>

#include "kernels.h"

namespace mla {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kChunk = 32;                     // dims per block
constexpr int kChunks = kDCkv / kChunk;        // grid.y

// One block per (request, 32-dim chunk).  The partials are read in their
// [slot][d/4][h][d%4] layout, consecutive threads on consecutive heads
// (coalesced); the merged chunk is staged in shared memory and written out
// row by row, 64 or 128 contiguous bytes per head.
template <bool kOutF32>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  const int e = blockIdx.x;
  if (e >= a.params->n_merge) return;
  const MergeEntry me = a.merge[e];
  const int H = a.num_heads;
  const int dq = blockIdx.y;
  __shared__ float tile[kMaxHeads][kChunk + 1];
  __shared__ float s_max[kMaxHeads], s_inv[kMaxHeads];
  const int t = threadIdx.x;
  if (t < H) {
    float M = -INFINITY, wsum = 0.f;
    for (int i = 0; i < me.n_slots; ++i)
      M = fmaxf(M, a.lse_part[lse_part_offset(me.first_slot + i, 0, t, H)]);
    for (int i = 0; i < me.n_slots; ++i)
      wsum += __expf(a.lse_part[lse_part_offset(me.first_slot + i, 0, t, H)] - M);
    s_max[t] = M;
    s_inv[t] = me.n_slots > 0 ? 1.f / wsum : 0.f;
    if (dq == 0) a.lse[static_cast<size_t>(me.req) * H + t] = me.n_slots > 0 ? M + __logf(wsum) : -INFINITY;
  }
  __syncthreads();
  // (kChunk / 4) * H <= kItems * kMergeThreads items of 4 dims; each thread
  // issues the loads of all its items for one slot before accumulating.
  constexpr int kItems = (kChunk / 4) * kMaxHeads / kMergeThreads;
  float4 acc[kItems];
  int hk[kItems], dk[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int idx = t + k * kMergeThreads;
    const int dg = idx / H;
    hk[k] = idx - dg * H;
    dk[k] = idx < (kChunk / 4) * H ? dq * kChunk + 4 * dg : -1;
  }
  for (int i = 0; i < me.n_slots; ++i) {
    const int slot = me.first_slot + i;
    float4 o[kItems];
    float l[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      if (dk[k] >= 0) {
        o[k] = *reinterpret_cast<const float4*>(a.o_part + part_offset(slot, hk[k], dk[k], H));
        l[k] = a.lse_part[lse_part_offset(slot, 0, hk[k], H)];
      }
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      if (dk[k] >= 0) {
        const float w = __expf(l[k] - s_max[hk[k]]);
        acc[k].x += w * o[k].x; acc[k].y += w * o[k].y; acc[k].z += w * o[k].z; acc[k].w += w * o[k].w;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    if (dk[k] >= 0) {
      const int h = hk[k], c = dk[k] - dq * kChunk;
      const float inv = s_inv[h];
      tile[h][c] = acc[k].x * inv;
      tile[h][c + 1] = acc[k].y * inv;
      tile[h][c + 2] = acc[k].z * inv;
      tile[h][c + 3] = acc[k].w * inv;
    }
  }
  __syncthreads();
  const size_t row0 = static_cast<size_t>(me.req) * H;
  if (kOutF32) {
    for (int idx = t; idx < H * (kChunk / 4); idx += kMergeThreads) {
      const int h = idx / (kChunk / 4), q = idx % (kChunk / 4);
      *reinterpret_cast<float4*>(static_cast<float*>(a.out) + (row0 + h) * kDCkv + dq * kChunk + 4 * q) =
          make_float4(tile[h][4 * q], tile[h][4 * q + 1], tile[h][4 * q + 2], tile[h][4 * q + 3]);
    }
  } else {
    for (int idx = t; idx < H * (kChunk / 8); idx += kMergeThreads) {
      const int h = idx / (kChunk / 8), q = idx % (kChunk / 8);
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(tile[h][8 * q + 2 * k], tile[h][8 * q + 2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + (row0 + h) * kDCkv + dq * kChunk + 8 * q) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, bool out_f32, cudaStream_t s) {
  if (a.merge_cap <= 0) return cudaSuccess;
  dim3 grid(a.merge_cap, kChunks);
  if (out_f32)
    merge_kernel<true><<<grid, kMergeThreads, 0, s>>>(a);
  else
    merge_kernel<false><<<grid, kMergeThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
