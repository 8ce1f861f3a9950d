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
#include "merge.h"

namespace mla {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kChunk = 32;                     // dims per block (the largest)
// Fewer heads, narrower chunks: with H <= 32 a block takes 8 dims, so a
// request spreads over 64 blocks and each block's threads split its slots
// into more groups.
__host__ __device__ inline int merge_chunk(int H) { return H <= 32 ? 8 : kChunk; }

// One block per (request, 32-dim chunk).  The partials are read in their
// [slot][d/8][h][d%8] layout, consecutive threads on consecutive heads
// (coalesced); the merged chunk is staged in shared memory and written out
// row by row, 64 or 128 contiguous bytes per head.  A long request can have
// a partial from every worker, so the slots are spread over the threads too:
// the per-head maximum and weight sum are reduced by G adjacent lanes per
// head, and with fewer than 32 heads the weighted sum is split over S thread
// groups (each in slot order, the groups then added in group order), every
// group loading kAhead slots before accumulating them.
template <bool kOutF32>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  // launched as a programmatic dependent of the decode kernel: wait for it
  // (a no-op in a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int e = blockIdx.x;
  if (e >= a.params->n_merge) return;
  const MergeEntry me = a.merge[e];
  const int H = a.num_heads;
  const int n = me.n_slots;
  const int dq = blockIdx.y;
  const int C = merge_chunk(H);
  __shared__ float tile[kMaxHeads][kChunk + 1];
  __shared__ float s_max[kMaxHeads], s_inv[kMaxHeads];
  __shared__ float4 s_part[kMergeThreads];
  const int t = threadIdx.x;
  constexpr int kAhead = 4;
  {
    int G = 1;   // lanes per head: a power of two, G * H <= threads
    while (G < 32 && 2 * G * H <= kMergeThreads) G *= 2;
    const int h = t / G, g = t % G;
    const bool act = h < H;
    // one pass, running maximum and the weight sum relative to it; four
    // slots' loads issued before they are folded in
    float M = -INFINITY, wsum = 0.f;
    if (act)
      for (int i0 = g; i0 < n; i0 += 4 * G) {
        float l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          l[j] = i0 + j * G < n ? a.lse_part[lse_part_offset(me.first_slot + i0 + j * G, 0, h, H)] : -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (l[j] == -INFINITY) continue;
          const float Mn = fmaxf(M, l[j]);
          wsum = wsum * __expf(M - Mn) + __expf(l[j] - Mn);
          M = Mn;
        }
      }
    for (int off = G / 2; off > 0; off >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, off);
      const float w2 = __shfl_xor_sync(0xffffffffu, wsum, off);
      const float Mn = fmaxf(M, M2);
      if (Mn != -INFINITY) {
        wsum = (M == -INFINITY ? 0.f : wsum * __expf(M - Mn)) + (M2 == -INFINITY ? 0.f : w2 * __expf(M2 - Mn));
        M = Mn;
      }
    }
    if (act && g == 0) {
      s_max[h] = M;
      s_inv[h] = n > 0 ? 1.f / wsum : 0.f;
      if (dq == 0) a.lse[static_cast<size_t>(me.req) * H + h] = n > 0 ? M + __logf(wsum) : -INFINITY;
    }
  }
  __syncthreads();
  const int items = (C / 4) * H;   // 4-dim items of this chunk
  if (items >= kMergeThreads) {
    // (kChunk / 4) * H <= kItems * kMergeThreads: several items per thread
    constexpr int kItems = (kChunk / 4) * kMaxHeads / kMergeThreads;
    float4 acc[kItems];
    int hk[kItems], dk[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int idx = t + k * kMergeThreads;
      const int dg = idx / H;
      hk[k] = idx - dg * H;
      dk[k] = idx < items ? dq * C + 4 * dg : -1;
    }
    for (int i0 = 0; i0 < n; i0 += kAhead) {
      float4 o[kAhead][kItems];
      float l[kAhead][kItems];
#pragma unroll
      for (int j = 0; j < kAhead; ++j)
#pragma unroll
        for (int k = 0; k < kItems; ++k)
          if (dk[k] >= 0 && i0 + j < n) {
            o[j][k] = *reinterpret_cast<const float4*>(a.o_part + part_offset(me.first_slot + i0 + j, hk[k], dk[k], H));
            l[j][k] = a.lse_part[lse_part_offset(me.first_slot + i0 + j, 0, hk[k], H)];
          }
#pragma unroll
      for (int j = 0; j < kAhead; ++j)
#pragma unroll
        for (int k = 0; k < kItems; ++k)
          if (dk[k] >= 0 && i0 + j < n) {
            const float w = __expf(l[j][k] - s_max[hk[k]]);
            acc[k].x += w * o[j][k].x; acc[k].y += w * o[j][k].y; acc[k].z += w * o[j][k].z; acc[k].w += w * o[j][k].w;
          }
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      if (dk[k] >= 0) {
        const int h = hk[k], c = dk[k] - dq * C;
        const float inv = s_inv[h];
        tile[h][c] = acc[k].x * inv;
        tile[h][c + 1] = acc[k].y * inv;
        tile[h][c + 2] = acc[k].z * inv;
        tile[h][c + 3] = acc[k].w * inv;
      }
    }
  } else {
    // one item per thread; S groups of threads take every S-th slot, each
    // loading kAheadSmall slots before folding them in
    constexpr int kAheadSmall = 8;
    int S = 1;
    while (2 * S * items <= kMergeThreads) S *= 2;
    const int item = t % items, sg = t / items;
    const int dg = item / H, h = item - dg * H, d = dq * C + 4 * dg;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (sg < S) {
      for (int i0 = sg; i0 < n; i0 += S * kAheadSmall) {
        float4 o[kAheadSmall];
        float l[kAheadSmall];
#pragma unroll
        for (int j = 0; j < kAheadSmall; ++j)
          if (i0 + S * j < n) {
            o[j] = *reinterpret_cast<const float4*>(a.o_part + part_offset(me.first_slot + i0 + S * j, h, d, H));
            l[j] = a.lse_part[lse_part_offset(me.first_slot + i0 + S * j, 0, h, H)];
          }
#pragma unroll
        for (int j = 0; j < kAheadSmall; ++j)
          if (i0 + S * j < n) {
            const float w = __expf(l[j] - s_max[h]);
            acc.x += w * o[j].x; acc.y += w * o[j].y; acc.z += w * o[j].z; acc.w += w * o[j].w;
          }
      }
    }
    s_part[t] = acc;
    __syncthreads();
    if (t < items) {
      float4 sum = s_part[t];
      for (int q = 1; q < S; ++q) {
        const float4 v = s_part[t + q * items];
        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
      }
      const int c = 4 * dg;
      const float inv = s_inv[h];
      tile[h][c] = sum.x * inv;
      tile[h][c + 1] = sum.y * inv;
      tile[h][c + 2] = sum.z * inv;
      tile[h][c + 3] = sum.w * inv;
    }
  }
  __syncthreads();
  const size_t row0 = static_cast<size_t>(me.req) * H;
  if (kOutF32) {
    for (int idx = t; idx < H * (C / 4); idx += kMergeThreads) {
      const int h = idx / (C / 4), q = idx % (C / 4);
      *reinterpret_cast<float4*>(static_cast<float*>(a.out) + (row0 + h) * kDCkv + dq * C + 4 * q) =
          make_float4(tile[h][4 * q], tile[h][4 * q + 1], tile[h][4 * q + 2], tile[h][4 * q + 3]);
    }
  } else {
    for (int idx = t; idx < H * (C / 8); idx += kMergeThreads) {
      const int h = idx / (C / 8), q = idx % (C / 8);
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(tile[h][8 * q + 2 * k], tile[h][8 * q + 2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + (row0 + h) * kDCkv + dq * C + 8 * q) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Two attention states of the same rows over disjoint token sets (a shared
// prefix and a request's own suffix, say) combined into one: one warp per
// row, 16 consecutive dims per lane (four 16-byte loads from each state), the
// whole row read before it is written, so the output may alias an input.
// The inputs may alias the outputs, so they are neither __restrict__ nor read
// through the read-only path: plain loads (cached in L2 only).
constexpr int kStatesWarps = 8;
template <bool kOutF32>
__global__ void __launch_bounds__(32 * kStatesWarps)
    merge_states_kernel(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                        void* out, float* lse_out, int rows) {
  const int row = blockIdx.x * kStatesWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const size_t base = static_cast<size_t>(row) * kDCkv + 16 * lane;
  const float la = __ldcg(lse_a + row), lb = __ldcg(lse_b + row);
  const float M = fmaxf(la, lb);
  float wa = 0.f, wb = 0.f, lse = -INFINITY;
  if (M != -INFINITY) {
    wa = __expf(la - M);
    wb = __expf(lb - M);
    const float inv = 1.f / (wa + wb);
    lse = M + __logf(wa + wb);
    wa *= inv;
    wb *= inv;
  }
  float4 a4[4], b4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a4[k] = __ldcg(reinterpret_cast<const float4*>(o_a + base) + k);
    b4[k] = __ldcg(reinterpret_cast<const float4*>(o_b + base) + k);
  }
  float v[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {   // a state without weight adds nothing, even where it holds NaN
    v[4 * k] = (wa != 0.f ? wa * a4[k].x : 0.f) + (wb != 0.f ? wb * b4[k].x : 0.f);
    v[4 * k + 1] = (wa != 0.f ? wa * a4[k].y : 0.f) + (wb != 0.f ? wb * b4[k].y : 0.f);
    v[4 * k + 2] = (wa != 0.f ? wa * a4[k].z : 0.f) + (wb != 0.f ? wb * b4[k].z : 0.f);
    v[4 * k + 3] = (wa != 0.f ? wa * a4[k].w : 0.f) + (wb != 0.f ? wb * b4[k].w : 0.f);
  }
  __syncwarp();
  if (kOutF32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + base);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  } else {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
      w[k] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + base);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  if (lane == 0) lse_out[row] = lse;
}

}  // namespace

cudaError_t launch_merge_states(const float* o_a, const float* lse_a, const float* o_b,
                                const float* lse_b, void* out, bool out_f32, float* lse_out,
                                int rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + kStatesWarps - 1) / kStatesWarps;
  if (out_f32)
    merge_states_kernel<true><<<grid, 32 * kStatesWarps, 0, s>>>(o_a, lse_a, o_b, lse_b, out, lse_out, rows);
  else
    merge_states_kernel<false><<<grid, 32 * kStatesWarps, 0, s>>>(o_a, lse_a, o_b, lse_b, out, lse_out, rows);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, bool out_f32, cudaStream_t s) {
  if (a.merge_cap <= 0) return cudaSuccess;
  // Programmatic dependent launch: the merge grid may be scheduled while the
  // decode kernel before it in the stream is still running (on SMs that
  // kernel has left); each block waits for that kernel to complete, and its
  // writes to be visible, before it reads a partial.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.merge_cap, kDCkv / merge_chunk(a.num_heads));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return out_f32 ? cudaLaunchKernelEx(&cfg, merge_kernel<true>, a) : cudaLaunchKernelEx(&cfg, merge_kernel<false>, a);
}

}  // namespace mla
