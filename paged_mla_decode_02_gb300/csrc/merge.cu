// Split-KV merge: combines the partial attentions of a request, each exact
// over its own token range, by log-sum-exp.  For request b, head h with
// partials (O_i, lse_i), i = 1..n (O_i already normalised by its own sum):
//   M = max_i lse_i,  w_i = exp(lse_i - M),
//   out = sum_i w_i O_i / sum_i w_i,   lse = M + log(sum_i w_i).
// This is the combination that cascade (multi-level) attention relies on,
// whose outputs were checked against plain attention in "[V1][Core]
// FlashInfer attention backend for V1" (vLLM PR #14061, "Outstanding items").
// A request with no tokens (n = 0) gets out = 0 and lse = -inf.
// Two kernels: a flat one for many heads (one thread per request, head and
// four dims) and a chunked one for few heads and many slots.
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

// Work items: (merged request, chunk of C dims), looped over by the grid in
// strides (the grid is sized for the plan's capacity, so a re-planned batch
// replays with the same launch and no block idles on an empty item).  The
// partials are read in their [slot][d/8][h][d%8] layout, consecutive threads
// on consecutive heads (coalesced); the merged chunk is staged in shared
// memory and written out row by row, 16 or 64 contiguous bytes per head.
// Each thread folds the slots into a running (maximum, weight sum, weighted
// output) in slot order, a partial and its log-sum-exp loaded together,
// two (four with few heads) slots at a time: an item takes one memory round
// trip per two (four) slots.  With few heads the slots are split over S thread groups (every
// S-th slot) whose states are then combined in group order.
__device__ __forceinline__ void fold_state(float& M, float& W, float4& acc, float l, const float4& o) {
  if (l == -INFINITY) return;   // a partial with no weight
  const float Mn = fmaxf(M, l);
  const float sa = __expf(M - Mn), sb = __expf(l - Mn);   // M = -inf: sa = 0 (acc, W are 0)
  acc.x = acc.x * sa + o.x * sb;
  acc.y = acc.y * sa + o.y * sb;
  acc.z = acc.z * sa + o.z * sb;
  acc.w = acc.w * sa + o.w * sb;
  W = W * sa + sb;
  M = Mn;
}

template <bool kOutF32>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  // launched as a programmatic dependent of the decode kernel: wait for it
  // (a no-op in a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel on the stream may be scheduled now; it waits for this
  // one to complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int H = a.num_heads;
  const int C = merge_chunk(H);
  const int nchunk = kDCkv / C;
  const int n_items = a.params->n_merge * nchunk;
  const int items = (C / 4) * H;   // 4-dim items of one chunk
  __shared__ float tile[kMaxHeads][kChunk + 1];
  __shared__ float4 s_acc[kMergeThreads];
  __shared__ float2 s_mw[kMergeThreads];
  const int t = threadIdx.x;
  for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
    const int e = w / nchunk, dq = w - e * nchunk;
    const MergeEntry me = a.merge[e];
    const int n = me.n_slots;
    const size_t row0 = static_cast<size_t>(me.req) * H;
    if (items >= kMergeThreads) {
      // several items per thread
      constexpr int kItems = (kChunk / 4) * kMaxHeads / kMergeThreads;
      constexpr int kAhead = 2;
      float4 acc[kItems];
      float M[kItems], W[kItems];
      int hk[kItems], dg[kItems];
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        M[k] = -INFINITY;
        W[k] = 0.f;
        const int idx = t + k * kMergeThreads;
        dg[k] = idx < items ? idx / H : -1;
        hk[k] = idx - (idx / H) * H;
      }
      for (int i0 = 0; i0 < n; i0 += kAhead) {
        float4 o[kAhead][kItems];
        float l[kAhead][kItems];
#pragma unroll
        for (int j = 0; j < kAhead; ++j)
#pragma unroll
          for (int k = 0; k < kItems; ++k)
            if (dg[k] >= 0 && i0 + j < n) {
              const int slot = me.first_slot + i0 + j;
              o[j][k] = *reinterpret_cast<const float4*>(a.o_part + part_offset(slot, hk[k], dq * C + 4 * dg[k], H));
              l[j][k] = a.lse_part[lse_part_offset(slot, 0, hk[k], H)];
            }
#pragma unroll
        for (int j = 0; j < kAhead; ++j)
#pragma unroll
          for (int k = 0; k < kItems; ++k)
            if (dg[k] >= 0 && i0 + j < n) fold_state(M[k], W[k], acc[k], l[j][k], o[j][k]);
      }
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        if (dg[k] < 0) continue;
        const int h = hk[k], c = 4 * dg[k];
        const float inv = W[k] > 0.f ? 1.f / W[k] : 0.f;
        tile[h][c] = acc[k].x * inv;
        tile[h][c + 1] = acc[k].y * inv;
        tile[h][c + 2] = acc[k].z * inv;
        tile[h][c + 3] = acc[k].w * inv;
        if (dq == 0 && dg[k] == 0) a.lse[row0 + h] = W[k] > 0.f ? M[k] + __logf(W[k]) : -INFINITY;
      }
    } else {
      // one item per thread; S groups of threads take every S-th slot, each
      // loading kAheadSmall slots before folding them in
      constexpr int kAheadSmall = 4;
      int S = 1;
      while (2 * S * items <= kMergeThreads) S *= 2;
      const int item = t % items, sg = t / items;
      const int dgi = item / H, h = item - dgi * H, d = dq * C + 4 * dgi;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float M = -INFINITY, W = 0.f;
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
            if (i0 + S * j < n) fold_state(M, W, acc, l[j], o[j]);
        }
      }
      s_acc[t] = acc;
      s_mw[t] = make_float2(M, W);
      __syncthreads();
      if (t < items) {
        for (int q = 1; q < S; ++q) {
          const float2 mw = s_mw[t + q * items];
          if (mw.y <= 0.f) continue;
          const float4 aq = s_acc[t + q * items];
          const float Mn = fmaxf(M, mw.x);
          const float sa = __expf(M - Mn), sb = __expf(mw.x - Mn);
          acc.x = acc.x * sa + aq.x * sb;
          acc.y = acc.y * sa + aq.y * sb;
          acc.z = acc.z * sa + aq.z * sb;
          acc.w = acc.w * sa + aq.w * sb;
          W = W * sa + mw.y * sb;
          M = Mn;
        }
        const int c = 4 * dgi;
        const float inv = W > 0.f ? 1.f / W : 0.f;
        tile[h][c] = acc.x * inv;
        tile[h][c + 1] = acc.y * inv;
        tile[h][c + 2] = acc.z * inv;
        tile[h][c + 3] = acc.w * inv;
        if (dq == 0 && dgi == 0) a.lse[row0 + h] = W > 0.f ? M + __logf(W) : -INFINITY;
      }
    }
    __syncthreads();
    if (kOutF32) {
      for (int idx = t; idx < H * (C / 4); idx += kMergeThreads) {
        const int h = idx / (C / 4), q = idx % (C / 4);
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + (row0 + h) * kDCkv + dq * C + 4 * q) =
            make_float4(tile[h][4 * q], tile[h][4 * q + 1], tile[h][4 * q + 2], tile[h][4 * q + 3]);
      }
    } else {
      for (int idx = t; idx < H * (C / 8); idx += kMergeThreads) {
        const int h = idx / (C / 8), q = idx % (C / 8);
        uint32_t wv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(tile[h][8 * q + 2 * k], tile[h][8 * q + 2 * k + 1]);
          wv[k] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + (row0 + h) * kDCkv + dq * C + 8 * q) =
            make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
    __syncthreads();   // the tile and the group states are reused by the next item
  }
}

// Many heads (H >= 64), the common split of a request into a few slots: one
// thread per (merged request, head, 4 dims), looped over by the grid in
// strides, each folding its slots four at a time (one memory round trip per
// four slots) with no shared memory and no block-wide barrier, so several
// blocks per SM keep many loads in flight.  Index i = ((e * 64 + d / 8) * H
// + h) * 2 + half: consecutive threads read consecutive 16 bytes of a
// partial; the two threads of (h, d / 8) join their halves through a shuffle
// and the even one writes 8 output dims (16 bytes in bf16).
constexpr int kFlatThreads = 256, kFlatBlocksPerSm = 4, kFlatAhead = 4;
template <bool kOutF32>
__global__ void __launch_bounds__(kFlatThreads, kFlatBlocksPerSm) merge_flat_kernel(const MergeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel on the stream may be scheduled now; it waits for this
  // one to complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int H = a.num_heads;
  const long long total = static_cast<long long>(a.params->n_merge) * (kDCkv / 8) * H * 2;
  const long long stride = static_cast<long long>(gridDim.x) * kFlatThreads;
  // every thread of a warp runs the same number of iterations (total is
  // even and the stride a multiple of 32), so the shuffle below is uniform
  for (long long i = static_cast<long long>(blockIdx.x) * kFlatThreads + threadIdx.x; i - (threadIdx.x & 31) < total;
       i += stride) {
    const bool live = i < total;
    const int half = static_cast<int>(i & 1);
    long long r = i >> 1;
    const int h = static_cast<int>(r % H);
    r /= H;
    const int d8 = static_cast<int>(r % (kDCkv / 8));
    const int e = static_cast<int>(r / (kDCkv / 8));
    const int d = 8 * d8 + 4 * half;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY, W = 0.f;
    MergeEntry me{0, 0, 0};
    if (live) {
      me = a.merge[e];
      for (int i0 = 0; i0 < me.n_slots; i0 += kFlatAhead) {
        float4 o[kFlatAhead];
        float l[kFlatAhead];
#pragma unroll
        for (int j = 0; j < kFlatAhead; ++j)
          if (i0 + j < me.n_slots) {
            const int slot = me.first_slot + i0 + j;
            o[j] = *reinterpret_cast<const float4*>(a.o_part + part_offset(slot, h, d, H));
            l[j] = a.lse_part[lse_part_offset(slot, 0, h, H)];
          }
#pragma unroll
        for (int j = 0; j < kFlatAhead; ++j)
          if (i0 + j < me.n_slots) fold_state(M, W, acc, l[j], o[j]);
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const float4 v = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    // the odd thread's four dims, for the even one
    const float4 u = make_float4(__shfl_down_sync(0xffffffffu, v.x, 1), __shfl_down_sync(0xffffffffu, v.y, 1),
                                 __shfl_down_sync(0xffffffffu, v.z, 1), __shfl_down_sync(0xffffffffu, v.w, 1));
    if (!live || half) continue;
    const size_t row = static_cast<size_t>(me.req) * H + h;
    if (kOutF32) {
      float* dst = static_cast<float*>(a.out) + row * kDCkv + d;
      *reinterpret_cast<float4*>(dst) = v;
      *reinterpret_cast<float4*>(dst + 4) = u;
    } else {
      const __nv_bfloat162 b0 = __floats2bfloat162_rn(v.x, v.y), b1 = __floats2bfloat162_rn(v.z, v.w);
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(u.x, u.y), b3 = __floats2bfloat162_rn(u.z, u.w);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + row * kDCkv + d) =
          make_uint4(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1),
                     *reinterpret_cast<const uint32_t*>(&b2), *reinterpret_cast<const uint32_t*>(&b3));
    }
    if (d8 == 0) a.lse[row] = W > 0.f ? M + __logf(W) : -INFINITY;
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
  // a programmatic dependent launch: wait for the kernel before it on the
  // stream (a no-op in a plain launch), then let the next one be scheduled
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + kStatesWarps - 1) / kStatesWarps);
  cfg.blockDim = dim3(32 * kStatesWarps);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return out_f32 ? cudaLaunchKernelEx(&cfg, merge_states_kernel<true>, o_a, lse_a, o_b, lse_b, out, lse_out, rows)
                 : cudaLaunchKernelEx(&cfg, merge_states_kernel<false>, o_a, lse_a, o_b, lse_b, out, lse_out, rows);
}

cudaError_t launch_merge(const MergeArgs& a, bool out_f32, cudaStream_t s) {
  if (a.merge_cap <= 0) return cudaSuccess;
  // Programmatic dependent launch: the merge grid may be scheduled while the
  // decode kernel before it in the stream is still running (on SMs that
  // kernel has left); each block waits for that kernel to complete, and its
  // writes to be visible, before it reads a partial.
  cudaLaunchConfig_t cfg = {};
  // a grid-stride loop over the plan's items: at most two blocks per SM
  // (the kernel's registers allow two)
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 1;
  }
  const bool flat = a.num_heads >= 64;
  if (flat) {
    // the flat kernel: a few blocks per SM, or fewer when the plan's capacity
    // needs fewer threads
    const long long cap_threads = static_cast<long long>(a.merge_cap) * (kDCkv / 8) * a.num_heads * 2;
    const long long blocks = (cap_threads + kFlatThreads - 1) / kFlatThreads;
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < kFlatBlocksPerSm * sms ? blocks : kFlatBlocksPerSm * sms));
    cfg.blockDim = dim3(kFlatThreads);
  } else {
    const int cap_items = a.merge_cap * (kDCkv / merge_chunk(a.num_heads));
    cfg.gridDim = dim3(cap_items < 2 * sms ? cap_items : 2 * sms);
    cfg.blockDim = dim3(kMergeThreads);
  }
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (flat)
    return out_f32 ? cudaLaunchKernelEx(&cfg, merge_flat_kernel<true>, a)
                   : cudaLaunchKernelEx(&cfg, merge_flat_kernel<false>, a);
  return out_f32 ? cudaLaunchKernelEx(&cfg, merge_kernel<true>, a) : cudaLaunchKernelEx(&cfg, merge_kernel<false>, a);
}

}  // namespace mla
