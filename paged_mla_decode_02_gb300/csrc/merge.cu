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

constexpr int kMergeThreads = 128;   // 4 dims per thread

template <bool kOutF32>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  const int e = blockIdx.x;
  if (e >= a.params->n_merge) return;
  const MergeEntry me = a.merge[e];
  const int H = a.num_heads;
  const int h = blockIdx.y;
  const int d = threadIdx.x * 4;
  const size_t orow = static_cast<size_t>(me.req) * H + h;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse_out = -INFINITY;
  if (me.n_slots > 0) {
    float M = -INFINITY;
    for (int i = 0; i < me.n_slots; ++i)
      M = fmaxf(M, a.lse_part[static_cast<size_t>(me.first_slot + i) * H + h]);
    float wsum = 0.f;
    for (int i = 0; i < me.n_slots; ++i) {
      const size_t row = static_cast<size_t>(me.first_slot + i) * H + h;
      const float w = __expf(a.lse_part[row] - M);
      const float4 o = *reinterpret_cast<const float4*>(a.o_part + row * kDCkv + d);
      acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
      wsum += w;
    }
    const float inv = 1.f / wsum;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    lse_out = M + __logf(wsum);
  }
  if (kOutF32) {
    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow * kDCkv + d) = acc;
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow * kDCkv + d) = v;
  }
  if (threadIdx.x == 0) a.lse[orow] = lse_out;
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, bool out_f32, cudaStream_t s) {
  if (a.merge_cap <= 0) return cudaSuccess;
  dim3 grid(a.merge_cap, a.num_heads);
  if (out_f32)
    merge_kernel<true><<<grid, kMergeThreads, 0, s>>>(a);
  else
    merge_kernel<false><<<grid, kMergeThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
