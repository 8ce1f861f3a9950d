// Paged MLA decode on the legacy warp-level tensor path (mma.sync m16n8k16,
// bf16 in, fp32 accumulate).  It is the simple, easily checked kernel kept
// for comparison with the tcgen05 kernel; it is selected only explicitly.
//
// One CTA (4 warps) handles one work unit (a contiguous tile range of one
// request) for 16 heads.  Per 64-token tile:
//   * cp.async gathers the tile's rows through the page table into shared
//     memory (rows past kv_len are zero-filled, so NaN or stale data after the
//     end of a request never reaches the PV product), double-buffered;
//   * warp w computes scores S[16 heads, tokens 16w..16w+15] over K = 576
//     (q_nope.ckv + q_pe.kpe as one contraction);
//   * an online softmax in the exp2 domain (running max m, running sum l)
//     gives P in bf16;
//   * warp w accumulates O[16 heads, dims 128w..128w+127] += P . ckv-tile.
// The epilogue writes out = O / l and lse = ln 2 * (m + log2 l), or the split
// partial (O / l, lse) for the merge kernel.
//
// Operation: absorbed MLA decode with one latent KV head of width 512 + 64
// ("[WIP] support flashinfer_mla", vLLM-metax PR #113, review of the
// decode_wrapper.plan parameters), no causal mask (causal=False there).
#include "device_utils.cuh"
#include "kernels.h"

namespace mla {
namespace {

constexpr int kHeadsPerCta = 16;
constexpr int kThreads = 128;
constexpr int kRowStride = kD + 8;          // 584 bf16 = 1168 B: conflict-free ldmatrix
constexpr int kPStride = kTileMma + 8;         // 72 bf16 = 144 B
constexpr int kRawRow = kD;                 // fp8 staging row: 576 bytes

template <bool kFp8>
struct SmemLayout {
  static constexpr int q_bytes = kHeadsPerCta * kRowStride * 2;
  static constexpr int kv_bytes = kTileMma * kRowStride * 2;             // one bf16 tile
  static constexpr int raw_bytes = kTileMma * kRawRow;                   // one fp8 tile
  static constexpr int n_kv = kFp8 ? 1 : 2;                           // bf16 tiles
  static constexpr int n_raw = kFp8 ? 2 : 0;                          // fp8 staging tiles
  static constexpr int p_bytes = kHeadsPerCta * kPStride * 2;
  static constexpr int red_bytes = 3 * 4 * kHeadsPerCta * 4;
  static constexpr int q_off = 0;
  static constexpr int kv_off = q_off + q_bytes;
  static constexpr int raw_off = kv_off + n_kv * kv_bytes;
  static constexpr int p_off = raw_off + n_raw * raw_bytes;
  static constexpr int red_off = p_off + p_bytes;
  static constexpr int total = red_off + red_bytes;
};

// Gather one 64-token tile (ckv 512 + kpe 64 per token) into shared memory.
template <bool kFp8>
__device__ __forceinline__ void load_tile(const DecodeArgs& a, const WorkUnit& u, int tile,
                                          int page_size, uint32_t dst_base) {
  constexpr int elem = kFp8 ? 1 : 2;
  constexpr int ckv_chunks = kDCkv * elem / 16;   // 64 (bf16) / 32 (fp8)
  constexpr int kpe_chunks = kDKpe * elem / 16;   // 8 / 4
  constexpr int row_chunks = ckv_chunks + kpe_chunks;
  constexpr int dst_row = kFp8 ? kRawRow : kRowStride * 2;
  const char* ckv = static_cast<const char*>(a.ckv);
  const char* kpe = static_cast<const char*>(a.kpe);
  for (int c = threadIdx.x; c < kTileMma * row_chunks; c += kThreads) {
    const int row = c / row_chunks;
    const int ch = c - row * row_chunks;
    const int tok = tile * kTileMma + row;
    const char* src = ckv;
    int bytes = 0;
    if (tok < u.tok_end) {
      const int page = a.kv_indices[u.page_base + tok / page_size];
      if (page >= 0 && page < a.num_pages) {
        const size_t slot = static_cast<size_t>(page) * page_size + (tok % page_size);
        src = ch < ckv_chunks ? ckv + slot * kDCkv * elem + ch * 16
                              : kpe + slot * kDKpe * elem + (ch - ckv_chunks) * 16;
        bytes = 16;
      } else {
        report_error(a.err, kErrBounds);
      }
    }
    cp_async_16(dst_base + row * dst_row + ch * 16, src, bytes);
  }
}

template <bool kFp8, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1) decode_mma_kernel(const DecodeArgs a) {
  using L = SmemLayout<kFp8>;
  extern __shared__ __align__(128) unsigned char smem[];
  const PlanDev prm = *a.params;
  const int unit_idx = blockIdx.x;
  if (unit_idx >= prm.n_units) return;
  const WorkUnit u = a.units[unit_idx];
  const int H = a.num_heads;
  const int head0 = blockIdx.y * kHeadsPerCta;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int page_size = prm.page_size;
  const float scale_log2 = prm.sm_scale * a.kv_scale * 1.4426950408889634f;

  const uint32_t q_s = smem_u32(smem + L::q_off);
  const uint32_t kv_s = smem_u32(smem + L::kv_off);
  const uint32_t raw_s = smem_u32(smem + L::raw_off);
  __nv_bfloat16* p_s = reinterpret_cast<__nv_bfloat16*>(smem + L::p_off);
  float* red_max = reinterpret_cast<float*>(smem + L::red_off);
  float* red_sum = red_max + 4 * kHeadsPerCta;
  float* red_xsum = red_sum + 4 * kHeadsPerCta;

  // Q rows of this head group (zero rows past num_heads).
  {
    const char* qn = static_cast<const char*>(a.q_nope);
    const char* qp = static_cast<const char*>(a.q_pe);
    for (int c = tid; c < kHeadsPerCta * 72; c += kThreads) {
      const int r = c / 72, ch = c % 72, h = head0 + r;
      const size_t bh = static_cast<size_t>(u.req) * H + h;
      const char* src = ch < 64 ? qn + bh * kDCkv * 2 + ch * 16 : qp + bh * kDKpe * 2 + (ch - 64) * 16;
      cp_async_16(q_s + r * kRowStride * 2 + ch * 16, h < H ? src : qn, h < H ? 16 : 0);
    }
  }
  const uint32_t stage0 = kFp8 ? raw_s : kv_s;
  const uint32_t stage_bytes = kFp8 ? L::raw_bytes : L::kv_bytes;
  const int t_begin = u.tok_begin / kTileMma;
  const int t_end = (u.tok_end + kTileMma - 1) / kTileMma;
  load_tile<kFp8>(a, u, t_begin, page_size, stage0);
  cp_async_commit();

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  // Per head (lane/4 and lane/4 + 8): running max m, the sum l of the
  // bf16-rounded weights that enter P.V (normalises the output consistently
  // with them) and the sum x of the unrounded fp32 weights (gives the lse).
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, x0 = 0.f, x1 = 0.f;
  const int hr0 = lane >> 2, hr1 = hr0 + 8;
  const int mi = lane >> 3, r8 = lane & 7;

  for (int t = t_begin; t < t_end; ++t) {
    const int it = t - t_begin;
    if (t + 1 < t_end)
      load_tile<kFp8>(a, u, t + 1, page_size, stage0 + ((it + 1) & 1) * stage_bytes);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    uint32_t kv = kv_s + (kFp8 ? 0 : (it & 1) * L::kv_bytes);
    if (kFp8) {
      // Widen the fp8 tile to bf16 in place of the single bf16 tile buffer.
      const unsigned char* raw = smem + L::raw_off + (it & 1) * L::raw_bytes;
      unsigned char* dst = smem + L::kv_off;
      for (int c = tid; c < kTileMma * 36; c += kThreads) {
        const int row = c / 36, ch = c % 36;
        const uint4 in = *reinterpret_cast<const uint4*>(raw + row * kRawRow + ch * 16);
        uint4 lo, hi;
        e4m3x16_to_bf16x16(in, lo, hi);
        uint4* d = reinterpret_cast<uint4*>(dst + row * kRowStride * 2 + ch * 32);
        d[0] = lo;
        d[1] = hi;
      }
      __syncthreads();
    }

    // ---- scores: warp w -> tokens 16w .. 16w+15 ----
    float s[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t af[4], bf[4];
      ldmatrix_x4(af, q_s + (((mi & 1) * 8 + r8) * kRowStride + kk * 16 + (mi >> 1) * 8) * 2);
      ldmatrix_x4(bf, kv + ((warp * 16 + (mi >> 1) * 8 + r8) * kRowStride + kk * 16 + (mi & 1) * 8) * 2);
      mma_bf16_16816(s[0], af, bf[0], bf[1]);
      mma_bf16_16816(s[1], af, bf[2], bf[3]);
    }

    // ---- online softmax (exp2 domain) ----
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = t * kTileMma + warp * 16 + j * 8 + 2 * (lane & 3) + e;
        const bool valid = tok < u.tok_end;
        s[j][e] = valid ? s[j][e] * scale_log2 : -INFINITY;
        s[j][2 + e] = valid ? s[j][2 + e] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[j][e]);
        mx1 = fmaxf(mx1, s[j][2 + e]);
      }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    if ((lane & 3) == 0) {
      red_max[warp * kHeadsPerCta + hr0] = mx0;
      red_max[warp * kHeadsPerCta + hr1] = mx1;
    }
    __syncthreads();
    float tm0 = red_max[hr0], tm1 = red_max[hr1];
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      tm0 = fmaxf(tm0, red_max[w * kHeadsPerCta + hr0]);
      tm1 = fmaxf(tm1, red_max[w * kHeadsPerCta + hr1]);
    }
    const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);   // finite: each tile has a valid token
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float sum0 = 0.f, sum1 = 0.f, xs0 = 0.f, xs1 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float e00 = exp2f(s[j][0] - mn0), e01 = exp2f(s[j][1] - mn0);
      const float e10 = exp2f(s[j][2] - mn1), e11 = exp2f(s[j][3] - mn1);
      xs0 += e00 + e01;
      xs1 += e10 + e11;
      const __nv_bfloat162 p0 = __floats2bfloat162_rn(e00, e01);
      const __nv_bfloat162 p1 = __floats2bfloat162_rn(e10, e11);
      sum0 += __bfloat162float(p0.x) + __bfloat162float(p0.y);
      sum1 += __bfloat162float(p1.x) + __bfloat162float(p1.y);
      const int col = warp * 16 + j * 8 + 2 * (lane & 3);
      *reinterpret_cast<__nv_bfloat162*>(p_s + hr0 * kPStride + col) = p0;
      *reinterpret_cast<__nv_bfloat162*>(p_s + hr1 * kPStride + col) = p1;
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      sum0 += __shfl_xor_sync(0xffffffffu, sum0, off);
      sum1 += __shfl_xor_sync(0xffffffffu, sum1, off);
      xs0 += __shfl_xor_sync(0xffffffffu, xs0, off);
      xs1 += __shfl_xor_sync(0xffffffffu, xs1, off);
    }
    if ((lane & 3) == 0) {
      red_sum[warp * kHeadsPerCta + hr0] = sum0;
      red_sum[warp * kHeadsPerCta + hr1] = sum1;
      red_xsum[warp * kHeadsPerCta + hr0] = xs0;
      red_xsum[warp * kHeadsPerCta + hr1] = xs1;
    }
    __syncthreads();
    float ts0 = 0.f, ts1 = 0.f, tx0 = 0.f, tx1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      ts0 += red_sum[w * kHeadsPerCta + hr0];
      ts1 += red_sum[w * kHeadsPerCta + hr1];
      tx0 += red_xsum[w * kHeadsPerCta + hr0];
      tx1 += red_xsum[w * kHeadsPerCta + hr1];
    }
    l0 = l0 * al0 + ts0;
    l1 = l1 * al1 + ts1;
    x0 = x0 * al0 + tx0;
    x1 = x1 * al1 + tx1;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= al0; o[j][1] *= al0;
      o[j][2] *= al1; o[j][3] *= al1;
    }

    // ---- O[16 heads, dims 128w..128w+127] += P . V ----
    const uint32_t p_addr = smem_u32(p_s);
#pragma unroll
    for (int kk = 0; kk < kTileMma / 16; ++kk) {
      uint32_t af[4];
      ldmatrix_x4(af, p_addr + (((mi & 1) * 8 + r8) * kPStride + kk * 16 + (mi >> 1) * 8) * 2);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t bf[4];
        ldmatrix_x4_trans(bf, kv + ((kk * 16 + (mi & 1) * 8 + r8) * kRowStride + warp * 128 +
                                    np * 16 + (mi >> 1) * 8) * 2);
        mma_bf16_16816(o[2 * np], af, bf[0], bf[1]);
        mma_bf16_16816(o[2 * np + 1], af, bf[2], bf[3]);
      }
    }
    __syncthreads();   // P, the reductions and this stage are rewritten next tile
  }
  cp_async_wait<0>();

  // ---- epilogue ----
  const float inv0 = a.kv_scale / l0, inv1 = a.kv_scale / l1;
  const float lse0 = (m0 + log2f(x0)) * 0.6931471805599453f;
  const float lse1 = (m1 + log2f(x1)) * 0.6931471805599453f;
  const int g0 = head0 + hr0, g1 = head0 + hr1;
  const bool partial = u.out_slot >= 0;
  const size_t row0 = partial ? static_cast<size_t>(u.out_slot) * H + g0 : static_cast<size_t>(u.req) * H + g0;
  const size_t row1 = row0 + 8;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int d = warp * 128 + j * 8 + 2 * (lane & 3);
    if (partial) {
      if (g0 < H)
        *reinterpret_cast<float2*>(a.o_part + part_offset(u.out_slot, g0, d, H)) =
            make_float2(o[j][0] * inv0, o[j][1] * inv0);
      if (g1 < H)
        *reinterpret_cast<float2*>(a.o_part + part_offset(u.out_slot, g1, d, H)) =
            make_float2(o[j][2] * inv1, o[j][3] * inv1);
    } else if (kOutF32) {
      float* out = static_cast<float*>(a.out);
      if (g0 < H) *reinterpret_cast<float2*>(out + row0 * kDCkv + d) = make_float2(o[j][0] * inv0, o[j][1] * inv0);
      if (g1 < H) *reinterpret_cast<float2*>(out + row1 * kDCkv + d) = make_float2(o[j][2] * inv1, o[j][3] * inv1);
    } else {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
      if (g0 < H) *reinterpret_cast<__nv_bfloat162*>(out + row0 * kDCkv + d) = __floats2bfloat162_rn(o[j][0] * inv0, o[j][1] * inv0);
      if (g1 < H) *reinterpret_cast<__nv_bfloat162*>(out + row1 * kDCkv + d) = __floats2bfloat162_rn(o[j][2] * inv1, o[j][3] * inv1);
    }
  }
  if (warp == 0 && (lane & 3) == 0) {
    if (partial) {
      if (g0 < H) a.lse_part[lse_part_offset(u.out_slot, 0, g0, H)] = lse0;
      if (g1 < H) a.lse_part[lse_part_offset(u.out_slot, 0, g1, H)] = lse1;
    } else {
      if (g0 < H) a.lse[row0] = lse0;
      if (g1 < H) a.lse[row1] = lse1;
    }
  }
}

template <bool kFp8, bool kOutF32>
cudaError_t launch_impl(const DecodeArgs& a, cudaStream_t s) {
  using L = SmemLayout<kFp8>;
  auto* k = decode_mma_kernel<kFp8, kOutF32>;
  static bool attr_set = false;   // set once, before any stream capture
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(a.units_cap, (a.num_heads + kHeadsPerCta - 1) / kHeadsPerCta);
  k<<<grid, kThreads, L::total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeArgs& a, bool kv_fp8, bool out_f32, cudaStream_t s) {
  if (kv_fp8) return out_f32 ? launch_impl<true, true>(a, s) : launch_impl<true, false>(a, s);
  return out_f32 ? launch_impl<false, true>(a, s) : launch_impl<false, false>(a, s);
}

}  // namespace mla
