// Paged MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Operation (absorbed multi-head latent attention, one query token, one
// latent KV head of width 512 + 64, no causal mask -- "[WIP] support
// flashinfer_mla", vLLM-metax PR #113, review of the decode_wrapper.plan
// parameters):  for request b, head h over the request's kv_len tokens
//   S   = sm_scale * (q_nope[b,h] . ckv_t + q_pe[b,h] . kpe_t)
//   out = softmax(S) . ckv,   lse = ln sum exp(S).
// Because all heads share the single latent KV head, both products are
// dense contractions with M = heads: S = Q[H x 576] . KV[T x 576]^T and
// O = P[H x T] . ckv[T x 512].
//
// Work decomposition.  A work unit (a token range of one request, from the
// host planner) is processed by a PAIR of CTAs; CTA half h in {0, 1} owns the
// output dims [256h, 256h + 256).  128 heads x 512 fp32 accumulators would
// fill all 512 TMEM columns of an SM, so each CTA keeps O[:, its 256 dims]
// in TMEM and both compute the full score tile S (the 576-wide contraction).
// The grid is persistent: one CTA pair per worker, each walking its units.
//
// Per CTA (192 threads):
//   warp 0      producer: TMA loads of Q (dims 0..255) and of the 32-token
//               KV tiles, gathered page by page through kv_indices into a
//               4-stage shared-memory ring (128-byte swizzle);
//   warp 1      allocates TMEM; one lane issues every tcgen05.mma:
//               QK(t) into one of two S buffers, then PV(t-1);
//   warps 2..5  softmax / epilogue, one thread per head row (TMEM lane):
//               online softmax in the exp2 domain with lazy rescaling
//               (the reference max moves only when a tile's max exceeds it
//               by more than 2^8), P to shared memory in bf16, O rescale in
//               TMEM when needed, zeroing of V rows past the request's end,
//               Q dims 256..575 into TMEM for the next unit, and the epilogue
//               O / l, lse.
// TMEM columns: O [0, 256) | S0 [256, 288) | S1 [288, 320) | Q dims 256..575
// as bf16 pairs [320, 480).
//
// Every wait is bounded (2 s); on expiry the kernel records
// MLA_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs, frees TMEM and
// returns.  Page ids outside [0, num_pages) are recorded as
// MLA_ERR_DEVICE_BOUNDS and never dereferenced.
#include <cuda_bf16.h>

#include "device_utils.cuh"
#include "kernels.h"
#include "tc_utils.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kT = kTileTc;               // 32 tokens per tile
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kPanelQ = 128 * 128;        // one 64-dim panel of Q: 128 rows x 128 B
constexpr int kPanelKV = kT * 128;        // one 64-dim panel of a KV tile: 32 rows x 128 B
constexpr int kStageBytes = 9 * kPanelKV; // 8 ckv panels + 1 kpe panel = 36 KB

// shared memory map (offsets from the 1024-byte aligned base)
constexpr int kOffQ = 0;                               // 4 panels: q_nope dims 0..255
constexpr int kOffKV = kOffQ + 4 * kPanelQ;            // 65536
constexpr int kOffP = kOffKV + kStages * kStageBytes;  // 212992: P [128 x 32] bf16, 64-byte swizzle
constexpr int kOffBar = kOffP + 128 * kT * 2;          // 221184
constexpr int kSmemBytes = kOffBar + 256 + 1024;       // + alignment slack

// barrier slots (8 bytes each)
enum Bar {
  kQFull = 0, kQTmemFull, kQEmpty, kKvFull0, kKvEmpty0 = kKvFull0 + kStages,
  kSFull0 = kKvEmpty0 + kStages, kSFree0 = kSFull0 + 2, kPFull = kSFree0 + 2, kPvDone,
  kOFree, kFinal, kNumBars
};
static_assert(kNumBars * 8 + 16 <= 256, "barrier area");

// TMEM columns
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320;
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P values stay below 2^8

__device__ __forceinline__ float tree_max32(const float (&v)[32]) {
  float t[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = fmaxf(v[j], v[j + 16]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
  return t[0];
}
__device__ __forceinline__ float tree_min32(const float (&v)[32]) {
  float t[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = fminf(v[j], v[j + 16]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = fminf(t[j], t[j + w]);
  return t[0];
}
__device__ __forceinline__ float tree_sum32(const float (&v)[32]) {
  float t[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = v[j] + v[j + 16];
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = t[j] + t[j + w];
  return t[0];
}

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) {
  return base + kOffBar + 8 * i;
}

// Q dims 256..575 of head row r into TMEM columns [kColQ, kColQ + 160) of lane r:
// 5 panels of 64 bf16, each 32 columns of packed pairs.
__device__ __forceinline__ void load_q_tmem(const DecodeArgs& a, int req, int r, uint32_t taddr) {
  const int H = a.num_heads;
  const bool ok = r < H;
  const size_t row = static_cast<size_t>(req) * H + (ok ? r : 0);
  const uint4* qn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_nope) +
                                                   row * kDCkv + 256);
  const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_pe) +
                                                   row * kDKpe);
#pragma unroll 1
  for (int p = 0; p < 5; ++p) {
    const uint4* src = p < 4 ? qn + p * 8 : qp;
    uint32_t v[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x = ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
    }
    tmem_st32(taddr + kColQ + 32 * p, v);
  }
  tmem_st_wait();
}

template <bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const DecodeArgs a, const __grid_constant__ TcMaps maps) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(sm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffBar + kNumBars * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + kNumBars * 8 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int worker = blockIdx.x >> 1, half = blockIdx.x & 1;
  const PlanDev prm = *a.params;
  const int H = a.num_heads;
  const int u0 = worker < prm.n_workers ? a.worker_ptr[worker] : 0;
  const int u1 = worker < prm.n_workers ? a.worker_ptr[worker + 1] : 0;

  // ---- setup ----
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kQTmemFull || i == kPFull || i == kOFree || i == kSFree0 || i == kSFree0 + 1) cnt = 4;
      mbar_init(bar_addr(base, i), cnt);
    }
    fence_barrier_init();
  }
  if (warp >= 2 && H < 128) {
    // Q rows past num_heads are never written by TMA: make them zero once.
    const int t = threadIdx.x - 64;
    for (int i = t; i < 4 * (128 - H) * 8; i += 128) {
      const int panel = i / ((128 - H) * 8), rem = i % ((128 - H) * 8);
      const int row = H + rem / 8, chunk = rem % 8;
      *reinterpret_cast<uint4*>(sm + kOffQ + panel * kPanelQ + row * 128 + chunk * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.q_nope);
    tma_prefetch_desc(&maps.ckv);
    tma_prefetch_desc(&maps.kpe);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0) {
    // ================= producer (whole warp, converged) =================
    const int P = prm.page_size;
    const int box = P < kT ? P : kT;
    int g = 0, uidx = 0;
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      if (uidx > 0 && !(ok = mbar_wait_warp(bar_addr(base, kQEmpty), (uidx - 1) & 1, abort_flag)))
        break;
      if (lane == 0) mbar_arrive_expect_tx(bar_addr(base, kQFull), 4 * H * 128);
      __syncwarp();
      if (lane < 4)
        tma_load_2d(base + kOffQ + lane * kPanelQ, &maps.q_nope, 64 * lane, u.req * H,
                    bar_addr(base, kQFull));
      for (int tok0 = u.tok_begin; tok0 < u.tok_end; tok0 += kT, ++g) {
        const int st = g % kStages;
        if (!(ok = mbar_wait_warp(bar_addr(base, kKvEmpty0 + st), ((g / kStages) & 1) ^ 1,
                                  abort_flag)))
          break;
        // lane l issues panel l % 9 of box l / 9 (a box = one page's rows of the tile)
        const int nbox = min(kT / box, (u.tok_end - tok0 + box - 1) / box);
        const int b = lane / 9, j = lane % 9;
        int row = 0;
        if (b < nbox) {
          const int t = tok0 + b * box;
          int page = a.kv_indices[u.page_base + t / P];
          if (page < 0 || page >= a.num_pages) {
            if (j == 0) report_error(a.err, kErrBounds);
            page = 0;
          }
          row = page * P + (t % P);
        }
        const uint32_t full = bar_addr(base, kKvFull0 + st);
        if (lane == 0) mbar_arrive_expect_tx(full, nbox * 9 * box * 128);
        __syncwarp();
        if (b < nbox) {
          const uint32_t dst = base + kOffKV + st * kStageBytes + j * kPanelKV + b * box * 128;
          if (j < 8)
            tma_load_2d(dst, &maps.ckv, 64 * j, row, full);
          else
            tma_load_2d(dst, &maps.kpe, 0, row, full);
        }
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    // Drain: every copy this warp issued has landed before the CTA exits.
    if (lane == 0)
      for (int k = 1; k <= kStages && k <= g; ++k) {
        const int gg = g - k;
        mbar_wait_drain(bar_addr(base, kKvFull0 + gg % kStages), (gg / kStages) & 1);
      }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (whole warp, converged; lane 0 issues) =================
    constexpr uint32_t id_qk = idesc_bf16_f32(128, kT, false, false);
    constexpr uint32_t id_pv = idesc_bf16_f32(128, 256, false, true);
    const uint32_t issue = lane == 0;
    const uint64_t q_desc0 = smem_desc(base + kOffQ, 16, 1024, kSw128);
    const uint64_t kv_desc0 = smem_desc(base + kOffKV, 16, 1024, kSw128);
    const uint64_t p_desc0 = smem_desc(base + kOffP, 16, 512, kSw64);
    const uint64_t v_desc0 = smem_desc(base + kOffKV + 4 * half * kPanelKV, kPanelKV, 1024, kSw128);
    int g = 0, uidx = 0;
    bool ok = true;
    auto pv = [&](int gg, bool first, int ux) -> bool {
      if (!mbar_wait_warp(bar_addr(base, kPFull), gg & 1, abort_flag)) return false;
      if (first && ux > 0 && !mbar_wait_warp(bar_addr(base, kOFree), (ux - 1) & 1, abort_flag))
        return false;
      tc_fence_after();
      const uint64_t vdesc = v_desc0 + static_cast<uint64_t>(((gg % kStages) * kStageBytes) >> 4);
#pragma unroll
      for (int k = 0; k < kT / 16; ++k)
        mma_ss(tmem + kColO, p_desc0 + static_cast<uint64_t>((k * 32) >> 4),
               vdesc + static_cast<uint64_t>((k * 2048) >> 4), id_pv, (first && k == 0) ? 0u : 1u,
               issue);
      mma_commit(bar_addr(base, kKvEmpty0 + gg % kStages), issue);
      mma_commit(bar_addr(base, kPvDone), issue);
      return true;
    };
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = (u.tok_end - u.tok_begin + kT - 1) / kT;
      if (!(ok = mbar_wait_warp(bar_addr(base, kQFull), uidx & 1, abort_flag) &&
                 mbar_wait_warp(bar_addr(base, kQTmemFull), uidx & 1, abort_flag)))
        break;
      tc_fence_after();
      for (int i = 0; i < n; ++i, ++g) {
        const int st = g % kStages, sb = g & 1;
        if (!(ok = mbar_wait_warp(bar_addr(base, kKvFull0 + st), (g / kStages) & 1, abort_flag) &&
                   mbar_wait_warp(bar_addr(base, kSFree0 + sb), ((g >> 1) & 1) ^ 1, abort_flag)))
          break;
        tc_fence_after();
        // descriptors differ only in their start-address field: add (offset >> 4)
        const uint64_t bdesc = kv_desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
        const uint32_t d = tmem + kColS + 32 * sb;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, q_desc0 + static_cast<uint64_t>((j * kPanelQ + kk * 32) >> 4),
                   bdesc + static_cast<uint64_t>((j * kPanelKV + kk * 32) >> 4), id_qk,
                   (j | kk) != 0, issue);
#pragma unroll
        for (int j = 4; j < 9; ++j)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(d, tmem + kColQ + (j - 4) * 32 + kk * 8,
                   bdesc + static_cast<uint64_t>((j * kPanelKV + kk * 32) >> 4), id_qk, 1u, issue);
        mma_commit(bar_addr(base, kSFull0 + sb), issue);
        if (i == n - 1) mma_commit(bar_addr(base, kQEmpty), issue);
        if (i > 0 && !(ok = pv(g - 1, i == 1, uidx))) break;
      }
      if (ok && n > 0) ok = pv(g - 1, n == 1, uidx);
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    // Drain: all MMAs issued by this warp complete before TMEM is freed.
    mma_commit(bar_addr(base, kFinal), issue);
    if (lane == 0) mbar_wait_drain(bar_addr(base, kFinal), 0);
    __syncwarp();
  } else {
    // ================= softmax / epilogue (warps 2..5) =================
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                 // head row == TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int t128 = threadIdx.x - 64;              // 0..127 for cooperative work
    const float c = prm.sm_scale * kLog2e;
    unsigned char* p_row = sm + kOffP + (r >> 3) * 512 + (r & 7) * 64;
    const uint32_t pswz = (r & 7) >> 1;
    int g = 0, uidx = 0;
    bool ok = true;
    if (u0 < u1) {
      load_q_tmem(a, a.units[u0].req, r, lane_addr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(base, kQTmemFull));
    }
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = (u.tok_end - u.tok_begin + kT - 1) / kT;
      float m = -INFINITY, lr = 0.f, lx = 0.f;
      for (int i = 0; i < n; ++i, ++g) {
        const int sb = g & 1;
        if (!(ok = mbar_wait_warp(bar_addr(base, kSFull0 + sb), (g >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(lane_addr + kColS + 32 * sb, sr);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(base, kSFree0 + sb));

        const int valid = min(kT, u.tok_end - (u.tok_begin + i * kT));
        // exponent of token j: s_j * c - m, one FFMA.  For c >= 0 the tile max
        // of s_j * c is c * max s_j (c < 0: c * min s_j).
        float sv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(sr[j]);
        float mx;
        if (valid == kT) {
          mx = c >= 0.f ? c * tree_max32(sv) : c * tree_min32(sv);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j >= valid) sv[j] = c >= 0.f ? -INFINITY : INFINITY;
          mx = c >= 0.f ? c * tree_max32(sv) : c * tree_min32(sv);
        }
        const bool move = mx > m + kRescaleThreshold;
        const float m_new = move ? mx : m;
        const float alpha = move ? exp2f(m - m_new) : 1.f;
        float ex[32], er[32];
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; ++j) ex[j] = exp2f(fmaf(sv[j], c, -m_new));
        if (valid < kT) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j >= valid) ex[j] = 0.f;        // masked tokens (also when c == 0)
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(ex[2 * j], ex[2 * j + 1]);
          er[2 * j] = __low2float(b2);
          er[2 * j + 1] = __high2float(b2);
          pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        const float sx = tree_sum32(ex), sr16 = tree_sum32(er);
        lx = lx * alpha + sx;
        lr = lr * alpha + sr16;
        m = m_new;

        // P buffer and O are free once PV of the previous tile completed.
        if (i > 0 && !(ok = mbar_wait_warp(bar_addr(base, kPvDone), (g - 1) & 1, abort_flag))) break;
        tc_fence_after();
        if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kColO + 32 * cc, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(lane_addr + kColO + 32 * cc, o);
          }
          tmem_st_wait();
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          *reinterpret_cast<uint4*>(p_row + ((ch ^ pswz) << 4)) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        if (valid < kT) {
          // rows past the request's end in this CTA's V panels -> 0
          unsigned char* v = sm + kOffKV + (g % kStages) * kStageBytes + 4 * half * kPanelKV;
          const int total = (kT - valid) * 32;
          for (int q = t128; q < total; q += 128) {
            const int row = valid + q / 32, rem = q % 32;
            *reinterpret_cast<uint4*>(v + (rem >> 3) * kPanelKV + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(base, kPFull));
        if (i == n - 1 && ui + 1 < u1) {
          // Q of the next unit: QK of this unit has completed (its S was read)
          load_q_tmem(a, a.units[ui + 1].req, r, lane_addr);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr(base, kQTmemFull));
        }
      }
      if (!ok) break;
      // ---- epilogue ----
      if (!(ok = mbar_wait_warp(bar_addr(base, kPvDone), (g - 1) & 1, abort_flag))) break;
      tc_fence_after();
      const bool partial = u.out_slot >= 0;
      const size_t orow = partial ? static_cast<size_t>(u.out_slot) * H + r
                                  : static_cast<size_t>(u.req) * H + r;
      const float inv = (r < H) ? a.kv_scale / lr : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t o[32];
        tmem_ld32(lane_addr + kColO + 32 * cc, o);
        tmem_ld_wait();
        if (r < H) {
          const int d0 = 256 * half + 32 * cc;
          if (partial || kOutF32) {
            float* dst = (partial ? a.o_part : static_cast<float*>(a.out)) + orow * kDCkv + d0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              reinterpret_cast<float4*>(dst)[j] =
                  make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                              __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + orow * kDCkv + d0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                    __uint_as_float(o[8 * j + 2 * e]) * inv, __uint_as_float(o[8 * j + 2 * e + 1]) * inv);
                w[e] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              reinterpret_cast<uint4*>(dst)[j] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(base, kOFree));
      if (half == 0 && r < H) {
        const float l2 = (m + log2f(lx)) * kLn2;
        (partial ? a.lse_part : a.lse)[orow] = l2;
      }
    }
    if (!ok) report_error(a.err, kErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kOutF32>
cudaError_t launch_impl(const DecodeArgs& a, const TcMaps& maps, cudaStream_t s) {
  auto* k = decode_tc_kernel<kOutF32>;
  static bool attr_set = false;   // set once, before any stream capture
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k<<<2 * a.n_workers, kThreads, kSmemBytes, s>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, const TcMaps& maps, bool out_f32, cudaStream_t s) {
  return out_f32 ? launch_impl<true>(a, maps, s) : launch_impl<false>(a, maps, s);
}

}  // namespace mla
