// Paged MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Operation (absorbed multi-head latent attention, one query token, one
// latent KV head of width 512 + 64, no causal mask -- "[WIP] support
// flashinfer_mla", vLLM-metax PR #113, review of the decode_wrapper.plan
// parameters):  for request b, head h over the request's kv_len tokens
//   S   = sm_scale * (q_nope[b,h] . ckv_t + q_pe[b,h] . kpe_t)
//   out = softmax(S) . ckv,   lse = ln sum exp(S).
// All heads share the single latent KV head, so both products are dense
// contractions with M = heads: S = Q[H x 576] . K[T x 576]^T and
// O = P[H x T] . ckv[T x 512].
//
// Work decomposition.  A work unit (a token range of one request, from the
// host planner) is processed by a PAIR of CTAs; CTA half h in {0, 1} owns the
// output dims [256h, 256h + 256).  128 heads x 512 fp32 accumulators would
// fill all 512 TMEM columns of an SM, so each CTA keeps O[:, its 256 dims]
// in TMEM and both compute the full score tile S.  The grid is persistent:
// one CTA pair per worker, each walking its units.
//
// Tiles are 128 tokens, so every score MMA is M=128 x N=128 x K=16 (a
// tcgen05.mma instruction costs about as much for N=32 as for N=128, so
// wide tiles keep the tensor pipe busy).  Per CTA (384 threads):
//   warp 0      K producer: TMA loads of Q dims 0..319 (per unit) and of
//               the 9 K panels (64 dims x 128 tokens, 16 KB) of every tile,
//               gathered page by page through kv_indices into a 5-slot ring,
//               after a contiguous L2 prefetch of the next tile's pages;
//   warp 1      allocates TMEM; lane 0 issues the QK(t) MMAs, panel by
//               panel, into S;
//   warp 11     lane 0 issues the PV(t) MMAs, chunk by chunk, into O (two
//               issuing warps keep the tensor pipe fed: a single warp can
//               issue a tcgen05.mma only every ~80-100 cycles);
//   warp 2      V producer: TMA loads of this CTA's 256 dims of ckv for PV,
//               16 tokens (8 KB) at a time into a 4-slot ring (a second
//               read of rows the K producer fetched shortly before, served
//               from L2); rows past the end of a request are zeroed;
//   warps 3..10 softmax / epilogue, two warps per 32 head rows (TMEM lane
//               quadrant): each owns 64 of the 128 tokens of a tile (one P
//               panel) and 128 of the 256 output dims.  S is drained from
//               TMEM to registers at once (so QK(t+1) can start; each warp
//               reads all 128 scores of its rows for the row max), online
//               softmax in the exp2 domain with lazy
//               rescaling (the reference max moves only when a tile's max
//               exceeds it by more than 2^8), P to shared memory in bf16,
//               O rescale in TMEM when needed, Q dims 320..575 into TMEM for
//               the next unit, and the epilogue O / l, lse.
// TMEM columns: O [0, 256) | S [256, 384) | Q dims 320..575 as bf16 pairs
// [384, 512).
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

constexpr int kT = kTileTc;                 // 128 tokens per tile
constexpr int kThreads = 384;
constexpr int kPvWarp = 11;
constexpr int kSoftmaxWarps = 8;
constexpr int kPanel = 128 * 128;           // 128 rows x 128 B (one 64-dim panel)
constexpr int kKSlots = 5;
constexpr int kVSlots = 4;
constexpr int kVChunkTok = 16;
constexpr int kVPanel = kVChunkTok * 128;   // 2 KB: 16 rows x 64 dims
constexpr int kVSlot = 4 * kVPanel;         // 8 KB: 16 rows x 256 dims
constexpr int kQSmemPanels = 5;             // Q dims 0..319 in shared memory

// shared memory map (offsets from the 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kQSmemPanels * kPanel;   // P [128 x 128] bf16: 2 panels
constexpr int kOffK = kOffP + 2 * kPanel;
constexpr int kOffV = kOffK + kKSlots * kPanel;
constexpr int kOffBar = kOffV + kVSlots * kVSlot;
constexpr int kBarBytes = 512;
constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

enum Bar {
  kQFull = 0, kQTmemFull, kQEmpty,
  kKFull0, kKEmpty0 = kKFull0 + kKSlots,
  kVFull0 = kKEmpty0 + kKSlots, kVEmpty0 = kVFull0 + kVSlots, kVTail0 = kVEmpty0 + kVSlots,
  kSFull = kVTail0 + kVSlots, kSFree, kPFull, kPvDone, kOFree, kFinal, kFinalPv,
  kXchg0, kNumBars = kXchg0 + 4   // per TMEM lane quadrant: the two softmax warps' row sums
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");

constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P values stay below 2^8

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + kOffBar + 8 * i; }

template <int N>
__device__ __forceinline__ float tree_max(float (&v)[N]) {
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) v[j] = fmaxf(v[j], v[j + w]);
  return v[0];
}
template <int N>
__device__ __forceinline__ float tree_min(float (&v)[N]) {
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) v[j] = fminf(v[j], v[j + w]);
  return v[0];
}
template <int N>
__device__ __forceinline__ float tree_sum(float (&v)[N]) {
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) v[j] = v[j] + v[j + w];
  return v[0];
}

// Q dims 320..575 of head row r into TMEM columns [kColQ, kColQ + 128) of
// lane r: q_nope dims 320..511 (3 panels of 64) then q_pe (64), each 32
// columns of packed bf16 pairs.  The warp of column half hc writes panels
// 2hc and 2hc + 1.
__device__ __forceinline__ void load_q_tmem(const DecodeArgs& a, int req, int r, int hc,
                                            uint32_t taddr) {
  const int H = a.num_heads;
  const bool ok = r < H;
  const size_t row = static_cast<size_t>(req) * H + (ok ? r : 0);
  const uint4* qn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_nope) +
                                                   row * kDCkv + 64 * kQSmemPanels);
  const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_pe) +
                                                   row * kDKpe);
#pragma unroll 1
  for (int p = 2 * hc; p < 2 * hc + 2; ++p) {
    const uint4* src = p < 3 ? qn + p * 8 : qp;
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
  const int P = prm.page_size;
  const int u0 = worker < prm.n_workers ? a.worker_ptr[worker] : 0;
  const int u1 = worker < prm.n_workers ? a.worker_ptr[worker + 1] : 0;

  // ---- setup ----
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar_addr(base, i),
                (i == kQTmemFull || i == kPFull || i == kOFree || i == kSFree) ? kSoftmaxWarps
                : i >= kXchg0                                                   ? 2
                                                                                : 1);
    fence_barrier_init();
  }
  if (warp >= 3 && warp < kPvWarp && H < 128) {
    // Q rows past num_heads are never written by TMA: make them zero once.
    const int t = threadIdx.x - 96;
    const int per_panel = (128 - H) * 8;
    for (int i = t; i < kQSmemPanels * per_panel; i += 32 * kSoftmaxWarps) {
      const int panel = i / per_panel, rem = i % per_panel;
      *reinterpret_cast<uint4*>(sm + kOffQ + panel * kPanel + (H + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.q_nope);
    tma_prefetch_desc(&maps.ckv_k);
    tma_prefetch_desc(&maps.kpe_k);
    tma_prefetch_desc(&maps.ckv_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0) {
    // ================= K producer =================
    int kc = 0, uidx = 0;
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      if (uidx > 0 && !(ok = mbar_wait_warp(bar_addr(base, kQEmpty), (uidx - 1) & 1, abort_flag)))
        break;
      if (lane == 0) mbar_arrive_expect_tx(bar_addr(base, kQFull), kQSmemPanels * H * 128);
      __syncwarp();
      if (lane < kQSmemPanels)
        tma_load_2d(base + kOffQ + lane * kPanel, &maps.q_nope, 64 * lane, u.req * H,
                    bar_addr(base, kQFull));
      for (int tok0 = u.tok_begin; tok0 < u.tok_end && ok; tok0 += kT) {
        // lane b < nbox owns page b of this tile (a box of P rows)
        const int nbox = (min(tok0 + kT, u.tok_end) - tok0 + P - 1) / P;
        int row = 0;
        if (lane < nbox) {
          int page = a.kv_indices[u.page_base + tok0 / P + lane];
          if (page < 0 || page >= a.num_pages) {
            report_error(a.err, kErrBounds);
            page = 0;
          }
          row = page * P;
        }
        {
          // The panels of a page are 128-byte slices of every 1 KB cache row;
          // fetched panel by panel, DRAM would open each row eight times.
          // Prefetch the next tile's pages whole (contiguous) into L2 instead,
          // so the panel copies below hit L2.
          int nu = ui, nt = tok0 + kT;
          if (nt >= u.tok_end) {
            nu = ui + 1;
            nt = nu < u1 ? a.units[nu].tok_begin : 0;
          }
          if (nu < u1) {
            const WorkUnit v = a.units[nu];
            const int nb = (min(nt + kT, v.tok_end) - nt + P - 1) / P;
            if (lane < nb) {
              const int page = a.kv_indices[v.page_base + nt / P + lane];
              if (page >= 0 && page < a.num_pages) {
                const size_t slot_row = static_cast<size_t>(page) * P;
                bulk_prefetch_l2(static_cast<const char*>(a.ckv) + slot_row * kDCkv * 2, P * kDCkv * 2);
                bulk_prefetch_l2(static_cast<const char*>(a.kpe) + slot_row * kDKpe * 2, P * kDKpe * 2);
              }
            }
          }
        }
        for (int j = 0; j < 9; ++j, ++kc) {
          const int slot = kc % kKSlots;
          if (!(ok = mbar_wait_warp(bar_addr(base, kKEmpty0 + slot), ((kc / kKSlots) & 1) ^ 1,
                                    abort_flag)))
            break;
          const uint32_t full = bar_addr(base, kKFull0 + slot);
          if (lane == 0) mbar_arrive_expect_tx(full, nbox * P * 128);
          __syncwarp();
          if (lane < nbox) {
            const uint32_t dst = base + kOffK + slot * kPanel + lane * P * 128;
            if (j < 8)
              tma_load_2d(dst, &maps.ckv_k, 64 * j, row, full);
            else
              tma_load_2d(dst, &maps.kpe_k, 0, row, full);
          }
        }
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    if (lane == 0)   // drain: the copies this warp issued land before the CTA exits
      for (int k = 1; k <= kKSlots && k <= kc; ++k)
        mbar_wait_drain(bar_addr(base, kKFull0 + (kc - k) % kKSlots), ((kc - k) / kKSlots) & 1);
    __syncwarp();
  } else if (warp == 2) {
    // ================= V producer (this CTA's 256 dims of ckv) =================
    int vc = 0;
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui) {
      const WorkUnit u = a.units[ui];
      for (int t = u.tok_begin; t < u.tok_end && ok; t += kVChunkTok, ++vc) {
        const int slot = vc % kVSlots;
        if (!(ok = mbar_wait_warp(bar_addr(base, kVEmpty0 + slot), ((vc / kVSlots) & 1) ^ 1,
                                  abort_flag)))
          break;
        int page = a.kv_indices[u.page_base + t / P];
        if (page < 0 || page >= a.num_pages) {
          if (lane == 0) report_error(a.err, kErrBounds);
          page = 0;
        }
        const int row = page * P + (t % P);
        const int rows = min(kVChunkTok, u.tok_end - t);
        const uint32_t full = bar_addr(base, kVFull0 + slot);
        const uint32_t dst = base + kOffV + slot * kVSlot;
        if (lane == 0) mbar_arrive_expect_tx(full, kVSlot);
        __syncwarp();
        if (lane < 4) tma_load_2d(dst + lane * kVPanel, &maps.ckv_v, 256 * half + 64 * lane, row, full);
        if (rows < kVChunkTok) {
          // Last chunk of a request: rows past kv_len may hold anything (even
          // NaN), and P = 0 there does not cancel NaN.  Wait for the copy,
          // zero those rows, then release the chunk through kVTail.
          if (!(ok = mbar_wait_warp(full, (vc / kVSlots) & 1, abort_flag))) break;
          for (int q = lane; q < (kVChunkTok - rows) * 32; q += 32) {
            const int rr = rows + q / 32, rem = q % 32;
            *reinterpret_cast<uint4*>(sm + kOffV + slot * kVSlot + (rem >> 3) * kVPanel + rr * 128 +
                                      (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr(base, kVTail0 + slot));
        }
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    if (lane == 0)
      for (int k = 1; k <= kVSlots && k <= vc; ++k)
        mbar_wait_drain(bar_addr(base, kVFull0 + (vc - k) % kVSlots), ((vc - k) / kVSlots) & 1);
    __syncwarp();
  } else if (warp == 1) {
    // ================= QK issuer (whole warp converged; lane 0 issues) =================
    constexpr uint32_t id_qk = idesc_bf16_f32(128, kT, false, false);
    const uint32_t issue = lane == 0;
    const uint64_t q_desc0 = smem_desc(base + kOffQ, 16, 1024, kSw128);
    const uint64_t k_desc0 = smem_desc(base + kOffK, 16, 1024, kSw128);
    int kc = 0, g = 0, uidx = 0;
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = (u.tok_end - u.tok_begin + kT - 1) / kT;
      if (!(ok = mbar_wait_warp(bar_addr(base, kQFull), uidx & 1, abort_flag) &&
                 mbar_wait_warp(bar_addr(base, kQTmemFull), uidx & 1, abort_flag)))
        break;
      tc_fence_after();
      for (int i = 0; i < n && ok; ++i, ++g) {
        // S is single-buffered: the softmax drains it to registers right away.
        if (!(ok = mbar_wait_warp(bar_addr(base, kSFree), (g & 1) ^ 1, abort_flag))) break;
        for (int j = 0; j < 9; ++j, ++kc) {
          const int slot = kc % kKSlots;
          if (!(ok = mbar_wait_warp(bar_addr(base, kKFull0 + slot), (kc / kKSlots) & 1, abort_flag)))
            break;
          tc_fence_after();
          const uint64_t bdesc = k_desc0 + static_cast<uint64_t>((slot * kPanel) >> 4);
          if (j < kQSmemPanels) {
            const uint64_t adesc = q_desc0 + static_cast<uint64_t>((j * kPanel) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + kColS, adesc + static_cast<uint64_t>((kk * 32) >> 4),
                     bdesc + static_cast<uint64_t>((kk * 32) >> 4), id_qk, (j | kk) != 0, issue);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + kColS, tmem + kColQ + (j - kQSmemPanels) * 32 + kk * 8,
                     bdesc + static_cast<uint64_t>((kk * 32) >> 4), id_qk, 1u, issue);
          }
          mma_commit(bar_addr(base, kKEmpty0 + slot), issue);
        }
        if (!ok) break;
        mma_commit(bar_addr(base, kSFull), issue);
        if (i == n - 1) mma_commit(bar_addr(base, kQEmpty), issue);
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    // Drain: all MMAs issued by this warp complete before TMEM is freed.
    mma_commit(bar_addr(base, kFinal), issue);
    if (lane == 0) mbar_wait_drain(bar_addr(base, kFinal), 0);
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ================= PV issuer (whole warp converged; lane 0 issues) =================
    constexpr uint32_t id_pv = idesc_bf16_f32(128, 256, false, true);
    const uint32_t issue = lane == 0;
    const uint64_t p_desc0 = smem_desc(base + kOffP, 16, 1024, kSw128);
    const uint64_t v_desc0 = smem_desc(base + kOffV, kVPanel, 1024, kSw128);
    int vc = 0, g = 0, uidx = 0;
    uint32_t tail_par = 0;   // per V slot: parity of its next tail-chunk release
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = (u.tok_end - u.tok_begin + kT - 1) / kT;
      for (int i = 0; i < n && ok; ++i, ++g) {
        const int valid = min(kT, u.tok_end - (u.tok_begin + i * kT));
        const int nch = (valid + kVChunkTok - 1) / kVChunkTok;
        if (!(ok = mbar_wait_warp(bar_addr(base, kPFull), g & 1, abort_flag))) break;
        // the first PV of a unit overwrites O: the previous epilogue must be done
        if (i == 0 && uidx > 0 &&
            !(ok = mbar_wait_warp(bar_addr(base, kOFree), (uidx - 1) & 1, abort_flag)))
          break;
        for (int c = 0; c < nch; ++c, ++vc) {
          const int slot = vc % kVSlots;
          if (c == nch - 1 && (valid % kVChunkTok) != 0) {
            if (!(ok = mbar_wait_warp(bar_addr(base, kVTail0 + slot), (tail_par >> slot) & 1,
                                      abort_flag)))
              break;
            tail_par ^= 1u << slot;
          } else if (!(ok = mbar_wait_warp(bar_addr(base, kVFull0 + slot), (vc / kVSlots) & 1,
                                           abort_flag))) {
            break;
          }
          tc_fence_after();
          mma_ss(tmem + kColO,
                 p_desc0 + static_cast<uint64_t>(((c >> 2) * kPanel + (c & 3) * 32) >> 4),
                 v_desc0 + static_cast<uint64_t>((slot * kVSlot) >> 4), id_pv,
                 (i == 0 && c == 0) ? 0u : 1u, issue);
          mma_commit(bar_addr(base, kVEmpty0 + slot), issue);
        }
        if (!ok) break;
        mma_commit(bar_addr(base, kPvDone), issue);
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    mma_commit(bar_addr(base, kFinalPv), issue);
    if (lane == 0) mbar_wait_drain(bar_addr(base, kFinalPv), 0);
    __syncwarp();
  } else {
    // ================= softmax / epilogue (warps 3..10) =================
    static_assert(kPvWarp == 3 + kSoftmaxWarps, "warp roles");
    const int quad = warp & 3;
    const int hc = (warp - 3) >> 2;                 // token half / P panel / O column half
    const int r = quad * 32 + lane;                 // head row == TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float c = prm.sm_scale * kLog2e;
    const float pad = c >= 0.f ? -INFINITY : INFINITY;   // neutral for the max of s * c
    unsigned char* p_row = sm + kOffP + hc * kPanel + (r >> 3) * 1024 + (r & 7) * 128;
    const int pswz = r & 7;
    int g = 0, uidx = 0;
    bool ok = true;
    if (u0 < u1) {
      load_q_tmem(a, a.units[u0].req, r, hc, lane_addr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(base, kQTmemFull));
    }
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = (u.tok_end - u.tok_begin + kT - 1) / kT;
      float m = -INFINITY, lr = 0.f, lx = 0.f;       // lr, lx: sums over this warp's tokens
      for (int i = 0; i < n; ++i, ++g) {
        if (!(ok = mbar_wait_warp(bar_addr(base, kSFull), g & 1, abort_flag))) break;
        tc_fence_after();
        const int valid = min(kT, u.tok_end - (u.tok_begin + i * kT));
        float s[64];
        float other;   // max (or min) over the partner warp's 64 tokens
        {
          uint32_t v[32];
          tmem_ld32(lane_addr + kColS + 64 * hc, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(v[j]);
          tmem_ld32(lane_addr + kColS + 64 * hc + 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(v[j]);
          const int ob = 64 * (1 - hc);
          float t[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) t[j] = pad;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            tmem_ld32(lane_addr + kColS + ob + 32 * q, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float y = ob + 32 * q + j < valid ? __uint_as_float(v[j]) : pad;
              t[j & 15] = c >= 0.f ? fmaxf(t[j & 15], y) : fminf(t[j & 15], y);
            }
          }
          other = c >= 0.f ? tree_max(t) : tree_min(t);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(base, kSFree));

        // exponent of token j: s_j * c - m (one FFMA); for c >= 0 the row max
        // of s_j * c is c * max s_j, for c < 0 it is c * min s_j.
        const int vb = 64 * hc;                      // first token of this warp's half
        float mx;
        {
          float t[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float lo = vb + j < valid ? s[j] : pad;
            const float hi = vb + 32 + j < valid ? s[32 + j] : pad;
            t[j] = c >= 0.f ? fmaxf(lo, hi) : fminf(lo, hi);
          }
          const float own = c >= 0.f ? tree_max(t) : tree_min(t);
          mx = c * (c >= 0.f ? fmaxf(own, other) : fminf(own, other));
        }
        const bool move = mx > m + kRescaleThreshold;
        const float m_new = move ? mx : m;
        const float alpha = move ? exp2f(m - m_new) : 1.f;
        uint32_t pk[32];
        float sx = 0.f, srd = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float ex[16], er[16];
          if (valid == kT) {
#pragma unroll
            for (int j = 0; j < 16; ++j) ex[j] = exp2f(fmaf(s[16 * q + j], c, -m_new));
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)   // masked tokens: 0 (also when c == 0)
              ex[j] = vb + 16 * q + j < valid ? exp2f(fmaf(s[16 * q + j], c, -m_new)) : 0.f;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(ex[2 * j], ex[2 * j + 1]);
            er[2 * j] = __low2float(b2);
            er[2 * j + 1] = __high2float(b2);
            pk[8 * q + j] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          sx += tree_sum(ex);
          srd += tree_sum(er);
        }
        lx = lx * alpha + sx;
        lr = lr * alpha + srd;
        m = m_new;

        // P buffer and O are free once PV of the previous tile completed.
        if (g > 0 && !(ok = mbar_wait_warp(bar_addr(base, kPvDone), (g - 1) & 1, abort_flag))) break;
        tc_fence_after();
        if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int cc = 4 * hc; cc < 4 * hc + 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kColO + 32 * cc, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(lane_addr + kColO + 32 * cc, o);
          }
          tmem_st_wait();
        }
        // P row r, this warp's panel: 16-byte chunk ch holds tokens 8ch .. 8ch+7
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(p_row + ((ch ^ pswz) << 4)) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(base, kPFull));
        if (i == n - 1 && ui + 1 < u1) {
          // Q of the next unit: every QK of this unit has completed (S was read)
          load_q_tmem(a, a.units[ui + 1].req, r, hc, lane_addr);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr(base, kQTmemFull));
        }
      }
      if (!ok) break;
      // ---- epilogue ----
      if (!(ok = mbar_wait_warp(bar_addr(base, kPvDone), (g - 1) & 1, abort_flag))) break;
      tc_fence_after();
      // Combine the two warps' row sums through their P rows (P is idle now).
      // Two phases of kXchg0 + quad per unit: "both written", "both read".
      float* xch = reinterpret_cast<float*>(p_row);
      xch[0] = lx;
      xch[1] = lr;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(base, kXchg0 + quad));
      if (!(ok = mbar_wait_warp(bar_addr(base, kXchg0 + quad), 0, abort_flag))) break;
      const float* pxch = reinterpret_cast<const float*>(p_row + (hc ? -kPanel : kPanel));
      const float lx_all = lx + pxch[0];
      const float lr_all = lr + pxch[1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(base, kXchg0 + quad));
      if (!(ok = mbar_wait_warp(bar_addr(base, kXchg0 + quad), 1, abort_flag))) break;
      const bool partial = u.out_slot >= 0;
      const size_t orow = partial ? static_cast<size_t>(u.out_slot) * H + r
                                  : static_cast<size_t>(u.req) * H + r;
      const float inv = (r < H) ? a.kv_scale / lr_all : 0.f;
#pragma unroll 1
      for (int cc = 4 * hc; cc < 4 * hc + 4; ++cc) {
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
      if (half == 0 && hc == 0 && r < H)
        (partial ? a.lse_part : a.lse)[orow] = (m + log2f(lx_all)) * kLn2;
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
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
