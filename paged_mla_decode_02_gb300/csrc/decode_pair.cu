// Paged MLA decode on a CTA pair: one tcgen05 MMA spans both SMs of a
// cluster (cta_group::2).
//
// Operation (absorbed multi-head latent attention, one query token, one
// latent KV head of width 512 + 64, no causal mask -- "[WIP] support
// flashinfer_mla", vLLM-metax PR #113, review of the decode_wrapper.plan
// parameters): for request b, head h over the request's kv_len tokens
//   S   = sm_scale * (q_nope[b,h] . ckv_t + q_pe[b,h] . kpe_t)
//   out = softmax(S) . ckv,   lse = ln sum exp(S).
//
// Both products are computed transposed, with the tokens or the latent dims
// as the MMA's M = 256 rows split over the two SMs:
//   S^T [256 tokens x 128 heads]  = K [256 tokens x 576] . Q^T         (QK)
//   O^T [512 dims x 128 heads]   += V^T [512 dims x 256 tokens] . P^T (PV, two MMAs of M = 256)
// For QK, CTA r holds the K rows of tokens [128 r, 128 r + 128) of each
// 256-token tile and the query of heads [64 r, 64 r + 64) (the B operand is
// split by N); it receives S^T of its own tokens for all heads.  For PV, CTA
// r holds V and O^T for latent dims [256 r, 256 r + 256) and P^T of heads
// [64 r, 64 r + 64).  So every score is computed once, the query is stored
// once per pair, and the only data the pair exchanges per tile are the
// per-head maxima and the half of P^T whose heads the other CTA holds
// (16 KB each way per 256 tokens).
//
// Per CTA: warp 0 producer (TMA: the query once per unit, then K panels and
// V chunks in exactly the order the MMAs consume them, through one ring of
// 16 KB slots); warp 1 allocates TMEM and, in the even CTA, issues every MMA
// of the pair (QK of tile g + 1, then PV of tile g, so the softmax of a tile
// overlaps the next tile's scores); in the odd CTA it relays "P^T complete"
// to the issuer; warps 2..9 softmax and epilogue (two warps per TMEM lane
// quadrant, each owning 64 heads).
//
// TMEM columns: S^T double-buffered [0, 128) and [128, 256); O^T [256, 512)
// (dims [256 r, 256 r + 128) then [256 r + 128, 256 r + 256), columns =
// heads).
//
// Softmax, per tile and head: the exact maximum over the tile's 256 tokens
// (warp butterfly, four lane quadrants, then the other CTA), a reference
// that moves only when that maximum exceeds it by more than 2^8 (then O^T
// and the running sums are rescaled), p = 2^(s log2e sm_scale - reference)
// rounded to bf16 for the MMA; the row sums are kept twice, exact and of the
// rounded p (the output is divided by the latter, the lse uses the former).
// Both CTAs derive every reference from the same values in the same order,
// so they agree bit for bit.
//
// Every wait is bounded (2 s); on expiry the kernel records
// MLA_ERR_DEVICE_TIMEOUT, lets its copies and MMAs land, frees TMEM and
// returns.  Page ids outside [0, num_pages) are recorded as
// MLA_ERR_DEVICE_BOUNDS and never dereferenced.
#include <cuda_bf16.h>

#include "device_utils.cuh"
#include "kernels.h"
#include "tc_utils.cuh"

namespace mla {
namespace {

using namespace tc;

#ifdef MLA_STALL_TEST
// Test build only: when nonzero, CTA 0's producer leaves out its
// g_pair_stall-th ring copy (1-based), so the issuer's wait for it runs out.
__device__ int g_pair_stall;
#endif

constexpr int kT = kTilePair;              // 256 tokens per tile
constexpr int kHalfT = kT / 2;             // tokens per CTA for the scores
constexpr int kThreads = 384;              // 12 warps
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kVProducerWarp = 10;
constexpr int kPvIssuerWarp = 11;
constexpr int kKSlots = 4, kVSlots = 3;    // rings of 16 KB slots
constexpr int kPBufs = 1;                  // P^T buffers (2: by tile parity)
constexpr int kSlotBytes = 16384;
constexpr int kVChunkTok = kTcVChunkTok;   // 32 tokens per V chunk
constexpr int kChunksPerTile = kT / kVChunkTok;
static_assert(kVChunkTok == 32, "V chunk: two 16-token MMA slices");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: p stays below 2^8

// shared memory (offsets from the 1024-byte aligned base)
constexpr int kOffQ = 0;                          // 9 panels x (64 heads x 128 B)
constexpr int kQPanel = 64 * 128;
constexpr int kOffP = kOffQ + 9 * kQPanel;        // P^T: 256 token rows x 128 B (64 heads)
constexpr int kPBuf = kT * 128;            // one P^T buffer: 32 KB
constexpr int kOffKRing = kOffP + kPBufs * kPBuf;
constexpr int kOffVRing = kOffKRing + kKSlots * kSlotBytes;
constexpr int kOffRed = kOffVRing + kVSlots * kSlotBytes;  // [4 quadrants][2 halves][32 lanes] float4
constexpr int kOffX = kOffRed + 4 * 2 * 32 * 16;          // peer maxima [2 parities][2 halves][32 lanes] float2
constexpr int kOffXs = kOffX + 2 * 2 * 32 * 8;            // peer sums [2 halves][32 lanes] float4
constexpr int kOffRef = kOffXs + 2 * 32 * 16;             // ref[128], alpha[128], inv[128], lse[128]
constexpr int kOffFlags = kOffRef + 4 * 128 * 4;          // abort, tmem slot, rescale flags
constexpr int kOffBar = kOffFlags + 64;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kOffKRing % 1024 == 0 && kOffVRing % 1024 == 0,
              "swizzle atoms");

enum Bar {
  kKFull0 = 0,                   // [kKSlots] even CTA: K slot loaded in both CTAs (1 arrival + both CTAs' bytes)
  kKEmpty0 = kKFull0 + kKSlots,  // [kKSlots] both: the MMAs reading the K slot completed
  kVFull0 = kKEmpty0 + kKSlots,  // [kVSlots] even CTA: V slot loaded in both CTAs
  kVEmpty0 = kVFull0 + kVSlots,  // [kVSlots] both
  kQFull = kVEmpty0 + kVSlots,   // even CTA: both query halves loaded (1 arrival + bytes)
  kQFree,                        // both: the unit's last QK completed
  kSFull0,                       // [2] both: S^T buffer written
  kSFree0 = kSFull0 + 2,         // [2] even CTA: S^T buffer read by all 16 softmax warps
  kPvDone0 = kSFree0 + 2,        // [2] by tile parity, both: the tile's PV completed
  kPIn0 = kPvDone0 + 2,          // [2] by tile parity, both: this CTA's P^T rows complete (8 warps + 16 KB from the peer)
  kPeerReady0 = kPIn0 + 2,       // [2] by tile parity, even CTA: the odd CTA's kPIn completed
  kOFree = kPeerReady0 + 2,                        // even CTA: both epilogues read O^T (16 arrivals)
  kRed0,                         // [2] both: per head half, the four quadrant warps posted
  kX0 = kRed0 + 2,               // [2 parities][2 halves] both: the peer's maxima landed
  kXs0 = kX0 + 4,                // [2] both: the peer's sums landed
  kRef = kXs0 + 2,               // both: references (or lse / 1/l) written by both combining warps
  kTail,                         // both: producer-local copy of a partial V chunk
  kTailReady,                    // even CTA: both CTAs zeroed the rows past the end of a partial V chunk
  kFinal,                        // even CTA: every QK MMA completed
  kFinalPv,                      // even CTA: every PV MMA completed
  kNumBars
};
constexpr int kSmemBytes = kOffBar + 8 * kNumBars + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t bar(uint32_t base, int i) { return base + kOffBar + 8 * i; }

__device__ __forceinline__ int tiles_of(const WorkUnit& u) { return (u.tok_end - u.tok_begin + kT - 1) / kT; }

// Reduce-scatter over the 32 lanes of a warp: v[64] holds one value per head
// (heads 0..63 of this lane's token); afterwards lane l holds the reduction
// over the warp of heads 2l and 2l + 1.  Step k (lane bit 4 - k) halves the
// live values: the lane keeps the half its bit selects and adds the partner's
// copy of it.
template <int kCnt, int kMask, bool kMax>
__device__ __forceinline__ void scatter_step(float (&v)[64], int lane) {
  constexpr int kHalf = kCnt / 2;
  const bool upper = (lane & kMask) != 0;
#pragma unroll
  for (int i = 0; i < kHalf; ++i) {
    const float keep = upper ? v[i + kHalf] : v[i];
    const float send = upper ? v[i] : v[i + kHalf];
    const float got = __shfl_xor_sync(0xffffffffu, send, kMask);
    v[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
}
template <bool kMax>
__device__ __forceinline__ float2 warp_scatter(float (&v)[64], int lane) {
  scatter_step<64, 16, kMax>(v, lane);
  scatter_step<32, 8, kMax>(v, lane);
  scatter_step<16, 4, kMax>(v, lane);
  scatter_step<8, 2, kMax>(v, lane);
  scatter_step<4, 1, kMax>(v, lane);
  return make_float2(v[0], v[1]);
}

template <bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const DecodeArgs a, const __grid_constant__ PairMaps maps) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(sm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffFlags + 4);
  volatile int* resc = reinterpret_cast<volatile int*>(sm + kOffFlags + 8);   // [2] rescale flags
  float* ref_s = reinterpret_cast<float*>(sm + kOffRef);
  float* alpha_s = ref_s + 128;
  float* inv_s = ref_s + 256;
  float* lse_s = ref_s + 384;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int worker = blockIdx.x >> 1;
  const int rank = static_cast<int>(cluster_ctarank());
  const int peer = rank ^ 1;
  const PlanDev prm = *a.params;
  const int H = a.num_heads;
  const int P = prm.page_size;
  const int u0 = worker < prm.n_workers ? a.worker_ptr[worker] : 0;
  const int u1 = worker < prm.n_workers ? a.worker_ptr[worker + 1] : 0;
  int n_tiles = 0;   // this worker's tiles over all its units
  for (int ui = u0; ui < u1; ++ui) n_tiles += tiles_of(a.units[ui]);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kTailReady) cnt = 2;
      if (i == kSFree0 || i == kSFree0 + 1 || i == kOFree) cnt = 16;
      if (i == kPIn0 || i == kPIn0 + 1) cnt = 8;
      if (i == kRed0 || i == kRed0 + 1) cnt = 4;
      if (i == kRef) cnt = 2;
      mbar_init(bar(base, i), cnt);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.q_nope);
    tma_prefetch_desc(&maps.q_pe);
    tma_prefetch_desc(&maps.ckv_k);
    tma_prefetch_desc(&maps.kpe_k);
    tma_prefetch_desc(&maps.ckv_v);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers initialised before any remote operation
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const uint32_t lead = static_cast<uint32_t>(0);   // the even CTA issues the MMAs

  if (warp == 0 || warp == kVProducerWarp) {
    // ================= producers (both CTAs) =================
    // Warp 0 loads the query (once per unit) and the K panels of every tile
    // into the K ring; warp 10 loads the V chunks into the V ring.  The two
    // streams (K mostly from DRAM, V mostly from L2, where the other CTA's K
    // copies of the same tokens left it) run concurrently.  Each copy of
    // both CTAs completes on the even CTA's full barrier of its slot, where
    // the even CTA's producer announces the bytes of both (the odd CTA only
    // issues its copies: an arrive at cluster scope per slot would cost a
    // fence each).
    const bool is_k = warp == 0;
    int rp = 0;            // slots of this ring used so far
    int tail_uses = 0;
    bool ok = true;
    int q_units = 0;       // query loads issued
    const int vbox = P >= kVChunkTok ? kVChunkTok : 16;
    const int nslots = is_k ? kKSlots : kVSlots;
    const int full0 = is_k ? kKFull0 : kVFull0, empty0 = is_k ? kKEmpty0 : kVEmpty0;
    const int ring = is_k ? kOffKRing : kOffVRing;
    auto next_slot = [&](int& slot) -> bool {
      slot = rp % nslots;
      const uint32_t par = ((rp / nslots) & 1) ^ 1;
      ++rp;
      return mbar_wait_warp(bar(base, empty0 + slot), par, abort_flag);
    };
#ifdef MLA_STALL_TEST
    auto stalled = [&]() { return g_pair_stall != 0 && blockIdx.x == 0 && !is_k && rp == g_pair_stall; };
#else
    auto stalled = [&]() { return false; };
#endif
    // page ids of one tile: lane b holds page b (P = 16: 16 pages, 32: 8, 64: 4)
    auto tile_pages = [&](const WorkUnit& v, int i) -> int {
      const int tok0 = v.tok_begin + i * kT;
      const int np = (min(tok0 + kT, v.tok_end) - tok0 + P - 1) / P;
      int page = 0;
      if (lane < np) {
        page = a.kv_indices[v.page_base + tok0 / P + lane];
        if (page < 0 || page >= a.num_pages) {
          report_error(a.err, kErrBounds);
          page = 0;
        }
      }
      return page;
    };
    auto emit_q = [&](const WorkUnit& v) -> bool {
      if (q_units > 0 && !(ok = mbar_wait_warp(bar(base, kQFree), (q_units - 1) & 1, abort_flag))) return false;
      ++q_units;
      if (lane == 0 && rank == 0) mbar_arrive_expect_tx(bar(base, kQFull), 2 * 9 * kQPanel);
      __syncwarp();
      if (lane < 9) {
        const int row = v.req * H + 64 * rank;   // rows past the batch are zero-filled
        if (lane < 8)
          tma_load_2d_pair(base + kOffQ + lane * kQPanel, &maps.q_nope, 64 * lane, row,
                           map_to_rank(bar(base, kQFull), lead));
        else
          tma_load_2d_pair(base + kOffQ + 8 * kQPanel, &maps.q_pe, 0, row, map_to_rank(bar(base, kQFull), lead));
      }
      return true;
    };
    auto emit_k = [&](const WorkUnit& v, int i, int pages) -> bool {
      const int t0 = v.tok_begin + i * kT + kHalfT * rank;
      const int cnt = max(0, min(kHalfT, v.tok_end - t0));
      const int nbox = (cnt + P - 1) / P;
      // the other CTA's half (announced by the even CTA)
      const int cnt1 = max(0, min(kHalfT, v.tok_end - (v.tok_begin + i * kT + kHalfT)));
      const int nbox_both = nbox + (cnt1 + P - 1) / P;
      const int pb = (kHalfT * rank) / P;   // first page of this half within the tile
      const int page = __shfl_sync(0xffffffffu, pages, min(pb + lane, 31));
      for (int j = 0; j < 9; ++j) {
        int slot;
        if (!(ok = next_slot(slot))) return false;
        const uint32_t full = map_to_rank(bar(base, kKFull0 + slot), lead);
        if (lane == 0 && rank == 0) mbar_arrive_expect_tx(bar(base, kKFull0 + slot), nbox_both * P * 128);
        __syncwarp();
        if (lane < nbox) {
          const uint32_t dst = base + kOffKRing + slot * kSlotBytes + lane * P * 128;
          if (j < 8)
            tma_load_2d_pair(dst, &maps.ckv_k, 64 * j, page * P, full);
          else
            tma_load_2d_pair(dst, &maps.kpe_k, 0, page * P, full);
        }
      }
      return true;
    };
    auto emit_v = [&](const WorkUnit& v, int i, int pages) -> bool {
      const int tok0 = v.tok_begin + i * kT;
      for (int c = 0; c < kChunksPerTile; ++c) {
        const int t = tok0 + kVChunkTok * c;
        const int rows = min(kVChunkTok, v.tok_end - t);
        if (rows <= 0) break;
        int slot;
        if (!(ok = next_slot(slot))) return false;
        const uint32_t full = map_to_rank(bar(base, kVFull0 + slot), lead);
        if (stalled()) continue;
        const int ncopy = (rows + vbox - 1) / vbox;
        const int tb = t + vbox * min(lane, ncopy - 1);
        const int page = __shfl_sync(0xffffffffu, pages, (tb - tok0) / P);
        const uint32_t dst = base + kOffVRing + slot * kSlotBytes + lane * vbox * 4 * 128;
        if (rows == kVChunkTok) {
          if (lane == 0 && rank == 0) mbar_arrive_expect_tx(bar(base, kVFull0 + slot), 2 * ncopy * vbox * 4 * 128);
          __syncwarp();
          if (lane < ncopy) tma_load_3d_pair(dst, &maps.ckv_v, 0, page * P + (tb % P), 4 * rank, full);
        } else {
          // last chunk of a request: rows past kv_len may hold anything (even
          // NaN) and p = 0 does not cancel NaN; copy locally, zero those
          // rows, then release the slot to the issuer
          const uint32_t tail = bar(base, kTail);
          if (lane == 0) mbar_arrive_expect_tx(tail, ncopy * vbox * 4 * 128);
          __syncwarp();
          if (lane < ncopy) tma_load_3d(dst, &maps.ckv_v, 0, page * P + (tb % P), 4 * rank, tail);
          if (!(ok = mbar_wait_warp(tail, tail_uses & 1, abort_flag))) return false;
          unsigned char* sv = sm + kOffVRing + slot * kSlotBytes;
          for (int q = lane; q < (kVChunkTok - rows) * 32; q += 32) {
            const int rr = rows + q / 32, pnl = (q % 32) >> 3, c16 = q & 7;
            const int off = vbox == kVChunkTok ? pnl * 4096 + rr * 128
                                               : (rr >> 4) * 8192 + pnl * 2048 + (rr & 15) * 128;
            *reinterpret_cast<uint4*>(sv + off + c16 * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          // both CTAs' rows zeroed: the even CTA then releases the slot
          if (rank == 0) {
            if (lane == 0) mbar_arrive(bar(base, kTailReady));
            if (!(ok = mbar_wait_cl_warp(bar(base, kTailReady), tail_uses & 1, abort_flag))) return false;
            if (lane == 0) mbar_arrive(bar(base, kVFull0 + slot));
          } else if (lane == 0) {
            mbar_arrive_cluster(map_to_rank(bar(base, kTailReady), lead));
          }
          ++tail_uses;
        }
      }
      return true;
    };
    for (int ui = u0; ui < u1 && ok; ++ui) {
      const WorkUnit v = a.units[ui];
      const int n = tiles_of(v);
      for (int i = 0; i < n && ok; ++i) {
        const int pages = tile_pages(v, i);
        if (is_k) {
          if (i == 0 && !emit_q(v)) break;
          if (!emit_k(v, i, pages)) break;
        } else if (!emit_v(v, i, pages)) {
          break;
        }
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
  } else if ((warp == 1 || warp == kPvIssuerWarp) && rank == 0) {
    // ================= MMA issuers (even CTA, whole warp, lane 0 issues) =================
    // Warp 1 issues the QK products of every tile, panel by panel from the K
    // ring; warp 11 the PV products, chunk by chunk from the V ring, once
    // the tile's P^T is complete in both CTAs.  Two issuers, because an
    // issuing thread cannot run ahead of the tensor pipe: the waits and
    // commits of one overlap the other's MMAs.
    const uint32_t issue = lane == 0;
    bool ok = true;
    if (warp == 1) {
      constexpr uint32_t id_qk = idesc_bf16_f32(256, 128, false, false);
      const uint64_t q_desc0 = smem_desc(base + kOffQ, 16, 1024, kSw128);
      const uint64_t k_desc0 = smem_desc(base + kOffKRing, 16, 1024, kSw128);
      int kc = 0, g = 0, unit_k = 0;
      for (int ui = u0; ui < u1 && ok; ++ui, ++unit_k) {
        const WorkUnit v = a.units[ui];
        const int n = tiles_of(v);
        if (!(ok = mbar_wait_warp(bar(base, kQFull), unit_k & 1, abort_flag))) break;
        for (int i = 0; i < n && ok; ++i, ++g) {
          if (g >= 2 && !(ok = mbar_wait_cl_warp(bar(base, kSFree0 + (g & 1)), ((g - 2) >> 1) & 1, abort_flag)))
            break;
          tc_fence_after();
          const uint32_t d = tmem + kColS + 128 * (g & 1);
          for (int j = 0; j < 9; ++j, ++kc) {
            const int slot = kc % kKSlots;
            if (!(ok = mbar_wait_warp(bar(base, kKFull0 + slot), (kc / kKSlots) & 1, abort_flag))) break;
            tc_fence_after();
            const uint64_t adesc = k_desc0 + static_cast<uint64_t>((slot * kSlotBytes) >> 4);
            const uint64_t bdesc = q_desc0 + static_cast<uint64_t>((j * kQPanel) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_pair(d, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2), id_qk,
                       (j | kk) != 0, issue);
            commit_pair(bar(base, kKEmpty0 + slot), 3, issue);
          }
          if (!ok) break;
          commit_pair(bar(base, kSFull0 + (g & 1)), 3, issue);
        }
        if (!ok) break;
        commit_pair(bar(base, kQFree), 3, issue);   // the unit's query no longer read
      }
      if (!ok && lane == 0) report_error(a.err, kErrTimeout);
      // drain: every MMA issued completes before TMEM is freed
      commit_pair(bar(base, kFinal), 1, issue);
      if (lane == 0) mbar_wait_cl_drain(bar(base, kFinal), 0);
      __syncwarp();
    } else {
      constexpr uint32_t id_pv = idesc_bf16_f32(256, 128, true, true);
      const uint64_t p_desc0 = smem_desc(base + kOffP, 16, 1024, kSw128);
      const bool v32 = P >= kVChunkTok;
      const uint64_t v_desc0 = smem_desc(base + kOffVRing, v32 ? 4096 : 2048, 1024, kSw128);
      const uint32_t v_kstep = v32 ? 2048 : 8192, v_block = v32 ? 8192 : 4096;
      int vc = 0, g = 0, unit_k = 0;
      for (int ui = u0; ui < u1 && ok; ++ui, ++unit_k) {
        const WorkUnit v = a.units[ui];
        const int n = tiles_of(v);
        // the first PV of a unit overwrites O^T: the previous epilogue must be done
        if (unit_k > 0 && !(ok = mbar_wait_cl_warp(bar(base, kOFree), (unit_k - 1) & 1, abort_flag))) break;
        for (int i = 0; i < n && ok; ++i, ++g) {
          if (!(ok = mbar_wait_warp(bar(base, kPIn0 + (g & 1)), (g >> 1) & 1, abort_flag) &&
                     mbar_wait_cl_warp(bar(base, kPeerReady0 + (g & 1)), (g >> 1) & 1, abort_flag)))
            break;
          tc_fence_after();
          const int valid = min(kT, v.tok_end - (v.tok_begin + i * kT));
          const int nch = (valid + kVChunkTok - 1) / kVChunkTok;
          for (int c = 0; c < nch; ++c, ++vc) {
            const int slot = vc % kVSlots;
            if (!(ok = mbar_wait_warp(bar(base, kVFull0 + slot), (vc / kVSlots) & 1, abort_flag))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint64_t bdesc = p_desc0 + static_cast<uint64_t>(
                                                   ((kPBufs == 2 ? (g & 1) : 0) * kPBuf + (kVChunkTok * c + 16 * kk) * 128) >> 4);
#pragma unroll
              for (int bb = 0; bb < 2; ++bb) {
                const uint64_t adesc =
                    v_desc0 + static_cast<uint64_t>((slot * kSlotBytes + kk * v_kstep + bb * v_block) >> 4);
                mma_pair(tmem + kColO + 128 * bb, adesc, bdesc, id_pv, (i == 0 && c == 0 && kk == 0) ? 0u : 1u,
                         issue);
              }
            }
            commit_pair(bar(base, kVEmpty0 + slot), 3, issue);
          }
          if (!ok) break;
          commit_pair(bar(base, kPvDone0 + (g & 1)), 3, issue);
        }
      }
      if (!ok && lane == 0) report_error(a.err, kErrTimeout);
      commit_pair(bar(base, kFinalPv), 1, issue);
      if (lane == 0) mbar_wait_cl_drain(bar(base, kFinalPv), 0);
      __syncwarp();
    }
  } else if (warp == 1) {
    // ================= relay (odd CTA): "my P^T rows are complete" =================
    bool ok = true;
    for (int g = 0; g < n_tiles && ok; ++g) {
      if (!(ok = mbar_wait_warp(bar(base, kPIn0 + (g & 1)), (g >> 1) & 1, abort_flag))) break;
      if (lane == 0) mbar_arrive_cluster(map_to_rank(bar(base, kPeerReady0 + (g & 1)), lead));
      __syncwarp();
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
  } else if (warp == kPvIssuerWarp) {
    // (odd CTA: no role)
  } else {
    // ================= softmax / epilogue (warps 2..9, both CTAs) =================
    const int sw = warp - kFirstSoftmaxWarp;
    const int q = warp & 3;                  // TMEM lane quadrant: tokens (S^T) or dims (O^T)
    const int hh = sw >> 2;                  // heads [64 hh, 64 hh + 64)
    const bool combiner = q == 0;            // one warp per head half combines and exchanges
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float c = prm.sm_scale * a.kv_scale * kLog2e;
    const int h0 = 64 * hh + 2 * lane;       // the two heads this lane reduces into
    // P^T rows of heads [64 hh, ..) live in CTA hh
    const bool p_local = hh == rank;
    int nred = 0;
    bool ok = true;
    int g = 0, unit_k = 0;
    for (int ui = u0; ui < u1 && ok; ++ui, ++unit_k) {
      const WorkUnit u = a.units[ui];
      const int n = tiles_of(u);
      float lx0 = 0.f, lx1 = 0.f, lr0 = 0.f, lr1 = 0.f;
      for (int i = 0; i < n && ok; ++i, ++g) {
        const bool first = i == 0;
        // ---- scores of this lane's token, 64 heads ----
        if (!(ok = mbar_wait_warp(bar(base, kSFull0 + (g & 1)), (g >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        float y[64];
        {
          uint32_t v0[32], v1[32];
          tmem_ld32(lane_addr + kColS + 128 * (g & 1) + 64 * hh, v0);
          tmem_ld32(lane_addr + kColS + 128 * (g & 1) + 64 * hh + 32, v1);
          tmem_ld_wait();
          const int tok = u.tok_begin + i * kT + kHalfT * rank + 32 * q + lane;
          const bool valid = tok < u.tok_end;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            y[j] = valid ? __uint_as_float(v0[j]) * c : -INFINITY;
            y[32 + j] = valid ? __uint_as_float(v1[j]) * c : -INFINITY;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(bar(base, kSFree0 + (g & 1)));
          else
            mbar_arrive_cluster(map_to_rank(bar(base, kSFree0 + (g & 1)), lead));
        }
        // ---- per-head maximum over the tile: warp, quadrants, then the peer ----
        {
          float t[64];
#pragma unroll
          for (int j = 0; j < 64; ++j) t[j] = y[j];
          const float2 mx = warp_scatter<true>(t, lane);
          float4* red = reinterpret_cast<float4*>(sm + kOffRed);
          *reinterpret_cast<float2*>(red + (q * 2 + hh) * 32 + lane) = mx;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(base, kRed0 + hh));
          if (combiner) {
            if (!(ok = mbar_wait_warp(bar(base, kRed0 + hh), nred & 1, abort_flag))) break;
            float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const float2 o = *reinterpret_cast<const float2*>(red + (qq * 2 + hh) * 32 + lane);
              m0 = fmaxf(m0, o.x);
              m1 = fmaxf(m1, o.y);
            }
            const int xp = g & 1;
            float2* xs = reinterpret_cast<float2*>(sm + kOffX) + (xp * 2 + hh) * 32;
            const uint32_t xbar = bar(base, kX0 + xp * 2 + hh);
            if (lane == 0) mbar_arrive_expect_tx(xbar, 32 * 8);
            __syncwarp();
            st_async_peer_v2f(map_to_rank(smem_u32(xs + lane), peer), m0, m1, map_to_rank(xbar, peer));
            if (!(ok = mbar_wait_warp(xbar, (g >> 1) & 1, abort_flag))) break;
            const float2 pm = xs[lane];
            m0 = fmaxf(m0, pm.x);
            m1 = fmaxf(m1, pm.y);
            float r0 = ref_s[h0], r1 = ref_s[h0 + 1];
            const float n0 = first || m0 > r0 + kRescaleThreshold ? m0 : r0;
            const float n1 = first || m1 > r1 + kRescaleThreshold ? m1 : r1;
            const float a0 = first ? 1.f : exp2f(r0 - n0), a1 = first ? 1.f : exp2f(r1 - n1);
            ref_s[h0] = n0;
            ref_s[h0 + 1] = n1;
            alpha_s[h0] = a0;
            alpha_s[h0 + 1] = a1;
            const bool moved = (h0 < H && a0 != 1.f) || (h0 + 1 < H && a1 != 1.f);
            const bool any = __any_sync(0xffffffffu, moved);
            if (lane == 0) resc[hh] = any && !first;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(base, kRef));
          }
          if (!(ok = mbar_wait_warp(bar(base, kRef), nred & 1, abort_flag))) break;
          ++nred;
        }
        // ---- p = 2^(y - reference), rounded to bf16; row sums ----
        uint32_t pk[32];
        {
          float px[64], pr[64];
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const float4 m4 = reinterpret_cast<const float4*>(ref_s + 64 * hh)[j4];
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) px[4 * j4 + e] = fast_exp2(y[4 * j4 + e] - mm[e]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(px[2 * j], px[2 * j + 1]);
            const uint32_t w = *reinterpret_cast<const uint32_t*>(&b2);
            pk[j] = w;
            pr[2 * j] = __uint_as_float(w << 16);
            pr[2 * j + 1] = __uint_as_float(w & 0xffff0000u);
          }
          const float2 sx = warp_scatter<false>(px, lane);
          const float2 sr = warp_scatter<false>(pr, lane);
          const float a0 = alpha_s[h0], a1 = alpha_s[h0 + 1];
          lx0 = first ? sx.x : fmaf(lx0, a0, sx.x);
          lx1 = first ? sx.y : fmaf(lx1, a1, sx.y);
          lr0 = first ? sr.x : fmaf(lr0, a0, sr.x);
          lr1 = first ? sr.y : fmaf(lr1, a1, sr.y);
        }
        // ---- the P^T buffer free (PV of the tile that used it done); for a
        // rescale, also the previous tile's PV (O^T current) ----
        const bool rescale = !first && (resc[0] | resc[1]);
        {
          const int tw = rescale ? g - 1 : g - kPBufs;
          if (tw >= 0 && !(ok = mbar_wait_warp(bar(base, kPvDone0 + (tw & 1)), (tw >> 1) & 1, abort_flag))) break;
          if (rescale && kPBufs == 2 && g >= 2 &&
              !(ok = mbar_wait_warp(bar(base, kPvDone0 + (g & 1)), ((g - 2) >> 1) & 1, abort_flag)))
            break;
        }
        tc_fence_after();
        if (rescale) {
          // O^T rows of this quadrant's dims, block hh: column h times alpha[h]
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            const uint32_t col = kColO + 128 * hh + 32 * cc;
            tmem_ld32(lane_addr + col, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha_s[32 * cc + j]);
            tmem_st32(lane_addr + col, o);
          }
          tmem_st_wait();
        }
        // ---- P^T row of this lane's token (64 heads = 128 bytes) ----
        {
          const uint32_t p_in_self = bar(base, kPIn0 + (g & 1));
          const uint32_t p_in_dst = p_local ? p_in_self : map_to_rank(p_in_self, peer);
          const int row = kHalfT * rank + 32 * q + lane;
          const int pb = kOffP + (kPBufs == 2 ? (g & 1) : 0) * kPBuf;
          const uint32_t rowaddr = base + pb + row * 128;
          if (p_local) {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(sm + pb + row * 128 + ((ch ^ (row & 7)) << 4)) =
                  make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            fence_proxy_async_smem();
          } else {
            const uint32_t rrow = map_to_rank(rowaddr, peer);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              st_async_peer(rrow + ((ch ^ (row & 7)) << 4),
                            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]), p_in_dst);
          }
          tc_fence_before();
          __syncwarp();
          // one local warp announces the 16 KB of rows the peer sends here
          if (lane == 0) {
            if (sw == 0)
              mbar_arrive_expect_tx(p_in_self, 128 * 128);
            else
              mbar_arrive(p_in_self);
          }
        }
      }
      if (!ok) break;
      // ================= epilogue of the unit =================
      {
        float4* red = reinterpret_cast<float4*>(sm + kOffRed);
        red[(q * 2 + hh) * 32 + lane] = make_float4(lx0, lr0, lx1, lr1);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(base, kRed0 + hh));
        if (combiner) {
          if (!(ok = mbar_wait_warp(bar(base, kRed0 + hh), nred & 1, abort_flag))) break;
          float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const float4 o = red[(qq * 2 + hh) * 32 + lane];
            s.x += o.x;
            s.y += o.y;
            s.z += o.z;
            s.w += o.w;
          }
          float4* xs = reinterpret_cast<float4*>(sm + kOffXs) + hh * 32;
          const uint32_t xbar = bar(base, kXs0 + hh);
          if (lane == 0) mbar_arrive_expect_tx(xbar, 32 * 16);
          __syncwarp();
          st_async_peer(map_to_rank(smem_u32(xs + lane), peer),
                        make_uint4(__float_as_uint(s.x), __float_as_uint(s.y), __float_as_uint(s.z),
                                   __float_as_uint(s.w)),
                        map_to_rank(xbar, peer));
          if (!(ok = mbar_wait_warp(xbar, unit_k & 1, abort_flag))) break;
          const float4 o = xs[lane];
          const float lx_0 = s.x + o.x, lr_0 = s.y + o.y, lx_1 = s.z + o.z, lr_1 = s.w + o.w;
          const float ls0 = (ref_s[h0] + log2f(lx_0)) * kLn2, ls1 = (ref_s[h0 + 1] + log2f(lx_1)) * kLn2;
          lse_s[h0] = ls0;
          lse_s[h0 + 1] = ls1;
          inv_s[h0] = a.kv_scale / lr_0;
          inv_s[h0 + 1] = a.kv_scale / lr_1;
          if (rank == 0) {
            const bool split = u.out_slot >= 0;
            if (h0 < H) {
              if (split) a.lse_part[lse_part_offset(u.out_slot, 0, h0, H)] = ls0;
              else a.lse[static_cast<size_t>(u.req) * H + h0] = ls0;
            }
            if (h0 + 1 < H) {
              if (split) a.lse_part[lse_part_offset(u.out_slot, 0, h0 + 1, H)] = ls1;
              else a.lse[static_cast<size_t>(u.req) * H + h0 + 1] = ls1;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(base, kRef));
        }
        if (!(ok = mbar_wait_warp(bar(base, kRef), nred & 1, abort_flag))) break;
        ++nred;
        if (!(ok = mbar_wait_warp(bar(base, kPvDone0 + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        // O^T: this lane's latent dim, all heads of block hh
        const int d = 256 * rank + 128 * hh + 32 * q + lane;
        const bool split = u.out_slot >= 0;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kColO + 128 * hh + 32 * cc, o);
          tmem_ld_wait();
          if (split) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int h = 32 * cc + j;
              if (h < H) a.o_part[part_offset(u.out_slot, h, d, H)] = __uint_as_float(o[j]) * inv_s[h];
            }
          } else if (kOutF32) {
            float* out = static_cast<float*>(a.out);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int h = 32 * cc + j;
              if (h < H) out[(static_cast<size_t>(u.req) * H + h) * kDCkv + d] = __uint_as_float(o[j]) * inv_s[h];
            }
          } else {
            // pairs of heads: even lanes store dims (d, d+1) of head h, odd
            // lanes dims (d-1, d) of head h+1 (4-byte bf16x2 stores)
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
            const bool odd = lane & 1;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const int h = 32 * cc + j;
              const float v0 = __uint_as_float(o[j]) * inv_s[h];
              const float v1 = __uint_as_float(o[j + 1]) * inv_s[h + 1];
              const float got = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
              const int hs = odd ? h + 1 : h;
              const int ds = odd ? d - 1 : d;
              const __nv_bfloat162 b2 = odd ? __floats2bfloat162_rn(got, v1) : __floats2bfloat162_rn(v0, got);
              if (hs < H)
                *reinterpret_cast<__nv_bfloat162*>(out + (static_cast<size_t>(u.req) * H + hs) * kDCkv + ds) = b2;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(bar(base, kOFree));
          else
            mbar_arrive_cluster(map_to_rank(bar(base, kOFree), lead));
        }
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
  }

  // On a device error some copies or remote stores may still be in flight
  // toward this CTA: give them time to land before it leaves.
  if (*abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the peer no longer addresses this CTA's shared memory or TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace

#ifdef MLA_STALL_TEST
// Test build only: the ring copy CTA 0's producer leaves out (0: none).
extern "C" int mla_test_set_pair_stall(int copy) {
  return static_cast<int>(cudaMemcpyToSymbol(g_pair_stall, &copy, sizeof(copy)));
}
#endif

namespace {
template <bool kOutF32>
cudaError_t set_pair_attributes() {
  static bool done = false;   // set once, before any stream capture
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<kOutF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    done = true;
  }
  return cudaSuccess;
}

cudaLaunchConfig_t pair_config(int clusters, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}
}  // namespace

cudaError_t decode_pair_max_workers(int* workers) {
  *workers = 0;
  cudaError_t e = set_pair_attributes<true>();
  if (e == cudaSuccess) e = set_pair_attributes<false>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(1, attr);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, decode_pair_kernel<false>, &cfg);
  if (e != cudaSuccess) return e;
  *workers = clusters;
  return cudaSuccess;
}

cudaError_t launch_decode_pair(const DecodeArgs& a, const PairMaps& maps, bool out_f32, cudaStream_t s) {
  cudaError_t e = out_f32 ? set_pair_attributes<true>() : set_pair_attributes<false>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(a.n_workers, attr);
  cfg.stream = s;
  return out_f32 ? cudaLaunchKernelEx(&cfg, decode_pair_kernel<true>, a, maps)
                 : cudaLaunchKernelEx(&cfg, decode_pair_kernel<false>, a, maps);
}

}  // namespace mla
