// Paged MLA decode on a CTA pair: one tcgen05 MMA spans both SMs of a
// cluster (cta_group::2), and the two SMs split the heads.
//
// Operation (absorbed multi-head latent attention, one query token, one
// latent KV head of width 512 + 64, no causal mask -- "[WIP] support
// flashinfer_mla", vLLM-metax PR #113, review of the decode_wrapper.plan
// parameters): for request b, head h over the request's kv_len tokens
//   S   = sm_scale * (q_nope[b,h] . ckv_t + q_pe[b,h] . kpe_t)
//   out = softmax(S) . ckv,   lse = ln sum exp(S).
//
// Both products are pair MMAs of M = 128 heads, each CTA holding 64 of them:
//   S [128 heads x 256 tokens]  = Q [128 x 576] . K^T            (QK, N = 256)
//   O [128 heads x 512 dims]   += P [128 x 256 tokens] . V        (PV, two MMAs of N = 256)
// CTA r supplies the rows of heads [64 r, 64 r + 64) of A (the query, then
// P) and half the N rows of B: for QK the K rows of tokens
// [128 r, 128 r + 128) of each 256-token tile, for PV the V columns of latent
// dims [256 r, 256 r + 256).  It receives the D rows of its own 64 heads,
// all N columns: TMEM lane l < 64 holds head 64 r + l over columns
// [0, N/2), lane 64 + l the same head over [N/2, N).  So every score and
// every output element of a head lands in one SM: the softmax of a head
// never leaves its CTA.  The pair exchanges only two signals per tile: "the
// scores were read" (the issuer may overwrite the S buffer) and "P is
// written" (the issuer may start P . V).
//
// Per CTA: warp 0 K producer (the shared-memory part of the query once per
// unit, then the K panels of every tile through a ring, two panels per slot
// for bf16), warp 10 V producer (32-token V chunks through a second ring);
// in the even CTA warp 1 issues every QK MMA of the pair and warp 11 every
// PV MMA, so the softmax of tile g overlaps the scores of tile g + 1 and the
// P . V of tile g - 1; warps 2..9 softmax and epilogue: warp w reads TMEM
// lane quadrant w % 4 and column half (w - 2) / 4, so each thread owns one
// head and 64 tokens of a tile, and the four threads of a head combine
// their maxima through shared memory.  For bf16 the softmax warps also store
// the query's dims [320, 576) into TMEM once per unit.
//
// TMEM columns: S [0, 128); bf16: the query's dims [320, 576) [128, 256);
// e4m3: a second S buffer [128, 256); O [256, 512) (lane l < 64: dims
// [0, 256) of head 64 r + l; lane 64 + l: dims [256, 512)).
//
// Softmax, per tile and head: the exact maximum over the tile's 256 tokens,
// a reference that moves only when that maximum exceeds it by more than 2^8
// (then O and the running sums are scaled by 2^(old - new) < 1), p =
// 2^(s log2e sm_scale - reference) rounded to bf16 for the MMA.  The row sums
// are kept twice per thread, exact and of the rounded p, and added over the
// four threads of a head at the end (the output is divided by the latter,
// the lse uses the former).
//
// fp8 (e4m3) caches (pages of 32 or 64 tokens): both products are e4m3
// MMAs (kind::f8f6f4) straight from the copied codes -- K panels of 64 dims
// (64-byte rows) and V chunks of 2 x 128 dims (128-byte rows, MN-major), in
// 8 KB ring slots.  The other operand of each product is split into two
// e4m3 terms, x = hi + lo (hi = e4m3(x), lo = e4m3(x - hi)), and both terms
// multiply the same codes into the same accumulator: the query once per
// unit under a power-of-two scale per head row (its largest magnitude in
// [2^7, 2^8): hi + lo is then the bf16 query exactly, but for elements
// below 2^-2 after the scaling), P per tile as p = 2^(s - reference) * 2^5
// with a reference that moves when the tile maximum exceeds it by more than
// 3.5 (p <= 2^8.5 < 448); hi + lo keeps 8 significant bits of p, as bf16
// does, down to 2^-2 (below, lo loses bits).  Two P buffers, by tile parity.
//
// Every wait is bounded (2 s); on expiry the kernel records
// MLA_ERR_DEVICE_TIMEOUT, lets its copies and MMAs land, frees TMEM and
// returns.  Page ids outside [0, num_pages) are recorded as
// MLA_ERR_DEVICE_BOUNDS and never dereferenced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "device_utils.cuh"
#include "kernels.h"
#include "tc_utils.cuh"

namespace mla {
namespace {

using namespace tc;

#ifdef MLA_STALL_TEST
// Test build only: when nonzero, CTA 0's V producer leaves out its
// g_pair_stall-th ring copy (1-based), so the issuer's wait for it runs out.
__device__ int g_pair_stall;
#endif

constexpr int kT = kTilePair;              // 256 tokens per tile
constexpr int kHalfT = kT / 2;             // K rows per CTA
constexpr int kThreads = 384;              // 12 warps
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kSoftmaxWarps = 8;
constexpr int kVProducerWarp = 10;
constexpr int kPvIssuerWarp = 11;
constexpr int kVChunkTok = kTcVChunkTok;   // 32 tokens per V chunk
constexpr int kChunksPerTile = kT / kVChunkTok;
static_assert(kVChunkTok == 32, "V chunk: two 16-token MMA slices");
// TMEM columns: S [0, 128) (e4m3: a second S buffer [128, 256)); bf16: the
// query's dims [320, 576) as the QK A operand in [128, 256), row 64 r + l of
// A in lanes l and 64 + l of CTA r; O [256, 512).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColQT = 128, kColO = 256;
constexpr int kQTDim0 = 320;               // first query dim held in TMEM (bf16)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// log2 units: the reference moves when a tile's maximum exceeds it by more
// than this; p = 2^(s - reference) stays below 2^8 (bf16), and e4m3 hi + lo
// take p * 2^5 <= 2^8.5 (the largest code is 448; a power of two keeps a
// lone token's p exact)
constexpr float kRescaleThreshold = 8.0f, kRescaleThresholdFp8 = 3.5f;
constexpr float kPOffsetFp8 = 5.0f, kPScaleFp8 = 32.0f;   // 2^kPOffsetFp8
// bf16: the K copies of tile t wait until the V copies have reached chunk
// 8 t - kKLeadChunks (8 chunks per tile): V re-reads the K rows from L2, and
// a K stream far ahead of V pushes them out first (measured on long
// requests at a high DRAM rate; the e4m3 path, with half the bytes in
// flight, gains nothing from the cap and pays for the count).
constexpr int kKLeadChunks = 12;

// shared memory (offsets from the 1024-byte aligned base)
constexpr int kOffQ = 0;                          // query panels x (64 heads x 128 B)
constexpr int kQPanel = 64 * 128;
constexpr int kPPanel = 64 * 128;
constexpr int kPBuf = 4 * kPPanel;                // one P buffer (4 token panels): 32 KB
constexpr int kOffRed = 221184;                   // 216 KB: query, P and the rings before it
constexpr int kOffSum = kOffRed + 2 * 4 * 64 * 4;          // sums [4 parts][64 heads] float2
constexpr int kOffQRed = kOffSum + 4 * 64 * 8;            // fp8: query row maxima [4 parts][64 heads] float
constexpr int kOffFlags = kOffQRed + 4 * 64 * 4;          // abort, tmem slot, V tiles issued
constexpr int kOffBar = kOffFlags + 64;

// The 216 KB before the reduction areas, per cache type:
// - bf16: the query's dims [0, 320) (5 panels, 40 KB; dims [320, 576) are
//   in TMEM), one P buffer (32 KB), 3 K ring slots of two 16 KB K panels
//   (128 tokens x 64 dims each: one barrier, one wait and one commit per two
//   panels -- each wait before an MMA issue costs the issuing thread over a
//   hundred cycles) and 3 V ring slots of 16 KB (a V chunk of 32 tokens x
//   256 dims);
// - e4m3: the whole query split into hi + lo terms (9 panels, 72 KB), two
//   P buffers (by tile parity: the softmax of a tile need not wait for the
//   previous tile's P . V), 8 KB ring slots (the same tokens and dims): 5
//   for K, 5 for V.
template <bool kFp8>
struct Ring {
  static constexpr bool kQTmem = !kFp8;   // part of the query in TMEM (then one S buffer)
  static constexpr int kQSmemPanels = kQTmem ? kQTDim0 / 64 : 9;
  static constexpr int kSBufs = kQTmem ? 1 : 2;
  static constexpr int kPBufs = kFp8 ? 2 : 1;
  static constexpr int kPanelBytes = kFp8 ? 8192 : 16384;   // one K panel (128 rows)
  static constexpr int kKPanelsPerSlot = kFp8 ? 1 : 2;
  static constexpr int kKSlotBytes = kPanelBytes * kKPanelsPerSlot;
  static constexpr int kVSlotBytes = kFp8 ? 8192 : 16384;   // one V chunk
  static constexpr int kKSlots = kFp8 ? 5 : 3;
  static constexpr int kVSlots = kFp8 ? 5 : 3;
  static constexpr int kVPanels = kFp8 ? 2 : 4;   // MN panels (128-byte rows) of a V chunk
  static constexpr int kOffP = kOffQ + kQSmemPanels * kQPanel;
  static constexpr int kOffKRing = kOffP + kPBufs * kPBuf;
  static constexpr int kOffVRing = kOffKRing + kKSlots * kKSlotBytes;
  static_assert(kOffVRing + kVSlots * kVSlotBytes <= kOffRed, "rings fit before the reduction areas");
  static_assert(kOffP % 1024 == 0 && kOffKRing % 1024 == 0 && kOffVRing % 1024 == 0, "swizzle atoms");
};
constexpr int kKSlotsMax = 5, kVSlotsMax = 5;

enum Bar {
  kKFull0 = 0,                      // [K slots] even CTA: K slot loaded in both CTAs (1 arrival + both CTAs' bytes)
  kKEmpty0 = kKFull0 + kKSlotsMax,  // [K slots] both: the MMAs reading the K slot completed
  kVFull0 = kKEmpty0 + kKSlotsMax,  // [V slots] even CTA: V slot loaded in both CTAs
  kVEmpty0 = kVFull0 + kVSlotsMax,  // [V slots] both
  kQFull = kVEmpty0 + kVSlotsMax,   // even CTA: both query halves loaded (1 arrival + bytes)
  kQFree,                        // both: the unit's last QK completed
  kSFull0,                       // [2] both: S buffer written
  kSFree0 = kSFull0 + 2,         // [2] even CTA: S buffer read by all 16 softmax warps
  kPvDone0 = kSFree0 + 2,        // [2] by tile parity, both: the tile's PV completed
  kPReady0 = kPvDone0 + 2,       // [2] by tile parity, even CTA: P written by all 16 softmax warps
  kOFree = kPReady0 + 2,         // even CTA: both epilogues read O (16 arrivals)
  kRed0,                         // [2] by tile parity, both: the 8 softmax warps posted their maxima
  kSum = kRed0 + 2,              // both: the 8 softmax warps posted their sums
  kTail,                         // both: producer-local copy of a partial V chunk
  kTailReady,                    // even CTA: both CTAs zeroed the rows past the end of a partial V chunk
  kFinal,                        // even CTA: every QK MMA completed
  kFinalPv,                      // even CTA: every PV MMA completed
  // fp8 caches only
  kQLand,                        // this CTA's query landed (1 arrival + bytes)
  kQRed,                         // the 8 softmax warps posted their query row maxima
  kQReady,                       // even CTA: both CTAs' query split into e4m3 terms (16 arrivals)
  kNumBars
};
constexpr int kSmemBytes = kOffBar + 8 * kNumBars + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t bar(uint32_t base, int i) { return base + kOffBar + 8 * i; }

__device__ __forceinline__ int tiles_of(const WorkUnit& u) { return (u.tok_end - u.tok_begin + kT - 1) / kT; }

// Arrive on a barrier of the even CTA (from the odd CTA through the cluster
// window).  What the signal publishes lives in the arriving CTA: its reads of
// S or O from its own TMEM are complete, or its P rows are written and fenced
// for the tensor core of its own SM.
__device__ __forceinline__ void arrive_lead(uint32_t local_bar, int rank) {
  if (rank == 0)
    mbar_arrive(local_bar);
  else
    mbar_arrive_remote(map_to_rank(local_bar, 0));
}

// ---------------------------------------------------------------------------
// fp8 (e4m3) caches: e4m3 x e4m3 -> f32 MMAs (kind::f8f6f4).  The instruction
// descriptor has the layout of kind::f16's; the format code 0 of A and B
// means e4m3 there.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                                   // D format: f32
         | (static_cast<uint32_t>(a_mn) << 15)       // A, B format: e4m3 (0)
         | (static_cast<uint32_t>(b_mn) << 16)
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// Two floats -> two e4m3 codes (round to nearest even, saturating to +-448;
// the first in the low byte), and back.
__device__ __forceinline__ uint32_t to_e4m3x2(float x0, float x1) {
  return __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 from_e4m3x2(uint32_t codes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
// x = hi + lo, each an e4m3 term: hi = e4m3(x), lo = e4m3(x - hi) (x - hi is
// exact in f32).  Two elements; returns (hi + lo) of both, added.
__device__ __forceinline__ float split_e4m3x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = to_e4m3x2(x0, x1);
  const float2 h = from_e4m3x2(hi);
  lo = to_e4m3x2(x0 - h.x, x1 - h.y);
  const float2 l = from_e4m3x2(lo);
  return (h.x + l.x) + (h.y + l.y);
}

template <bool kOutF32, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const DecodeArgs a, const __grid_constant__ PairMaps maps) {
  // launched as a programmatic dependent of the previous kernel on the
  // stream: nothing is read before that kernel has completed and its writes
  // are visible (a no-op in a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel on the stream may be scheduled now; it waits for this
  // one to complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(sm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffFlags + 4);

  constexpr int kKSlots = Ring<kFp8>::kKSlots, kVSlots = Ring<kFp8>::kVSlots;
  constexpr int kVPanels = Ring<kFp8>::kVPanels;
  constexpr int kPanelBytes = Ring<kFp8>::kPanelBytes, kKPanelsPerSlot = Ring<kFp8>::kKPanelsPerSlot;
  constexpr int kKSlotBytes = Ring<kFp8>::kKSlotBytes, kVSlotBytes = Ring<kFp8>::kVSlotBytes;
  constexpr int kPBufs = Ring<kFp8>::kPBufs, kSBufs = Ring<kFp8>::kSBufs;
  constexpr int kQSmemPanels = Ring<kFp8>::kQSmemPanels;
  constexpr bool kQTmem = Ring<kFp8>::kQTmem;
  constexpr int kOffP = Ring<kFp8>::kOffP;
  constexpr int kOffKRing = Ring<kFp8>::kOffKRing, kOffVRing = Ring<kFp8>::kOffVRing;
  static_assert(kKSlots <= kKSlotsMax && kVSlots <= kVSlotsMax, "barrier slots");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int worker = blockIdx.x >> 1;
  const int rank = static_cast<int>(cluster_ctarank());
  const PlanDev prm = *a.params;
  const int H = a.num_heads;
  const int P = prm.page_size;
  const int u0 = worker < prm.n_workers ? a.worker_ptr[worker] : 0;
  const int u1 = worker < prm.n_workers ? a.worker_ptr[worker + 1] : 0;

  volatile int* v_tiles = reinterpret_cast<volatile int*>(sm + kOffFlags + 8);
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *v_tiles = 0;
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kTailReady) cnt = 2;
      if (i == kSFree0 || i == kSFree0 + 1 || i == kPReady0 || i == kPReady0 + 1 || i == kOFree)
        cnt = 2 * kSoftmaxWarps;
      if (i == kRed0 || i == kRed0 + 1 || i == kSum || i == kQRed) cnt = kSoftmaxWarps;
      // all 8 softmax warps of both CTAs: split the query (e4m3), store its
      // TMEM part (bf16)
      if (i == kQReady) cnt = 2 * kSoftmaxWarps;
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
    // streams (K mostly from DRAM, V mostly from L2, where the K copies of
    // the same tokens left it) run concurrently.  Each copy of both CTAs
    // completes on the even CTA's full barrier of its slot, where the even
    // CTA's producer announces the bytes of both (the odd CTA only issues
    // its copies: an arrive at cluster scope per slot would cost a fence
    // each).  An fp8 cache is copied as its e4m3 codes, which the MMAs read
    // as they are.
    const bool is_k = warp == 0;
    int rp = 0;            // slots of this ring used so far
    int tail_uses = 0;
    bool ok = true;
    int q_units = 0;       // query loads issued
    const int vbox = P >= kVChunkTok ? kVChunkTok : 16;
    const int nslots = is_k ? kKSlots : kVSlots;
    const int empty0 = is_k ? kKEmpty0 : kVEmpty0;
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
      if constexpr (kFp8) {
        // this CTA's query lands here; the softmax warps split it into e4m3
        // terms
        if (lane == 0) mbar_arrive_expect_tx(bar(base, kQLand), 9 * kQPanel);
        __syncwarp();
        if (lane < 9) {
          const int row = v.req * H + 64 * rank;   // rows past the batch are zero-filled
          if (lane < 8)
            tma_load_2d(base + kOffQ + lane * kQPanel, &maps.q_nope, 64 * lane, row, bar(base, kQLand));
          else
            tma_load_2d(base + kOffQ + 8 * kQPanel, &maps.q_pe, 0, row, bar(base, kQLand));
        }
        return true;
      }
      // bf16: the query's dims [0, 320) into shared memory (the rest goes to
      // TMEM, loaded by the softmax warps)
      if (lane == 0 && rank == 0) mbar_arrive_expect_tx(bar(base, kQFull), 2 * kQSmemPanels * kQPanel);
      __syncwarp();
      if (lane < kQSmemPanels) {
        const int row = v.req * H + 64 * rank;   // rows past the batch are zero-filled
        tma_load_2d_pair(base + kOffQ + lane * kQPanel, &maps.q_nope, 64 * lane, row,
                         map_to_rank(bar(base, kQFull), lead));
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
      // a panel row: 64 dims, 128 bytes (bf16) or 64 (e4m3)
      constexpr int row_bytes = kFp8 ? 64 : 128;
      // lane -> (panel jj of the slot, page box b): lanes [0, np * nbox)
      const int b = lane % max(nbox, 1), jj = lane / max(nbox, 1);
      const int page = __shfl_sync(0xffffffffu, pages, min(pb + b, 31));
      for (int j0 = 0; j0 < 9; j0 += kKPanelsPerSlot) {
        const int np = min(kKPanelsPerSlot, 9 - j0);   // panels j0 .. j0 + np - 1 in this slot
        int slot;
        if (!(ok = next_slot(slot))) return false;
        const uint32_t full = map_to_rank(bar(base, kKFull0 + slot), lead);
        if (lane == 0 && rank == 0)
          mbar_arrive_expect_tx(bar(base, kKFull0 + slot), np * nbox_both * P * row_bytes);
        __syncwarp();
        if (lane < np * nbox) {
          const int j = j0 + jj;
          const uint32_t dst = base + kOffKRing + slot * kKSlotBytes + jj * kPanelBytes + b * P * row_bytes;
          if (j < 8)
            tma_load_2d_pair(dst, &maps.ckv_k, 64 * j, page * P, full);
          else
            tma_load_2d_pair(dst, &maps.kpe_k, 0, page * P, full);
        }
      }
      return true;
    };
    auto emit_v = [&](const WorkUnit& v, int i, int pages, int vt) -> bool {
      const int tok0 = v.tok_begin + i * kT;
      for (int c = 0; c < kChunksPerTile; ++c) {
        const int t = tok0 + kVChunkTok * c;
        const int rows = min(kVChunkTok, v.tok_end - t);
        if (rows <= 0) break;
        int slot;
        if (!(ok = next_slot(slot))) return false;
        const uint32_t full = map_to_rank(bar(base, kVFull0 + slot), lead);
        if (!kFp8 && lane == 0 && c > 0) *v_tiles = 8 * vt + c;   // chunks before this one issued
        if (stalled()) continue;
        // one copy: vbox rows of kVPanels panels (128-byte rows), this CTA's
        // 256 dims
        const int ncopy = (rows + vbox - 1) / vbox;
        const int tb = t + vbox * min(lane, ncopy - 1);
        const int page = __shfl_sync(0xffffffffu, pages, (tb - tok0) / P);
        const int copy_bytes = vbox * kVPanels * 128;
        const uint32_t dst = base + kOffVRing + slot * kVSlotBytes + lane * copy_bytes;
        if (rows == kVChunkTok) {
          if (lane == 0 && rank == 0) mbar_arrive_expect_tx(bar(base, kVFull0 + slot), 2 * ncopy * copy_bytes);
          __syncwarp();
          if (lane < ncopy) tma_load_3d_pair(dst, &maps.ckv_v, 0, page * P + (tb % P), kVPanels * rank, full);
        } else {
          // last chunk of a request: rows past kv_len may hold anything (even
          // NaN) and p = 0 does not cancel NaN; copy locally, zero those
          // rows, then release the slot to the issuer
          const uint32_t tail = bar(base, kTail);
          if (lane == 0) mbar_arrive_expect_tx(tail, ncopy * copy_bytes);
          __syncwarp();
          if (lane < ncopy) tma_load_3d(dst, &maps.ckv_v, 0, page * P + (tb % P), kVPanels * rank, tail);
          if (!(ok = mbar_wait_warp(tail, tail_uses & 1, abort_flag))) return false;
          unsigned char* sv = sm + kOffVRing + slot * kVSlotBytes;
          // 16-byte chunks of the rows past the end: 8 per panel row
          for (int q = lane; q < (kVChunkTok - rows) * kVPanels * 8; q += 32) {
            const int rr = rows + q / (kVPanels * 8), pnl = (q % (kVPanels * 8)) >> 3, c16 = q & 7;
            const int off = vbox == kVChunkTok ? pnl * (kVChunkTok * 128) + rr * 128
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
            mbar_arrive_remote(map_to_rank(bar(base, kTailReady), lead));
          }
          ++tail_uses;
        }
      }
      return true;
    };
    int t = 0;   // tiles of this CTA so far
    for (int ui = u0; ui < u1 && ok; ++ui) {
      const WorkUnit v = a.units[ui];
      const int n = tiles_of(v);
      for (int i = 0; i < n && ok; ++i, ++t) {
        const int pages = tile_pages(v, i);
        if (is_k) {
          if (i == 0 && !emit_q(v)) break;
          // at most kKLeadChunks V chunks ahead of the V copies (bounded wait)
          if (!kFp8 && 8 * t > kKLeadChunks) {
            const uint64_t t0 = globaltimer_ns();
            while (*v_tiles < 8 * t - kKLeadChunks) {
              if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                ok = false;
                break;
              }
              __nanosleep(64);
            }
            __syncwarp();
            if (!(ok = __all_sync(0xffffffffu, ok))) break;
          }
          if (!emit_k(v, i, pages)) break;
        } else {
          if (!emit_v(v, i, pages, t)) break;
          __syncwarp();
          if (!kFp8 && lane == 0) *v_tiles = 8 * (t + 1);   // a short tile counts as 8 chunks
        }
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
  } else if ((warp == 1 || warp == kPvIssuerWarp) && rank == 0) {
    // ================= MMA issuers (even CTA, whole warp, lane 0 issues) =================
    // Warp 1 issues the QK products of every tile, panel by panel from the K
    // ring; warp 11 the PV products, chunk by chunk from the V ring, once
    // the tile's P is written in both CTAs.  Two issuers, because an issuing
    // thread cannot run ahead of the tensor pipe: the waits and commits of
    // one overlap the other's MMAs.
    const uint32_t issue = lane == 0;
    bool ok = true;
    if (warp == 1) {
      constexpr uint32_t id_qk = kFp8 ? idesc_e4m3_f32(128, 256, false, false) : idesc_bf16_f32(128, 256, false, false);
      const uint64_t q_desc0 = smem_desc(base + kOffQ, 16, 1024, kSw128);
      // K panels: 128-byte rows, 128-byte swizzle (bf16) or 64-byte rows and
      // swizzle (e4m3); 8-row groups 1024 or 512 bytes apart
      const uint64_t k_desc0 = kFp8 ? smem_desc(base + kOffKRing, 16, 512, kSw64)
                                    : smem_desc(base + kOffKRing, 16, 1024, kSw128);
      int kc = 0, g = 0, unit_k = 0;
      for (int ui = u0; ui < u1 && ok; ++ui, ++unit_k) {
        const WorkUnit v = a.units[ui];
        const int n = tiles_of(v);
        // the unit's query: split into e4m3 terms in both CTAs (fp8), or its
        // shared-memory part copied and its TMEM part stored (bf16)
        if ((kFp8 || kQTmem) && !(ok = mbar_wait_cl_warp(bar(base, kQReady), unit_k & 1, abort_flag))) break;
        if (!kFp8 && !(ok = mbar_wait_warp(bar(base, kQFull), unit_k & 1, abort_flag))) break;
        for (int i = 0; i < n && ok; ++i, ++g) {
          // the S buffer this tile writes was read by the softmax
          if (kSBufs == 2 && g >= 2 &&
              !(ok = mbar_wait_cl_warp(bar(base, kSFree0 + (g & 1)), ((g - 2) >> 1) & 1, abort_flag)))
            break;
          if (kSBufs == 1 && g >= 1 && !(ok = mbar_wait_cl_warp(bar(base, kSFree0), (g - 1) & 1, abort_flag)))
            break;
          tc_fence_after();
          const uint32_t d = tmem + kColS + 128 * (kSBufs == 2 ? (g & 1) : 0);
          for (int j0 = 0; j0 < 9; j0 += kKPanelsPerSlot, ++kc) {
            const int slot = kc % kKSlots;
            const uint32_t par = (kc / kKSlots) & 1;
            if (!(ok = mbar_wait_warp(bar(base, kKFull0 + slot), par, abort_flag))) break;
            tc_fence_after();
            for (int j = j0; j < j0 + kKPanelsPerSlot && j < 9; ++j) {
              const uint64_t adesc = q_desc0 + static_cast<uint64_t>((j * kQPanel) >> 4);
              const uint64_t bdesc =
                  k_desc0 + static_cast<uint64_t>((slot * kKSlotBytes + (j - j0) * kPanelBytes) >> 4);
              if constexpr (kFp8) {
                // dims [64 j + 32 kk, + 32): the query's hi codes at byte 32 kk
                // of its row, its lo codes at 64 + 32 kk, the K codes at 32 kk
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                  const uint64_t b = bdesc + static_cast<uint64_t>(kk * 2);
                  mma_pair_e4m3(d, adesc + static_cast<uint64_t>(kk * 2), b, id_qk, (j | kk) != 0, issue);
                  mma_pair_e4m3(d, adesc + static_cast<uint64_t>(4 + kk * 2), b, id_qk, 1u, issue);
                }
              } else if (j < kQSmemPanels) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_pair(d, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2), id_qk,
                           (j | kk) != 0, issue);
              } else {
                // dims [64 j, 64 j + 64) of the query from TMEM: 8 columns per
                // 16-dim K step
                const uint32_t a_t = tmem + kColQT + (64 * j - kQTDim0) / 2;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_pair_ts(d, a_t + 8 * kk, bdesc + static_cast<uint64_t>(kk * 2), id_qk, 1u, issue);
              }
            }
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
      constexpr uint32_t id_pv = kFp8 ? idesc_e4m3_f32(128, 256, false, true) : idesc_bf16_f32(128, 256, false, true);
      const uint64_t p_desc0 = smem_desc(base + kOffP, 16, 1024, kSw128);
      const bool v32 = P >= kVChunkTok;
      // V chunks, MN-major: panels of 128-byte rows (64 bf16 or 128 e4m3
      // dims), 128-byte swizzle, 8-row groups 1024 bytes apart
      const uint64_t v_desc0 = smem_desc(base + kOffVRing, v32 ? 4096 : 2048, 1024, kSw128);
      const uint32_t v_kstep = v32 ? 2048 : 8192, v_block = v32 ? 8192 : 4096;
      int vc = 0, g = 0, unit_k = 0;
      for (int ui = u0; ui < u1 && ok; ++ui, ++unit_k) {
        const WorkUnit v = a.units[ui];
        const int n = tiles_of(v);
        // the first PV of a unit overwrites O: the previous epilogue must be done
        if (unit_k > 0 && !(ok = mbar_wait_cl_warp(bar(base, kOFree), (unit_k - 1) & 1, abort_flag))) break;
        for (int i = 0; i < n && ok; ++i, ++g) {
          if (!(ok = mbar_wait_cl_warp(bar(base, kPReady0 + (g & 1)), (g >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          const int valid = min(kT, v.tok_end - (v.tok_begin + i * kT));
          const int nch = (valid + kVChunkTok - 1) / kVChunkTok;
          const uint32_t pbuf = (g % kPBufs) * kPBuf;
          for (int c = 0; c < nch; ++c, ++vc) {
            const int slot = vc % kVSlots;
            const uint32_t par = (vc / kVSlots) & 1;
            if (!(ok = mbar_wait_warp(bar(base, kVFull0 + slot), par, abort_flag))) break;
            tc_fence_after();
            if constexpr (kFp8) {
              // tokens [32 c, 32 c + 32): P's hi codes at byte 32 (c & 1) of
              // the rows of token panel c / 2, its lo codes 64 bytes further;
              // V panel bb (128 dims) of the chunk for O columns [128 bb, ..)
              const uint64_t a_hi =
                  p_desc0 + static_cast<uint64_t>((pbuf + (c >> 1) * kPPanel + 32 * (c & 1)) >> 4);
#pragma unroll
              for (int bb = 0; bb < 2; ++bb) {
                const uint64_t bdesc =
                    v_desc0 + static_cast<uint64_t>((slot * kVSlotBytes + bb * kVChunkTok * 128) >> 4);
                mma_pair_e4m3(tmem + kColO + 128 * bb, a_hi, bdesc, id_pv, (i == 0 && c == 0) ? 0u : 1u, issue);
                mma_pair_e4m3(tmem + kColO + 128 * bb, a_hi + 4, bdesc, id_pv, 1u, issue);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const int t = kVChunkTok * c + 16 * kk;   // first token of the K step
                const uint64_t adesc =
                    p_desc0 + static_cast<uint64_t>((pbuf + (t >> 6) * kPPanel + (t & 63) * 2) >> 4);
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                  const uint64_t bdesc =
                      v_desc0 + static_cast<uint64_t>((slot * kVSlotBytes + kk * v_kstep + bb * v_block) >> 4);
                  mma_pair(tmem + kColO + 128 * bb, adesc, bdesc, id_pv, (i == 0 && c == 0 && kk == 0) ? 0u : 1u,
                           issue);
                }
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
  } else if (warp == 1 || warp == kPvIssuerWarp) {
    // odd CTA: no role (the even CTA issues the pair's MMAs)
  } else {
    // ================= softmax / epilogue (warps 2..9, both CTAs) =================
    const int sw = warp - kFirstSoftmaxWarp;
    const int q = warp & 3;                  // TMEM lane quadrant
    const int ch = sw >> 2;                  // S columns [64 ch, 64 ch + 64), O columns [128 ch, 128 ch + 128)
    const int hl = 32 * (q & 1) + lane;      // head within this CTA
    const int h = 64 * rank + hl;
    const int tq = q >> 1;                   // S: tokens [128 tq, 128 tq + 128) of the tile; O: dims [256 tq, ..)
    const int part = 2 * tq + ch;            // which of the head's four threads this is
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float c = prm.sm_scale * a.kv_scale * kLog2e;
    // several query tokens packed into the rows: this row's token j sees all
    // but the request's last q_len - 1 - j tokens (0 with one token per row)
    const int row_hide = prm.q_len > 1 && prm.heads_per_token > 0 && h < H
                             ? prm.q_len - 1 - h / prm.heads_per_token
                             : 0;
    float* red = reinterpret_cast<float*>(sm + kOffRed);
    float2* sums = reinterpret_cast<float2*>(sm + kOffSum);
    bool ok = true;
    // fp8: a unit's query, split into e4m3 terms by these warps -- the
    // first unit's at the start, every later unit's as soon as the previous
    // unit's last P is written (its query has landed by then or soon after:
    // it is loaded once the previous unit's last scores are done), so the
    // split overlaps that unit's last P . V and epilogue, and the next
    // scores can start meanwhile.  Returns false when a wait runs out; sets
    // cq_next to the score scale of this thread's head.
    float cq_next = c;
    auto split_query = [&](uint32_t parity) -> bool {
      // ---- the unit's query (this CTA's 64 heads) split in place into
      // e4m3 terms: row hl is scaled by 2^e so that its largest magnitude
      // lies in [2^7, 2^8) (then hi + lo is the scaled bf16 value exactly
      // down to magnitudes of 2^-2), and the scores by 2^-e.  Each 128-byte
      // row of a panel (64 bf16 dims) becomes the 64 hi codes followed by
      // the 64 lo codes of the same dims, in the same row (128-byte
      // swizzle).  The head's four threads take panels part, part + 4, ..
      // of its 9, whole rows, so no thread reads what another writes ----
      if (!mbar_wait_warp(bar(base, kQLand), parity, abort_flag)) return false;
      auto qchunk = [&](int pj, int k) -> uint4* {
        return reinterpret_cast<uint4*>(sm + kOffQ + pj * kQPanel + hl * 128 + ((k ^ (hl & 7)) << 4));
      };
      float mx = 0.f;
      for (int pj = part; pj < 9; pj += 4) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = *qchunk(pj, k);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int m = 0; m < 4; ++m)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[m] << 16)), fabsf(__uint_as_float(w[m] & 0xffff0000u))));
        }
      }
      float* qred = reinterpret_cast<float*>(sm + kOffQRed);
      qred[part * 64 + hl] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(base, kQRed));
      if (!mbar_wait_warp(bar(base, kQRed), parity, abort_flag)) return false;
      const float rm = fmaxf(fmaxf(qred[hl], qred[64 + hl]), fmaxf(qred[128 + hl], qred[192 + hl]));
      // rows of zeros (heads past H) keep e = 0
      int e = 0;
      if (rm > 0.f && rm < INFINITY) e = min(max(7 - (((__float_as_int(rm) >> 23) & 0xff) - 127), -100), 100);
      const float up = __int_as_float((127 + e) << 23);
      for (int pj = part; pj < 9; pj += 4) {
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = *qchunk(pj, k);
          w[4 * k] = v.x;
          w[4 * k + 1] = v.y;
          w[4 * k + 2] = v.z;
          w[4 * k + 3] = v.w;
        }
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {   // dims 4 m .. 4 m + 3
          uint32_t h01, l01, h23, l23;
          split_e4m3x2(__uint_as_float(w[2 * m] << 16) * up, __uint_as_float(w[2 * m] & 0xffff0000u) * up, h01,
                       l01);
          split_e4m3x2(__uint_as_float(w[2 * m + 1] << 16) * up, __uint_as_float(w[2 * m + 1] & 0xffff0000u) * up,
                       h23, l23);
          hi[m] = h01 | (h23 << 16);
          lo[m] = l01 | (l23 << 16);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          *qchunk(pj, k) = make_uint4(hi[4 * k], hi[4 * k + 1], hi[4 * k + 2], hi[4 * k + 3]);
          *qchunk(pj, 4 + k) = make_uint4(lo[4 * k], lo[4 * k + 1], lo[4 * k + 2], lo[4 * k + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) arrive_lead(bar(base, kQReady), rank);
      cq_next = c * __int_as_float((127 - e) << 23);
      return true;
    };
    // bf16: the query's dims [320, 576) of this thread's head (request req)
    // into TMEM columns [128, 256) of this thread's lane, where the QK MMAs
    // read them as A (column half ch: dims [320 + 128 ch, + 128)).  Every
    // row is held twice, in lanes hl and 64 + hl (quadrants q and q + 2 have
    // the same heads): an M = 128 pair MMA reads A row 64 r + l from lane l
    // for the D columns of this CTA's half of B and from lane 64 + l for the
    // other CTA's half.  The previous unit's QK MMAs read the same columns:
    // unless wait_parity < 0, wait for them (kQFree) first.  Returns false
    // when the wait runs out.
    auto load_query_tmem = [&](int req, int wait_parity) -> bool {
      uint32_t w0[32], w1[32];
      if (h < H) {
        const size_t row = static_cast<size_t>(req) * H + h;
        const uint4* src0 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_nope) +
                                                            row * kDCkv + kQTDim0 + 128 * ch);
        // ch 0: dims [320, 448) of q_nope; ch 1: [448, 512) of q_nope, then q_pe
        const uint4* src1 =
            ch == 0 ? src0 + 8 : reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_pe) + row * kDKpe);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v0 = src0[k], v1 = src1[k];
          w0[4 * k] = v0.x, w0[4 * k + 1] = v0.y, w0[4 * k + 2] = v0.z, w0[4 * k + 3] = v0.w;
          w1[4 * k] = v1.x, w1[4 * k + 1] = v1.y, w1[4 * k + 2] = v1.z, w1[4 * k + 3] = v1.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) w0[k] = w1[k] = 0u;
      }
      if (wait_parity >= 0 && !mbar_wait_warp(bar(base, kQFree), static_cast<uint32_t>(wait_parity), abort_flag))
        return false;
      tc_fence_after();
      tmem_st32(lane_addr + kColQT + 64 * ch, w0);
      tmem_st32(lane_addr + kColQT + 64 * ch + 32, w1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_lead(bar(base, kQReady), rank);
      return true;
    };
    int g = 0, unit_k = 0;
    for (int ui = u0; ui < u1 && ok; ++ui, ++unit_k) {
      const WorkUnit u = a.units[ui];
      const int n = tiles_of(u);
      if (kQTmem && unit_k == 0 && !(ok = load_query_tmem(u.req, -1))) break;
      float ref = 0.f;                       // the head's reference (the same in its four threads)
      float lx = 0.f, lr = 0.f;              // this thread's share of the row sums
      float cq = c;                          // score scale of this thread's head
      if constexpr (kFp8) {
        if (unit_k == 0 && !(ok = split_query(0))) break;
        cq = cq_next;
      }
      for (int i = 0; i < n && ok; ++i, ++g) {
        const bool first = i == 0;
        // ---- scores: this thread's head, 64 tokens ----
        if (!(ok = mbar_wait_warp(bar(base, kSFull0 + (g & 1)), (g >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        float y[64];
        float mx = -INFINITY;
        {
          uint32_t v0[32], v1[32];
          const uint32_t col = kColS + 128 * (kSBufs == 2 ? (g & 1) : 0) + 64 * ch;
          tmem_ld32(lane_addr + col, v0);
          tmem_ld32(lane_addr + col + 32, v1);
          tmem_ld_wait();
          const int row_end = min(u.tok_end, u.kv_len - row_hide);
          const int nvalid = row_end - (u.tok_begin + i * kT + kHalfT * tq + 64 * ch);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            y[j] = j < nvalid ? __uint_as_float(v0[j]) * cq : -INFINITY;
            y[32 + j] = 32 + j < nvalid ? __uint_as_float(v1[j]) * cq : -INFINITY;
          }
#pragma unroll
          for (int j = 0; j < 64; ++j) mx = fmaxf(mx, y[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_lead(bar(base, kSFree0 + (kSBufs == 2 ? (g & 1) : 0)), rank);
        // ---- the head's maximum over the tile (its four threads) ----
        float* rd = red + (g & 1) * 4 * 64;
        rd[part * 64 + hl] = mx;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(base, kRed0 + (g & 1)));
        if (!(ok = mbar_wait_warp(bar(base, kRed0 + (g & 1)), (g >> 1) & 1, abort_flag))) break;
        const float mt = fmaxf(fmaxf(rd[hl], rd[64 + hl]), fmaxf(rd[128 + hl], rd[192 + hl]));
        // the reference moves up only (alpha < 1): nothing is ever scaled up
        float alpha = 1.f;
        if (first) {
          ref = mt;
        } else if (mt > ref + (kFp8 ? kRescaleThresholdFp8 : kRescaleThreshold)) {
          alpha = exp2f(ref - mt);
          ref = mt;
        }
        // ---- p = 2^(y - reference) rounded to bf16, or 2^(y - reference)
        // * 2^5 as e4m3 hi + lo terms (this thread's 64 tokens: hi codes in
        // words 0..15, lo codes in words 16..31); row sums.  A packed row
        // with no visible token so far keeps the reference -inf and p = 0
        // (its y are all -inf; the exponent then uses 0) ----
        uint32_t pk[32];
        {
          const float rexp = ref == -INFINITY ? 0.f : ref;
          float sx = 0.f, sr = 0.f;
          if constexpr (kFp8) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const float p0 = fast_exp2(y[4 * m] - rexp) * kPScaleFp8, p1 = fast_exp2(y[4 * m + 1] - rexp) * kPScaleFp8;
              const float p2 = fast_exp2(y[4 * m + 2] - rexp) * kPScaleFp8;
              const float p3 = fast_exp2(y[4 * m + 3] - rexp) * kPScaleFp8;
              sx += (p0 + p1) + (p2 + p3);
              uint32_t h01, l01, h23, l23;
              sr += split_e4m3x2(p0, p1, h01, l01) + split_e4m3x2(p2, p3, h23, l23);
              pk[m] = h01 | (h23 << 16);
              pk[16 + m] = l01 | (l23 << 16);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float p0 = fast_exp2(y[2 * j] - rexp), p1 = fast_exp2(y[2 * j + 1] - rexp);
              sx += p0 + p1;
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
              const uint32_t w = *reinterpret_cast<const uint32_t*>(&b2);
              pk[j] = w;
              sr += __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
            }
          }
          lx = first ? sx : fmaf(lx, alpha, sx);
          lr = first ? sr : fmaf(lr, alpha, sr);
        }
        // ---- the P buffer free (PV of the tile that used it done); for a
        // rescale, also the previous tile's PV (O current) ----
        const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
        {
          const int tw = rescale ? g - 1 : g - kPBufs;
          if (tw >= 0 && !(ok = mbar_wait_warp(bar(base, kPvDone0 + (tw & 1)), (tw >> 1) & 1, abort_flag))) break;
        }
        tc_fence_after();
        if (rescale) {
          // this thread's 128 columns of O (its head), times alpha
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            const uint32_t col = kColO + 128 * ch + 32 * cc;
            tmem_ld32(lane_addr + col, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(lane_addr + col, o);
          }
          tmem_st_wait();
        }
        // ---- P row of this head over this thread's 64 tokens: one 128-byte
        // row of token panel 2 tq + ch (K-major, 128-byte swizzle; e4m3: the
        // 64 hi codes, then the 64 lo codes) ----
        {
          unsigned char* prow = sm + kOffP + (g % kPBufs) * kPBuf + part * kPPanel + hl * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(prow + ((k ^ (hl & 7)) << 4)) =
                make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_lead(bar(base, kPReady0 + (g & 1)), rank);
        }
      }
      if (!ok) break;
      if (kFp8 && ui + 1 < u1 && !(ok = split_query((unit_k + 1) & 1))) break;
      if (kQTmem && ui + 1 < u1 && !(ok = load_query_tmem(a.units[ui + 1].req, unit_k & 1))) break;
      // ================= epilogue of the unit =================
      {
        sums[part * 64 + hl] = make_float2(lx, lr);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(base, kSum));
        if (!(ok = mbar_wait_warp(bar(base, kSum), unit_k & 1, abort_flag))) break;
        float sx = 0.f, sr = 0.f;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const float2 s = sums[pp * 64 + hl];
          sx += s.x;
          sr += s.y;
        }
        // (e4m3 P carries the factor 2^5, in both sums)
        const float ls = (ref - (kFp8 ? kPOffsetFp8 : 0.f) + log2f(sx)) * kLn2;
        const float inv = sr > 0.f ? a.kv_scale / sr : 0.f;   // a row with no visible token: out 0
        const bool split = u.out_slot >= 0;
        if (part == 0 && h < H) {
          if (split)
            a.lse_part[lse_part_offset(u.out_slot, 0, h, H)] = ls;
          else
            a.lse[static_cast<size_t>(u.req) * H + h] = ls;
        }
        if (!(ok = mbar_wait_warp(bar(base, kPvDone0 + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        // O: this thread's head, dims [256 tq + 128 ch, + 128)
        const int d0 = kHalfT * 2 * tq + 128 * ch;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kColO + 128 * ch + 32 * cc, o);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * inv);
          if (h < H) {
            const int d = d0 + 32 * cc;
            if (split) {
#pragma unroll
              for (int j = 0; j < 4; ++j) st_global_v8(a.o_part + part_offset(u.out_slot, h, d + 8 * j, H), &o[8 * j]);
            } else if (kOutF32) {
              float* dst = static_cast<float*>(a.out) + (static_cast<size_t>(u.req) * H + h) * kDCkv + d;
#pragma unroll
              for (int j = 0; j < 4; ++j) st_global_v8(dst + 8 * j, &o[8 * j]);
            } else {
              uint32_t w[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const __nv_bfloat162 b2 =
                    __floats2bfloat162_rn(__uint_as_float(o[2 * j]), __uint_as_float(o[2 * j + 1]));
                w[j] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(u.req) * H + h) * kDCkv + d;
              st_global_v8(dst, &w[0]);
              st_global_v8(dst + 16, &w[8]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_lead(bar(base, kOFree), rank);
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
  }

  // On a device error some copies may still be in flight toward this CTA:
  // give them time to land before it leaves.
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
template <bool kOutF32, bool kFp8>
cudaError_t set_pair_attributes() {
  static bool done = false;   // set once, before any stream capture
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<kOutF32, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
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
  cudaError_t e = set_pair_attributes<true, false>();
  if (e == cudaSuccess) e = set_pair_attributes<false, false>();
  if (e == cudaSuccess) e = set_pair_attributes<true, true>();
  if (e == cudaSuccess) e = set_pair_attributes<false, true>();
  if (e != cudaSuccess) return e;
  // the instantiations share the launch shape and the shared-memory size
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(1, attr);
  int clusters = 0, clusters_fp8 = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, decode_pair_kernel<false, false>, &cfg);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters_fp8, decode_pair_kernel<false, true>, &cfg);
  if (e != cudaSuccess) return e;
  *workers = clusters < clusters_fp8 ? clusters : clusters_fp8;
  return cudaSuccess;
}

cudaError_t launch_decode_pair(const DecodeArgs& a, const PairMaps& maps, bool out_f32, bool kv_fp8,
                               cudaStream_t s) {
  cudaError_t e = kv_fp8 ? (out_f32 ? set_pair_attributes<true, true>() : set_pair_attributes<false, true>())
                         : (out_f32 ? set_pair_attributes<true, false>() : set_pair_attributes<false, false>());
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(a.n_workers, attr);
  cfg.stream = s;
  // a programmatic dependent launch: the grid is scheduled while the previous
  // kernel drains, and waits for it at its first instruction
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  if (kv_fp8)
    return out_f32 ? cudaLaunchKernelEx(&cfg, decode_pair_kernel<true, true>, a, maps)
                   : cudaLaunchKernelEx(&cfg, decode_pair_kernel<false, true>, a, maps);
  return out_f32 ? cudaLaunchKernelEx(&cfg, decode_pair_kernel<true, false>, a, maps)
                 : cudaLaunchKernelEx(&cfg, decode_pair_kernel<false, false>, a, maps);
}

}  // namespace mla
