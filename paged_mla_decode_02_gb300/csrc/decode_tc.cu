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
// host planner) is processed by a cluster of C CTAs (C = kTcCluster = 2; the
// same source builds C = 4).  CTA `rank` owns the output dims
// [512/C rank, 512/C (rank + 1)): 128 heads x 512 fp32 accumulators would
// fill all 512 TMEM columns of one SM.  The unit's 128-token tiles rotate
// over the cluster's CTAs: the owner of tile g (g mod C == rank) loads its K,
// computes S = Q K^T and the softmax, and sends P (bf16) with the tile's
// reference max and row sums to the other CTAs through distributed shared
// memory (bulk copies on three barriers: the row info, the first 64 tokens
// of P, the other 64, so the receiver applies the tile and starts P . V on
// the first half while the rest lands).  Every CTA then accumulates P . V over its
// own dims.  So every score tile is computed once.  The grid is persistent:
// one cluster per worker, walking its units.
//
// Per CTA (384 threads, 12 warps), for C = 2:
//   warp 0      K producer (own tiles): TMA loads of Q dims 0..319 (per
//               unit) and of the 9 K panels (64 dims x 128 tokens) of the
//               tile, page by page through kv_indices, into a 3-slot ring;
//   warp 1      allocates TMEM; lane 0 issues the QK MMAs (M=128 heads,
//               N=128 tokens, K=16) of own tiles into S;
//   warp 2      V producer (every tile): this CTA's 256 dims of ckv,
//               32 tokens (16 KB) at a time into a 3-slot ring; rows past the
//               end of a request are zeroed;
//   warps 3..10 softmax: two warps per 32 head rows (TMEM lane quadrant),
//               each owning 64 tokens of a tile (one P panel) and half of
//               this CTA's output dims.  For an own tile: drain S, row max over
//               the tile, lazy-rescaled exp2 (the reference max moves only
//               when a tile's max exceeds it by more than 2^8), P to local and
//               remote shared memory.  For every tile, in order: take its
//               reference (own, or received), rescale O in TMEM when the
//               reference moved, update the row sums, release it to PV.
//               Then the epilogue O / l, lse;
//   warp 11     lane 0 issues the PV MMAs (M=128, N=256 dims, K=16 tokens).
// TMEM columns: O [0, 256) | S [256, 384) | Q dims 320..575 as bf16 pairs
// [384, 512).  (C = 4: O 128 columns, Q dims 64..575 in TMEM, two P buffers,
// deeper rings; measured slower on the DeepSeek shape -- each owner then
// pushes three copies of P -- so C = 2 is the launched configuration.)
//
// Reference max of tile g (every CTA uses the value the owner sends): the
// owner takes the lazy update of the two latest references it has already
// applied, so no CTA's softmax waits on another's.  O and the
// row sums are kept relative to the reference of the last applied tile.
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

#ifdef MLA_STALL_TEST
// Test build only: when nonzero, CTA 0's V producer leaves out its
// g_stall_chunk-th copy (1-based), so the PV warp's wait for it runs out.
__device__ int g_stall_chunk;
#endif

constexpr int kT = kTileTc;                 // 128 tokens per tile
constexpr int kThreads = 384;
constexpr int kSoftmaxWarps = 8;
constexpr int kPvWarp = 11;
constexpr int kPanel = 128 * 128;           // 128 rows x 128 B (one 64-dim panel)
constexpr int kVChunkTok = kTcVChunkTok;    // tokens per V chunk (32: two PV MMAs)
static_assert(kVChunkTok == 16 || kVChunkTok == 32, "V chunk: one or two 16-token MMA slices");
constexpr int kVPanel = kVChunkTok * 128;   // 4 KB: 32 rows x 64 dims
// A tile's row info, per softmax warp: 32 heads x {ref max, lx, lr, -} (16 B);
// laid out [token half][head] so each warp's block is contiguous.
constexpr int kInfoRow = 16;
constexpr int kInfoBytes = 2 * 128 * kInfoRow;
constexpr int kRecvBytes = 2 * kPanel + kInfoBytes;   // P (both token halves) + info
constexpr int kBarBytes = 640;
constexpr uint32_t kTmemCols = 512;

// Layout for clusters of C CTAs (C = 2 or 4).  CTA `rank` owns output dims
// [512 / C * rank, 512 / C * (rank + 1)); its O accumulator takes 512 / C TMEM
// columns, S 128, and Q's upper dims the rest (as bf16 pairs); Q's lower
// dims stay in shared memory.  With four CTAs the freed TMEM takes all of Q
// but one panel, and the freed shared memory buys a second P buffer and
// deeper copy rings.
template <int C>
struct Cfg {
  static constexpr int kDims = kDCkv / C;                 // output dims per CTA
  static constexpr uint32_t kColO = 0, kColS = kDims, kColQ = kDims + 128;
  static constexpr int kQTmemPanels = (kTmemCols - kColQ) / 32;   // 64-dim Q panels in TMEM
  static constexpr int kQSmemPanels = 9 - kQTmemPanels;           // Q dims below, in smem
  static constexpr int kPBufs = C == 2 ? 1 : 2;           // P buffers (by tile parity when 2)
  static constexpr int kKSlots = C == 2 ? 3 : 5;
  static constexpr int kVPanels = kDims / 64;             // V panels per chunk (this CTA's dims)
  static constexpr int kVSlot = kVPanels * kVPanel;       // 16 KB (C = 2) or 8 KB (C = 4)
  static constexpr int kVSlots = C == 2 ? 3 : 6;
  // shared memory map (offsets from the 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  // P buffer b: P [128 x 128] bf16 (2 panels) followed by the tile's row
  // info, so one copy carries both to another CTA
  static constexpr int kPStride = kRecvBytes;
  static constexpr int kOffP = kOffQ + kQSmemPanels * kPanel;
  static constexpr int kOffK = kOffP + kPBufs * kPStride;
  static constexpr int kOffV = kOffK + kKSlots * kPanel;
  static constexpr int kOffXchg = kOffV + kVSlots * kVSlot;             // 128 x (lx, lr) x 2 halves
  static constexpr int kOffMaxX = kOffXchg + 128 * 16;                  // [own tile parity][half][128] maxima
  static constexpr int kOffBar = kOffMaxX + 2 * 2 * 128 * 4;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;         // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffBar % 8 == 0, "barrier alignment");
  static_assert(kPStride % 1024 == 0 && kOffP % 1024 == 0, "P buffers on swizzle-atom boundaries");
  static_assert(kQTmemPanels * 32 + kColQ == kTmemCols, "TMEM budget");
};

constexpr int kMaxKSlots = 5, kMaxVSlots = 6;   // ring barriers sized for the deepest rings
static_assert(Cfg<2>::kKSlots <= kMaxKSlots && Cfg<4>::kKSlots <= kMaxKSlots, "K ring");
static_assert(Cfg<2>::kVSlots <= kMaxVSlots && Cfg<4>::kVSlots <= kMaxVSlots, "V ring");

enum Bar {
  kQFull = 0, kQTmemFull, kQEmpty,
  kKFull0, kKEmpty0 = kKFull0 + kMaxKSlots,
  kVFull0 = kKEmpty0 + kMaxKSlots, kVEmpty0 = kVFull0 + kMaxVSlots, kVTail0 = kVEmpty0 + kMaxVSlots,
  kSFull = kVTail0 + kMaxVSlots, kSFree,
  kPFree0,          // 2, by tile parity: every CTA's PV of the tile done (its P buffer reusable)
  kPRecv0 = kPFree0 + 2,   // 2, by P buffer: a peer's row info for a tile it owns has landed
  kPReady0 = kPRecv0 + 2,  // 2, by tile parity: tile released to PV (O rescaled, P in place)
  kPvDone0 = kPReady0 + 2,   // 2, by tile parity: this CTA's PV of the tile completed
  kOFree = kPvDone0 + 2, kFinal, kFinalPv,
  kXchg0, kMaxX0 = kXchg0 + 4,   // 4, per lane quadrant: the two warps' row maxima posted
  kMergeB = kMaxX0 + 4,   // split unit: merge-or-publish decided (flag in shared memory)
  kPWritten,              // own tile: all 8 softmax warps wrote their P rows and row info
  kPRecvB0,               // 2, by P buffer: a peer's P token panel 1 has landed
  kPRecvP0 = kPRecvB0 + 2,  // 2, by P buffer: a peer's P token panel 0 has landed
  kKReady0 = kPRecvP0 + 2,  // kMaxKSlots, by K slot (fp8 cache): panel expanded to bf16
  kNumBars = kKReady0 + kMaxKSlots
};
static_assert(kNumBars * 8 + 16 + 4 * kMaxVSlots <= kBarBytes, "barrier area");

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P values stay below 2^8
// A tile applied with a reference more than kDropLog2 below the running one
// (its owner had not yet seen the previous tile's far larger maximum) weighs
// below 2^-(kDropLog2 - kRescaleThreshold) per token against the rows already
// summed, beneath fp32 resolution; moving O up to its reference instead
// could overflow.  Such a row keeps its state and its P row is zeroed.
constexpr float kDropLog2 = 64.0f;
constexpr int kMergeRegs = 8;               // split request slots whose weights stay in registers

template <int C>
__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + Cfg<C>::kOffBar + 8 * i; }

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

// Q dims above the shared-memory panels (64 * kQSmemPanels .. 575) of head row
// r into TMEM columns [kColQ, 512) of lane r: the remaining q_nope panels
// then q_pe, each 64 dims = 32 columns of packed bf16 pairs.  The warp of
// column half hc writes the first or the second half of those panels.
template <int C>
__device__ __forceinline__ void load_q_tmem(const DecodeArgs& a, int req, int r, int hc,
                                            uint32_t taddr) {
  using L = Cfg<C>;
  constexpr int kPer = L::kQTmemPanels / 2;
  const int H = a.num_heads;
  const bool ok = r < H;
  const size_t row = static_cast<size_t>(req) * H + (ok ? r : 0);
  const uint4* qn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_nope) +
                                                   row * kDCkv + 64 * L::kQSmemPanels);
  const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_pe) +
                                                   row * kDKpe);
#pragma unroll
  for (int p = kPer * hc; p < kPer * hc + kPer; ++p) {
    const uint4* src = p < L::kQTmemPanels - 1 ? qn + p * 8 : qp;
    uint32_t v[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x = ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
    }
    tmem_st32(taddr + L::kColQ + 32 * p, v);
  }
  tmem_st_wait();
}

__device__ __forceinline__ int tiles_of(const WorkUnit& u) { return (u.tok_end - u.tok_begin + kT - 1) / kT; }

// 32 consecutive dims of one output row: 32-byte stores when out is 32-byte
// aligned (rows then are too), else 16-byte stores.
template <bool kOutF32>
__device__ __forceinline__ void store_out_row32(void* out, size_t orow, int d0, const float (&v)[32],
                                                bool out32) {
  uint32_t w[32];
  if (kOutF32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(v[j]);
    float* dst = static_cast<float*>(out) + orow * kDCkv + d0;
    if (out32) {
#pragma unroll
      for (int j = 0; j < 4; ++j) st_global_v8(dst + 8 * j, &w[8 * j]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        reinterpret_cast<uint4*>(dst)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      w[e] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + orow * kDCkv + d0;
    if (out32) {
      st_global_v8(dst, &w[0]);
      st_global_v8(dst + 16, &w[8]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        reinterpret_cast<uint4*>(dst)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
  }
}

// fp8 (e4m3) caches: a copy lands as rows of 64 codes (64 bytes) in the upper
// half of a shared-memory slot, 64-byte swizzled (16-byte chunk c of row r at
// chunk c ^ ((r >> 1) & 3), every destination 512-byte aligned), and a warp
// expands it in place to the bf16 rows of the 128-byte-swizzled panel the
// MMA reads (chunk c of row r at chunk c ^ (r & 7)).  One lane per row: the
// 64-byte swizzle puts the 8 rows of each 8-lane phase on distinct banks
// for the reads, and the 128-byte one for the writes.  Each step reads its 32 rows before any lane
// writes: a bf16 row r covers the bytes of fp8 rows 2r - 128 and 2r - 127 of
// a 128-row panel (of the same or earlier steps), and for a V chunk bf16
// panel p covers fp8 panels 2p - 4 and 2p - 3 (of the same or earlier panels).
__device__ __forceinline__ void expand_row_fp8(unsigned char* dst_row, int r, const uint4 (&q)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 lo, hi;
    e4m3x16_to_bf16x16(q[k], lo, hi);
    *reinterpret_cast<uint4*>(dst_row + (((2 * k) ^ (r & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(dst_row + (((2 * k + 1) ^ (r & 7)) << 4)) = hi;
  }
}

// A K panel slot: 128 rows (tokens) of 64 dims.  Warp-wide.
__device__ __forceinline__ void expand_k_panel(unsigned char* slot, int lane) {
#pragma unroll 1
  for (int it = 0; it < 4; ++it) {
    const int r = 32 * it + lane;
    const uint4* src = reinterpret_cast<const uint4*>(slot + kPanel / 2 + 64 * r);
    uint4 q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = src[k ^ ((r >> 1) & 3)];
    __syncwarp();
    expand_row_fp8(slot + 128 * r, r, q);
    __syncwarp();
  }
}

// A V chunk slot: kPanels panels of kVChunkTok rows; rows >= rows_valid
// (past the request's last token) become zeros.  Warp-wide.
template <int kPanels>
__device__ __forceinline__ void expand_v_chunk(unsigned char* slot, int lane, int rows_valid) {
  static_assert(kVChunkTok == 32, "one row per lane");
#pragma unroll 1
  for (int p = 0; p < kPanels; ++p) {
    const uint4* src = reinterpret_cast<const uint4*>(slot + kPanels * kVPanel / 2 + p * (kVPanel / 2) + 64 * lane);
    uint4 q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = lane < rows_valid ? src[k ^ ((lane >> 1) & 3)] : make_uint4(0, 0, 0, 0);
    __syncwarp();
    expand_row_fp8(slot + p * kVPanel + 128 * lane, lane, q);
    __syncwarp();
  }
}

template <bool kOutF32, int C, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const DecodeArgs a, const __grid_constant__ TcMaps maps) {
  using L = Cfg<C>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(sm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kOffBar + kNumBars * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kOffBar + kNumBars * 8 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int worker = blockIdx.x / C;
  const int rank = static_cast<int>(cluster_ctarank());   // == blockIdx.x % C
  const PlanDev prm = *a.params;
  const int H = a.num_heads;
  const int P = prm.page_size;
  const int u0 = worker < prm.n_workers ? a.worker_ptr[worker] : 0;
  const int u1 = worker < prm.n_workers ? a.worker_ptr[worker + 1] : 0;

  // ---- setup ----
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kQTmemFull || i == kSFree || i == kPReady0 || i == kPReady0 + 1 || i == kOFree ||
          i == kPWritten)
        cnt = kSoftmaxWarps;
      if (i == kPFree0 || i == kPFree0 + 1) cnt = C;              // every CTA's PV commit
      if (i >= kXchg0 && i < kMergeB) cnt = 2;                    // kXchg*, kMaxX*
      mbar_init(bar_addr<C>(base, i), cnt);
    }
    fence_barrier_init();
  }
  if (warp >= 3 && warp < kPvWarp && H < 128) {
    // Q rows past num_heads are never written by TMA: make them zero once.
    const int t = threadIdx.x - 96;
    const int per_panel = (128 - H) * 8;
    for (int i = t; i < L::kQSmemPanels * per_panel; i += 32 * kSoftmaxWarps) {
      const int panel = i / per_panel, rem = i % per_panel;
      *reinterpret_cast<uint4*>(sm + L::kOffQ + panel * kPanel + (H + rem / 8) * 128 + (rem % 8) * 16) =
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
  cluster_sync_all();   // both CTAs' barriers initialised before any remote operation
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0) {
    // ================= K producer (own tiles) =================
    int kc = 0, g = 0, uidx = 0;
    bool ok = true;
    // fp8 cache: the even panels of a tile (j = 0, 2, .., 8) are expanded to
    // bf16 here, panel k once panel k + 1 has been issued (one behind: a
    // longer lag would chain the expansion of panel k behind the MMAs of
    // panel k - 1 through the ring), and every issued one before this warp
    // waits on anything the QK warp signals; the QK warp expands the odd
    // panels itself
    int kx = 0;   // next panel to expand
    auto expand_upto = [&](int end) {
      for (; kx < end && ok; ++kx) {
        if ((kx % 9) & 1) continue;
        const int slot = kx % L::kKSlots;
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kKFull0 + slot), (kx / L::kKSlots) & 1, abort_flag)))
          break;
        expand_k_panel(sm + L::kOffK + slot * kPanel, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr<C>(base, kKReady0 + slot));
      }
    };
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      if (kFp8) expand_upto(kc);
      if (uidx > 0 && ok && !(ok = mbar_wait_warp(bar_addr<C>(base, kQEmpty), (uidx - 1) & 1, abort_flag)))
        break;
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(bar_addr<C>(base, kQFull), L::kQSmemPanels * H * 128);
      __syncwarp();
      if (lane < L::kQSmemPanels)
        tma_load_2d(base + L::kOffQ + lane * kPanel, &maps.q_nope, 64 * lane, u.req * H,
                    bar_addr<C>(base, kQFull));
      for (int tok0 = u.tok_begin; tok0 < u.tok_end && ok; tok0 += kT, ++g) {
        if (g % C != rank) continue;
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
        for (int j = 0; j < 9; ++j, ++kc) {
          const int slot = kc % L::kKSlots;
          if (!(ok = mbar_wait_warp(bar_addr<C>(base, kKEmpty0 + slot), ((kc / L::kKSlots) & 1) ^ 1,
                                    abort_flag)))
            break;
          const uint32_t full = bar_addr<C>(base, kKFull0 + slot);
          constexpr int kRowBytes = kFp8 ? 64 : 128;   // one row of a panel as copied
          if (lane == 0) mbar_arrive_expect_tx(full, nbox * P * kRowBytes);
          __syncwarp();
          if (lane < nbox) {
            const uint32_t dst = base + L::kOffK + slot * kPanel + (kFp8 ? kPanel / 2 : 0) + lane * P * kRowBytes;
            if (j < 8)
              tma_load_2d(dst, &maps.ckv_k, 64 * j, row, full);
            else
              tma_load_2d(dst, &maps.kpe_k, 0, row, full);
          }
          if (kFp8) expand_upto(kc);
        }
      }
    }
    if (kFp8) expand_upto(kc);
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    if (lane == 0)   // drain: the copies this warp issued land before the CTA exits
      for (int k = 1; k <= L::kKSlots && k <= kc; ++k)
        mbar_wait_drain(bar_addr<C>(base, kKFull0 + (kc - k) % L::kKSlots), ((kc - k) / L::kKSlots) & 1);
    __syncwarp();
  } else if (warp == 2) {
    // ================= V producer (this CTA's 256 dims of ckv, every tile) =================
    // The page ids of a tile are read once (lane b: page b), one tile ahead,
    // so no chunk waits on a dependent load of kv_indices.
    auto tile_pages = [&](int ui, int i) -> int {
      const WorkUnit v = a.units[ui];
      const int tok0 = v.tok_begin + i * kT;
      const int nb = (min(tok0 + kT, v.tok_end) - tok0 + P - 1) / P;
      int page = 0;
      if (lane < nb) {
        page = a.kv_indices[v.page_base + tok0 / P + lane];
        if (page < 0 || page >= a.num_pages) {
          report_error(a.err, kErrBounds);
          page = 0;
        }
      }
      return page;
    };
    int vc = 0, vslot = 0;
    uint32_t vphase = 0;   // parity of the current pass over the ring
    bool ok = true;
    // fp8 cache: the even chunks of a tile are expanded to bf16 here (rows
    // past the request's end zeroed), chunk k once chunk k + 1 has been
    // issued (one behind, as for K); the PV warp expands the odd ones.  A chunk's valid row
    // count (and bit 16: odd in its tile) waits in shared memory, one entry
    // per slot.
    volatile int* vrows = reinterpret_cast<volatile int*>(sm + L::kOffBar + kNumBars * 8 + 16);
    int vx = 0;   // next chunk to expand
    auto expand_upto = [&](int end) {
      for (; vx < end && ok; ++vx) {
        const int slot = vx % L::kVSlots;
        const int info = vrows[slot];
        if (info >> 16) continue;
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kVFull0 + slot), (vx / L::kVSlots) & 1, abort_flag)))
          break;
        expand_v_chunk<L::kVPanels>(sm + L::kOffV + slot * L::kVSlot, lane, info);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr<C>(base, kVTail0 + slot));
      }
    };
    int pg_cur = u0 < u1 ? tile_pages(u0, 0) : 0;
    for (int ui = u0, i = 0; ui < u1 && ok;) {
      const WorkUnit u = a.units[ui];
      const int tok0 = u.tok_begin + i * kT;
      // next tile in the flattened sequence of this worker's tiles
      int ui2 = ui, i2 = i + 1;
      if (i2 >= tiles_of(u)) {
        ++ui2;
        i2 = 0;
      }
      const int pg_next = ui2 < u1 ? tile_pages(ui2, i2) : 0;
      for (int t = tok0; t < min(tok0 + kT, u.tok_end) && ok; t += kVChunkTok, ++vc) {
        const int slot = vslot;
        const uint32_t ph = vphase;
        if (++vslot == L::kVSlots) {
          vslot = 0;
          vphase ^= 1;
        }
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kVEmpty0 + slot), ph ^ 1, abort_flag))) break;
        // One 3-D copy per page run of the chunk brings this CTA's kVPanels
        // panels: pages of >= 32 rows give one 32-row copy (panels 4 KB apart),
        // 16-row pages two 16-row copies (panels 2 KB apart, the second copy
        // half a slot in).
        const int rows = min(kVChunkTok, u.tok_end - t);
        const int vbox = P >= kVChunkTok ? kVChunkTok : 16;   // rows of the V map's box
        const int ncopy = (rows + vbox - 1) / vbox;
        const uint32_t full = bar_addr<C>(base, kVFull0 + slot);
        constexpr int kRowBytes = kFp8 ? 64 : 128;   // one row of a panel as copied
        const uint32_t dst = base + L::kOffV + slot * L::kVSlot + (kFp8 ? L::kVSlot / 2 : 0);
#ifdef MLA_STALL_TEST
        const bool skip = g_stall_chunk != 0 && blockIdx.x == 0 && vc + 1 == g_stall_chunk;
#else
        constexpr bool skip = false;
#endif
        if (lane == 0 && !skip) {
          if (kFp8) vrows[slot] = rows | ((((t - tok0) / kVChunkTok) & 1) << 16);
          mbar_arrive_expect_tx(full, ncopy * vbox * L::kVPanels * kRowBytes);
        }
        __syncwarp();
        // lane c < ncopy issues copy c (lanes past it mirror the last one for the shuffle)
        const int tb = t + vbox * min(lane, ncopy - 1);
        const int page = __shfl_sync(0xffffffffu, pg_cur, (tb - tok0) / P);
        if (lane < ncopy && !skip)
          tma_load_3d(dst + lane * vbox * L::kVPanels * kRowBytes, &maps.ckv_v, 0, page * P + (tb % P),
                      L::kVPanels * rank, full);
        if (kFp8) {
          expand_upto(vc);
        } else if (rows < kVChunkTok) {
          // Last chunk of a request: rows past kv_len may hold anything (even
          // NaN), and P = 0 there does not cancel NaN.  Wait for the copy,
          // zero those rows, then release the chunk through kVTail.
          if (!(ok = mbar_wait_warp(full, ph, abort_flag))) break;
          constexpr int kRowChunks = L::kVPanels * 8;   // 16-byte pieces of one chunk row
          for (int q = lane; q < (kVChunkTok - rows) * kRowChunks; q += 32) {
            const int rr = rows + q / kRowChunks, pnl = (q % kRowChunks) >> 3, c16 = q & 7;
            const int off = vbox == kVChunkTok
                                ? pnl * kVPanel + rr * 128
                                : (rr >> 4) * (L::kVSlot / 2) + pnl * (kVPanel / 2) + (rr & 15) * 128;
            *reinterpret_cast<uint4*>(sm + L::kOffV + slot * L::kVSlot + off + c16 * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr<C>(base, kVTail0 + slot));
        }
      }
      if (!ok) break;
      pg_cur = pg_next;
      ui = ui2;
      i = i2;
    }
    if (kFp8) expand_upto(vc);
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    if (lane == 0)
      for (int k = 1; k <= L::kVSlots && k <= vc; ++k)
        mbar_wait_drain(bar_addr<C>(base, kVFull0 + (vc - k) % L::kVSlots), ((vc - k) / L::kVSlots) & 1);
    __syncwarp();
  } else if (warp == 1) {
    // ================= QK issuer (own tiles; whole warp converged, lane 0 issues) =================
    constexpr uint32_t id_qk = idesc_bf16_f32(128, kT, false, false);
    const uint32_t issue = lane == 0;
    const uint64_t q_desc0 = smem_desc(base + L::kOffQ, 16, 1024, kSw128);
    const uint64_t k_desc0 = smem_desc(base + L::kOffK, 16, 1024, kSw128);
    int g = 0, gl = 0, uidx = 0, kslot = 0;
    uint32_t kphase = 0;
    uint32_t ready_par = 0;   // fp8: per K slot, parity of its next kKReady phase
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = tiles_of(u);
      if (!(ok = mbar_wait_warp(bar_addr<C>(base, kQFull), uidx & 1, abort_flag) &&
                 mbar_wait_warp(bar_addr<C>(base, kQTmemFull), uidx & 1, abort_flag)))
        break;
      tc_fence_after();
      for (int i = 0; i < n && ok; ++i, ++g) {
        if (g % C != rank) continue;
        // S is single-buffered: the softmax drains it to registers right away.
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kSFree), (gl & 1) ^ 1, abort_flag))) break;
        tc_fence_after();
        for (int j = 0; j < 9; ++j) {
          const int slot = kslot;
          const uint32_t ph = kphase;
          if (++kslot == L::kKSlots) {
            kslot = 0;
            kphase ^= 1;
          }
          if (kFp8 && (j & 1)) {
            // fp8, odd panel: expanded here once its copy has landed
            if (!(ok = mbar_wait_warp(bar_addr<C>(base, kKFull0 + slot), ph, abort_flag))) break;
            expand_k_panel(sm + L::kOffK + slot * kPanel, lane);
            fence_proxy_async_smem();
            __syncwarp();
          } else if (kFp8) {
            // fp8, even panel: the K producer expanded it (kKReady counts even panels only)
            if (!(ok = mbar_wait_warp(bar_addr<C>(base, kKReady0 + slot), (ready_par >> slot) & 1, abort_flag)))
              break;
            ready_par ^= 1u << slot;
          } else if (!(ok = mbar_wait_warp(bar_addr<C>(base, kKFull0 + slot), ph, abort_flag))) {
            break;
          }
          const uint64_t bdesc = k_desc0 + static_cast<uint64_t>((slot * kPanel) >> 4);
          if (j < L::kQSmemPanels) {
            const uint64_t adesc = q_desc0 + static_cast<uint64_t>((j * kPanel) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + L::kColS, adesc + static_cast<uint64_t>((kk * 32) >> 4),
                     bdesc + static_cast<uint64_t>((kk * 32) >> 4), id_qk, (j | kk) != 0, issue);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + L::kColS, tmem + L::kColQ + (j - L::kQSmemPanels) * 32 + kk * 8,
                     bdesc + static_cast<uint64_t>((kk * 32) >> 4), id_qk, 1u, issue);
          }
          mma_commit(bar_addr<C>(base, kKEmpty0 + slot), issue);
        }
        if (!ok) break;
        mma_commit(bar_addr<C>(base, kSFull), issue);
        ++gl;
      }
      if (!ok) break;
      mma_commit(bar_addr<C>(base, kQEmpty), issue);   // Q of this unit no longer read
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    // Drain: all MMAs issued by this warp complete before TMEM is freed.
    mma_commit(bar_addr<C>(base, kFinal), issue);
    if (lane == 0) mbar_wait_drain(bar_addr<C>(base, kFinal), 0);
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ================= PV issuer (every tile; lane 0 issues) =================
    constexpr uint32_t id_pv = idesc_bf16_f32(128, L::kDims, false, true);
    const uint32_t issue = lane == 0;
    const uint64_t p_desc0 = smem_desc(base + L::kOffP, 16, 1024, kSw128);
    // V chunk layout (see the V producer): panels 4 KB apart and the two
    // 16-token slices 2 KB apart, or for 16-row pages 2 KB and 8 KB
    const bool v32 = P >= kVChunkTok;
    const uint64_t v_desc0 = smem_desc(base + L::kOffV, v32 ? kVPanel : kVPanel / 2, 1024, kSw128);
    const uint32_t v_kstep = v32 ? 16 * 128 : L::kVSlot / 2;
    int g = 0, uidx = 0, vslot = 0;
    uint32_t vphase = 0;
    uint32_t tail_par = 0;   // per V slot: parity of its next tail-chunk release
    uint32_t recvb_par = 0;  // per P buffer: parity of its next token-panel-1 receive
    uint32_t recvp_par = 0;  // per P buffer: parity of its next token-panel-0 receive
    bool ok = true;
    const volatile int* merge_flag = reinterpret_cast<const volatile int*>(sm + L::kOffBar + kNumBars * 8 + 8);
    // After unit v's epilogue released O (kOFree): if v is a split unit that
    // does not merge, its stored share becomes visible GPU-wide and is counted
    // as published (the fence orders the softmax warps' stores, seen through
    // the barrier, before the count).
    auto publish = [&](const WorkUnit& v) {
      if (v.n_slots > 0 && *merge_flag == 0 && lane == 0) {
        __threadfence();
        atomicAdd(a.counters + 8 * v.req + 4 + rank, 1);
      }
    };
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = tiles_of(u);
      // the first PV of a unit overwrites O: the previous epilogue must be done
      if (uidx > 0) {
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kOFree), (uidx - 1) & 1, abort_flag))) break;
        publish(a.units[ui - 1]);
      }
      for (int i = 0; i < n && ok; ++i, ++g) {
        const int valid = min(kT, u.tok_end - (u.tok_begin + i * kT));
        const int nch = (valid + kVChunkTok - 1) / kVChunkTok;
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kPReady0 + (g & 1)), (g >> 1) & 1, abort_flag)))
          break;
        tc_fence_after();
        const uint64_t p_desc = p_desc0 + static_cast<uint64_t>(((L::kPBufs == 2 ? (g & 1) : 0) * L::kPStride) >> 4);
        // A received tile's P arrives in two token panels after its row info
        // (which the softmax warps waited for): each is waited for before the
        // first MMA that reads it.
        const int bb = L::kPBufs == 2 ? (g & 1) : 0;
        bool have_b = g % C == rank;
        if (g % C != rank) {
          if (!(ok = mbar_wait_warp(bar_addr<C>(base, kPRecvP0 + bb), (recvp_par >> bb) & 1, abort_flag))) break;
          recvp_par ^= 1u << bb;
        }
        for (int c = 0; c < nch; ++c) {
          if (!have_b && c * kVChunkTok >= 64) {
            if (!(ok = mbar_wait_warp(bar_addr<C>(base, kPRecvB0 + bb), (recvb_par >> bb) & 1, abort_flag))) break;
            recvb_par ^= 1u << bb;
            have_b = true;
          }
          const int slot = vslot;
          const uint32_t ph = vphase;
          if (++vslot == L::kVSlots) {
            vslot = 0;
            vphase ^= 1;
          }
          if (kFp8 && (c & 1)) {
            // fp8, odd chunk of the tile: expanded here once its copy has landed
            if (!(ok = mbar_wait_warp(bar_addr<C>(base, kVFull0 + slot), ph, abort_flag))) break;
            expand_v_chunk<L::kVPanels>(sm + L::kOffV + slot * L::kVSlot, lane,
                                        min(kVChunkTok, valid - kVChunkTok * c));
            fence_proxy_async_smem();
            __syncwarp();
          } else if (kFp8 || (c == nch - 1 && (valid % kVChunkTok) != 0)) {
            if (!(ok = mbar_wait_warp(bar_addr<C>(base, kVTail0 + slot), (tail_par >> slot) & 1,
                                      abort_flag)))
              break;
            tail_par ^= 1u << slot;
          } else if (!(ok = mbar_wait_warp(bar_addr<C>(base, kVFull0 + slot), ph, abort_flag))) {
            break;
          }
#pragma unroll
          for (int kk = 0; kk < kVChunkTok / 16; ++kk) {
            const int tok = kVChunkTok * c + 16 * kk;   // first token of this MMA's K slice
            mma_ss(tmem + L::kColO,
                   p_desc + static_cast<uint64_t>(((tok >> 6) * kPanel + (tok & 63) * 2) >> 4),
                   v_desc0 + static_cast<uint64_t>((slot * L::kVSlot + kk * v_kstep) >> 4), id_pv,
                   (i == 0 && c == 0 && kk == 0) ? 0u : 1u, issue);
          }
          mma_commit(bar_addr<C>(base, kVEmpty0 + slot), issue);
        }
        if (!ok) break;
        if (!have_b) {
          if (!(ok = mbar_wait_warp(bar_addr<C>(base, kPRecvB0 + bb), (recvb_par >> bb) & 1, abort_flag))) break;
          recvb_par ^= 1u << bb;
        }
        mma_commit(bar_addr<C>(base, kPvDone0 + (g & 1)), issue);
        // the tile's P buffer is reusable once every CTA's PV of the tile is done
        mma_commit_mc(bar_addr<C>(base, kPFree0 + (g & 1)), static_cast<uint16_t>((1u << C) - 1), issue);
      }
    }
    if (ok && uidx > 0) {   // the last unit's share
      if ((ok = mbar_wait_warp(bar_addr<C>(base, kOFree), (uidx - 1) & 1, abort_flag)))
        publish(a.units[u1 - 1]);
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
    mma_commit(bar_addr<C>(base, kFinalPv), issue);
    if (lane == 0) mbar_wait_drain(bar_addr<C>(base, kFinalPv), 0);
    __syncwarp();
  } else {
    // ================= softmax / epilogue (warps 3..10) =================
    static_assert(kPvWarp == 3 + kSoftmaxWarps, "warp roles");
    const int quad = warp & 3;
    const int hc = (warp - 3) >> 2;                 // token half / P panel / O column half
    const int r = quad * 32 + lane;                 // head row == TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    // scores on the stored cache values: kv_scale folds the fp8 dequantisation
    // in (1 for a bf16 cache); the epilogue multiplies O by it too
    const float c = prm.sm_scale * a.kv_scale * kLog2e;
    const float pad = c >= 0.f ? -INFINITY : INFINITY;   // neutral for the max of s * c
    // P of tile g lives in buffer g & 1 in both CTAs; this row's chunk area:
    const uint32_t p_off = hc * kPanel + (r >> 3) * 1024 + (r & 7) * 128;
    const int pswz = r & 7;
    const uint32_t info_off = (hc * 128 + r) * kInfoRow;
    constexpr int kCh = L::kDims / 64;              // 32-dim O chunks per warp
    int g = 0, gl = 0, uidx = 0, nsplit = 0;
    uint32_t recv_par = 0;                          // bit b: parity of P buffer b's next receive
    bool ok = true;
    volatile int* merge_flag = reinterpret_cast<volatile int*>(sm + L::kOffBar + kNumBars * 8 + 8);
    // Requests without tokens: out = 0, lse = -inf (merge entries with no
    // slots, dealt round-robin over the workers).
    if (worker < prm.n_workers && r < H) {
      for (int e = worker; e < prm.n_merge; e += prm.n_workers) {
        const MergeEntry me = a.merge[e];
        if (me.n_slots != 0) continue;
        const size_t orow = static_cast<size_t>(me.req) * H + r;
        const int d0 = L::kDims * rank + (L::kDims / 2) * hc;
        uint4* dst = kOutF32 ? reinterpret_cast<uint4*>(static_cast<float*>(a.out) + orow * kDCkv + d0)
                             : reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * kDCkv + d0);
#pragma unroll 4
        for (int j = 0; j < (kOutF32 ? L::kDims / 8 : L::kDims / 16); ++j) dst[j] = make_uint4(0, 0, 0, 0);
        if (rank == 0 && hc == 0) a.lse[orow] = -INFINITY;
      }
    }
    if (u0 < u1) {
      load_q_tmem<C>(a, a.units[u0].req, r, hc, lane_addr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr<C>(base, kQTmemFull));
    }
    for (int ui = u0; ui < u1 && ok; ++ui, ++uidx) {
      const WorkUnit u = a.units[ui];
      const int n = tiles_of(u);
      const int g0 = g;
      // split request: the unit counts itself one tile before its last (near
      // its end, so the last to count is about the last to finish); the result
      // is first needed a tile later, which hides the atomic's latency
      int end_count = 0;
      const int i_count = max(n - 2, 0);
      // references: m_last = of the last applied tile, m_prev = the one before
      float m_last = -INFINITY, m_prev = -INFINITY;
      float lx = 0.f, lr = 0.f;                        // this warp's token half
      // the own tile computed but not yet applied
      float own_m = -INFINITY, own_lx = 0.f, own_lr = 0.f;
      for (int i = 0; i <= n && ok; ++i) {
        const bool own_now = i < n && (g0 + i) % C == rank;
        if (u.n_slots > 0 && warp == 3 && lane == 0) {
          if (i == i_count) end_count = atomicAdd(a.counters + 8 * u.req + rank, 1);
          if (i == i_count + 1 && end_count == u.n_slots - 1) {
            // this unit will merge: bring the other units' shares of this
            // CTA's dims (contiguous kDims / 8 x H x 32 bytes per slot) into L2
            constexpr int kGroups = L::kDims / 8;
            for (int k = u.slot0; k < u.slot0 + u.n_slots; ++k) {
              if (k == u.out_slot) continue;
              const char* src = reinterpret_cast<const char*>(a.o_part + part_offset(k, 0, L::kDims * rank, H));
              for (int off = 0; off < kGroups * H * 32; off += 32768)
                bulk_prefetch_l2(src + off, min(32768, kGroups * H * 32 - off));
            }
          }
        }
        uint32_t pk[32];
        if (own_now) {
          // ---------- own tile g0 + i: scores -> P (registers) ----------
          const int gg = g0 + i;
          if (!(ok = mbar_wait_warp(bar_addr<C>(base, kSFull), gl & 1, abort_flag))) break;
          tc_fence_after();
          const int valid = min(kT, u.tok_end - (u.tok_begin + i * kT));
          const int vb = 64 * hc;                      // first token of this warp's half
          float s[64];
          {
            uint32_t v0[32], v1[32];
            tmem_ld32(lane_addr + L::kColS + vb, v0);
            tmem_ld32(lane_addr + L::kColS + vb + 32, v1);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              s[j] = __uint_as_float(v0[j]);
              s[32 + j] = __uint_as_float(v1[j]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr<C>(base, kSFree));
          ++gl;

          // max (min when c < 0) of s over this warp's valid tokens, then
          // combined with the partner warp's half of the row
          float hmx;
          {
            float t[32];
            if (valid >= vb + 64) {
#pragma unroll
              for (int j = 0; j < 32; ++j) t[j] = c >= 0.f ? fmaxf(s[j], s[32 + j]) : fminf(s[j], s[32 + j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float lo = vb + j < valid ? s[j] : pad;
                const float hi = vb + 32 + j < valid ? s[32 + j] : pad;
                t[j] = c >= 0.f ? fmaxf(lo, hi) : fminf(lo, hi);
              }
            }
            hmx = c >= 0.f ? tree_max(t) : tree_min(t);
          }
          float* mx_slot = reinterpret_cast<float*>(sm + L::kOffMaxX) + ((gl & 1) * 2 + hc) * 128 + r;
          *mx_slot = hmx;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr<C>(base, kMaxX0 + quad));
          // phase k of this barrier: both warps of the quadrant posted own tile k
          if (!(ok = mbar_wait_warp(bar_addr<C>(base, kMaxX0 + quad), (gl - 1) & 1, abort_flag))) break;
          const float other = mx_slot[(1 - 2 * hc) * 128];
          const float mx = c * (c >= 0.f ? fmaxf(hmx, other) : fminf(hmx, other));
          // lazy reference: the latest two applied references, moved only when
          // this tile's max exceeds them by more than the threshold
          const float m_known = fmaxf(m_last, m_prev);
          const float m_new = mx > m_known + kRescaleThreshold ? mx : m_known;
          float sx = 0.f, srd = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float ex[16], er[16];
            if (valid >= vb + 64) {
#pragma unroll
              for (int j = 0; j < 16; ++j) ex[j] = fast_exp2(fmaf(s[16 * q + j], c, -m_new));
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)   // masked tokens: 0 (also when c == 0)
                ex[j] = vb + 16 * q + j < valid ? fast_exp2(fmaf(s[16 * q + j], c, -m_new)) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(ex[2 * j], ex[2 * j + 1]);
              const uint32_t w = *reinterpret_cast<const uint32_t*>(&b2);
              er[2 * j] = __uint_as_float(w << 16);
              er[2 * j + 1] = __uint_as_float(w & 0xffff0000u);
              pk[8 * q + j] = w;
            }
            sx += tree_sum(ex);
            srd += tree_sum(er);
          }
          own_m = m_new;
          own_lx = sx;
          own_lr = srd;

        }
        if (i > 0) {
        // ---------- apply tile t = g0 + i - 1 (own or received), release it to PV ----------
        const int t = g0 + i - 1;
        const int tb = L::kPBufs == 2 ? (t & 1) : 0;   // P buffer (and received info) of tile t
        const bool recv = t % C != rank;
        const uint32_t tpar = (recv_par >> tb) & 1;   // phase parity of tile t's receive barriers
        float mt, tlx, tlr;
        if (!recv) {
          mt = own_m;
          tlx = own_lx;
          tlr = own_lr;
        } else {
          const int b = tb;
          if (warp == 3 && lane == 0) {
            mbar_arrive_expect_tx(bar_addr<C>(base, kPRecvB0 + b), kPanel);
            mbar_arrive_expect_tx(bar_addr<C>(base, kPRecvP0 + b), kPanel);
            mbar_arrive_expect_tx(bar_addr<C>(base, kPRecv0 + b), kInfoBytes);
          }
          if (!(ok = mbar_wait_warp(bar_addr<C>(base, kPRecv0 + b), tpar, abort_flag)))
            break;
          recv_par ^= 1u << b;
          const float* info =
              reinterpret_cast<const float*>(sm + L::kOffP + b * L::kPStride + 2 * kPanel + info_off);
          mt = info[0];
          tlx = info[1];
          tlr = info[2];
        }
        // Stay at most two tiles ahead of PV (PV(t-2) complete): with one
        // kPvDone barrier per tile parity, every wait below is then less
        // than two phases away, so its parity is unambiguous.
        if (t >= 2 && !(ok = mbar_wait_warp(bar_addr<C>(base, kPvDone0 + (t & 1)), ((t - 2) >> 1) & 1,
                                            abort_flag)))
          break;
        const bool first = t == g0;
        const bool drop = !first && m_last - mt > kDropLog2;
        if (__any_sync(0xffffffffu, drop)) {
          // zero the dropped rows' P (this warp's token half) in this CTA's
          // copy; a received panel must have landed first
          if (recv && !(ok = mbar_wait_warp(bar_addr<C>(base, (hc == 0 ? kPRecvP0 : kPRecvB0) + tb), tpar,
                                            abort_flag)))
            break;
          if (drop) {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(sm + L::kOffP + tb * L::kPStride + p_off + (ch << 4)) =
                  make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        const float alpha = first ? 0.f : drop ? 1.f : exp2f(m_last - mt);
        if (!first && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O holds P . V of earlier tiles relative to m_last: move it to mt
          if (!(ok = mbar_wait_warp(bar_addr<C>(base, kPvDone0 + ((t - 1) & 1)), ((t - 1) >> 1) & 1,
                                    abort_flag)))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = kCh * hc; cc < kCh * hc + kCh; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_addr + L::kColO + 32 * cc, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(lane_addr + L::kColO + 32 * cc, o);
          }
          tmem_st_wait();
        }
        if (!drop) {
          lx = first ? tlx : lx * alpha + tlx;
          lr = first ? tlr : lr * alpha + tlr;
          m_prev = m_last;
          m_last = mt;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr<C>(base, kPReady0 + (t & 1)));
        }
        if (own_now) {
          // ---------- own tile g0 + i: P to this CTA and the peer ----------
          // (after tile g0 + i - 1 was released above: its PV, in both CTAs,
          // is what frees the P buffers)
          const int gg = g0 + i;
          // The tile's P buffer (in every CTA) is free once every CTA's PV of
          // the tile that last used it -- kPBufs tiles back -- is done.
          const int gw = gg - L::kPBufs;
          if (gw >= 0 && !(ok = mbar_wait_warp(bar_addr<C>(base, kPFree0 + (gw & 1)), (gw >> 1) & 1,
                                               abort_flag)))
            break;
          const int b = L::kPBufs == 2 ? (gg & 1) : 0;
          const uint32_t pbuf = L::kOffP + b * L::kPStride;
          const uint32_t prow = pbuf + p_off;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(sm + prow + ((ch ^ pswz) << 4)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
          *reinterpret_cast<float4*>(sm + pbuf + 2 * kPanel + info_off) =
              make_float4(own_m, own_lx, own_lr, 0.f);
          // Once all eight warps wrote their rows, one thread sends the buffer
          // to every other CTA of the cluster by bulk copies on three
          // barriers: the row info (all the peer's softmax warps need), token
          // panel 0, token panel 1 -- so the peer applies the tile and starts
          // its PV on tokens 0..63 while the rest is in flight.  The
          // copy engine moves distributed shared memory far faster than
          // remote stores, and a few large copies cost much less than one per
          // warp.
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr<C>(base, kPWritten));
          if (warp == 3 && lane == 0) {
            if (!mbar_wait(bar_addr<C>(base, kPWritten), (gl - 1) & 1, abort_flag)) {
              report_error(a.err, kErrTimeout);
            } else {
#pragma unroll
              for (int pr = 1; pr < C; ++pr) {
                const uint32_t peer = static_cast<uint32_t>(rank ^ pr);
                const uint32_t ra = map_to_rank(bar_addr<C>(base, kPRecv0 + b), peer);
                bulk_copy_to_peer(map_to_rank(base + pbuf + 2 * kPanel, peer), base + pbuf + 2 * kPanel, kInfoBytes, ra);
                bulk_copy_to_peer(map_to_rank(base + pbuf, peer), base + pbuf, kPanel,
                                  map_to_rank(bar_addr<C>(base, kPRecvP0 + b), peer));
                bulk_copy_to_peer(map_to_rank(base + pbuf + kPanel, peer), base + pbuf + kPanel, kPanel,
                                  map_to_rank(bar_addr<C>(base, kPRecvB0 + b), peer));
              }
            }
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      g = g0 + n;
      if (ui + 1 < u1) {
        // Q of the next unit: every own QK of this unit has been drained, and
        // the QK warp has finished the unit (so it consumed this unit's
        // kQTmemFull phase before the next one is signalled)
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kQEmpty), uidx & 1, abort_flag))) break;
        load_q_tmem<C>(a, a.units[ui + 1].req, r, hc, lane_addr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr<C>(base, kQTmemFull));
      }
      // ---- epilogue ----
      if (!(ok = mbar_wait_warp(bar_addr<C>(base, kPvDone0 + ((g - 1) & 1)), ((g - 1) >> 1) & 1,
                                abort_flag)))
        break;
      tc_fence_after();
      // Combine the two warps' row sums through shared memory; two phases of
      // kXchg0 + quad per unit.
      float* xch = reinterpret_cast<float*>(sm + L::kOffXchg + r * 16);
      xch[2 * hc] = lx;
      xch[2 * hc + 1] = lr;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr<C>(base, kXchg0 + quad));
      if (!(ok = mbar_wait_warp(bar_addr<C>(base, kXchg0 + quad), 0, abort_flag))) break;
      const float lx_all = xch[0] + xch[2];
      const float lr_all = xch[1] + xch[3];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr<C>(base, kXchg0 + quad));
      if (!(ok = mbar_wait_warp(bar_addr<C>(base, kXchg0 + quad), 1, abort_flag))) break;
      // A split request is combined by its unit that counted last (warp 3
      // lane 0 holds that count): the others publish their
      // share (partial O and lse of each CTA half), the last one waits for
      // them -- they counted first, so they are running and wait on nothing
      // of this unit -- and merges them with its own O straight from TMEM.
      const bool split = u.n_slots > 0;
      bool last = false;
      if (split) {
        if (warp == 3 && lane == 0) {
          const bool me_last = end_count == u.n_slots - 1;
          if (me_last) {
            int32_t* cnt = a.counters + 8 * u.req;
            if (!wait_count_acquire(cnt + 4 + rank, u.n_slots - 1, abort_flag)) {
              report_error(a.err, kErrTimeout);
            } else {
              cnt[rank] = 0;       // every unit counted and published: clean for the next launch
              cnt[4 + rank] = 0;
            }
          }
          *merge_flag = me_last;
          mbar_arrive(bar_addr<C>(base, kMergeB));
        }
        if (!(ok = mbar_wait_warp(bar_addr<C>(base, kMergeB), nsplit & 1, abort_flag))) break;
        ++nsplit;
        last = *merge_flag != 0;
      }
      // rows of out are 32-byte aligned when out is (the ABI asks for 16)
      const bool out32 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
      const size_t orow = static_cast<size_t>(u.req) * H + r;
      const float lse_own = (m_last + log2f(lx_all)) * kLn2;
      const float inv = (r < H) ? a.kv_scale / lr_all : 0.f;
      if (last) {
        // Slots are combined in slot order, this unit's own slot (from TMEM,
        // O * inv: bit-identical to the share it would have stored) in its
        // place, so the result does not depend on which unit merges.
        // The published shares are visible here: warp 3 saw their counts with
        // an acquire load and released that to these warps through kMergeB;
        // they are read from L2 (.cg), past this SM's L1.
        const int rr = r < H ? r : H - 1;
        const int ns = u.n_slots, own = u.out_slot - u.slot0;
        auto slot_lse = [&](int k) {   // k: index within the request's slots
          return k == own ? lse_own : __ldcg(a.lse_part + lse_part_offset(u.slot0 + k, rank, rr, H));
        };
        // the first kMergeRegs slot lse values are loaded together (static
        // indices keep them in registers); more slots are re-read
        float lk[kMergeRegs];
#pragma unroll
        for (int k = 0; k < kMergeRegs; ++k) lk[k] = k < ns ? slot_lse(k) : -INFINITY;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMergeRegs; ++k) M = fmaxf(M, lk[k]);
        for (int k = kMergeRegs; k < ns; ++k) M = fmaxf(M, slot_lse(k));
        float W = 0.f;
#pragma unroll
        for (int k = 0; k < kMergeRegs; ++k) W += k < ns ? __expf(lk[k] - M) : 0.f;
        for (int k = kMergeRegs; k < ns; ++k) W += __expf(slot_lse(k) - M);
        const float winv = 1.f / W;
        auto weight = [&](int k) { return __expf(slot_lse(k) - M) * winv; };
        if (ns == 2) {
          // the common split in two: the other share's loads and the TMEM
          // load of each chunk are in flight together
          const int other = u.slot0 + (1 - own);
          const float w0 = __expf(lk[0] - M) * winv, w1 = __expf(lk[1] - M) * winv;
#pragma unroll 1
          for (int cc = kCh * hc; cc < kCh * hc + kCh; ++cc) {
            const int d0 = L::kDims * rank + 32 * cc;
            uint32_t o[32];
            tmem_ld32(lane_addr + L::kColO + 32 * cc, o);   // in flight with the loads below
            float4 q[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              q[j] = __ldcg(reinterpret_cast<const float4*>(a.o_part + part_offset(other, rr, d0 + 4 * j, H)));
            tmem_ld_wait();
            float acc[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float vo[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float mine = __uint_as_float(o[4 * j + e]) * inv;
                acc[4 * j + e] = own == 0 ? fmaf(w1, vo[e], w0 * mine) : fmaf(w1, mine, w0 * vo[e]);
              }
            }
            if (r < H) store_out_row32<kOutF32>(a.out, orow, d0, acc, out32);
          }
        } else {
#pragma unroll 1
          for (int cc = kCh * hc; cc < kCh * hc + kCh; ++cc) {
            const int d0 = L::kDims * rank + 32 * cc;
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
#pragma unroll 1
            for (int k = 0; k < ns; ++k) {
              const float w = weight(k);
              float v[32];
              if (k == own) {
                uint32_t o[32];
                tmem_ld32(lane_addr + L::kColO + 32 * cc, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(o[j]) * inv;
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 q = __ldcg(reinterpret_cast<const float4*>(
                      a.o_part + part_offset(u.slot0 + k, rr, d0 + 4 * j, H)));
                  v[4 * j] = q.x;
                  v[4 * j + 1] = q.y;
                  v[4 * j + 2] = q.z;
                  v[4 * j + 3] = q.w;
                }
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) acc[j] = fmaf(w, v[j], acc[j]);
            }
            if (r < H) store_out_row32<kOutF32>(a.out, orow, d0, acc, out32);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr<C>(base, kOFree));
        if (rank == 0 && hc == 0 && r < H) a.lse[orow] = M + __logf(W);
      } else {
#pragma unroll 1
        for (int cc = kCh * hc; cc < kCh * hc + kCh; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_addr + L::kColO + 32 * cc, o);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * inv);
          if (r < H) {
            const int d0 = L::kDims * rank + 32 * cc;
            if (split) {
              // lanes hold consecutive heads: each store covers 1 KB of contiguous memory
#pragma unroll
              for (int j = 0; j < 4; ++j)
                st_global_v8(a.o_part + part_offset(u.out_slot, r, d0 + 8 * j, H), &o[8 * j]);
            } else {
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(o[j]);
              store_out_row32<kOutF32>(a.out, orow, d0, v, out32);
            }
          }
        }
        if (split && hc == 0 && r < H) a.lse_part[lse_part_offset(u.out_slot, rank, r, H)] = lse_own;
        // O may be overwritten now; for a split unit this also hands the
        // stored share to the PV warp, which publishes it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr<C>(base, kOFree));
        if (!split && rank == 0 && hc == 0 && r < H) a.lse[orow] = lse_own;
      }
    }
    if (!ok && lane == 0) report_error(a.err, kErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync_all();   // no CTA leaves while its peer may still address its shared memory
}

// The launched kernel: clusters of kTcCluster CTAs.
template <bool kOutF32, bool kFp8>
cudaError_t set_attributes() {
  using L = Cfg<kTcCluster>;
  static bool attr_set = false;   // set once, before any stream capture
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<kOutF32, kTcCluster, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return cudaSuccess;
}

cudaLaunchConfig_t cluster_config(int clusters, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kTcCluster * clusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<kTcCluster>::kSmemBytes;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTcCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bool kOutF32, bool kFp8>
cudaError_t launch_impl(const DecodeArgs& a, const TcMaps& maps, cudaStream_t s) {
  cudaError_t e = set_attributes<kOutF32, kFp8>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(a.n_workers, attr);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<kOutF32, kTcCluster, kFp8>, a, maps);
}

}  // namespace

cudaError_t decode_tc_max_workers(int* workers) {
  *workers = 0;
  cudaError_t e = set_attributes<true, false>();
  if (e == cudaSuccess) e = set_attributes<false, false>();
  if (e == cudaSuccess) e = set_attributes<true, true>();
  if (e == cudaSuccess) e = set_attributes<false, true>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(1, attr);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, decode_tc_kernel<false, kTcCluster, false>, &cfg);
  if (e != cudaSuccess) return e;
  *workers = clusters;
  return cudaSuccess;
}

#ifdef MLA_STALL_TEST
// Test build only: set the copy CTA 0's V producer leaves out (0: none).
extern "C" int mla_test_set_stall(int chunk) {
  return static_cast<int>(cudaMemcpyToSymbol(g_stall_chunk, &chunk, sizeof(chunk)));
}
#endif

cudaError_t launch_decode_tc(const DecodeArgs& a, const TcMaps& maps, bool out_f32, bool kv_fp8,
                             cudaStream_t s) {
  if (kv_fp8) return out_f32 ? launch_impl<true, true>(a, maps, s) : launch_impl<false, true>(a, maps, s);
  return out_f32 ? launch_impl<true, false>(a, maps, s) : launch_impl<false, false>(a, maps, s);
}

}  // namespace mla
