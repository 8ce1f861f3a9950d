// Kernel arguments and host launchers (internal).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "mla_internal.h"

namespace mla {

struct DecodeArgs {
  const void* q_nope;          // [B,H,512] bf16
  const void* q_pe;            // [B,H,64] bf16
  const void* ckv;             // [num_pages,P,512] bf16 or e4m3
  const void* kpe;             // [num_pages,P,64]
  const int32_t* kv_indices;   // page ids
  const WorkUnit* units;
  const int32_t* worker_ptr;   // [n_workers+1]
  const PlanDev* params;
  void* out;                   // [B,H,512] bf16 or fp32
  float* lse;                  // [B,H]
  float* o_part;               // partial outputs, fp32, layout of part_offset()
  float* lse_part;             // [slots][2][H]: one copy per CTA half (lse_part_offset)
  const MergeEntry* merge;     // split and empty requests
  int32_t* counters;           // [max_batch][8]: per cluster CTA (up to 4), units
                               // counted and shares published; zero between launches
  int32_t* err;
  int num_pages;
  int num_heads;
  float kv_scale;
  int units_cap;
  int n_workers;
};

// Element (slot, head h, dim d) of the fp32 partial outputs.  Dims are
// grouped by eight and the heads of a group are adjacent:
//   [slot][d / 8][h][d % 8]
// so a warp holding 32 consecutive heads x 8 dims stores (or loads) 1 KB of
// contiguous memory with 32-byte accesses, where a [slot][h][d] layout would
// touch 32 separate rows per instruction.
__host__ __device__ inline size_t part_offset(int slot, int h, int d, int H) {
  return ((static_cast<size_t>(slot) * (kDCkv / 8) + d / 8) * H + h) * 8 + (d & 7);
}

// Log-sum-exp of partial slot `slot`, head h: each CTA of a tcgen05 cluster
// keeps its own copy (up to four; copy 0 is the one the merge kernel reads).
constexpr int kLsePartCopies = 4;
__host__ __device__ inline size_t lse_part_offset(int slot, int copy, int h, int H) {
  return (static_cast<size_t>(slot) * kLsePartCopies + copy) * H + h;
}

struct MergeArgs {
  const MergeEntry* merge;
  const PlanDev* params;
  const float* o_part;
  const float* lse_part;
  void* out;
  float* lse;
  int num_heads;
  int merge_cap;
};

// Legacy warp-level tensor path (mma.sync m16n8k16): one CTA per (unit, 16-head group).
cudaError_t launch_decode_mma(const DecodeArgs& a, bool kv_fp8, bool out_f32, cudaStream_t s);

// tcgen05 / TMEM path: persistent clusters of kTcCluster CTAs, one per worker.
constexpr int kTcCluster = 2;
// Tokens per V chunk of the tcgen05 kernel; its V tensor map copies boxes of
// min(page_size, kTcVChunkTok) rows (host encoding and kernel share this).
constexpr int kTcVChunkTok = 32;
struct TcMaps {
  CUtensorMap q_nope;   // [B*H, 512] bf16, box 64 x H
  CUtensorMap ckv_k;    // [pages*P, 512] bf16 (fp8), box 64 x P (one page of a K panel)
  CUtensorMap kpe_k;    // [pages*P, 64] bf16 (fp8), box 64 x P
  CUtensorMap ckv_v;    // (64, pages*P, 8 panels) view of ckv, box 64 x min(P, 32) x 4 panels
};
// kv_fp8: e4m3 cache (byte maps, 64-byte swizzle, page_size >= 32); the
// kernel expands each copy to bf16 in shared memory and scales by kv_scale.
cudaError_t launch_decode_tc(const DecodeArgs& a, const TcMaps& maps, bool out_f32, bool kv_fp8,
                             cudaStream_t s);
// Host: the tensor maps launch_decode_tc takes, for one batch (false when the
// driver's encoder is unavailable or rejects an argument).
bool encode_tc_maps(TcMaps* maps, const void* q_nope, const void* ckv_cache, const void* kpe_cache,
                    int batch, int num_heads, int page_size, int num_pages, bool kv_fp8 = false);
// Clusters of two CTAs of the tcgen05 kernel that can be resident at once
// (the persistent grid uses at most that many workers).
cudaError_t decode_tc_max_workers(int* workers);

// CTA-pair kernel (one tcgen05 MMA over both SMs of a cluster, cta_group::2):
// persistent, one pair per worker; split requests leave normalised partials
// (part_offset layout, lse copy 0) for launch_merge.
// An fp8 (e4m3) cache is read through byte maps with a 64-byte swizzle (the
// same boxes in elements) and needs page_size >= 32.
struct PairMaps {
  CUtensorMap q_nope;   // [B*H, 512] bf16, box 64 x 64 (64 heads)
  CUtensorMap q_pe;     // [B*H, 64] bf16, box 64 x 64
  CUtensorMap ckv_k;    // [pages*P, 512] bf16 / e4m3, box 64 x P
  CUtensorMap kpe_k;    // [pages*P, 64] bf16 / e4m3, box 64 x P
  CUtensorMap ckv_v;    // (64, pages*P, 8 panels) view of ckv, box 64 x min(P, 32) x 4 panels
};
cudaError_t launch_decode_pair(const DecodeArgs& a, const PairMaps& maps, bool out_f32, bool kv_fp8,
                               cudaStream_t s);
bool encode_pair_maps(PairMaps* maps, const void* q_nope, const void* q_pe, const void* ckv_cache,
                      const void* kpe_cache, int batch, int num_heads, int page_size, int num_pages,
                      bool kv_fp8);
cudaError_t decode_pair_max_workers(int* workers);

// LSE merge of split partials (and zero-fill of empty requests); the mma.sync
// and CTA-pair paths -- the one-CTA tcgen05 kernel merges in its own epilogue.
cudaError_t launch_merge(const MergeArgs& a, bool out_f32, cudaStream_t s);

}  // namespace mla
