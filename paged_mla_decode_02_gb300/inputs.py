"""Seeded synthetic inputs for paged MLA decode.

This module only draws numbers and lays them out in the paged-cache format.
It holds none of the attention arithmetic, so both the float64 oracle and
the CUDA path can be fed from it without sharing any of the method's code.

Layout (the one the C ABI takes):
  q_nope  [B, H, 512]        bf16 (stored here as uint16 bit patterns)
  q_pe    [B, H, 64]         bf16 bits
  ckv     [pool, P, 512]     bf16 bits (uint16) or fp8-e4m3 codes (uint8)
  kpe     [pool, P, 64]      same dtype as ckv
  kv_indptr  int32 [B + 1]   CSR offsets into kv_indices, in pages
  kv_indices int32 [nnz]     page ids into the pool
  kv_len     int32 [B]       tokens per request

The paging arrays follow the plan arguments discussed for the FlashInfer MLA
wrapper (vLLM-metax PR #113, review of the ``decode_wrapper.plan`` call and of
the host-side ``paged_kv_indptr_cpu`` / ``paged_kv_len_arr_cpu`` slices).

Draw order for every config, from one ``numpy.random.Generator(PCG64(seed))``:
kv_len -> page permutation -> q_nope -> q_pe -> ckv -> kpe.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

D_CKV = 512  # kv_lora_rank
D_KPE = 64   # qk_rope_head_dim

BF16_NAN_BITS = np.uint16(0x7FC0)
FP8_E4M3_NAN_CODE = np.uint8(0x7F)


@dataclasses.dataclass
class MLAInputs:
    name: str
    q_nope: np.ndarray      # uint16 [B,H,512], or [B,Q,H,512] with several query tokens
    q_pe: np.ndarray        # uint16 [B,H,64], or [B,Q,H,64]
    ckv: np.ndarray         # uint16 or uint8 [pool,P,512]
    kpe: np.ndarray         # uint16 or uint8 [pool,P,64]
    kv_indptr: np.ndarray   # int32 [B+1]
    kv_indices: np.ndarray  # int32 [nnz]
    kv_len: np.ndarray      # int32 [B]
    page_size: int
    sm_scale: float
    kv_dtype: str           # "bf16" | "fp8_e4m3"
    kv_scale: float = 1.0

    @property
    def batch(self) -> int:
        return int(self.kv_len.shape[0])

    @property
    def q_len(self) -> int:
        return 1 if self.q_nope.ndim == 3 else int(self.q_nope.shape[1])

    @property
    def num_heads(self) -> int:
        return int(self.q_nope.shape[-2])

    @property
    def num_pages(self) -> int:
        return int(self.ckv.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.kv_len.astype(np.int64).sum())


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 -> bf16 (round-to-nearest-even) via torch's CPU cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32_to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Saturating round-to-nearest-even float32 -> fp8 e4m3fn codes (torch's cast)."""
    import torch
    x = np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0)
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _normal_codes(rng: np.random.Generator, shape, scale: float, kv_dtype: str,
                  kv_scale: float = 1.0, chunk_rows: int = 1 << 16) -> np.ndarray:
    """Draw N(0,1)*scale in float32, in row chunks, and encode as bf16 bits or fp8 codes."""
    shape = tuple(int(s) for s in shape)
    rows = shape[0]
    per_row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out_dtype = np.uint16 if kv_dtype == "bf16" else np.uint8
    out = np.empty((rows, per_row), dtype=out_dtype)
    step = max(1, chunk_rows * 512 // max(per_row, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = rng.standard_normal((r1 - r0, per_row), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        if kv_dtype == "bf16":
            out[r0:r1] = f32_to_bf16_bits(x)
        elif kv_dtype == "fp8_e4m3":
            out[r0:r1] = f32_to_e4m3_codes(x / np.float32(kv_scale))
        else:
            raise ValueError(f"unknown kv dtype {kv_dtype!r}")
    return out.reshape(shape)


def make_inputs(name: str, kv_len, num_heads: int, page_size: int, *,
                seed: int = 0, rng: np.random.Generator | None = None,
                pool_pages: int | None = None, key_scale: float = 1.0,
                kv_dtype: str = "bf16", kv_scale: float = 1.0,
                sm_scale: float = 1.0 / math.sqrt(192.0),
                poison: bool = False, slack_pages: int = 0, q_len: int = 0) -> MLAInputs:
    """Build one paged batch.

    ``kv_len`` is either a sequence of ints or a callable ``rng -> int array``
    (drawn first, so the draw order above holds).  Request pages are taken, in
    request order, from a random permutation of the pool.  ``poison`` fills
    every pool page no request uses, and every slot past ``kv_len`` in a
    request's last page, with NaN, so a kernel that reads them and lets them
    reach an output fails parity.  ``q_len`` > 0 draws that many query tokens
    per request (q arrays [B,Q,H,.]); 0 keeps the single-token layout [B,H,.].
    """
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    if callable(kv_len):
        kv_len = kv_len(rng)
    kv_len = np.asarray(kv_len, dtype=np.int64)
    if kv_len.ndim != 1 or (kv_len < 0).any():
        raise ValueError("kv_len must be a 1-D array of non-negative ints")
    batch = kv_len.shape[0]
    npages = (kv_len + page_size - 1) // page_size
    nnz = int(npages.sum())
    pool = nnz + int(slack_pages) if pool_pages is None else int(pool_pages)
    if pool < nnz:
        raise ValueError("pool smaller than the pages the batch needs")
    perm = rng.permutation(pool).astype(np.int32)
    kv_indices = perm[:nnz].copy()
    kv_indptr = np.zeros(batch + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(npages)

    qs = (batch, num_heads) if q_len == 0 else (batch, q_len, num_heads)
    q_nope = _normal_codes(rng, qs + (D_CKV,), 1.0, "bf16")
    q_pe = _normal_codes(rng, qs + (D_KPE,), 1.0, "bf16")
    ckv = _normal_codes(rng, (pool, page_size, D_CKV), key_scale, kv_dtype, kv_scale)
    kpe = _normal_codes(rng, (pool, page_size, D_KPE), key_scale, kv_dtype, kv_scale)

    if poison:
        nan = BF16_NAN_BITS if kv_dtype == "bf16" else FP8_E4M3_NAN_CODE
        used = np.zeros(pool, dtype=bool)
        used[kv_indices] = True
        ckv[~used] = nan
        kpe[~used] = nan
        for b in range(batch):
            L = int(kv_len[b])
            if L == 0:
                continue
            tail = L - (int(npages[b]) - 1) * page_size
            last = kv_indices[kv_indptr[b + 1] - 1]
            ckv[last, tail:] = nan
            kpe[last, tail:] = nan

    return MLAInputs(name=name, q_nope=q_nope, q_pe=q_pe, ckv=ckv, kpe=kpe,
                     kv_indptr=kv_indptr, kv_indices=kv_indices,
                     kv_len=kv_len.astype(np.int32), page_size=page_size,
                     sm_scale=float(sm_scale), kv_dtype=kv_dtype,
                     kv_scale=float(kv_scale))


def plant_dominant_tokens(x: MLAInputs, where, gap: float) -> MLAInputs:
    """Make token ``pos`` of request ``b`` score about ``gap`` natural-log
    units above the request's other tokens, in every head, for each (b, pos)
    in ``where``.  Every head of such a request gets head 0's q_pe, and the
    token's kpe row becomes that vector times gap / (sm_scale |q_pe|^2), so
    the rope term of its score rises by about ``gap`` (the stored values are
    rounded to the cache dtype; the exact scores follow from them).  An
    attention-sink token at position 0, or one late sharp maximum, is the
    case this builds.  Returns a modified copy."""
    y = dataclasses.replace(x, q_pe=x.q_pe.copy(), kpe=x.kpe.copy())
    for b, pos in where:
        if not 0 <= pos < int(x.kv_len[b]):
            raise ValueError(f"token {pos} is outside request {b}")
        y.q_pe[b, ...] = y.q_pe[b, ..., :1, :] if y.q_pe.ndim == 3 else y.q_pe[b, :, :1, :]
        u = _bits_to_f32(y.q_pe[b].reshape(-1, D_KPE)[0])
        k = np.float32(gap / (x.sm_scale * float(np.dot(u.astype(np.float64), u))))
        row = (u * k).reshape(1, D_KPE)
        page = x.kv_indices[x.kv_indptr[b] + pos // x.page_size]
        if x.kv_dtype == "bf16":
            y.kpe[page, pos % x.page_size] = f32_to_bf16_bits(row)[0]
        else:
            y.kpe[page, pos % x.page_size] = f32_to_e4m3_codes(row / np.float32(x.kv_scale))[0]
    return y


def _bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _ragged_lengths(rng):
    return rng.integers(1, 8193, size=128)


def _lognormal_lengths(rng):
    x = np.exp(rng.normal(math.log(2048.0), 0.8, size=256))
    return np.minimum(16384, np.maximum(1, np.rint(x))).astype(np.int64)


# Workload recipes: shapes of DeepSeek-V3-style absorbed MLA decode
# (kv_lora_rank 512, qk_rope_head_dim 64, 128 query heads).
CONFIGS = {
    "tiny": dict(kv_len=[33, 70], num_heads=16, page_size=16, pool_pages=16),
    "deepseek": dict(kv_len=[4096] * 64, num_heads=128, page_size=64),
    "deepseek_mtp2": dict(kv_len=[4096] * 64, num_heads=128, page_size=64, q_len=2),
    "ragged": dict(kv_len=_ragged_lengths, num_heads=128, page_size=16),
    "long_b1": dict(kv_len=[131072], num_heads=16, page_size=64, key_scale=3.0),
    "long_b4": dict(kv_len=[131072] * 4, num_heads=16, page_size=64, key_scale=3.0),
    "long_b4_mtp4": dict(kv_len=[131072] * 4, num_heads=16, page_size=64, key_scale=3.0, q_len=4),
    "fp8": dict(kv_len=_lognormal_lengths, num_heads=128, page_size=64,
                kv_dtype="fp8_e4m3", kv_scale=1.0),
}

CONFIG_DESCRIPTIONS = {
    "tiny": "B2 H16 P16 L{33,70} pool16 bf16",
    "deepseek": "B64 H128 P64 L4096 bf16",
    "deepseek_mtp2": "B64 H128 P64 L4096 bf16, 2 query tokens per request",
    "ragged": "B128 H128 P16 L~U[1,8192] bf16",
    "long_b1": "B1 H16 P64 L131072 bf16 keys x3",
    "long_b4": "B4 H16 P64 L131072 bf16 keys x3",
    "long_b4_mtp4": "B4 H16 P64 L131072 bf16 keys x3, 4 query tokens per request",
    "fp8": "B256 H128 P64 L~lognormal(2048,0.8)<=16384 fp8-e4m3",
}


def make_config(name: str, seed: int = 0, poison: bool = False) -> MLAInputs:
    """Build one of the named workloads with the draw order above."""
    if name not in CONFIGS:
        raise KeyError(f"unknown config {name!r}; known: {sorted(CONFIGS)}")
    kw = dict(CONFIGS[name])
    if poison and "pool_pages" not in kw:
        kw["slack_pages"] = 8
    return make_inputs(name, seed=seed, poison=poison, **kw)


def config_lengths(name: str, seed: int = 0) -> np.ndarray:
    """Only the kv_len draw of a named config (cheap: no cache is generated)."""
    kw = CONFIGS[name]
    rng = np.random.Generator(np.random.PCG64(seed))
    kl = kw["kv_len"]
    return np.asarray(kl(rng) if callable(kl) else kl, dtype=np.int64)
