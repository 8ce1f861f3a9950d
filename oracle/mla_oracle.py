"""Float64 CPU oracle for paged MLA decode.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The library
never calls it, and it shares no code with the CUDA path: it decodes the
stored bf16 / fp8 codes itself, gathers pages itself and evaluates exact
softmax attention in float64 with numpy.

What it computes (absorbed multi-head latent attention, decode, q_len = 1;
``mla_decode_multi`` extends it to several query tokens per request):
for request b with pages ``kv_indices[kv_indptr[b]:kv_indptr[b+1]]`` and
``L = kv_len[b]`` tokens, C = the first L gathered ckv rows [L, 512] and
R = the first L gathered kpe rows [L, 64]; for every head h

    s   = sm_scale * (C @ q_nope[b,h] + R @ q_pe[b,h])          [L]
    lse = log(sum_i exp(s_i))          (natural log, of the scaled scores)
    out = sum_i exp(s_i - lse) * C_i                              [512]

Sources on the pages:
  * one latent KV head per token, ckv width = kv_lora_rank and kpe width =
    qk_rope_head_dim: "[WIP] support flashinfer_mla" (vLLM-metax PR #113),
    review comment on the ``decode_wrapper.plan`` parameters (num_kv_heads is 1
    for MLA; head_dim_ckv is the compressed-cache width);
  * no causal mask for decode: same review comment, ``causal=False``;
  * request addressing by a page-count CSR (indptr) and per-request token
    counts: same PR, review comment on slicing ``paged_kv_indptr_cpu`` and
    ``paged_kv_len_arr_cpu`` to the decode requests;
  * a KV-cache dtype that differs from the query dtype: "[V1][Core] FlashInfer
    attention backend for V1" (vLLM PR #14061), "Current limitations";
  * partial attentions combined by log-sum-exp (cascade attention):
    same PR, "Outstanding items".
The formula itself is the standard absorbed-MLA decode; the pages give only
its dimensions and parameters.

Readings where the pages are silent: sm_scale is a caller argument; lse is the
natural log-sum-exp of the scaled scores; an empty request (L = 0) gives
out = 0 and lse = -inf; fp8 codes are OCP E4M3 (e4m3fn) times a per-tensor
scale.
"""
from __future__ import annotations

import numpy as np

D_CKV = 512
D_KPE = 64


# ---------------------------------------------------------------------------
# Stored-value decoding
# ---------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64.  bf16 is the top half of an IEEE float32."""
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):          # signalling-NaN patterns stay NaN
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """fp8 E4M3 (OCP 'e4m3fn') codes -> float64, from the format definition.

    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
    subnormal (m/8 * 2^-6); there is no infinity and S.1111.111 is NaN.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    val = sign * np.where(e == 0, subnormal, normal)
    return np.where((e == 15) & (m == 7), np.nan, val)


def dequantize(codes: np.ndarray, kv_dtype: str, kv_scale: float = 1.0) -> np.ndarray:
    """Cache codes -> float64 values as stored (fp8 values times kv_scale)."""
    if kv_dtype == "bf16":
        return decode_bf16(codes)
    if kv_dtype == "fp8_e4m3":
        return decode_e4m3(codes) * float(kv_scale)
    raise ValueError(f"unknown kv dtype {kv_dtype!r}")


# ---------------------------------------------------------------------------
# Paging
# ---------------------------------------------------------------------------

def gather_request(cache: np.ndarray, kv_indptr, kv_indices, b: int, kv_len: int,
                   page_size: int) -> np.ndarray:
    """Rows of request b in page-table order, truncated to kv_len: [L, width]."""
    pages = np.asarray(kv_indices[int(kv_indptr[b]):int(kv_indptr[b + 1])], dtype=np.int64)
    if kv_len == 0:
        return cache.reshape(-1, cache.shape[-1])[:0]
    if len(pages) * page_size < kv_len:
        raise ValueError("request has fewer pages than its kv_len needs")
    rows = cache[pages]                      # [npages, P, width]
    return rows.reshape(-1, cache.shape[-1])[:kv_len]


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def attend(q_nope: np.ndarray, q_pe: np.ndarray, C: np.ndarray, R: np.ndarray,
           sm_scale: float):
    """Exact softmax attention of H query heads over one latent KV head.

    q_nope [H,512], q_pe [H,64], C [L,512], R [L,64], all float64.
    Returns out [H,512] and lse [H] (natural log of the scaled scores).
    """
    H = q_nope.shape[0]
    L = C.shape[0]
    if L == 0:
        return np.zeros((H, C.shape[1])), np.full(H, -np.inf)
    s = sm_scale * (q_nope @ C.T + q_pe @ R.T)          # [H, L]
    m = s.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        raise FloatingPointError("non-finite score: a cache row that should not be read was read")
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    lse = m + np.log(l)                                  # [H, 1]
    out = np.exp(s - lse) @ C                            # [H, 512]
    return out, lse[:, 0]


def mla_decode(q_nope, q_pe, ckv, kpe, kv_indptr, kv_indices, kv_len, page_size: int,
               sm_scale: float, kv_dtype: str = "bf16", kv_scale: float = 1.0,
               requests=None):
    """Oracle for a whole paged batch.

    q_nope / q_pe are bf16 bit arrays [B,H,512] / [B,H,64]; ckv / kpe are cache
    codes [pool,P,512] / [pool,P,64].  Returns float64 out [b,H,512] and lse
    [b,H] for the requests listed in ``requests`` (all when None), in order.
    """
    B = len(kv_len)
    reqs = range(B) if requests is None else list(requests)
    H = q_nope.shape[1]
    out = np.zeros((len(reqs), H, D_CKV))
    lse = np.zeros((len(reqs), H))
    for i, b in enumerate(reqs):
        L = int(kv_len[b])
        Cc = gather_request(ckv, kv_indptr, kv_indices, b, L, page_size)
        Rc = gather_request(kpe, kv_indptr, kv_indices, b, L, page_size)
        C = dequantize(Cc, kv_dtype, kv_scale)
        R = dequantize(Rc, kv_dtype, kv_scale)
        qn = decode_bf16(q_nope[b])
        qp = decode_bf16(q_pe[b])
        out[i], lse[i] = attend(qn, qp, C, R, sm_scale)
    return out, lse


def mla_decode_multi(q_nope, q_pe, ckv, kpe, kv_indptr, kv_indices, kv_len, page_size: int,
                     sm_scale: float, kv_dtype: str = "bf16", kv_scale: float = 1.0,
                     requests=None):
    """Oracle for decode steps of several query tokens per request.

    q_nope / q_pe are bf16 bit arrays [B,Q,H,512] / [B,Q,H,64]: the Q newest
    tokens of each request, whose keys are the last Q of its kv_len cached
    tokens.  Query j (0-based) sits at position L - Q + j and sees the tokens
    at positions 0 .. L - Q + j: a causal mask inside the query block, none
    before it.  Returns float64 out [b,Q,H,512] and lse [b,Q,H].

    Sources: decode with short query lengths, which the prefill wrapper serves
    poorly ("[V1][Core] FlashInfer attention backend for V1", vLLM PR #14061,
    review discussion of the wrapper's decode performance).  The mask is the
    reading for speculative or multi-token decode: each new token attends to
    the cache up to and including itself.
    """
    B = len(kv_len)
    reqs = range(B) if requests is None else list(requests)
    Q, H = q_nope.shape[1], q_nope.shape[2]
    out = np.zeros((len(reqs), Q, H, D_CKV))
    lse = np.zeros((len(reqs), Q, H))
    for i, b in enumerate(reqs):
        L = int(kv_len[b])
        if L < Q:
            raise ValueError("a request holds fewer cached tokens than query tokens")
        C = dequantize(gather_request(ckv, kv_indptr, kv_indices, b, L, page_size), kv_dtype, kv_scale)
        R = dequantize(gather_request(kpe, kv_indptr, kv_indices, b, L, page_size), kv_dtype, kv_scale)
        pos = np.arange(L)
        for j in range(Q):
            qn = decode_bf16(q_nope[b, j])                      # [H,512]
            qp = decode_bf16(q_pe[b, j])                        # [H,64]
            s = sm_scale * (qn @ C.T + qp @ R.T)                # [H,L]
            s = np.where(pos[None, :] <= L - Q + j, s, -np.inf)  # causal inside the block
            m = s.max(axis=1, keepdims=True)
            if not np.all(np.isfinite(m)):
                raise FloatingPointError("non-finite score in the visible tokens")
            l = np.exp(s - m).sum(axis=1, keepdims=True)
            lse_j = m + np.log(l)
            out[i, j] = np.exp(s - lse_j) @ C
            lse[i, j] = lse_j[:, 0]
    return out, lse


def mla_decode_inputs(x, requests=None):
    """``mla_decode`` on an ``MLAInputs``-like object (any object with its fields)."""
    return mla_decode(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                      x.kv_len, x.page_size, x.sm_scale, x.kv_dtype, x.kv_scale,
                      requests=requests)


def lse_merge(outs, lses):
    """Combine partial attentions over disjoint KV chunks by log-sum-exp.

    outs: list of [H,D] float64, lses: list of [H].  Chunks with lse = -inf
    (empty) carry no weight.  Returns (out [H,D], lse [H]).
    This is the combination behind cascade attention ("[V1][Core] FlashInfer
    attention backend for V1", "Outstanding items"): each chunk's softmax is
    exact on its own, and re-weighting by exp(lse_i - lse_total) restores the
    softmax over the union.
    """
    lses = np.stack([np.asarray(x, dtype=np.float64) for x in lses])   # [S,H]
    outs = np.stack([np.asarray(x, dtype=np.float64) for x in outs])   # [S,H,D]
    M = lses.max(axis=0)                                                # [H]
    safe_M = np.where(np.isfinite(M), M, 0.0)
    w = np.exp(lses - safe_M)                                           # [S,H]
    tot = w.sum(axis=0)
    lse = np.where(tot > 0, safe_M + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    out = np.einsum("sh,shd->hd", w, outs) / np.where(tot > 0, tot, 1.0)[:, None]
    return out, lse


def absorb_q(q_nope_raw, W_UK):
    """The decode's q_nope from a head's own query: per head h,
    q_nope[b,h] = W_UK[h] @ q_raw[b,h], mapping the head's dn-wide no-rope
    query into the 512-wide latent space of the compressed cache (so the
    scores need no up-projection of the keys).

    q_nope_raw bf16 bits [B,H,dn]; W_UK bf16 bits [H,512,dn].  Returns float64
    [B,H,512].  Sources: the decode runs on the compressed cache of width
    kv_lora_rank with the query's rope part kept apart (head_dim_ckv =
    kv_lora_rank, head_dim_kpe = qk_rope_head_dim: "[WIP] support
    flashinfer_mla", review of the decode_wrapper.plan parameters), which
    needs the query taken into that space first.
    """
    return np.einsum("hnd,bhd->bhn", decode_bf16(W_UK), decode_bf16(q_nope_raw))


def project_out(out, W_UV):
    """A head's value output from the decode's latent output: per head h,
    o[b,h] = out[b,h] @ W_UV[h] (512 -> dv).  out float64 [B,H,512] (or bf16
    bits); W_UV bf16 bits [H,512,dv].  Returns float64 [B,H,dv]."""
    o = decode_bf16(out) if np.asarray(out).dtype == np.uint16 else np.asarray(out, np.float64)
    return np.einsum("bhn,hnv->bhv", o, decode_bf16(W_UV))


def unabsorbed_attention(q_nope_orig, q_pe, C, R, W_UK, W_UV, sm_scale: float):
    """MLA attention in its explicit (un-absorbed) form, for pinning ``attend``.

    Per head h: K_h = [C @ W_UK[h], R] and V_h = C @ W_UV[h];
    o_h = softmax(sm_scale * [q_nope_orig_h, q_pe_h] . K_h^T) @ V_h.
    q_nope_orig [H,dn], q_pe [H,64], C [L,512], R [L,64],
    W_UK [H,512,dn], W_UV [H,512,dv].  Returns o [H,dv].
    """
    H = q_nope_orig.shape[0]
    o = np.zeros((H, W_UV.shape[2]))
    for h in range(H):
        K = np.concatenate([C @ W_UK[h], R], axis=1)           # [L, dn+64]
        V = C @ W_UV[h]                                        # [L, dv]
        q = np.concatenate([q_nope_orig[h], q_pe[h]])          # [dn+64]
        s = sm_scale * (K @ q)
        p = np.exp(s - s.max())
        o[h] = (p / p.sum()) @ V
    return o
