"""Pins for the float64 oracle, independent of the oracle's own code.

Each check ties the oracle to something other than itself: a hand-worked
example, a library conversion routine, a closed form, an algebraic identity
(the un-absorbed form of MLA), an invariant, or a brute-force scalar loop.
A second group plants plausible mistakes in copies of the oracle and checks
that at least one pin catches each of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=1):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------------------
# stored-value decoding, pinned to torch's conversions
# ---------------------------------------------------------------------------

def test_decode_bf16_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.decode_bf16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_decode_e4m3_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2                       # 0x7F and 0xFF
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


# ---------------------------------------------------------------------------
# hand-worked example (tests/golden/worked_example_3tok.txt)
# ---------------------------------------------------------------------------

def _worked_example_inputs():
    P, pool = 2, 3
    ckv = np.full((pool, P, 512), I.BF16_NAN_BITS, dtype=np.uint16)
    kpe = np.full((pool, P, 64), I.BF16_NAN_BITS, dtype=np.uint16)
    vals_c = np.zeros((3, 512), np.float32)
    vals_r = np.zeros((3, 64), np.float32)
    vals_c[0, :3] = [1, 7, 0.5]
    vals_c[1, :3] = [0, -7, 0.25]
    vals_c[2, :3] = [0, 14, -1]
    vals_r[0, 0] = 1
    vals_r[1, 0] = 1
    slots = [(2, 0), (2, 1), (0, 0)]
    for t, (pg, sl) in enumerate(slots):
        ckv[pg, sl] = I.f32_to_bf16_bits(vals_c[t])
        kpe[pg, sl] = I.f32_to_bf16_bits(vals_r[t])
    qn = np.zeros((1, 2, 512), np.float32)
    qp = np.zeros((1, 2, 64), np.float32)
    qn[0, 0, 0] = 1
    qp[0, 0, 0] = 1
    return dict(q_nope=I.f32_to_bf16_bits(qn), q_pe=I.f32_to_bf16_bits(qp), ckv=ckv, kpe=kpe,
                kv_indptr=np.array([0, 2], np.int32), kv_indices=np.array([2, 0], np.int32),
                kv_len=np.array([3], np.int32), page_size=P, sm_scale=math.log(2.0))


def test_golden_worked_example():
    rows = np.loadtxt(os.path.join(GOLDEN, "worked_example_3tok.txt"), comments="#")
    out, lse = O.mla_decode(**_worked_example_inputs())
    for h in range(2):
        assert abs(lse[0, h] - rows[h, 1]) < 1e-13
        assert np.allclose(out[0, h, :3], rows[h, 2:5], rtol=0, atol=1e-13)
        assert np.all(out[0, h, 3:] == 0)


# ---------------------------------------------------------------------------
# algebraic identity: absorbed == un-absorbed MLA
# ---------------------------------------------------------------------------

def _unabsorbed_error(attend_fn, seed=3):
    rng = _rng(seed)
    H, L, dn, dv = 4, 37, 128, 128
    C = rng.standard_normal((L, 512))
    R = rng.standard_normal((L, 64))
    W_UK = rng.standard_normal((H, 512, dn)) / math.sqrt(512)
    W_UV = rng.standard_normal((H, 512, dv)) / math.sqrt(512)
    q_orig = rng.standard_normal((H, dn))
    q_pe = rng.standard_normal((H, 64))
    sm_scale = 1.0 / math.sqrt(dn + 64)
    ref = O.unabsorbed_attention(q_orig, q_pe, C, R, W_UK, W_UV, sm_scale)
    q_abs = np.einsum("hkd,hd->hk", W_UK, q_orig)       # fold W_UK into the query
    out, _ = attend_fn(q_abs, q_pe, C, R, sm_scale)
    got = np.einsum("hk,hkv->hv", out, W_UV)            # fold W_UV into the output
    return np.abs(got - ref).max()


def test_absorbed_matches_unabsorbed():
    assert _unabsorbed_error(O.attend) < 1e-10


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def test_single_token_closed_form():
    rng = _rng(4)
    C = rng.standard_normal((1, 512))
    R = rng.standard_normal((1, 64))
    qn = rng.standard_normal((3, 512))
    qp = rng.standard_normal((3, 64))
    out, lse = O.attend(qn, qp, C, R, 0.1)
    assert np.array_equal(out, np.repeat(C, 3, axis=0))
    s0 = 0.1 * (qn @ C[0] + qp @ R[0])
    assert np.allclose(lse, s0, rtol=0, atol=1e-12)


def test_dominant_token_closed_form():
    # one token scoring ~200 natural-log units above the rest: the softmax is
    # that token alone (the others weigh below e^-190), so out is its ckv row
    # and lse its score, computed here by scalar loops on the decoded values
    x = I.make_inputs("dominant", [300, 130], 4, 64, seed=21)
    y = I.plant_dominant_tokens(x, [(0, 0), (1, 129)], 200.0)
    out, lse = O.mla_decode_inputs(y)

    def bf16(bits):
        return [float(v) for v in (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)]

    for b, pos in ((0, 0), (1, 129)):
        page = y.kv_indices[y.kv_indptr[b] + pos // 64]
        c = bf16(y.ckv[page, pos % 64])
        k = bf16(y.kpe[page, pos % 64])
        for h in range(y.num_heads):
            qn, qp = bf16(y.q_nope[b, h]), bf16(y.q_pe[b, h])
            s = y.sm_scale * math.fsum([a * w for a, w in zip(qn, c)] + [a * w for a, w in zip(qp, k)])
            assert abs(lse[b, h] - s) <= 1e-9 * max(1.0, abs(s))
            assert np.allclose(out[b, h], c, rtol=0, atol=1e-12)


def _uniform_error(attend_fn):
    rng = _rng(5)
    L = 29
    C = rng.standard_normal((L, 512))
    R = np.tile(rng.standard_normal((1, 64)), (L, 1))      # identical keys
    qp = rng.standard_normal((2, 64))
    qn = np.zeros((2, 512))
    out, lse = attend_fn(qn, qp, C, R, 0.3)
    s = 0.3 * (qp @ R[0])
    e1 = np.abs(out - C.mean(axis=0)).max()
    e2 = np.abs(lse - (s + math.log(L))).max()
    # sm_scale = 0 gives the same mean with lse = ln L
    qn2 = rng.standard_normal((2, 512))
    out2, lse2 = attend_fn(qn2, qp, C, rng.standard_normal((L, 64)), 0.0)
    e3 = np.abs(out2 - C.mean(axis=0)).max()
    e4 = np.abs(lse2 - math.log(L)).max()
    return max(e1, e2, e3, e4)


def test_identical_keys_give_mean_of_values():
    assert _uniform_error(O.attend) < 1e-12


def test_empty_request():
    x = I.make_inputs("e", [0, 5], 4, 16, seed=6)
    out, lse = O.mla_decode_inputs(x)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_page_table_permutation_is_bitwise_invariant():
    x = I.make_inputs("p", [70, 33, 129], 8, 16, seed=7, slack_pages=5)
    out, lse = O.mla_decode_inputs(x)
    rng = _rng(8)
    perm = rng.permutation(x.num_pages)        # new position of old page p is perm[p]
    ckv2 = np.empty_like(x.ckv)
    kpe2 = np.empty_like(x.kpe)
    ckv2[perm] = x.ckv
    kpe2[perm] = x.kpe
    idx2 = perm[x.kv_indices].astype(np.int32)
    out2, lse2 = O.mla_decode(x.q_nope, x.q_pe, ckv2, kpe2, x.kv_indptr, idx2, x.kv_len,
                              x.page_size, x.sm_scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def _split_merge_error(attend_fn, seed=9):
    rng = _rng(seed)
    H, L = 6, 300
    C = rng.standard_normal((L, 512)) * 2
    R = rng.standard_normal((L, 64)) * 2
    qn = rng.standard_normal((H, 512))
    qp = rng.standard_normal((H, 64))
    ref_out, ref_lse = attend_fn(qn, qp, C, R, 0.07)
    cuts = np.sort(rng.choice(np.arange(1, L), size=4, replace=False))
    bounds = [0, *cuts.tolist(), L]
    parts = [attend_fn(qn, qp, C[a:b], R[a:b], 0.07) for a, b in zip(bounds[:-1], bounds[1:])]
    parts.append(attend_fn(qn, qp, C[:0], R[:0], 0.07))        # an empty chunk
    out, lse = O.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    return max(np.abs(out - ref_out).max(), np.abs(lse - ref_lse).max())


def test_split_and_merge_matches_unsplit():
    assert _split_merge_error(O.attend) < 1e-12


def _bruteforce(q_nope, q_pe, ckv, kpe, kv_indptr, kv_indices, kv_len, page_size, sm_scale):
    """Scalar loops with math.exp / math.fsum over decoded python floats."""
    def f(bits):
        return float(torch.tensor(int(np.int16(np.uint16(bits).view(np.int16))),
                                  dtype=torch.int16).view(torch.bfloat16).item())
    B, H = q_nope.shape[:2]
    outs, lses = [], []
    for b in range(B):
        toks = []
        for t in range(int(kv_len[b])):
            page = int(kv_indices[int(kv_indptr[b]) + t // page_size])
            toks.append((page, t % page_size))
        for h in range(H):
            qn = [f(v) for v in q_nope[b, h]]
            qp = [f(v) for v in q_pe[b, h]]
            scores, rows = [], []
            for page, slot in toks:
                c = [f(v) for v in ckv[page, slot]]
                r = [f(v) for v in kpe[page, slot]]
                s = math.fsum([qn[i] * c[i] for i in range(512)] + [qp[i] * r[i] for i in range(64)])
                scores.append(sm_scale * s)
                rows.append(c)
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            tot = math.fsum(w)
            outs.append([math.fsum(w[i] * rows[i][d] for i in range(len(w))) / tot for d in range(512)])
            lses.append(m + math.log(tot))
    return np.array(outs).reshape(B, H, 512), np.array(lses).reshape(B, H)


def test_bruteforce_scalar_loops():
    x = I.make_inputs("bf", [5, 3], 2, 2, seed=10, slack_pages=1, poison=True)
    out, lse = O.mla_decode_inputs(x)
    bo, bl = _bruteforce(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                         x.kv_len, x.page_size, x.sm_scale)
    assert np.abs(out - bo).max() < 1e-12
    assert np.abs(lse - bl).max() < 1e-12


def test_poison_pages_never_read():
    a = I.make_config("tiny")
    b = I.make_config("tiny", poison=True)
    assert np.isnan(O.decode_bf16(b.ckv)).any()
    oa, la = O.mla_decode_inputs(a)
    ob, lb = O.mla_decode_inputs(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_fp8_cache_equals_bf16_cache_of_same_values():
    """Every e4m3 value is exact in bf16: converting the codes with torch and
    running the bf16 path must give identical results (kv_scale = 1)."""
    x = I.make_inputs("f8", [40, 7], 4, 16, seed=11, kv_dtype="fp8_e4m3")
    def to_bf16(codes):
        t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    o8, l8 = O.mla_decode_inputs(x)
    o16, l16 = O.mla_decode(x.q_nope, x.q_pe, to_bf16(x.ckv), to_bf16(x.kpe), x.kv_indptr,
                            x.kv_indices, x.kv_len, x.page_size, x.sm_scale)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)
    # kv_scale multiplies the stored values
    o8s, _ = O.mla_decode(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices, x.kv_len,
                          x.page_size, x.sm_scale / 2.0, "fp8_e4m3", 2.0)
    assert np.allclose(o8s, 2.0 * o8, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# ---------------------------------------------------------------------------

def _mutant_drop_kpe(qn, qp, C, R, sc):
    return O.attend(qn, np.zeros_like(qp), C, R, sc)


def _mutant_sign(qn, qp, C, R, sc):
    return O.attend(qn, qp, C, R, -sc)


def _mutant_log2_lse(qn, qp, C, R, sc):
    out, lse = O.attend(qn, qp, C, R, sc)
    return out, lse / math.log(2.0)


def _mutant_unnormalised(qn, qp, C, R, sc):
    out, lse = O.attend(qn, qp, C, R, sc)
    return out * C.shape[0] ** 0.5 if C.shape[0] else out, lse


def _mutant_skip_last_token(qn, qp, C, R, sc):
    if C.shape[0] > 1:
        return O.attend(qn, qp, C[:-1], R[:-1], sc)
    return O.attend(qn, qp, C, R, sc)


def _mutant_values_from_kpe_width(qn, qp, C, R, sc):
    out, lse = O.attend(qn, qp, C, R, sc)
    out = out.copy()
    out[:, :64] = np.exp(sc * (qn @ C.T + qp @ R.T) - lse[:, None]) @ R if C.shape[0] else 0
    return out, lse


@pytest.mark.parametrize("mutant", [_mutant_drop_kpe, _mutant_sign, _mutant_log2_lse,
                                    _mutant_unnormalised, _mutant_skip_last_token,
                                    _mutant_values_from_kpe_width])
def test_pins_catch_planted_mistakes(mutant):
    caught = (_unabsorbed_error(mutant) > 1e-6 or _uniform_error(mutant) > 1e-6
              or _split_merge_error(mutant) > 1e-6)
    if not caught:
        x = I.make_inputs("bf", [5, 3], 2, 2, seed=10, slack_pages=1)
        bo, bl = _bruteforce(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                             x.kv_len, x.page_size, x.sm_scale)
        orig = O.attend
        try:
            O.attend = mutant
            out, lse = O.mla_decode_inputs(x)
        finally:
            O.attend = orig
        caught = np.abs(out - bo).max() > 1e-6 or np.abs(lse - bl).max() > 1e-6
    assert caught


def test_pins_catch_page_indexing_mistake():
    """Reading the page table one entry off, or ignoring it, breaks brute force."""
    x = I.make_inputs("bf", [5, 3], 2, 2, seed=10, slack_pages=1)
    bo, _ = _bruteforce(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                        x.kv_len, x.page_size, x.sm_scale)
    shifted = np.roll(x.kv_indices, 1)
    out, _ = O.mla_decode(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, shifted, x.kv_len,
                          x.page_size, x.sm_scale)
    assert np.abs(out - bo).max() > 1e-3


# ---------------------------------------------------------------------------
# several query tokens per request (causal inside the query block)
# ---------------------------------------------------------------------------

def _multi(lens, heads, P, Q, seed=31):
    return I.make_inputs("mq", lens, heads, P, seed=seed, q_len=Q, slack_pages=2, poison=True)


def _multi_oracle(x):
    return O.mla_decode_multi(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                              x.kv_len, x.page_size, x.sm_scale)


def test_multi_token_single_query_is_decode():
    x = _multi([37, 5, 64], 4, 16, 1)
    out, lse = _multi_oracle(x)
    o1, l1 = O.mla_decode(x.q_nope[:, 0], x.q_pe[:, 0], x.ckv, x.kpe, x.kv_indptr,
                          x.kv_indices, x.kv_len, x.page_size, x.sm_scale)
    assert np.array_equal(out[:, 0], o1) and np.array_equal(lse[:, 0], l1)


@pytest.mark.parametrize("Q", [2, 3, 5])
def test_multi_token_query_j_is_decode_of_the_prefix(Q):
    """Query j of a block of Q sees exactly the first L - Q + 1 + j tokens: it
    equals single-token decode of the request cut to that length (through the
    page table, so cut inside a page too), and differs from the lengths one
    shorter or longer (an off-by-one or a missing mask is caught)."""
    x = _multi([37, 5, 64], 4, 16, Q)
    out, lse = _multi_oracle(x)
    for j in range(Q):
        cut = x.kv_len - Q + 1 + j
        oj, lj = O.mla_decode(x.q_nope[:, j], x.q_pe[:, j], x.ckv, x.kpe, x.kv_indptr,
                              x.kv_indices, cut, x.page_size, x.sm_scale)
        assert np.abs(out[:, j] - oj).max() < 1e-12 and np.abs(lse[:, j] - lj).max() < 1e-12
        for d in (-1, 1):
            alt = np.clip(cut + d, 1, x.kv_len)
            oa, _ = O.mla_decode(x.q_nope[:, j], x.q_pe[:, j], x.ckv, x.kpe, x.kv_indptr,
                                 x.kv_indices, alt, x.page_size, x.sm_scale)
            moved = alt != cut
            if moved.any():
                assert np.abs(out[moved, j] - oa[moved]).max(axis=(1, 2)).min() > 1e-6


def test_multi_token_bruteforce():
    x = _multi([6, 4], 2, 2, 3, seed=12)
    out, lse = _multi_oracle(x)
    for j in range(3):
        bo, bl = _bruteforce(x.q_nope[:, j], x.q_pe[:, j], x.ckv, x.kpe, x.kv_indptr,
                             x.kv_indices, x.kv_len - 3 + 1 + j, x.page_size, x.sm_scale)
        assert np.abs(out[:, j] - bo).max() < 1e-12 and np.abs(lse[:, j] - bl).max() < 1e-12


def test_multi_token_needs_the_query_tokens_in_the_cache():
    x = _multi([2, 9], 2, 16, 3)
    with pytest.raises(ValueError):
        _multi_oracle(x)


# ---------------------------------------------------------------------------
# the projections around the latent decode
# ---------------------------------------------------------------------------

def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_absorb_decode_project_equals_unabsorbed_attention():
    """absorb_q -> decode -> project_out is the explicit MLA attention with
    up-projected keys and values (on the same bf16 values)."""
    rng = _rng(21)
    B, H, dn, dv, P = 2, 3, 128, 128, 16
    x = I.make_inputs("ab", [40, 23], H, P, seed=22)
    q_raw = _bf16_bits(rng.standard_normal((B, H, dn)))
    W_UK = _bf16_bits(rng.standard_normal((H, 512, dn)) / math.sqrt(dn))
    W_UV = _bf16_bits(rng.standard_normal((H, 512, dv)) / math.sqrt(512))
    q_abs = O.absorb_q(q_raw, W_UK)
    # the decode takes bf16 queries: feed it the exact absorbed values through
    # an fp64 attend (the decode's own rounding is tested elsewhere)
    got = np.zeros((B, H, dv))
    for b in range(B):
        C = O.decode_bf16(O.gather_request(x.ckv, x.kv_indptr, x.kv_indices, b, int(x.kv_len[b]), P))
        R = O.decode_bf16(O.gather_request(x.kpe, x.kv_indptr, x.kv_indices, b, int(x.kv_len[b]), P))
        out, _ = O.attend(q_abs[b], O.decode_bf16(x.q_pe[b]), C, R, x.sm_scale)
        got[b] = O.project_out(out[None], W_UV)[0]
        ref = O.unabsorbed_attention(O.decode_bf16(q_raw[b]), O.decode_bf16(x.q_pe[b]), C, R,
                                     O.decode_bf16(W_UK), O.decode_bf16(W_UV), x.sm_scale)
        assert np.abs(got[b] - ref).max() < 1e-9


def test_projections_catch_transposed_weights():
    """Using a head's weight transposed (or another head's) changes the result."""
    rng = _rng(23)
    q_raw = _bf16_bits(rng.standard_normal((2, 2, 128)))
    W = _bf16_bits(rng.standard_normal((2, 512, 128)))
    good = O.absorb_q(q_raw, W)
    swapped = O.absorb_q(q_raw, W[::-1].copy())
    assert np.abs(good - swapped).max() > 1e-3
    out = rng.standard_normal((2, 2, 512))
    Wv = _bf16_bits(rng.standard_normal((2, 512, 128)))
    assert np.abs(O.project_out(out, Wv) - O.project_out(out, Wv[::-1].copy())).max() > 1e-3
