"""Which operands the fp8-cache products may take (host only, no GPU).

An fp8 e4m3 cache feeds kind::f8f6f4 tensor-core products only if the other
operand of each product is e4m3 too: the query (for the scores) and the
probabilities P (for P . V).  This test emulates that arithmetic on an
fp8-cache batch in float64, with the operands rounded as the MMA would see
them, and compares it with the oracle (the exact attention over the
dequantised cache) at the parity bar: max-abs <= 1e-2, relative L2 <= 5e-3,
|delta lse| <= 1e-3.
- bf16 operands (every e4m3 code is exact in bf16) stay inside the bar.
- A single e4m3 query (per-row scale to the e4m3 range) or e4m3 P breaks it.
- Two e4m3 terms per operand, x = hi + lo with hi = e4m3(x) and
  lo = e4m3(x - hi), stay inside it, computed the way the CTA-pair kernel
  does: the query scaled per row so that its largest magnitude lies in
  [2^7, 2^8) (hi + lo is then the bf16 query exactly, but for elements
  below 2^-2 after the scaling, which keep 2^-10), P in 256-token tiles
  as 2^(s - reference) * 2^5 with a reference that moves when a tile's
  maximum exceeds it by more than 3.5 (log2 units), the output divided by
  the sum of the hi + lo values and the lse taken from the exact sum.
"""
import math
import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import inputs as I

BAR = (1e-2, 5e-3, 1e-3)


def _e4m3(x):
    t = torch.from_numpy(np.clip(x, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16(x):
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.fixture(scope="module")
def batch():
    # lengths around the fp8 workload's median (2048), 128 heads, 64-token pages
    x = I.make_inputs("fp8_operands", [2048, 3100, 900, 4500], 128, 64, seed=41, kv_dtype="fp8_e4m3")
    ref_out, ref_lse = O.mla_decode_inputs(x)
    return x, ref_out, ref_lse


def _emulate(x, q_e4m3, p_e4m3):
    qn, qp = O.decode_bf16(x.q_nope), O.decode_bf16(x.q_pe)
    outs, lses = [], []
    for b in range(x.batch):
        pages = x.kv_indices[x.kv_indptr[b]:x.kv_indptr[b + 1]]
        L = int(x.kv_len[b])
        C = O.decode_e4m3(x.ckv[pages].reshape(-1, 512))[:L] * x.kv_scale
        R = O.decode_e4m3(x.kpe[pages].reshape(-1, 64))[:L] * x.kv_scale
        q1, q2 = qn[b], qp[b]
        if q_e4m3:
            s1 = np.abs(q1).max(axis=1, keepdims=True) / 448.0
            s2 = np.abs(q2).max(axis=1, keepdims=True) / 448.0
            q1, q2 = _e4m3(q1 / s1) * s1, _e4m3(q2 / s2) * s2
        s = x.sm_scale * (q1 @ C.T + q2 @ R.T)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        lses.append(m[:, 0] + np.log(p.sum(axis=1)))
        pq = _e4m3(p) if p_e4m3 else _bf16(p)
        outs.append((pq @ C) / pq.sum(axis=1, keepdims=True))
    return np.stack(outs), np.stack(lses)


def _f32(x):
    return x.astype(np.float32).astype(np.float64)


def _split(x):
    hi = _e4m3(x)
    return hi, _e4m3(_f32(x - hi))


def _emulate_split(x, threshold=3.5, offset=5.0, tile=256):
    qn, qp = O.decode_bf16(x.q_nope), O.decode_bf16(x.q_pe)
    log2e = 1.0 / math.log(2.0)
    outs, lses = [], []
    for b in range(x.batch):
        pages = x.kv_indices[x.kv_indptr[b]:x.kv_indptr[b + 1]]
        L = int(x.kv_len[b])
        C = O.decode_e4m3(x.ckv[pages].reshape(-1, 512))[:L]
        R = O.decode_e4m3(x.kpe[pages].reshape(-1, 64))[:L]
        q = np.concatenate([qn[b], qp[b]], axis=1)
        K = np.concatenate([C, R], axis=1)
        rm = np.abs(q).max(axis=1, keepdims=True)
        e = np.where(rm > 0, 7 - np.floor(np.log2(np.where(rm > 0, rm, 1.0))), 0.0)
        qs = q * 2.0 ** e
        qh, ql = _split(qs)
        # the bf16 query exactly from magnitude 2^-2 up; below, to 2^-10 (half
        # the e4m3 subnormal step)
        big = np.abs(qs) >= 0.25
        assert np.array_equal((qh + ql)[big], qs[big])
        assert np.abs(qh + ql - qs).max() <= 2.0 ** -10
        y = _f32(_f32(qh @ K.T + ql @ K.T) * (x.sm_scale * x.kv_scale * log2e * 2.0 ** -e))
        H = y.shape[0]
        o, lx, lr, ref = np.zeros((H, 512)), np.zeros(H), np.zeros(H), None
        for t0 in range(0, L, tile):
            yt = y[:, t0:t0 + tile]
            mt = yt.max(axis=1)
            if ref is None:
                ref, alpha = mt.copy(), np.ones(H)
            else:
                up = mt > ref + threshold
                alpha = np.where(up, 2.0 ** (ref - mt), 1.0)
                ref = np.where(up, mt, ref)
            p = _f32(2.0 ** (yt - ref[:, None])) * 2.0 ** offset
            assert p.max() < 448.0
            ph, pl = _split(p)
            lx = lx * alpha + p.sum(axis=1)
            lr = lr * alpha + (ph + pl).sum(axis=1)
            o = o * alpha[:, None] + (ph + pl) @ C[t0:t0 + tile]
        outs.append(o / lr[:, None] * x.kv_scale)
        lses.append((ref - offset + np.log2(lx)) * math.log(2.0))
    return np.stack(outs), np.stack(lses)


def _errors(out, lse, ref_out, ref_lse):
    err = out - ref_out
    return (float(np.abs(err).max()), float(np.linalg.norm(err) / np.linalg.norm(ref_out)),
            float(np.abs(lse - ref_lse).max()))


def _inside(e):
    return all(v <= b for v, b in zip(e, BAR))


def test_bf16_operands_meet_the_bar(batch):
    x, ref_out, ref_lse = batch
    e = _errors(*_emulate(x, False, False), ref_out, ref_lse)
    assert _inside(e), e


@pytest.mark.parametrize("q_e4m3, p_e4m3", [(True, False), (False, True), (True, True)])
def test_e4m3_operands_break_the_bar(batch, q_e4m3, p_e4m3):
    x, ref_out, ref_lse = batch
    e = _errors(*_emulate(x, q_e4m3, p_e4m3), ref_out, ref_lse)
    assert not _inside(e), e


def test_split_e4m3_operands_meet_the_bar(batch):
    x, ref_out, ref_lse = batch
    e = _errors(*_emulate_split(x), ref_out, ref_lse)
    assert _inside(e), e
    # with margin: a tenth of the bar on the output, a hundredth on the lse
    assert e[0] <= 1e-3 and e[1] <= 5e-4 and e[2] <= 1e-5, e
