"""Why the fp8-cache path multiplies in bf16 (host only, no GPU).

An fp8 e4m3 cache could feed kind::f8f6f4 tensor-core products, but then both
operands of each product are e4m3: the query (for the scores) and the
probabilities P (for P . V).  This test emulates that arithmetic on an
fp8-cache batch in float64, with the operands rounded as the MMA would see
them, and compares it with the oracle (the exact attention over the
dequantised cache) at the parity bar: max-abs <= 1e-2, relative L2 <= 5e-3,
|delta lse| <= 1e-3.  bf16 operands (what the kernels use: every e4m3 code is
exact in bf16) stay inside the bar; an e4m3 query (per-row scale to the e4m3
range) or e4m3 P each break it.
"""
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
