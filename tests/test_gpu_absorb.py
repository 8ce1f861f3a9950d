"""The per-head projections around the latent decode (mla_absorb_q,
mla_project_out), each against the oracle, and the whole absorbed chain
against explicit (un-absorbed) MLA attention on the same bf16 values."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from gpu_helpers import to_device
from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import inputs as I
from paged_mla_decode_02_gb300 import mla

pytestmark = pytest.mark.gpu


def _bf16(rng, shape, scale=1.0):
    """bf16 bit patterns of N(0, scale^2) values and the device tensor."""
    t = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.cuda()


def _check_rounded(got, ref, what):
    """got = bf16 of an fp32 accumulation of ref's terms: within one bf16 ulp
    of ref (rounding of fp32 sums near a bf16 boundary may go either way),
    and close to ref overall."""
    ulp = np.maximum(np.abs(ref), 1e-30) * 2.0 ** -7
    assert np.all(np.abs(got - ref) <= ulp + 1e-5), f"{what}: more than one bf16 ulp off"
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 3e-3, f"{what}: rel-L2 {rel:.2e}"


@pytest.mark.parametrize("B, H, dn", [(5, 3, 128), (64, 128, 128), (200, 4, 64)])
def test_absorb_q_matches_oracle(B, H, dn):
    rng = np.random.Generator(np.random.PCG64(B * 7 + dn))
    q_bits, q = _bf16(rng, (B, H, dn))
    w_bits, w = _bf16(rng, (H, 512, dn), 1.0 / math.sqrt(dn))
    out = mla.mla_absorb_q(q, w, check_status=True)
    ref = O.absorb_q(q_bits, w_bits)
    _check_rounded(out.double().cpu().numpy(), ref, f"absorb B={B} H={H} dn={dn}")


@pytest.mark.parametrize("B, H, dv", [(5, 3, 128), (64, 128, 128), (200, 4, 64)])
def test_project_out_matches_oracle(B, H, dv):
    rng = np.random.Generator(np.random.PCG64(B * 11 + dv))
    o_bits, o = _bf16(rng, (B, H, 512))
    w_bits, w = _bf16(rng, (H, 512, dv), 1.0 / math.sqrt(512))
    got = mla.mla_project_out(o, w, check_status=True)
    ref = O.project_out(o_bits, w_bits)
    _check_rounded(got.double().cpu().numpy(), ref, f"project B={B} H={H} dv={dv}")


@pytest.mark.parametrize("lens, heads, P", [([40, 700, 33, 1500], 16, 16), ([2000, 90], 128, 64)])
def test_absorbed_chain_matches_unabsorbed_attention(lens, heads, P):
    """q_raw -> absorb -> decode -> project against attention with explicit
    keys C.W_UK and values C.W_UV (float64 on the same bf16 inputs).  Three
    bf16 roundings sit on the path (the absorbed query, the decode output and
    the projected output), each ~2^-9 relative, plus the decode's own error
    (within its bar): the chain is held to rel-L2 <= 1e-2."""
    x = I.make_inputs("abs", lens, heads, P, seed=8)
    d = to_device(x)
    rng = np.random.Generator(np.random.PCG64(9))
    dn = dv = 128
    q_bits, q_raw = _bf16(rng, (x.batch, heads, dn))
    wk_bits, w_uk = _bf16(rng, (heads, 512, dn), 1.0 / math.sqrt(dn))
    wv_bits, w_uv = _bf16(rng, (heads, 512, dv), 1.0 / math.sqrt(512))

    q_nope = mla.mla_absorb_q(q_raw, w_uk, check_status=True)
    dec = mla.MLADecoder(x.batch, heads)
    try:
        dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, P, x.sm_scale)
        out, _ = dec.run(q_nope, d["q_pe"], d["ckv"], d["kpe"], out_dtype=torch.bfloat16)
        dec.check_status()
    finally:
        dec.close()
    o = mla.mla_project_out(out, w_uv, check_status=True).double().cpu().numpy()

    ref = np.zeros_like(o)
    for b in range(x.batch):
        L = int(x.kv_len[b])
        C = O.decode_bf16(O.gather_request(x.ckv, x.kv_indptr, x.kv_indices, b, L, P))
        R = O.decode_bf16(O.gather_request(x.kpe, x.kv_indptr, x.kv_indices, b, L, P))
        ref[b] = O.unabsorbed_attention(O.decode_bf16(q_bits[b]), O.decode_bf16(x.q_pe[b]), C, R,
                                        O.decode_bf16(wk_bits), O.decode_bf16(wv_bits), x.sm_scale)
    rel = np.linalg.norm(o - ref) / np.linalg.norm(ref)
    assert rel <= 1e-2, f"absorbed chain rel-L2 {rel:.2e}"


def test_chain_back_to_back_equals_synchronised_chain():
    """absorb -> decode (+ merge) -> project launched back to back on one
    stream, each kernel a programmatic dependent launch of the one before it
    (it waits for that kernel at its first instruction), eagerly and from a
    CUDA graph: the same bits as the chain with a synchronisation after
    every call.  The intermediate and output buffers hold NaN before each
    run, so a kernel that read its input early would show."""
    x = I.make_inputs("abs_b2b", [2000, 90, 30000], 128, 64, seed=18)   # the last request split
    d = to_device(x)
    rng = np.random.Generator(np.random.PCG64(19))
    _, q_raw = _bf16(rng, (x.batch, 128, 128))
    _, w_uk = _bf16(rng, (128, 512, 128), 1.0 / math.sqrt(128))
    _, w_uv = _bf16(rng, (128, 512, 128), 1.0 / math.sqrt(512))
    q_nope = torch.empty((x.batch, 128, 512), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((x.batch, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((x.batch, 128), dtype=torch.float32, device="cuda")
    o = torch.empty((x.batch, 128, 128), dtype=torch.bfloat16, device="cuda")
    dec = mla.MLADecoder(x.batch, 128)
    try:
        dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, 64, x.sm_scale)
        torch.cuda.synchronize()
        assert dec.info()["num_partial_slots"] > 0      # the merge kernel has work

        def poison():
            for t in (q_nope, out, lse, o):
                t.fill_(float("nan"))

        def chain(sync):
            mla.mla_absorb_q(q_raw, w_uk, q_nope)
            if sync:
                torch.cuda.synchronize()
            dec.run(q_nope, d["q_pe"], d["ckv"], d["kpe"], out, lse)
            if sync:
                torch.cuda.synchronize()
            mla.mla_project_out(out, w_uv, o)
            if sync:
                torch.cuda.synchronize()

        poison()
        chain(True)
        ref_o, ref_lse = o.clone(), lse.clone()
        assert not torch.isnan(ref_o).any()
        for _ in range(3):
            poison()
            chain(False)
            torch.cuda.synchronize()
            assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain(False)
        for _ in range(3):
            poison()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
        dec.check_status()
    finally:
        dec.close()


def test_projection_arguments_are_checked():
    q = torch.zeros((2, 3, 96), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((3, 512, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_absorb_q(q, w)
    assert ei.value.status == mla.ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        mla.mla_absorb_q(q.float(), w)
