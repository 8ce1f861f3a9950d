"""Two-level (cascade) decode: a prefix shared by every request and each
request's own suffix decoded as two batches, their states combined by
``mla_merge_states``; checked against the float64 oracle on the concatenated
pages, and the merge itself against the oracle's log-sum-exp merge."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import assert_parity, bf16_round, run_decode, to_device
from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import inputs as I
from paged_mla_decode_02_gb300 import mla

pytestmark = pytest.mark.gpu


def _states(rows, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    o_a = rng.normal(size=(rows, 512))
    o_b = rng.normal(size=(rows, 512))
    lse_a = rng.normal(scale=4.0, size=rows)
    lse_b = rng.normal(scale=4.0, size=rows)
    lse_a[::7] = -np.inf          # one side empty
    lse_b[3::11] = -np.inf
    lse_a[5] = lse_b[5] = -np.inf  # both empty
    o_a[np.isinf(lse_a)] = np.nan  # an empty state's o carries no weight, whatever it holds
    return o_a, lse_a, o_b, lse_b


def _cuda32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_states_matches_oracle(out_dtype):
    rows = 1000
    o_a, lse_a, o_b, lse_b = _states(rows, 3)
    out = torch.empty((rows, 512), dtype=out_dtype, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    mla.mla_merge_states(_cuda32(o_a), _cuda32(lse_a), _cuda32(o_b), _cuda32(lse_b), out, lse)
    torch.cuda.synchronize()
    # oracle on the values the kernel saw (fp32-rounded inputs)
    f = lambda a: a.astype(np.float32).astype(np.float64)
    ref_o, ref_l = O.lse_merge([np.nan_to_num(f(o_a)), f(o_b)], [f(lse_a), f(lse_b)])
    got = out.double().cpu().numpy()
    if out_dtype == torch.bfloat16:
        ref_o = bf16_round(ref_o)
        assert np.abs(got - ref_o).max() <= 2.0 ** -7 * np.abs(ref_o).max()
    else:
        assert np.abs(got - ref_o).max() <= 1e-5 * max(1.0, np.abs(ref_o).max())
    gl = lse.double().cpu().numpy()
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.abs(gl[fin] - ref_l[fin]).max() < 1e-5
    assert np.all(got[~fin] == 0.0)


def test_merge_states_in_place():
    rows = 64
    o_a, lse_a, o_b, lse_b = _states(rows, 4)
    o_a = np.nan_to_num(o_a)
    a, la = _cuda32(o_a), _cuda32(lse_a)
    ref = torch.empty_like(a), torch.empty_like(la)
    mla.mla_merge_states(a, la, _cuda32(o_b), _cuda32(lse_b), ref[0], ref[1])
    mla.mla_merge_states(a, la, _cuda32(o_b), _cuda32(lse_b), a, la)   # out aliases o_a, lse_a
    torch.cuda.synchronize()
    assert torch.equal(a, ref[0]) and torch.equal(la, ref[1])


@pytest.mark.parametrize("kernel", ["pair", "tcgen05", "mma_sync"])
@pytest.mark.parametrize("prefix_pages, suffix, heads, P", [
    (5, [37, 0, 200, 64], 16, 16),        # a request without a suffix of its own
    (40, [700, 1300, 5], 128, 64),        # a long shared prefix, 128 heads
])
def test_cascade_prefix_and_suffix_merge_to_full_decode(kernel, prefix_pages, suffix, heads, P):
    # request 0 of the generated batch holds the shared prefix; requests 1..
    # hold the suffixes and give the queries
    plen = prefix_pages * P
    x = I.make_inputs("cas", [plen] + suffix, heads, P, seed=17, poison=True, slack_pages=2)
    B = len(suffix)
    pre_pages = x.kv_indices[x.kv_indptr[0]:x.kv_indptr[1]]
    d = to_device(x)
    dev = torch.device("cuda")
    qn, qp = d["q_nope"][1:].contiguous(), d["q_pe"][1:].contiguous()

    def decode(indptr, indices, lens):
        idx = torch.from_numpy(indices.astype(np.int32)).to(dev)
        dec = mla.MLADecoder(B, heads, kernel)
        try:
            dec.plan(indptr, idx, lens, P, x.sm_scale)
            out, lse = dec.run(qn, qp, d["ckv"], d["kpe"], out_dtype=torch.float32)
            dec.check_status()
            return out, lse
        finally:
            dec.close()

    # level 0: the shared prefix, once per request; level 1: own suffixes
    o0, l0 = decode(np.arange(B + 1, dtype=np.int32) * prefix_pages, np.tile(pre_pages, B),
                    np.full(B, plen, np.int32))
    o1, l1 = decode(x.kv_indptr[1:] - x.kv_indptr[1], x.kv_indices[x.kv_indptr[1]:],
                    x.kv_len[1:])
    out = torch.empty_like(o0)
    lse = torch.empty_like(l0)
    mla.mla_merge_states(o0, l0, o1, l1, out, lse)
    torch.cuda.synchronize()

    # oracle: one decode over the prefix pages followed by each suffix's pages
    indptr = np.zeros(B + 1, np.int32)
    indices = []
    for b in range(B):
        own = x.kv_indices[x.kv_indptr[b + 1]:x.kv_indptr[b + 2]]
        indices.append(np.concatenate([pre_pages, own]))
        indptr[b + 1] = indptr[b] + len(indices[-1])
    full_len = (plen + x.kv_len[1:]).astype(np.int32)
    ref_out, ref_lse = O.mla_decode(x.q_nope[1:], x.q_pe[1:], x.ckv, x.kpe, indptr,
                                    np.concatenate(indices), full_len, P, x.sm_scale)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                  f"cascade {kernel} {prefix_pages} {suffix}")
