"""Decode steps of several query tokens per request (causal inside the query
block), through the C ABI, against the float64 oracle's multi-token decode."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import assert_parity, run_decode, to_device
from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import inputs as I
from paged_mla_decode_02_gb300 import mla

pytestmark = pytest.mark.gpu

KERNELS = ["pair", "tcgen05", "mma_sync"]


def _run_multi(x, d, kernel, out_dtype=torch.float32):
    dec = mla.MLADecoder(x.batch * x.q_len, x.num_heads, kernel)
    try:
        dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, x.page_size, x.sm_scale, q_len=x.q_len)
        out, lse = dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out_dtype=out_dtype)
        dec.check_status()
        assert tuple(out.shape) == (x.batch, x.q_len, x.num_heads, 512)
        return out.double().cpu().numpy(), lse.double().cpu().numpy()
    finally:
        dec.close()


def _oracle(x, requests=None):
    return O.mla_decode_multi(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                              x.kv_len, x.page_size, x.sm_scale, requests=requests)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("lens, heads, P, Q", [
    ([37, 5, 64, 200], 16, 16, 2),      # the block cut inside a page, ragged tails
    ([130, 129, 128, 300], 32, 32, 3),  # the mask edge on a tile boundary
    ([700, 4], 128, 64, 4),             # a request holding exactly its query tokens
    ([1500, 2900], 64, 16, 2),          # split across workers
])
def test_multi_token_matches_oracle(kernel, lens, heads, P, Q):
    x = I.make_inputs("mq", lens, heads, P, seed=41, q_len=Q, poison=True, slack_pages=3)
    d = to_device(x)
    out, lse = _run_multi(x, d, kernel)
    ref_out, ref_lse = _oracle(x)
    assert_parity(out, lse, ref_out, ref_lse, f"{kernel} Q={Q} {lens}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_single_query_plan_equals_plain_plan(kernel):
    x1 = I.make_inputs("mq1", [33, 700, 9], 16, 16, seed=5, q_len=1)
    d = to_device(x1)
    out, lse = _run_multi(x1, d, kernel)
    x0 = I.make_inputs("mq1", [33, 700, 9], 16, 16, seed=5)
    d0 = to_device(x0)
    ref_out, ref_lse = run_decode(x0, d0, kernel, torch.float32)
    assert np.array_equal(out[:, 0], ref_out) and np.array_equal(lse[:, 0], ref_lse)


def test_multi_token_deepseek_shape_mtp2():
    """Two query tokens per request on the decode shape of the bench (64
    requests x 4096 tokens, 128 heads): every request against the oracle."""
    x = I.make_inputs("mtp2", [4096] * 64, 128, 64, seed=3, q_len=2)
    d = to_device(x)
    out, lse = _run_multi(x, d, "tcgen05")
    ref_out, ref_lse = _oracle(x)
    assert_parity(out, lse, ref_out, ref_lse, "deepseek mtp2")


@pytest.mark.parametrize("bad, status", [
    (dict(q_len=0), mla.ERR_INVALID_ARG),
    (dict(q_len=10), mla.ERR_INVALID_ARG),        # a request shorter than its query block
    (dict(q_len=3, max_batch=5), mla.ERR_CAPACITY),
])
def test_multi_token_plan_rejects_bad_arguments(bad, status):
    x = I.make_inputs("mqbad", [9, 40], 16, 16, seed=2)
    d = to_device(x)
    dec = mla.MLADecoder(bad.get("max_batch", 64), 16, "tcgen05")
    try:
        with pytest.raises(mla.MLAError) as ei:
            mla.mla_decode_plan_multi(dec.handle, x.kv_indptr, d["kv_indices"], x.kv_len,
                                      bad["q_len"], 16, 512, 64, 16, x.sm_scale)
        assert ei.value.status == status
    finally:
        dec.close()
