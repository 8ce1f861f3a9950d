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


@pytest.mark.parametrize("kernel", ["tcgen05", "default"])
def test_multi_token_deepseek_shape_mtp2(kernel):
    """Two query tokens per request on the decode shape of the bench (64
    requests x 4096 tokens, 128 heads): every request against the oracle.
    On the CTA-pair plan the 128 planned requests are not split: the merge
    pass over 128 shares of 128 heads would cost more than the unevenness
    of whole requests (32 against 27 tiles on the slowest worker)."""
    x = I.make_inputs("mtp2", [4096] * 64, 128, 64, seed=3, q_len=2)
    d = to_device(x)
    if kernel == "default":
        dec, out_t, lse_t = _run_multi_dec(x, d, kernel)
        try:
            assert dec.info()["num_partial_slots"] == 0
        finally:
            dec.close()
        out, lse = out_t.double().cpu().numpy(), lse_t.double().cpu().numpy()
    else:
        out, lse = _run_multi(x, d, kernel)
    ref_out, ref_lse = _oracle(x)
    assert_parity(out, lse, ref_out, ref_lse, f"deepseek mtp2 {kernel}")


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


# ---------------------------------------------------------------------------
# the CTA-pair kernel packs the query tokens of a request into its MMA rows
# (q_len x heads <= 128): one plan request per request, each row masked to
# its own prefix
# ---------------------------------------------------------------------------

def _run_multi_dec(x, d, kernel, max_batch=None):
    dec = mla.MLADecoder(max_batch or x.batch * x.q_len, x.num_heads, kernel)
    dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, x.page_size, x.sm_scale, q_len=x.q_len)
    out, lse = dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], kv_scale=x.kv_scale,
                       out_dtype=torch.float32)
    dec.check_status()
    return dec, out, lse


def _oracle_x(x):
    return O.mla_decode_multi(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                              x.kv_len, x.page_size, x.sm_scale, x.kv_dtype, x.kv_scale)


@pytest.mark.parametrize("lens, heads, P, Q, kv_dtype", [
    ([20000, 4, 777], 16, 64, 4, "bf16"),     # a request split over many workers; one of exactly Q tokens
    ([40000], 16, 64, 8, "bf16"),             # 128 rows, one request over every worker
    ([300, 257, 9], 32, 32, 3, "bf16"),       # 96 rows: the odd CTA's last 32 rows unused
    ([5000, 700, 2], 16, 64, 2, "fp8_e4m3"),  # e4m3 cache (hi + lo query and P)
])
def test_packed_query_tokens_match_oracle(lens, heads, P, Q, kv_dtype):
    x = I.make_inputs("mqp", lens, heads, P, seed=47, q_len=Q, poison=True, slack_pages=3,
                      kv_dtype=kv_dtype)
    d = to_device(x)
    dec, out, lse = _run_multi_dec(x, d, "pair")
    try:
        assert dec.info()["batch"] == x.batch      # one plan request per request: packed
        ref_out, ref_lse = _oracle_x(x)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      f"packed Q={Q} H={heads} {lens} {kv_dtype}")
        # split shares are combined in slot order: repeated runs are bit-identical
        out2, lse2 = dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], kv_scale=x.kv_scale,
                             out_dtype=torch.float32)
        dec.check_status()
        assert torch.equal(out, out2) and torch.equal(lse, lse2)
    finally:
        dec.close()


@pytest.mark.parametrize("kernel, heads, Q, packed", [
    ("pair", 16, 8, True),
    ("pair", 64, 2, True),
    ("pair", 128, 2, False),      # 256 rows do not fit one pair MMA: one plan request per token
    ("tcgen05", 16, 4, False),
    ("mma_sync", 16, 4, False),
])
def test_which_plans_pack(kernel, heads, Q, packed):
    x = I.make_inputs("mqw", [600, 64], heads, 64, seed=3, q_len=Q)
    d = to_device(x)
    dec, out, lse = _run_multi_dec(x, d, kernel)
    try:
        assert dec.info()["batch"] == (x.batch if packed else x.batch * Q)
        ref_out, ref_lse = _oracle_x(x)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      f"{kernel} H={heads} Q={Q}")
    finally:
        dec.close()


def test_packed_full_size_long_b4_mtp4():
    """The bench's long_b4_mtp4 workload (4 x 131072 tokens, 16 heads, 4 query
    tokens per request, packed) against the oracle, every request."""
    x = I.make_config("long_b4_mtp4")
    d = to_device(x)
    dec, out, lse = _run_multi_dec(x, d, "default")
    try:
        assert dec.info()["batch"] == x.batch
        ref_out, ref_lse = _oracle_x(x)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      "long_b4_mtp4")
    finally:
        dec.close()


def test_packed_plan_graph_replay_after_replan():
    """A packed run (3 query tokens x 32 heads = 96 rows per request) captured
    in a CUDA graph replays after a re-plan with the same q_len, new lengths,
    pages and cache contents in the same buffers."""
    Q, H, P = 3, 32, 64
    x = I.make_inputs("mqg1", [900, 3, 5000], H, P, seed=51, q_len=Q, pool_pages=100)
    x2 = I.make_inputs("mqg2", [4100, 777, 64], H, P, seed=52, q_len=Q, pool_pages=100)
    d, d2 = to_device(x), to_device(x2)
    idx = torch.zeros(100, dtype=torch.int32, device="cuda")
    idx[: len(x.kv_indices)].copy_(d["kv_indices"])
    qn, qp, ckv, kpe = (d[k].clone() for k in ("q_nope", "q_pe", "ckv", "kpe"))
    out = torch.empty((x.batch, Q, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((x.batch, Q, H), dtype=torch.float32, device="cuda")
    dec = mla.MLADecoder(x.batch * Q, H, "default")
    try:
        dec.plan(x.kv_indptr, idx, x.kv_len, P, x.sm_scale, q_len=Q)
        assert dec.info()["batch"] == x.batch
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            dec.run(qn, qp, ckv, kpe, out, lse)
        g.replay()
        torch.cuda.synchronize()
        dec.check_status()
        ref_out, ref_lse = _oracle_x(x)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse, "captured")
        for k, t in (("q_nope", qn), ("q_pe", qp), ("ckv", ckv), ("kpe", kpe)):
            t.copy_(d2[k])
        idx.zero_()
        idx[: len(x2.kv_indices)].copy_(d2["kv_indices"])
        dec.plan(x2.kv_indptr, idx, x2.kv_len, P, x2.sm_scale, q_len=Q)
        g.replay()
        torch.cuda.synchronize()
        dec.check_status()
        r2o, r2l = _oracle_x(x2)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), r2o, r2l, "re-planned")
    finally:
        dec.close()
