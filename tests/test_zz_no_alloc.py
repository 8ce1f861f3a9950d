"""The decode entry point that allocates nothing (fixed scratch inside the
library), called through the C ABI and compared with the plan / run entry
points on the same inputs, two calls in a row.  The file is collected last so
it also runs after every other GPU test has used the library."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import assert_parity, run_decode, to_device
from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import inputs as I
from paged_mla_decode_02_gb300 import mla

pytestmark = pytest.mark.gpu


def _noalloc(x, d, out_dtype=torch.float32):
    out = torch.empty((x.batch, x.num_heads, 512), dtype=out_dtype, device="cuda")
    lse = torch.empty((x.batch, x.num_heads), dtype=torch.float32, device="cuda")
    mla.mla_decode_noalloc(x.kv_indptr, d["kv_indices"], x.kv_len, x.page_size, x.sm_scale,
                           d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out, lse,
                           kv_scale=x.kv_scale, check_status=True)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("name, lens, heads, P", [
    ("na_small", [33, 70, 0, 200], 16, 16),      # an empty request, ragged last pages
    ("na_split", [1500, 7, 3000, 64], 128, 32),  # requests split across workers
    ("na_long", [20000], 128, 64),               # one request over many units
])
def test_noalloc_matches_plan_and_run(name, lens, heads, P):
    x = I.make_inputs(name, lens, heads, P, seed=21, poison=True, slack_pages=2)
    d = to_device(x)
    ref_out, ref_lse = run_decode(x, d, "tcgen05")
    for _ in range(2):
        out, lse = _noalloc(x, d)
        assert_parity(out, lse, ref_out, ref_lse, f"{name}: no-alloc vs plan/run")
    o_ref, l_ref = O.mla_decode_inputs(x)
    assert_parity(out, lse, o_ref, l_ref, f"{name}: no-alloc vs oracle")


def test_noalloc_bf16_output_matches_plan_and_run():
    x = I.make_inputs("na_bf16", [700, 33, 4096], 128, 64, seed=5)
    d = to_device(x)
    ref_out, ref_lse = run_decode(x, d, "tcgen05", torch.bfloat16)
    for _ in range(2):
        out, lse = _noalloc(x, d, torch.bfloat16)
        assert_parity(out, lse, ref_out, ref_lse, "bf16 out: no-alloc vs plan/run")


def test_noalloc_rejects_batches_beyond_its_scratch():
    x = I.make_inputs("na_big", [1] * 4097, 16, 16, seed=1)
    d = to_device(x)
    out = torch.empty((x.batch, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((x.batch, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_noalloc(x.kv_indptr, d["kv_indices"], x.kv_len, 16, x.sm_scale,
                               d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out, lse)
    assert ei.value.status == mla.ERR_CAPACITY


def test_noalloc_error_is_kept_until_a_checking_call():
    # A step that does not check (check_status 0) and meets a page id out of
    # range: its error stays recorded, and the next call that checks reports
    # it even though that call's own inputs are good; the call after it is
    # clean again.
    x = I.make_inputs("na_err", [40, 20], 16, 16, seed=2)
    d = to_device(x)
    bad = d["kv_indices"].clone()
    bad[1] = x.num_pages + 5                     # checked by the kernel before any read
    out = torch.empty((x.batch, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((x.batch, 16), dtype=torch.float32, device="cuda")
    args = (x.kv_indptr, None, x.kv_len, x.page_size, x.sm_scale, d["q_nope"], d["q_pe"],
            d["ckv"], d["kpe"], out, lse)

    def call(idx, check):
        a = list(args)
        a[1] = idx
        mla.mla_decode_noalloc(*a, check_status=check)

    call(bad, False)
    with pytest.raises(mla.MLAError) as ei:
        call(d["kv_indices"], True)
    assert ei.value.status == mla.ERR_DEVICE_BOUNDS
    call(d["kv_indices"], True)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                  "after the reported error")


def test_noalloc_rejects_a_dequantisation_scale():
    x = I.make_inputs("na_scale", [40], 16, 16, seed=3)
    d = to_device(x)
    out = torch.empty((1, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_noalloc(x.kv_indptr, d["kv_indices"], x.kv_len, 16, x.sm_scale,
                               d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out, lse, kv_scale=0.5)
    assert ei.value.status == mla.ERR_UNSUPPORTED
