"""GPU parity on sharp score jumps: one token scores tens to hundreds of
natural-log units above the rest of its request (an attention sink at
position 0, a maximum at the first token of a later tile, at a request's last
token, inside a request split over several work units).  The online softmax
must neither overflow nor lose that token; every output element is compared
with the float64 oracle at the usual bar.
"""
import functools

import numpy as np
import pytest
import torch

from gpu_helpers import assert_parity, run_decode, to_device
from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import build as B
from paged_mla_decode_02_gb300 import inputs as I
from paged_mla_decode_02_gb300 import mla

pytestmark = pytest.mark.gpu

KERNELS = ["pair", "tcgen05", "mma_sync"]
GAPS = [40.0, 60.0, 100.0, 200.0]


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    mla.load_library()


@functools.lru_cache(maxsize=4)
def _batch(gap, heads, kv_dtype="bf16"):
    # request 0: sink at token 0 (the first tile); request 1: maximum at token
    # 128 (first token of the second 128-token tile); request 2: at its last
    # token; request 3: none; request 4: a single token
    x = I.make_inputs("dominant", [4000, 4000, 1000, 300, 1], heads, 64, seed=17,
                      kv_dtype=kv_dtype, poison=True, slack_pages=4)
    return I.plant_dominant_tokens(x, [(0, 0), (1, 128), (2, 999), (4, 0)], gap)


def _check(x, kernel, what):
    d = to_device(x)
    out, lse = run_decode(x, d, kernel, torch.float32)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert np.isfinite(out).all() and np.isfinite(lse).all(), f"{what}: non-finite output"
    return assert_parity(out, lse, ref_out, ref_lse, what)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("gap", GAPS)
@pytest.mark.parametrize("heads", [128, 16])
def test_dominant_token(kernel, gap, heads):
    _check(_batch(gap, heads), kernel, f"gap {gap} heads {heads}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("gap", [60.0, 200.0])
def test_dominant_token_in_split_requests(kernel, gap):
    # two requests long enough to be cut into many units: the maximum sits in
    # the first unit of one and the middle of the other, so it lands in a unit
    # other than the one that combines the request
    x = I.make_inputs("dominant_split", [40000, 40000, 64], 128, 64, seed=19)
    x = I.plant_dominant_tokens(x, [(0, 5), (1, 20000)], gap)
    d = to_device(x)
    dec = mla.MLADecoder(x.batch, x.num_heads, kernel)
    dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, x.page_size, x.sm_scale)
    assert dec.info()["num_partial_slots"] >= 4, "the requests were meant to be split"
    out, lse = dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out_dtype=torch.float32)
    dec.check_status()
    dec.close()
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                  f"split gap {gap}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_dominant_token_fp8_cache(kernel):
    _check(_batch(100.0, 128, "fp8_e4m3"), kernel, "fp8 gap 100")
