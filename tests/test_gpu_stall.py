"""A device wait that runs out, on purpose, in a test build of the library.

The test build (``-DMLA_STALL_TEST``, a separate shared library that the
product never loads) gives every bounded wait of the decode kernels a 1 ms
limit and has a knob per kernel that makes CTA 0's V producer leave out one
copy (the one-CTA tcgen05 kernel and the CTA-pair kernel).  The PV issuer
waiting for that copy gives up, the other roles of the cluster see the abort
or run out of time on their own waits, drain what they issued, free TMEM and
return: the kernel ends by itself.  The host then reads
MLA_ERR_DEVICE_TIMEOUT from the plan's status word, and the next run of the
same plan, knob off, must match the oracle (the kernel left no state behind).
No trap, fault or endless loop is involved: the wait is bounded by design.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from gpu_helpers import assert_parity, to_device
from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import build as B
from paged_mla_decode_02_gb300 import inputs as I
from paged_mla_decode_02_gb300 import mla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def testlib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = mla.bind_library(B.build_variant("stalltest", ["-DMLA_STALL_TEST"]))
    for fn in (lib.mla_test_set_stall, lib.mla_test_set_pair_stall):
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_int]
    return lib


KNOBS = {"tcgen05": (mla.KERNEL_TCGEN05, "mla_test_set_stall"),
         "pair": (mla.KERNEL_PAIR, "mla_test_set_pair_stall")}


def _plan(lib, x, d, kernel):
    h = ctypes.c_void_p()
    assert lib.mla_plan_create(x.batch, x.num_heads, KNOBS[kernel][0], ctypes.byref(h)) == mla.OK
    indptr = np.ascontiguousarray(x.kv_indptr, np.int32)
    lens = np.ascontiguousarray(x.kv_len, np.int32)
    st = lib.mla_decode_plan(h, indptr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                             d["kv_indices"].data_ptr(),
                             lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), x.batch,
                             x.num_heads, 512, 64, x.page_size, x.sm_scale,
                             torch.cuda.current_stream().cuda_stream)
    assert st == mla.OK
    return h


def _run(lib, h, x, d, out, lse):
    st = lib.mla_decode_run(h, d["q_nope"].data_ptr(), d["q_pe"].data_ptr(), mla.DTYPE_BF16,
                            d["ckv"].data_ptr(), d["kpe"].data_ptr(), mla.DTYPE_BF16, 1.0,
                            x.num_pages, out.data_ptr(), mla.DTYPE_FP32, lse.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    assert st == mla.OK


@pytest.mark.parametrize("kernel", ["tcgen05", "pair"])
@pytest.mark.parametrize("lens, chunk", [
    ([600, 300], 3),               # one unit per request
    ([9000, 40], 7),               # a request split over several units
])
def test_expired_wait_is_reported_and_leaves_no_state(testlib, kernel, lens, chunk):
    x = I.make_inputs("stall", lens, 128, 64, seed=31)
    d = to_device(x)
    out = torch.empty((x.batch, x.num_heads, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((x.batch, x.num_heads), dtype=torch.float32, device="cuda")
    h = _plan(testlib, x, d, kernel)
    knob = getattr(testlib, KNOBS[kernel][1])
    try:
        assert knob(chunk) == 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        _run(testlib, h, x, d, out, lse)
        assert testlib.mla_plan_check_status(h) == mla.ERR_DEVICE_TIMEOUT
        assert time.perf_counter() - t0 < 5.0      # the kernel ended by itself
        assert testlib.mla_plan_check_status(h) == mla.OK   # the word was cleared
        # knob off: the same plan, no re-plan, runs clean and right
        assert knob(0) == 0
        _run(testlib, h, x, d, out, lse)
        assert testlib.mla_plan_check_status(h) == mla.OK
        ref_out, ref_lse = O.mla_decode_inputs(x)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      "after the expired wait")
    finally:
        knob(0)
        testlib.mla_plan_destroy(h)
