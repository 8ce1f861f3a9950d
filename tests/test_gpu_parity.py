"""GPU parity: the CUDA path, called through the C ABI, against the float64
oracle on the same seeded inputs.

Floating-point bar (fp32 output): max-abs <= 1e-2, relative L2 <= 5e-3 and
|delta lse| <= 1e-3.  A bf16 output must equal the RNE bf16 rounding of the
fp32 output to within one bf16 ulp.  Every batch, the full-size workloads
included, is compared element by element over all of its requests.
"""
import functools

import numpy as np
import pytest
import torch

from gpu_helpers import assert_parity, bf16_round, run_decode, to_device
from oracle import mla_oracle as O
from paged_mla_decode_02_gb300 import build as B
from paged_mla_decode_02_gb300 import inputs as I
from paged_mla_decode_02_gb300 import mla

pytestmark = pytest.mark.gpu

KERNELS = ["pair", "tcgen05", "mma_sync"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    mla.load_library()


@functools.lru_cache(maxsize=2)
def _config(name, poison=False):
    return I.make_config(name, poison=poison)


@functools.lru_cache(maxsize=2)
def _oracle(name):
    return O.mla_decode_inputs(_config(name))


def _check_all(x, kernel, out_dtype=torch.float32, what=""):
    d = to_device(x)
    out, lse = run_decode(x, d, kernel, out_dtype)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    return assert_parity(out, lse, ref_out, ref_lse, what or x.name)


# ---------------------------------------------------------------------------
# small batches, every output compared
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny(kernel):
    _check_all(_config("tiny"), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny_poisoned_pool(kernel):
    # unused pool pages and the slots past kv_len in last pages hold NaN
    _check_all(_config("tiny", poison=True), kernel)


SHAPES = [
    # (kv_len list, heads, page_size)
    ([1], 16, 16),
    ([1, 2, 31, 32, 33], 16, 16),
    ([64, 65, 127, 128, 129], 32, 32),
    ([200, 17, 1000], 128, 64),
    ([5, 300], 1, 16),
    ([257, 96, 3], 64, 32),
    ([4000, 1, 777], 128, 16),
    ([2048] * 3, 100, 64),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("lens, heads, P", SHAPES)
def test_small_shapes(kernel, lens, heads, P):
    x = I.make_inputs("shape", lens, heads, P, seed=11, poison=True, slack_pages=3)
    _check_all(x, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_sharp_softmax(kernel):
    # keys x3 as in the long-context workload: scores spread over ~+-15 sigma
    x = I.make_inputs("sharp", [3000, 129], 16, 64, seed=3, key_scale=3.0)
    _check_all(x, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("sm_scale", [0.0, -0.05, 1.0 / 24.0])
def test_degenerate_and_negative_scales(kernel, sm_scale):
    # sm_scale 0: uniform weights (out = mean of the ckv rows, lse = ln L);
    # a negative scale flips the ordering of the scores
    x = I.make_inputs("scale", [45, 100, 7], 32, 16, seed=12, sm_scale=sm_scale, poison=True,
                      slack_pages=2)
    _check_all(x, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_empty_requests(kernel):
    x = I.make_inputs("empty", [0, 40, 0, 1], 16, 16, seed=5, poison=True, slack_pages=2)
    d = to_device(x)
    out, lse = run_decode(x, d, kernel)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    assert_parity(out, lse, ref_out, ref_lse, "empty")


@pytest.mark.parametrize("kernel", KERNELS)
def test_bf16_output_is_rounded_fp32_output(kernel):
    x = I.make_inputs("bf16out", [700, 33, 64], 128, 16, seed=9)
    d = to_device(x)
    o32, l32 = run_decode(x, d, kernel, torch.float32)
    o16, l16 = run_decode(x, d, kernel, torch.bfloat16)
    r = bf16_round(o32)
    ulp = np.abs(r) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(o16 - r) <= ulp)
    np.testing.assert_array_equal(l16, l32)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(o32, l32, ref_out, ref_lse, "bf16out fp32")


@pytest.mark.parametrize("kernel", KERNELS)
def test_page_table_permutation_invariance(kernel):
    x = I.make_inputs("perm", [300, 77], 32, 16, seed=4)
    d = to_device(x)
    o1, l1 = run_decode(x, d, kernel)
    rng = np.random.Generator(np.random.PCG64(99))
    perm = rng.permutation(x.num_pages)          # new position of each old page
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    x2 = I.MLAInputs(**{**x.__dict__})
    x2.ckv = x.ckv[inv]
    x2.kpe = x.kpe[inv]
    x2.kv_indices = perm[x.kv_indices].astype(np.int32)
    o2, l2 = run_decode(x2, to_device(x2), kernel)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("kernel", KERNELS)
def test_out_of_range_page_is_reported(kernel):
    x = I.make_inputs("oob", [40, 20], 16, 16, seed=2)
    d = to_device(x)
    bad = d["kv_indices"].clone()
    bad[1] = x.num_pages + 5                     # checked by the kernel before any read
    dec = mla.MLADecoder(x.batch, x.num_heads, kernel)
    dec.plan(x.kv_indptr, bad, x.kv_len, x.page_size, x.sm_scale)
    dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out_dtype=torch.float32)
    with pytest.raises(mla.MLAError) as ei:
        dec.check_status()
    assert ei.value.status == mla.ERR_DEVICE_BOUNDS
    dec.check_status()                           # the error word was cleared
    dec.close()


# ---------------------------------------------------------------------------
# streams, graphs, host-buffer entry point, re-planning
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_nondefault_stream_and_graph_replay(kernel):
    x = I.make_inputs("graph", [500, 1200, 64], 128, 64, seed=8, pool_pages=40)
    d = to_device(x)
    idx = torch.zeros(40, dtype=torch.int32, device="cuda")     # page-table buffer, fixed address
    idx[: len(x.kv_indices)].copy_(d["kv_indices"])
    ref_out, ref_lse = O.mla_decode_inputs(x)
    dec = mla.MLADecoder(x.batch, x.num_heads, kernel)
    s = torch.cuda.Stream()
    out = torch.empty((x.batch, x.num_heads, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((x.batch, x.num_heads), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        dec.plan(x.kv_indptr, idx, x.kv_len, x.page_size, x.sm_scale)
        dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out, lse)
    s.synchronize()
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse, "stream")
    out.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], out, lse)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    dec.check_status()
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse, "graph")
    # new lengths, new page table and new cache contents in the same buffers:
    # re-plan with the same plan object and replay the captured graph
    x2 = I.make_inputs("graph2", [64, 1300, 999], 128, 64, seed=21, pool_pages=40)
    d2 = to_device(x2)
    for k in ("q_nope", "q_pe", "ckv", "kpe"):
        d[k].copy_(d2[k])
    idx[: len(x2.kv_indices)].copy_(d2["kv_indices"])
    dec.plan(x2.kv_indptr, idx, x2.kv_len, x2.page_size, x2.sm_scale)
    g.replay()
    torch.cuda.synchronize()
    dec.check_status()
    r2o, r2l = O.mla_decode_inputs(x2)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), r2o, r2l, "replan+replay")
    dec.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_graph_replay_after_replan_to_a_smaller_batch(kernel):
    """A run captured at batch 3 replays after the same plan is re-planned
    for batch 2 (new lengths, pages and cache contents in the same buffers):
    the captured query and output extents cover the smaller batch."""
    x = I.make_inputs("g3", [700, 64, 1500], 128, 64, seed=31, pool_pages=48)
    x2 = I.make_inputs("g2", [1300, 257], 128, 64, seed=32, pool_pages=48)
    d, d2 = to_device(x), to_device(x2)
    idx = torch.zeros(48, dtype=torch.int32, device="cuda")
    idx[: len(x.kv_indices)].copy_(d["kv_indices"])
    qn, qp, ckv, kpe = (d[k].clone() for k in ("q_nope", "q_pe", "ckv", "kpe"))
    out = torch.empty((x.batch, x.num_heads, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((x.batch, x.num_heads), dtype=torch.float32, device="cuda")
    dec = mla.MLADecoder(x.batch, x.num_heads, kernel)
    dec.plan(x.kv_indptr, idx, x.kv_len, x.page_size, x.sm_scale)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec.run(qn, qp, ckv, kpe, out, lse)
    g.replay()
    torch.cuda.synchronize()
    dec.check_status()
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse, "batch 3")
    qn[:2].copy_(d2["q_nope"])
    qp[:2].copy_(d2["q_pe"])
    ckv.copy_(d2["ckv"])
    kpe.copy_(d2["kpe"])
    idx.zero_()
    idx[: len(x2.kv_indices)].copy_(d2["kv_indices"])
    dec.plan(x2.kv_indptr, idx, x2.kv_len, x2.page_size, x2.sm_scale)
    g.replay()
    torch.cuda.synchronize()
    dec.check_status()
    r2o, r2l = O.mla_decode_inputs(x2)
    assert_parity(out[:2].double().cpu().numpy(), lse[:2].double().cpu().numpy(), r2o, r2l,
                  "re-planned to batch 2")
    dec.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_run_host_entry_point(kernel):
    x = I.make_inputs("host", [100, 3000], 128, 64, seed=6)
    d = to_device(x)
    dec = mla.MLADecoder(x.batch, x.num_heads, kernel)
    dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, x.page_size, x.sm_scale)
    qn = d["q_nope"].cpu().pin_memory()
    qp = d["q_pe"].cpu().pin_memory()
    out = torch.empty((x.batch, x.num_heads, 512), dtype=torch.float32).pin_memory()
    lse = torch.empty((x.batch, x.num_heads), dtype=torch.float32).pin_memory()
    mla.mla_decode_run_host(dec.handle, qn, qp, d["ckv"], d["kpe"], out, lse)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(out.double().numpy(), lse.double().numpy(), ref_out, ref_lse, "run_host")
    dec.close()


def test_bad_arguments_are_errors():
    x = I.make_inputs("args", [40], 16, 16, seed=1)
    d = to_device(x)
    dec = mla.MLADecoder(4, 16)
    with pytest.raises(mla.MLAError) as ei:
        dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"])
    assert ei.value.status == mla.ERR_NOT_PLANNED
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_plan(dec.handle, x.kv_indptr, d["kv_indices"], x.kv_len, 16, 16, 64, 16, 0.1)
    assert ei.value.status == mla.ERR_UNSUPPORTED        # num_kv_heads passed as head_dim_ckv
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_plan(dec.handle, x.kv_indptr, d["kv_indices"], x.kv_len, 32, 512, 64, 16, 0.1)
    assert ei.value.status == mla.ERR_INVALID_ARG        # heads differ from the plan's
    big = I.make_inputs("big", [1] * 5, 16, 16, seed=1)
    with pytest.raises(mla.MLAError) as ei:
        dec.plan(big.kv_indptr, to_device(big)["kv_indices"], big.kv_len, 16, 0.1)
    assert ei.value.status == mla.ERR_CAPACITY
    dec.close()


# ---------------------------------------------------------------------------
# full-size workloads, every request
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("cfg", ["deepseek", "ragged", "long_b1", "long_b4", "fp8"])
def test_full_size_config(kernel, cfg):
    # the launch configuration the bench times (the same plan over the whole
    # batch), every output element against the oracle
    x = _config(cfg)
    d = to_device(x)
    out, lse = run_decode(x, d, kernel, torch.float32)
    ref_out, ref_lse = _oracle(cfg)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert_parity(out, lse, ref_out, ref_lse, cfg)
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", ["deepseek", "fp8"])
def test_default_kernel_full_size(cfg):
    # DEFAULT plans for the CTA-pair kernel, which runs both caches here
    x = _config(cfg)
    d = to_device(x)
    dec = mla.MLADecoder(x.batch, x.num_heads, "default")
    out, lse = run_decode(x, d, "default", torch.float32, decoder=dec)
    info = dec.info()
    assert info["kernel"] == mla.KERNEL_PAIR and info["tile_tokens"] == 256
    dec.close()
    ref_out, ref_lse = _oracle(cfg)
    assert_parity(out, lse, ref_out, ref_lse, cfg + " default")
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("lens", [[20000, 1, 777, 0, 300], [9000] * 9 + [40]])
def test_default_kernel_fp8_split_requests(lens):
    # fp8 split requests on the default kernel (partials combined by the merge
    # kernel); repeated runs are bit-identical
    x = I.make_inputs("default_fp8", lens, 128, 64, seed=23, kv_dtype="fp8_e4m3")
    d = to_device(x)
    dec = mla.MLADecoder(x.batch, x.num_heads, "default")
    o0, l0 = run_decode(x, d, "default", torch.float32, decoder=dec)
    assert dec.info()["num_partial_slots"] > 0, "the batch was meant to split requests"
    o1, l1 = run_decode(x, d, "default", torch.float32, decoder=dec)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    dec.close()
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(o0, l0, ref_out, ref_lse, "default fp8 splits")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("cfg, lens, heads, P", [
    ("split_many", [20000, 1, 777], 128, 16),  # one request over ~two dozen units
    ("ragged", None, None, None),              # many requests split in two or three
])
def test_split_requests_deterministic(kernel, cfg, lens, heads, P):
    # Split requests are combined by whichever unit finishes last; the result
    # must not depend on which one that is: repeated runs are bit-identical.
    x = _config(cfg) if lens is None else I.make_inputs(cfg, lens, heads, P, seed=13)
    d = to_device(x)
    dec = mla.MLADecoder(x.batch, x.num_heads, kernel)
    o0, l0 = run_decode(x, d, kernel, torch.float32, decoder=dec)
    for _ in range(3):
        o1, l1 = run_decode(x, d, kernel, torch.float32, decoder=dec)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    dec.close()
    ref_out, ref_lse = _oracle(cfg) if lens is None else O.mla_decode_inputs(x)
    assert_parity(o0, l0, ref_out, ref_lse, cfg)
    del d
    torch.cuda.empty_cache()
