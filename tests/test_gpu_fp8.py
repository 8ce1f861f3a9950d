"""fp8 (e4m3) caches on every kernel against the oracle on the dequantised
values: the CTA-pair kernel multiplies the copied codes as they are with
e4m3 MMAs, against the query (scaled per row by a power of two) and P each
split into two e4m3 terms; the one-CTA tcgen05 kernel expands each copied
tile to bf16 (every e4m3 value is exact in it); both fold kv_scale into the
scores and the output; the mma.sync kernel converts while staging."""
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


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("lens, heads, P, scale", [
    ([1, 31, 32, 33, 200], 16, 32, 1.0),     # ragged tails inside a V chunk and a page
    ([129, 4000, 64], 128, 64, 0.5),         # split request, a power-of-two scale
    ([700, 2, 1500], 64, 64, 0.37),          # a scale that is not a power of two
])
def test_fp8_cache_matches_oracle(kernel, lens, heads, P, scale):
    x = I.make_inputs("f8", lens, heads, P, seed=19, kv_dtype="fp8_e4m3", kv_scale=scale,
                      poison=True, slack_pages=2)
    d = to_device(x)
    out, lse = run_decode(x, d, kernel, torch.float32)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(out, lse, ref_out, ref_lse, f"fp8 {kernel} {lens} P={P} scale={scale}")


def test_fp8_tcgen05_matches_bf16_cache_of_the_same_values():
    """An fp8 cache and the bf16 cache holding the same (exact) values give the
    same result up to summation order on the tcgen05 kernel."""
    x = I.make_inputs("f8b", [300, 1000, 77], 128, 64, seed=23, kv_dtype="fp8_e4m3")
    d = to_device(x)
    o8, l8 = run_decode(x, d, "tcgen05", torch.float32)
    d16 = dict(d, ckv=d["ckv"].to(torch.bfloat16), kpe=d["kpe"].to(torch.bfloat16))
    x16 = I.MLAInputs(**{**x.__dict__, "kv_dtype": "bf16"})
    o16, l16 = run_decode(x16, d16, "tcgen05", torch.float32)
    assert np.abs(o8 - o16).max() < 1e-4 and np.abs(l8 - l16).max() < 1e-4


@pytest.mark.parametrize("kernel", ["pair", "tcgen05", "default"])
def test_fp8_tensor_core_kernels_reject_16_token_pages(kernel):
    x = I.make_inputs("f8p16", [40, 9], 16, 16, seed=2, kv_dtype="fp8_e4m3")
    d = to_device(x)
    with pytest.raises(mla.MLAError) as ei:
        run_decode(x, d, kernel, torch.float32)
    assert ei.value.status == mla.ERR_UNSUPPORTED


def test_fp8_pair_query_row_scales():
    """Query rows of very different magnitudes (2^-20 .. 2^4 times N(0,1), one
    row of zeros): each row is scaled by its own power of two (largest
    magnitude into [2^7, 2^8)) before its split into two e4m3 terms, so every
    row keeps its precision (unscaled, e4m3 would flush the small rows'
    values below 2^-10 to zero)."""
    x = I.make_inputs("f8q", [700, 130], 128, 64, seed=43, kv_dtype="fp8_e4m3")
    rng = np.random.Generator(np.random.PCG64(7))
    exps = rng.integers(-20, 5, size=(x.batch, x.num_heads)).astype(np.float64)
    exps[0, 5] = np.nan                                   # a zero row
    for name in ("q_nope", "q_pe"):
        q = O.decode_bf16(getattr(x, name))
        f = np.where(np.isnan(exps), 0.0, np.exp2(np.nan_to_num(exps)))[..., None]
        q32 = torch.from_numpy((q * f).astype(np.float32)).to(torch.bfloat16)
        setattr(x, name, q32.view(torch.int16).numpy().view(np.uint16))
    d = to_device(x)
    out, lse = run_decode(x, d, "pair", torch.float32)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert_parity(out, lse, ref_out, ref_lse, "fp8 pair, scaled query rows")


@pytest.mark.parametrize("kernel", KERNELS)
def test_kv_scale_is_ignored_for_bf16_caches(kernel):
    """kv_scale dequantises fp8 codes; a bf16 cache holds its values as they are."""
    x = I.make_inputs("s16", [90, 500], 32, 32, seed=29)
    d = to_device(x)
    o1, l1 = run_decode(x, d, kernel, torch.float32)
    x2 = I.MLAInputs(**{**x.__dict__, "kv_scale": 3.0})
    o2, l2 = run_decode(x2, d, kernel, torch.float32)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_cache_of_the_wrong_width_is_rejected_before_any_launch():
    """fp8 codes reinterpreted as bf16 (rows half as wide as the layout says)
    would make the kernel read past the buffer: the binding refuses them."""
    x = I.make_inputs("f8w", [100, 30], 16, 32, seed=3, kv_dtype="fp8_e4m3")
    d = to_device(x)
    as_bf16 = d["ckv"].view(torch.uint8).view(torch.bfloat16)       # [pages, P, 256]
    kpe16 = d["kpe"].view(torch.uint8).view(torch.bfloat16)         # [pages, P, 32]
    dec = mla.MLADecoder(x.batch, x.num_heads, "tcgen05")
    try:
        dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, x.page_size, x.sm_scale)
        with pytest.raises(ValueError):
            dec.run(d["q_nope"], d["q_pe"], as_bf16, kpe16)
    finally:
        dec.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_every_finite_fp8_code_converts_exactly(kernel):
    """Requests of one token: the output is that token's ckv row itself
    (softmax of one score is 1), so it must equal the stored values exactly.
    The row holds every finite e4m3 code, subnormals included; the scores
    (lse) come from the same converted values."""
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)   # 254 codes
    row = np.concatenate([finite, finite[::-1], np.zeros(4, np.uint8)])               # 512
    rng = np.random.Generator(np.random.PCG64(5))
    x = I.make_inputs("codes", [1, 1, 1, 1], 16, 32, seed=31, kv_dtype="fp8_e4m3")
    for b in range(x.batch):
        page = x.kv_indices[x.kv_indptr[b]]
        x.ckv[page, 0, :] = np.roll(row, 37 * b)
        x.kpe[page, 0, :] = rng.choice(finite, size=64)
    d = to_device(x)
    out, lse = run_decode(x, d, kernel, torch.float32)
    ref_out, ref_lse = O.mla_decode_inputs(x)
    assert np.array_equal(out, ref_out), "a converted code differs from its e4m3 value"
    assert np.abs(lse - ref_lse).max() < 1e-3
