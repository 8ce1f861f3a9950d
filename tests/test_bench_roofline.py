"""The algorithmic bytes and flops bench.py divides by (the roofline's
numerator), recomputed here from the layout of the data the kernel must
touch."""
from __future__ import annotations

from types import SimpleNamespace

import numpy as np
import pytest

import bench


def _shape(batch, heads, kv_len, page, q_len=1, kv_dtype="bf16"):
    lens = np.full(batch, kv_len, np.int32)
    pages = batch * -(-kv_len // page)
    return SimpleNamespace(total_tokens=int(lens.sum()), kv_dtype=kv_dtype, num_heads=heads,
                           batch=batch, q_len=q_len, kv_len=lens,
                           kv_indices=np.zeros(pages, np.int32))


def test_deepseek_shape_totals():
    # cache: 64 x 4096 tokens x (512 + 64) bf16; per (request, head): q_nope
    # + q_pe in (576 bf16), out (512 bf16), lse (fp32); one int32 page id per
    # page, 8 bytes of lengths per request
    x = _shape(64, 128, 4096, 64)
    nbytes, flops = bench.algorithmic(x)
    cache = 64 * 4096 * 576 * 2
    per_row = 64 * 128 * (576 * 2 + 512 * 2 + 4)
    assert nbytes == cache + per_row + 64 * 64 * 4 + 64 * 8 == 319_865_344
    # QK^T: 576 multiply-adds per token and head, P.V: 512
    assert flops == 64 * 4096 * 128 * 2 * (576 + 512) == 73_014_444_032


def test_fp8_cache_counts_one_byte_per_element():
    b16, f16 = bench.algorithmic(_shape(4, 16, 1000, 32))
    b8, f8 = bench.algorithmic(_shape(4, 16, 1000, 32, kv_dtype="fp8_e4m3"))
    assert b16 - b8 == 4 * 1000 * 576 and f16 == f8


@pytest.mark.parametrize("Q", [1, 2, 3])
def test_query_tokens_see_their_own_prefix(Q):
    # query j of a request attends to kv_len - Q + 1 + j tokens
    x = _shape(3, 8, 50, 16, q_len=Q)
    _, flops = bench.algorithmic(x)
    seen = 3 * sum(50 - Q + 1 + j for j in range(Q))
    assert flops == seen * 8 * 2 * (576 + 512)
