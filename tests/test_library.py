"""CPU tests of the C ABI library: it loads without a GPU, exports every
symbol the public header declares, and its host planner partitions batches
correctly and rejects malformed ones with the documented status codes."""
import math
import os
import re

import numpy as np
import pytest

from paged_mla_decode_02_gb300 import build as B
from paged_mla_decode_02_gb300 import mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return mla.load_library()


def _declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(mla_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert {"mla_decode_plan", "mla_decode_run"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(mla.EXPORTED) == declared


def test_status_strings(lib):
    for code in range(8):
        assert mla.status_string(code)
    assert mla.status_string(0) == "ok"


def _batch(lens, P):
    lens = np.asarray(lens, np.int32)
    pages = (lens + P - 1) // P
    indptr = np.zeros(len(lens) + 1, np.int32)
    indptr[1:] = np.cumsum(pages)
    return indptr, lens


def _check_partition(lens, P, W, T):
    indptr, lens = _batch(lens, P)
    units, wptr, merge, n_slots = mla.mla_plan_partition_host(indptr, lens, W, T, P)
    # worker ranges are contiguous in the unit list
    assert wptr[0] == 0 and wptr[-1] == len(units) and np.all(np.diff(wptr) >= 0)
    # every request's tokens covered exactly once, in order, tile-aligned
    cover = {b: [] for b in range(len(lens))}
    for req, t0, t1, slot, base, L in units:
        assert base == indptr[req] and L == lens[req]
        assert t0 % T == 0 and 0 <= t0 < t1 <= L
        cover[req].append((t0, t1, slot))
    for b, L in enumerate(lens):
        segs = cover[b]
        if L == 0:
            assert segs == []
            continue
        assert segs[0][0] == 0 and segs[-1][1] == L
        for (a0, a1, _), (b0, b1, _) in zip(segs, segs[1:]):
            assert a1 == b0
        if len(segs) == 1:
            assert segs[0][2] == -1
    # balance under the planner's cost model (quarter tiles): a tile costs
    # TILE, a unit UNIT more, a unit of a split request SPLIT more again.  The
    # largest worker cost stays within a fixed margin of the perfect share of
    # the work that cannot be avoided (tiles and one unit per request); every
    # piece of a split request has at least MIN_PIECE tiles.
    TILE, UNIT, SPLIT, MIN_PIECE = 4, 8, 4, 4
    tiles = np.zeros(W, np.int64)
    cost = np.zeros(W, np.int64)
    for w in range(W):
        for u in units[wptr[w]:wptr[w + 1]]:
            n = (u[2] - u[1] + T - 1) // T
            tiles[w] += n
            cost[w] += TILE * n + UNIT + (SPLIT if u[3] >= 0 else 0)
    total = int(((lens + T - 1) // T).sum())
    assert tiles.sum() == total
    share = (TILE * total + UNIT * int((lens > 0).sum())) / W
    assert cost.max() <= share + 2 * (UNIT + SPLIT) + TILE * MIN_PIECE, (cost.max(), share)
    assert len(units) <= W + len(lens)
    for b in range(len(lens)):
        if len(cover[b]) > 1:
            assert min((t1 - t0 + T - 1) // T for t0, t1, _ in cover[b]) >= MIN_PIECE
    # merge entries: split requests get consecutive slots, empty ones n_slots 0
    used = []
    for req, first, n in merge:
        if lens[req] == 0:
            assert n == 0
            continue
        slots = [s for (_, _, s) in cover[req]]
        assert n == len(slots) >= 2 and slots == list(range(first, first + n))
        used += slots
    assert sorted(used) == list(range(n_slots))
    return units, merge


@pytest.mark.parametrize("T", [64, 128])
@pytest.mark.parametrize("P", [16, 32, 64])
def test_partition_random_batches(lib, T, P):
    rng = np.random.Generator(np.random.PCG64(7))
    for trial in range(30):
        B_ = int(rng.integers(1, 40))
        lens = rng.integers(0, 3000, size=B_)
        lens[rng.random(B_) < 0.1] = 0
        W = int(rng.integers(1, 100))
        _check_partition(lens, P, W, T)


def test_partition_named_shapes(lib):
    _check_partition([33, 70], 16, 76, 128)
    _check_partition([4096] * 64, 64, 76, 128)
    _check_partition([131072], 64, 76, 128)
    _check_partition([0, 0, 5], 16, 3, 128)


def test_partition_long_request_split_over_the_workers(lib):
    # 1024 tiles on 76 workers: pieces of at most 14 tiles (the smallest
    # whole-tile share), one per worker, all merged as one request
    units, merge = _check_partition([131072], 64, 76, 128)
    pieces = (units[:, 2] - units[:, 1] + 127) // 128
    assert pieces.max() == 14 and len(units) == 74
    assert merge.shape[0] == 1 and merge[0, 2] == len(units)


@pytest.mark.parametrize("bad, status", [
    (dict(head_dim_ckv=1), mla.ERR_UNSUPPORTED),      # e.g. the KV-head count passed by mistake
    (dict(head_dim_kpe=128), mla.ERR_UNSUPPORTED),
    (dict(page_size=8), mla.ERR_UNSUPPORTED),
    (dict(sm_scale=math.inf), mla.ERR_INVALID_ARG),
    (dict(sm_scale=math.nan), mla.ERR_INVALID_ARG),
    (dict(tile_tokens=32), mla.ERR_UNSUPPORTED),
])
def test_partition_rejects_bad_arguments(lib, bad, status):
    indptr, lens = _batch([33, 70], 16)
    kw = dict(head_dim_ckv=512, head_dim_kpe=64, page_size=16, sm_scale=0.1, tile_tokens=128)
    kw.update(bad)
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_plan_partition_host(indptr, lens, 4, kw["tile_tokens"], kw["page_size"],
                                    kw["head_dim_ckv"], kw["head_dim_kpe"], kw["sm_scale"])
    assert ei.value.status == status


def test_partition_rejects_inconsistent_paging(lib):
    indptr, lens = _batch([33, 70], 16)
    bad = indptr.copy()
    bad[1] += 1                                  # request 0 claims 4 pages for 33 tokens
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_plan_partition_host(bad, lens, 4, 128, 16)
    assert ei.value.status == mla.ERR_INVALID_ARG
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_plan_partition_host(indptr, np.array([33, -1], np.int32), 4, 128, 16)
    assert ei.value.status == mla.ERR_INVALID_ARG
    nz = indptr.copy()
    nz[0] = 1
    with pytest.raises(mla.MLAError):
        mla.mla_plan_partition_host(nz, lens, 4, 128, 16)


# the planner's cost constants (tile, unit, split, minimum piece) per tile size
COSTS = {128: (4, 8, 4, 4), 256: (4, 4, 2, 2)}


def _greedy_fits(lens, W, T, budget):
    """The planner's fill rule, restated: requests in order, whole while they
    fit, else cut where the worker fills up (both pieces >= MIN_PIECE tiles)."""
    TILE, UNIT, SPLIT, MIN_PIECE = COSTS[T]
    w, used = 0, 0
    for L in lens:
        n = (int(L) + T - 1) // T
        t, split = 0, False
        while t < n:
            if w >= W:
                return False
            whole = UNIT + TILE * (n - t) + (SPLIT if split else 0)
            if used + whole <= budget:
                used += whole
                break
            take = min((budget - used - UNIT - SPLIT) // TILE, n - t - MIN_PIECE)
            if take < MIN_PIECE:
                if used == 0:
                    return False
                w, used = w + 1, 0
                continue
            t += take
            split = True
            w, used = w + 1, 0
    return True


@pytest.mark.parametrize("T", [128, 256])
def test_partition_makespan_is_the_smallest_feasible_budget(lib, T):
    # The fill's success is not monotone in the budget, so a bisection alone
    # can stop above the best budget (one request of 19 tiles on 5 workers:
    # 40 against 32).  The planner's largest worker cost must equal the
    # smallest budget a linear scan finds.
    P = 64
    TILE, UNIT, SPLIT, _ = COSTS[T]
    rng = np.random.Generator(np.random.PCG64(23))
    cases = [([19 * T], 5)]
    for _ in range(40):
        B_ = int(rng.integers(1, 6))
        cases.append((list(rng.integers(1, 40 * T, size=B_)), int(rng.integers(1, 12))))
    for lens, W in cases:
        indptr, l32 = _batch(lens, P)
        units, wptr, _, _ = mla.mla_plan_partition_host(indptr, l32, W, T, P)
        cost = [sum(TILE * ((u[2] - u[1] + T - 1) // T) + UNIT + (SPLIT if u[3] >= 0 else 0)
                    for u in units[wptr[w]:wptr[w + 1]]) for w in range(W)]
        best = next(b for b in range(1, 10 ** 6) if _greedy_fits(l32, W, T, b))
        assert max(cost) <= best, (lens, W, max(cost), best)
