"""Pins for the oracle's FlatParameter layout, pack, views and all-gather.

The oracle is checked against the worked example of "Infra: Data Parallel"
(FSDP1 figure, fixture in tests/golden) and against invariants checked by
element tracking, by brute force over every small unit."""
import itertools
import os
import random

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_worked_example_24_elements():
    rows = _read_fixture("fsdp1_worked_example.txt")
    kv = {r[0]: r[1:] for r in rows if r[0] in ("shapes", "nd", "total", "padded", "shard")}
    shapes = [tuple(int(x) for x in s.split("x")) for s in kv["shapes"]]
    nd = int(kv["nd"][0])
    # W1, W2, W3 with distinct element values so every element can be traced
    tensors = [np.arange(1, 9, dtype=np.float32).reshape(s) + 100 * (t + 1)
               for t, s in enumerate(shapes)]
    flat, lay = oracle.flat_pack(tensors, nd)
    assert lay.total == int(kv["total"][0])
    assert lay.padded == int(kv["padded"][0])
    assert lay.shard == int(kv["shard"][0])
    shards = [oracle.shard_of(flat, lay, r) for r in range(nd)]
    for r in range(nd):
        assert shards[r].shape == (lay.shard,)
    for _, r, t, first, count in (x for x in rows if x[0] == "piece"):
        r, t, first, count = int(r), int(t), int(first), int(count)
        view = oracle.sharded_views(shards[r], lay, r)[t]
        assert view.size == count
        assert np.array_equal(view, tensors[t].reshape(-1)[first:first + count])
    for _, r, t, rowlist in (x for x in rows if x[0] == "rows"):
        r, t = int(r), int(t)
        view = oracle.sharded_views(shards[r], lay, r)[t]
        want = [] if rowlist == "-" else [int(i) for i in rowlist.split(",")]
        got = tensors[t][want].reshape(-1) if want else np.zeros(0, np.float32)
        assert np.array_equal(view, got)
    full, views = oracle.ag_unpack(shards, lay, shapes)
    for t in range(3):
        assert views[t].shape == shapes[t]
        assert np.array_equal(views[t], tensors[t])


def _check_unit(numels, nd, dtype=np.uint16):
    # element (t, k) carries the id 1 + (offset of t) + k, padding stays 0
    tensors = []
    nxt = 1
    for n in numels:
        tensors.append(np.arange(nxt, nxt + n, dtype=np.int64).astype(dtype))
        nxt += n
    flat, lay = oracle.flat_pack(tensors, nd)
    T = sum(numels)
    assert lay.total == T
    assert lay.padded % nd == 0 and 0 <= lay.padded - T < nd
    assert lay.shard * nd == lay.padded
    # flat: tensors back to back in registration order, zeros after
    assert np.array_equal(flat[:T], np.arange(1, T + 1).astype(dtype))
    assert not flat[T:].any()
    shards = [oracle.shard_of(flat, lay, r) for r in range(nd)]
    # the union of the shards, in rank order, is the whole flat buffer
    assert np.array_equal(np.concatenate(shards) if shards else flat, flat)
    # every element of every tensor sits in exactly one rank's view, in order
    for t, ten in enumerate(tensors):
        pieces = [oracle.sharded_views(shards[r], lay, r)[t] for r in range(nd)]
        assert np.array_equal(np.concatenate(pieces), ten)
        for r in range(nd):
            lo, hi = lay.lo[r][t], lay.hi[r][t]
            assert 0 <= lo <= hi <= lay.shard
            # the piece is exactly the overlap of the tensor with the shard
            a, b = lay.offsets[t], lay.offsets[t] + ten.size
            ov = max(0, min(b, (r + 1) * lay.shard) - max(a, r * lay.shard))
            assert hi - lo == ov
    full, views = oracle.ag_unpack(shards, lay)
    assert np.array_equal(full, flat)
    for ten, v in zip(tensors, views):
        assert np.array_equal(v, ten)


def test_brute_force_small_units():
    for K in range(0, 4):
        for numels in itertools.product(range(0, 8), repeat=K):
            for nd in range(1, 6):
                _check_unit(list(numels), nd)


def test_random_units_four_tensors():
    rng = random.Random(0)
    for _ in range(400):
        numels = [rng.randrange(0, 40) for _ in range(4)]
        _check_unit(numels, rng.randrange(1, 9))


@pytest.mark.parametrize("dtype", [np.uint16, np.float32])
def test_pack_is_a_bit_copy(dtype):
    rng = np.random.default_rng(1)
    nbits = 16 if dtype == np.uint16 else 32
    raw = [rng.integers(0, 1 << nbits, size=n, dtype=np.uint64) for n in (5, 11, 3)]
    itype = np.uint16 if dtype == np.uint16 else np.uint32
    tensors = [r.astype(itype).view(dtype) for r in raw]   # includes NaN patterns for fp32
    flat, lay = oracle.flat_pack(tensors, 4)
    back = oracle.unpack_views(flat, lay)
    for a, b in zip(tensors, back):
        assert a.view(itype).tobytes() == b.view(itype).tobytes()


def test_rank_with_no_piece_of_a_tensor_gets_empty_view():
    # one tensor of 3 elements spread over 4 ranks: rank 3 holds only padding
    lay = oracle.layout([3], 4)
    assert (lay.padded, lay.shard) == (4, 1)
    sizes = [lay.hi[r][0] - lay.lo[r][0] for r in range(4)]
    assert sizes == [1, 1, 1, 0]


def test_layout_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.layout([1, 2], 0)
    with pytest.raises(ValueError):
        oracle.layout([-1], 2)


# ---------------------------------------- element sources (the inverse of pack)

def _tagged(numels, u=0):
    # tensor t's element k holds the value u * 10^6 + (t + 1) * 10^4 + k (exact in
    # float64), so every element of a packed buffer names its source
    return [(u * 10 ** 6 + (t + 1) * 10 ** 4 + np.arange(n)).astype(np.float64)
            for t, n in enumerate(numels)]


def test_element_source_inverts_flat_pack_by_brute_force():
    for nd in range(1, 6):
        for k in range(0, 4):
            for numels in itertools.product(range(0, 6), repeat=k):
                flat, lay = oracle.flat_pack(_tagged(numels), nd) if k else \
                    (np.zeros(0), oracle.layout([], nd))
                t, kk = oracle.element_source(lay, np.arange(lay.padded))
                for f in range(lay.padded):
                    if t[f] < 0:
                        assert f >= lay.total and flat[f] == 0
                    else:
                        assert flat[f] == (t[f] + 1) * 10 ** 4 + kk[f]


def test_element_source_on_the_worked_example():
    # [W1(8) | W2(8) | W3(8)] on two ranks: element 12 (rank 1's first) is W2
    # row 2 column 0, i.e. W2's element 4; element 23 is W3's last
    lay = oracle.layout([8, 8, 8], 2)
    t, k = oracle.element_source(lay, [0, 11, 12, 15, 16, 23])
    assert list(t) == [0, 1, 1, 1, 2, 2]
    assert list(k) == [0, 3, 4, 7, 0, 7]


def test_rank_view_sources_match_the_concatenated_shards():
    rnd = random.Random(5)
    for _ in range(200):
        nd = rnd.randint(1, 6)
        units = [[rnd.randint(0, 9) for _ in range(rnd.randint(1, 4))]
                 for _ in range(rnd.randint(1, 4))]
        packed = [oracle.flat_pack(_tagged(n, u), nd) for u, n in enumerate(units)]
        layouts = [lay for _, lay in packed]
        for r in range(nd):
            view = np.concatenate([oracle.shard_of(f, lay, r) for f, lay in packed])
            u, t, k = oracle.rank_view_sources(layouts, r, np.arange(view.size))
            for i in range(view.size):
                if t[i] < 0:
                    assert view[i] == 0
                else:
                    assert view[i] == u[i] * 10 ** 6 + (t[i] + 1) * 10 ** 4 + k[i]
            with pytest.raises(IndexError):
                oracle.rank_view_sources(layouts, r, [view.size])
