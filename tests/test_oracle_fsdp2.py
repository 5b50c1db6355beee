"""Pins for the oracle's FSDP2 per-parameter Shard(0): the examples of the
"Infra: Data Parallel" FSDP2 figure and text (fixture in tests/golden),
torch.chunk along dim 0 (the library routine DTensor's Shard(0) placement
follows), and brute-force round trips with element tracking."""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "fsdp2_shard0_examples.txt")):
        line = line.split("#", 1)[0].split()
        if not line:
            continue
        if line[0] == "case":
            cur = {"nd": int(line[3]), "shapes": [tuple(int(d) for d in x.split("x"))
                                                    for x in line[5:]],
                   "local": {}, "rows": {}}
            cases.append(cur)
        elif line[0] == "local":
            cur["local"][int(line[1])] = [tuple(int(d) for d in x.split("x")) for x in line[2:]]
        elif line[0] == "rows":
            cur["rows"][int(line[1])] = [tuple(int(d) for d in x.split("-")) for x in line[2:]]
        elif line[0] == "elements":
            cur["elements"] = int(line[1])
    return cases


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"nd{c['nd']}")
def test_page_examples(case):
    shapes, nd = case["shapes"], case["nd"]
    lay = oracle.fsdp2_layout(shapes, nd)
    tensors = [np.arange(int(np.prod(s)), dtype=np.float32).reshape(s) + 1000 * t
               for t, s in enumerate(shapes)]
    assert lay.local == case["elements"]
    for r in range(nd):
        loc = oracle.local_shards(tensors, lay, r)
        assert [x.shape for x in loc] == case["local"][r]
        for t, (a, b) in enumerate(case["rows"][r]):
            assert np.array_equal(loc[t], tensors[t][a:b + 1])
        assert sum(x.size for x in loc) == case["elements"]
    # the global shape is kept: gathering the local pieces gives the tensors
    bufs = [oracle.local_buffer(tensors, lay, r) for r in range(nd)]
    for t, full in enumerate(oracle.all_gather_copy_out(bufs, lay)):
        assert full.shape == shapes[t] and np.array_equal(full, tensors[t])


def test_local_shards_follow_torch_chunk_along_dim0():
    for d0 in range(0, 12):
        for nd in range(1, 7):
            x = np.arange(d0 * 3, dtype=np.float32).reshape(d0, 3)
            lay = oracle.fsdp2_layout([(d0, 3)], nd)
            chunks = torch.from_numpy(x).chunk(nd, dim=0) if d0 else ()
            for r in range(nd):
                want = chunks[r].numpy() if r < len(chunks) else np.zeros((0, 3), np.float32)
                got = oracle.local_shards([x], lay, r)[0]
                assert got.shape == want.shape and np.array_equal(got, want), (d0, nd, r)


def _check(shapes, nd):
    lay = oracle.fsdp2_layout(shapes, nd)
    nxt = 1
    tensors = []
    for s in shapes:
        n = int(np.prod(s))
        tensors.append(np.arange(nxt, nxt + n, dtype=np.int64).reshape(s))
        nxt += n
    assert lay.local == sum(-(-s[0] // nd) * int(np.prod(s[1:])) for s in shapes)
    cc = oracle.chunk_cat(tensors, lay)
    assert cc.size == nd * lay.local
    seen = np.zeros(nxt, dtype=np.int64)
    for r in range(nd):
        buf = oracle.local_buffer(tensors, lay, r)
        assert np.array_equal(buf, cc[r * lay.local:(r + 1) * lay.local])
        for t, s in enumerate(shapes):
            seg = buf[lay.offset[t]:lay.offset[t] + lay.chunk[t] * lay.row[t]]
            k = lay.rows_of(r, t) * lay.row[t]
            # the rank's rows first, then zero padding rows
            assert not seg[k:].any()
            seen[seg[:k]] += 1
        pieces = oracle.local_shards(tensors, lay, r)
        for t, p in enumerate(pieces):
            assert p.shape[1:] == tuple(shapes[t][1:])
    assert np.all(seen[1:] == 1)           # every element in exactly one rank
    for t, s in enumerate(shapes):          # local pieces stack back in rank order
        stacked = np.concatenate([oracle.local_shards(tensors, lay, r)[t] for r in range(nd)])
        assert np.array_equal(stacked, tensors[t])
    bufs = [oracle.local_buffer(tensors, lay, r) for r in range(nd)]
    for a, b in zip(oracle.all_gather_copy_out(bufs, lay), tensors):
        assert np.array_equal(a, b)


def test_brute_force_small_groups():
    dims = [(0,), (1,), (3,), (5,), (2, 3), (7, 1), (4, 2), (5, 2, 2)]
    for n in range(1, 4):
        for shapes in itertools.product(dims, repeat=n):
            for nd in (1, 2, 3, 4, 5):
                _check(list(shapes), nd)


def test_sharded_mean_equals_sliced_full_mean():
    # reduce-scatter of the chunk-cat buffers = rows of the mean of the full
    # gradients (the per-parameter layout changes only where elements live)
    rng = np.random.default_rng(0)
    shapes, nd = [(7, 3), (5,), (9, 2)], 4
    lay = oracle.fsdp2_layout(shapes, nd)
    grads = [[rng.standard_normal(s) for s in shapes] for _ in range(nd)]
    cc = [oracle.chunk_cat(g, lay) for g in grads]
    means = [oracle.rs_avg(cc, r, lay.local) for r in range(nd)]
    full_mean = [sum(grads[q][t] for q in range(nd)) / nd for t in range(len(shapes))]
    gathered = oracle.all_gather_copy_out(means, lay)
    for a, b in zip(gathered, full_mean):
        assert np.allclose(a, b, rtol=0, atol=1e-15)


def test_layout_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.fsdp2_layout([(2, 2)], 0)
    with pytest.raises(ValueError):
        oracle.fsdp2_layout([()], 2)
