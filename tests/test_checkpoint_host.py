"""CPU checks of the native sharded checkpoint (host memory only, no GPU):
rank files written from FlatParameter shards load back under any rank count
equal to the oracle's resharding; the reshard plan matches the oracle's brute
force; checksums catch a flipped byte; a truncated file is refused."""
import ctypes
import itertools
import os

import numpy as np
import pytest

import oracle
import sharded_optimizer_step_gb300 as ss
from oracle import checkpoint as ock
from sharded_optimizer_step_gb300 import _capi
from sharded_optimizer_step_gb300 import checkpoint as ck


@pytest.fixture(scope="module", autouse=True)
def built():
    ss.build()


def _units(seed):
    rng = np.random.default_rng(seed)
    return [int(x) for x in (1000, 1, 777, 4096, 13)]


def _save(directory, totals, nd, step, seed=0):
    """Rank files for nd ranks from seeded master/m/v flat states; returns
    the per-unit per-kind flat states."""
    rng = np.random.default_rng(seed)
    flats = [[rng.standard_normal(T).astype(np.float32) for _ in range(3)] for T in totals]
    for r in range(nd):
        keep = []
        secs = (_capi.CkptSection * (3 * len(totals)))()
        k = 0
        for u, T in enumerate(totals):
            lay = oracle.layout([T], nd)
            for kind in range(3):
                full = np.zeros(lay.padded, np.float32)
                full[:T] = flats[u][kind]
                sh = np.ascontiguousarray(full[r * lay.shard:(r + 1) * lay.shard])
                keep.append(sh)
                secs[k] = _capi.CkptSection(u, kind, sh.nbytes, sh.ctypes.data)
                k += 1
        _capi.check("save", _capi.lib().shardstep_ckpt_save_rank(
            ck.rank_file(directory, r).encode(), nd, r, step, _capi.i64_array(totals),
            len(totals), secs, k))
    return flats


def _load(directory, totals, new_nd, r):
    old_nd, step, saved = ck.info(directory)
    assert saved == totals
    out = []
    for u, T in enumerate(totals):
        S = -(-T // new_nd)
        per_kind = []
        for kind in range(3):
            buf = np.zeros(S, np.float32)
            for q, off, new_off, n in ck.plan(T, old_nd, new_nd, r):
                _capi.check("read", _capi.lib().shardstep_ckpt_read(
                    ck.rank_file(directory, q).encode(), u, kind, off * 4, n * 4,
                    ctypes.c_void_p(buf.ctypes.data + new_off * 4)))
            per_kind.append(buf)
        out.append(per_kind)
    return out


@pytest.mark.parametrize("old_nd", [1, 3, 8])
def test_load_under_any_rank_count_equals_oracle_reshard(tmp_path, old_nd):
    totals = _units(0)
    flats = _save(str(tmp_path), totals, old_nd, step=17)
    nd, step, _ = ck.info(str(tmp_path))
    assert (nd, step) == (old_nd, 17)
    ck.verify(str(tmp_path))
    for new_nd in (1, 2, 4, 5, 8, 16):
        for r in range(new_nd):
            got = _load(str(tmp_path), totals, new_nd, r)
            for u, T in enumerate(totals):
                lay = oracle.layout([T], old_nd)
                for kind in range(3):
                    full = np.zeros(lay.padded, np.float32)
                    full[:T] = flats[u][kind]
                    old = [full[q * lay.shard:(q + 1) * lay.shard] for q in range(old_nd)]
                    want = ock.reshard(old, T, new_nd, r)
                    assert got[u][kind].tobytes() == want.tobytes()


def test_plan_matches_oracle_brute_force():
    for total in (0, 1, 5, 24, 97, 1000):
        for old_nd, new_nd in itertools.product((1, 2, 3, 5, 8), repeat=2):
            for r in range(new_nd):
                assert ck.plan(total, old_nd, new_nd, r) == ock.plan(total, old_nd, new_nd, r)


def test_checksum_catches_a_flipped_byte(tmp_path):
    totals = [5000]
    _save(str(tmp_path), totals, 2, step=1)
    path = ck.rank_file(str(tmp_path), 1)
    data = bytearray(open(path, "rb").read())
    data[-100] ^= 0x10
    open(path, "wb").write(bytes(data))
    with pytest.raises(ss.ShardstepError) as e:
        ck.verify(str(tmp_path))
    assert e.value.code == _capi.ERR_IO


def test_truncated_or_foreign_files_are_refused(tmp_path):
    totals = [64, 64]
    _save(str(tmp_path), totals, 1, step=3)
    path = ck.rank_file(str(tmp_path), 0)
    data = open(path, "rb").read()
    open(path, "wb").write(data[:80])
    with pytest.raises(ss.ShardstepError):
        ck.info(str(tmp_path))
    open(path, "wb").write(b"not a checkpoint" * 8)
    with pytest.raises(ss.ShardstepError):
        ck.info(str(tmp_path))
    assert not os.path.exists(path + ".tmp")


def test_bad_arguments_are_refused(tmp_path):
    L = _capi.lib()
    p = str(tmp_path / "x.shst").encode()
    assert L.shardstep_ckpt_save_rank(p, 0, 0, 1, None, 0, None, 0) == _capi.ERR_INVALID
    assert L.shardstep_ckpt_save_rank(p, 2, 2, 1, None, 0, None, 0) == _capi.ERR_INVALID
    n = _capi.c_i32()
    assert L.fsdp_reshard_plan(10, 2, 4, 4, None, 0, ctypes.byref(n)) == _capi.ERR_INVALID
    pieces = (_capi.CkptPiece * 1)()
    assert L.fsdp_reshard_plan(100, 8, 1, 0, pieces, 1, ctypes.byref(n)) == _capi.ERR_CAPACITY
    assert n.value == 8


# ---- the rank-file format, restated here from its description: header of 64
# bytes, unit totals, section table (unit, kind, bytes, offset, checksum),
# sections at 4096-byte aligned offsets; FNV-1a over little-endian 64-bit words

_BASIS, _PRIME, _MASK = 14695981039346656037, 1099511628211, (1 << 64) - 1


def _words(data: bytes):
    data = data + b"\0" * (-len(data) % 8)
    return np.frombuffer(data, "<u8").tolist()


def _fnv_chain(words, h=_BASIS):
    for w in words:
        h = ((h ^ w) * _PRIME) & _MASK
    return h


def _four_lane(data: bytes):
    w = _words(data)
    lanes = [_fnv_chain(w[k::4]) for k in range(4)]
    return _fnv_chain(lanes)


def _section_table(raw: bytes):
    import struct
    magic, version, hb, nd, rank, n_units, n_sec, step = struct.unpack_from("<8sIIiiiiq", raw, 0)
    off = 64 + 8 * n_units
    return version, [struct.unpack_from("<iiqqQ", raw, off + 32 * s) for s in range(n_sec)]


def test_section_checksums_are_four_interleaved_fnv1a_chains(tmp_path):
    # sizes whose word counts end on every chain, and a trailing partial word
    totals = [1000, 1, 777, 4096, 13]
    _save(str(tmp_path), totals, 3, step=2, seed=4)
    for r in range(3):
        raw = open(ck.rank_file(str(tmp_path), r), "rb").read()
        version, table = _section_table(raw)
        assert version == 2
        for unit, kind, nbytes, offset, checksum in table:
            data = raw[offset:offset + nbytes]
            assert checksum == _four_lane(data), (r, unit, kind)
            if nbytes > 8:
                assert checksum != _fnv_chain(_words(data))


def _version1_file(path, totals, nd, rank, step, sections):
    """A rank file of the first format version (every checksum one chain)."""
    import struct
    n_u, n_s = len(totals), len(sections)
    off = -(-(64 + 8 * n_u + 32 * n_s) // 4096) * 4096
    table, body = [], b""
    for unit, kind, data in sections:
        table.append((unit, kind, len(data), off, _fnv_chain(_words(data))))
        off = -(-(off + len(data)) // 4096) * 4096
    totals_b = struct.pack(f"<{n_u}q", *totals)
    table_b = b"".join(struct.pack("<iiqqQ", *e) for e in table)
    tsum = _fnv_chain(_words(table_b), _fnv_chain(_words(totals_b)))
    raw = bytearray(struct.pack("<8sIIiiiiqQ16s", b"SHSTCKPT", 1, 64, nd, rank, n_u, n_s, step,
                                tsum, b"\0" * 16) + totals_b + table_b)
    for (unit, kind, data), e in zip(sections, table):
        raw += b"\0" * (e[3] - len(raw)) + data
    open(path, "wb").write(bytes(raw))


def test_version1_files_are_still_read_and_verified(tmp_path):
    rng = np.random.default_rng(9)
    totals = [10, 21]
    secs = [(0, 0, rng.standard_normal(10).astype(np.float32).tobytes()),
            (1, 0, rng.standard_normal(11).astype(np.float32).tobytes())]
    path = ck.rank_file(str(tmp_path), 0)
    _version1_file(path, totals, 2, 0, 5, secs)
    nd, step, saved = ck.info(str(tmp_path))
    assert (nd, step, saved) == (2, 5, totals)
    L = _capi.lib()
    assert L.shardstep_ckpt_verify(path.encode()) == _capi.OK
    got = np.empty(11, np.float32)
    assert L.shardstep_ckpt_read(path.encode(), 1, 0, 0, got.nbytes,
                                 got.ctypes.data_as(ctypes.c_void_p)) == _capi.OK
    assert got.tobytes() == secs[1][2]
    raw = bytearray(open(path, "rb").read())
    raw[-3] ^= 0x40
    open(path, "wb").write(bytes(raw))
    assert L.shardstep_ckpt_verify(path.encode()) == _capi.ERR_IO


def test_four_lane_checksum_across_read_chunks(tmp_path):
    """A section longer than the 4 MB pieces verify reads it in, with a
    partial last piece: the chains continue across the pieces."""
    totals = [2_100_003]
    _save(str(tmp_path), totals, 1, step=1, seed=11)
    path = ck.rank_file(str(tmp_path), 0)
    raw = open(path, "rb").read()
    _, table = _section_table(raw)
    unit, kind, nbytes, offset, checksum = table[0]
    assert nbytes > 2 * (1 << 22)
    assert checksum == _four_lane(raw[offset:offset + nbytes])
    assert _capi.lib().shardstep_ckpt_verify(path.encode()) == _capi.OK
