"""Cache files on the host: the oracle's restatement of the layout and load rules
(oracle/kvcache_file.py) pinned to what the pages fix, and the library's header check
(kvq_cache_probe, host only) on files the oracle wrote.  colibri PR #399: Commit 1
(".coli_kv v2 ... quantize-on-upgrade from v1, reject-on-mismatch, self-heal"), Commit 6
(the magic encodes the tier; a header word carries codec << 8 | bits), the review thread
(refuse, never misread; refuse containers whose byte counts do not add up)."""
import struct

import numpy as np
import pytest

import workloads as W
from oracle import kvcache_file as KF


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_fp8_gb300 as k
    return k


def planes(orc, fmt, T=40, seed=0):
    rows = W.unit_rows(T, seed=seed)
    if fmt == KF.FP8:
        lat, ls = orc.encode_fp8(rows.c)
    else:
        lat, ls = orc.encode_tq(rows.c, W.sign_bits(seed), KF.BITS[fmt])
    rope, rs = orc.encode_fp8(rows.k_rope)
    return dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs), rows


@pytest.mark.parametrize("fmt", [KF.FP8, KF.TQ3, KF.TQ4, KF.TQ6])
def test_oracle_round_trip_and_header(orc, tmp_path, fmt):
    p, _ = planes(orc, fmt, seed=fmt)
    signs = W.sign_bits(fmt) if fmt in KF.BITS else None
    path = tmp_path / "c.kvq"
    path.write_bytes(KF.file_bytes(fmt, p, signs))
    w = struct.unpack("<16I", path.read_bytes()[:64])
    # the magic names the tier; word 7 is codec << 8 | bits
    assert path.read_bytes()[:4] == {KF.FP8: b"KVQ2"}.get(fmt, b"KVQ3")
    assert w[7] == (8 if fmt == KF.FP8 else (1 << 8) | KF.BITS[fmt])
    f = KF.read(path)
    assert f["n_rows"] == 40 and f["trailing"] == 0
    for k in p:
        assert np.array_equal(f["planes"][k], p[k])
    assert len(path.read_bytes()) == 64 + (64 if signs is not None else 0) + 40 * KF.record_bytes(fmt)


def test_oracle_refuses_other_modes_and_upgrades_f32(orc, tmp_path):
    p8, rows = planes(orc, KF.FP8, seed=3)
    a = tmp_path / "a.kvq"
    a.write_bytes(KF.file_bytes(KF.FP8, p8))
    with pytest.raises(KF.Mismatch):
        KF.load_as(a, KF.TQ4, W.sign_bits(3))
    p4, _ = planes(orc, KF.TQ4, seed=3)
    b = tmp_path / "b.kvq"
    b.write_bytes(KF.file_bytes(KF.TQ4, p4, W.sign_bits(3)))
    with pytest.raises(KF.Mismatch):
        KF.load_as(b, KF.TQ6, W.sign_bits(3))                  # same tier, other width
    with pytest.raises(KF.Mismatch):
        KF.load_as(b, KF.TQ4, W.sign_bits(4))                  # other rotation
    c = tmp_path / "c.kvq"
    c.write_bytes(KF.f32_file_bytes(rows.c, rows.k_rope))
    up = KF.load_as(c, KF.FP8)                                 # quantize on load
    assert np.array_equal(up["lat"], p8["lat"]) and np.array_equal(up["rope"], p8["rope"])


def test_oracle_append_self_heals(orc, tmp_path):
    p, _ = planes(orc, KF.FP8, T=30, seed=5)
    path = tmp_path / "c.kvq"
    full = KF.file_bytes(KF.FP8, p, rows=20)
    path.write_bytes(full + b"\x01" * 100)                    # an interrupted append
    assert KF.read(path)["trailing"] == 100
    out = KF.append_bytes(path, KF.FP8, p, 20, 10)
    assert out == KF.file_bytes(KF.FP8, p, rows=30)


@pytest.mark.parametrize("fmt", [KF.FP8, KF.TQ6])
def test_library_probe_reads_oracle_files(kvq, orc, tmp_path, fmt):
    p, _ = planes(orc, fmt, seed=7)
    signs = W.sign_bits(7) if fmt in KF.BITS else None
    path = tmp_path / "c.kvq"
    path.write_bytes(KF.file_bytes(fmt, p, signs) + b"\x00" * 33)
    info = kvq.kvq_cache_probe(path)
    assert (info.format, info.n_rows, info.record_bytes, info.trailing_bytes) == \
        (fmt, 40, KF.record_bytes(fmt), 33)
    assert (info.codec, info.bits) == ((0, 8) if fmt == KF.FP8 else (1, 6))


def test_library_probe_refuses_bad_containers(kvq, orc, tmp_path):
    p, _ = planes(orc, KF.FP8, seed=9)
    good = KF.file_bytes(KF.FP8, p)
    bad = {"short": good[:40], "truncated": good[:-5], "magic": b"KVQ9" + good[4:],
           "reserved": good[:60] + b"\x01\x00\x00\x00" + good[64:],
           "record": good[:32] + struct.pack("<I", 999) + good[36:]}
    for name, data in bad.items():
        path = tmp_path / f"{name}.kvq"
        path.write_bytes(data)
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_cache_probe(path)
        assert e.value.status == 9, name
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_cache_probe(tmp_path / "missing.kvq")
    assert e.value.status == 9
