"""Cache files through the GPU: kvq_cache_save / save_f32 write exactly the bytes of the
oracle's layout restatement; kvq_cache_load reads oracle-written files into the device
planes, quantizes fp32 files on load byte-exactly like the oracle's encoders, and refuses
files of another mode (KVQ_EMISMATCH) or with missing bytes (KVQ_EIO) without writing;
kvq_cache_append self-heals an interrupted append.  colibri PR #399, Commits 1 and 6 and
the review thread."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import kvcache_file as KF

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_fp8_gb300 as k
    return k


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_planes(orc, fmt, T, seed):
    rows = W.unit_rows(T, seed=seed)
    if fmt == KF.FP8:
        lat, ls = orc.encode_fp8(rows.c)
    else:
        lat, ls = orc.encode_tq(rows.c, W.sign_bits(seed), KF.BITS[fmt])
    rope, rs = orc.encode_fp8(rows.k_rope)
    return dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs), rows


def empty_planes(fmt, T, fill=0x5A):
    lb = KF.lat_bytes(fmt)
    return dict(lat=torch.full((T, lb), fill, dtype=torch.uint8, device="cuda"),
                lat_scale=torch.full((T,), -7.0, device="cuda"),
                rope=torch.full((T, 64), fill, dtype=torch.uint8, device="cuda"),
                rope_scale=torch.full((T,), -7.0, device="cuda"))


def to_host(p):
    return {k: v.cpu().numpy() for k, v in p.items()}


@pytest.mark.parametrize("fmt", [KF.FP8, KF.TQ3, KF.TQ4, KF.TQ6])
def test_save_matches_oracle_and_load_round_trips(kvq, orc, tmp_path, fmt):
    T = 5000                                                 # two chunks of records
    hp, _ = host_planes(orc, fmt, T, seed=fmt)
    signs = W.sign_bits(fmt)
    path = tmp_path / "c.kvq"
    kvq.kvq_cache_save(path, fmt, {k: dev(v) for k, v in hp.items()}, T,
                       signs=dev(signs) if fmt in KF.BITS else None)
    torch.cuda.synchronize()
    assert path.read_bytes() == KF.file_bytes(fmt, hp, signs if fmt in KF.BITS else None)
    out = empty_planes(fmt, T + 3)
    n = kvq.kvq_cache_load(path, fmt, out, signs=dev(signs) if fmt in KF.BITS else None)
    assert n == T
    got = to_host(out)
    for k in hp:
        assert np.array_equal(got[k][:T], hp[k])
    assert np.all(got["lat"][T:] == 0x5A)                    # rows past the file untouched


@pytest.mark.parametrize("fmt", [KF.FP8, KF.TQ4, KF.TQ6])
def test_f32_file_quantizes_on_load(kvq, orc, tmp_path, fmt):
    T = 4500
    rows = W.magnitude_rows(T, seed=11, lo=1e-3, hi=40.0)
    path = tmp_path / "v1.kvq"
    kvq.kvq_cache_save_f32(path, dev(rows.c), dev(rows.k_rope))
    torch.cuda.synchronize()
    assert path.read_bytes() == KF.f32_file_bytes(rows.c, rows.k_rope)
    before = path.read_bytes()
    signs = W.sign_bits(11)
    out = empty_planes(fmt, T)
    ws = torch.empty(kvq.kvq_cache_load_workspace(), dtype=torch.uint8, device="cuda")
    n = kvq.kvq_cache_load(path, fmt, out, signs=dev(signs), workspace=ws)
    assert n == T
    ref = KF.load_as(path, fmt, signs)
    got = to_host(out)
    for k in ref:
        assert np.array_equal(got[k], ref[k]), k
    assert path.read_bytes() == before                      # the file is left as it was
    with pytest.raises(kvq.KvqError) as e:                  # an upgrade needs the workspace
        kvq.kvq_cache_load(path, fmt, out, signs=dev(signs))
    assert e.value.status == 5


def test_other_modes_and_short_files_are_refused_untouched(kvq, orc, tmp_path):
    T = 300
    h4, _ = host_planes(orc, KF.TQ4, T, seed=21)
    s21 = W.sign_bits(21)
    path = tmp_path / "c.kvq"
    path.write_bytes(KF.file_bytes(KF.TQ4, h4, s21))
    cases = [(KF.FP8, s21, 8), (KF.TQ6, s21, 8), (KF.TQ4, W.sign_bits(22), 8)]
    for fmt, signs, status in cases:
        out = empty_planes(fmt, T)
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_cache_load(path, fmt, out, signs=dev(signs))
        assert e.value.status == status
        assert np.all(out["lat"].cpu().numpy() == 0x5A)      # nothing written
    short = tmp_path / "short.kvq"
    short.write_bytes(KF.file_bytes(KF.TQ4, h4, s21)[:-10])
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_cache_load(short, KF.TQ4, empty_planes(KF.TQ4, T), signs=dev(s21))
    assert e.value.status == 9
    with pytest.raises(kvq.KvqError) as e:                   # capacity
        kvq.kvq_cache_load(path, KF.TQ4, empty_planes(KF.TQ4, T - 1), signs=dev(s21))
    assert e.value.status == 1


def test_append_self_heals_and_refuses_other_modes(kvq, orc, tmp_path):
    T = 600
    hp, _ = host_planes(orc, KF.FP8, T, seed=31)
    path = tmp_path / "c.kvq"
    path.write_bytes(KF.file_bytes(KF.FP8, hp, rows=400) + b"\xEE" * 777)   # interrupted
    expect = KF.append_bytes(path, KF.FP8, hp, 400, 200)
    dp = {k: dev(v) for k, v in hp.items()}
    kvq.kvq_cache_append(path, KF.FP8, dp, 400, 200)
    assert path.read_bytes() == expect == KF.file_bytes(KF.FP8, hp)
    out = empty_planes(KF.FP8, T)
    assert kvq.kvq_cache_load(path, KF.FP8, out) == T
    assert np.array_equal(out["lat"].cpu().numpy(), hp["lat"])
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_cache_append(path, KF.TQ4, dp, 0, 10)
    assert e.value.status == 8
