"""GPU parity of the codecs, the q4_0 paged append/gather and the row gather: every
byte, scale bit pattern and gathered binary16 bit pattern must equal the oracle's."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_fp8_gb300 as k
    return k


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_fp8(kvq, x):
    x = dev(x)
    R, D = x.shape
    codes = torch.full((R, D), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((R,), -1.0, dtype=torch.float32, device="cuda")
    kvq.kvq_encode_fp8(x, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


# ---------------------------------------------------------------------------- fp8 ------

@pytest.mark.parametrize("T", [1, 17, 1024])
def test_fp8_encode_tiny_workload(kvq, orc, T):
    rows = W.fp8_tiny_rows(T, seed=0)
    for x in (rows.c, rows.k_rope):
        codes, scales = gpu_fp8(kvq, x)
        oc, os_ = orc.encode_fp8(x)
        assert np.array_equal(codes, oc)
        assert np.array_equal(bits(scales), bits(os_))


@pytest.mark.parametrize("dim", [64, 100, 128, 256, 576, 1024, 3])
def test_fp8_encode_dims_and_edges(kvq, orc, dim):
    g = np.random.default_rng(dim)
    x = (g.standard_normal((77, dim)) * np.exp(g.uniform(-12, 6, (77, 1)))).astype(np.float32)
    x[5] = 0.0                                         # zero row
    x[6, :] = -0.0
    x[7, 0] = 448.0 * 3                                # saturation path of the row max
    x[8, :] = 2.0 ** -130                              # subnormal inputs
    x[9, ::2] = -x[9, ::2]
    codes, scales = gpu_fp8(kvq, x)
    oc, os_ = orc.encode_fp8(x)
    assert np.array_equal(codes, oc)
    assert np.array_equal(bits(scales), bits(os_))


def test_fp8_encode_strided(kvq, orc):
    """ldx / ldc larger than dim: the MLA row layout written as two strided encodes."""
    rows = W.unit_rows(300, seed=4)
    full = np.concatenate([rows.c, rows.k_rope], axis=1)          # [T][576]
    x = dev(full)
    codes = torch.zeros(300, 576, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(300, 2, dtype=torch.float32, device="cuda")
    s0 = torch.empty(300, dtype=torch.float32, device="cuda")
    s1 = torch.empty(300, dtype=torch.float32, device="cuda")
    kvq.kvq_encode_fp8(x[:, :512], codes[:, :512], s0)
    kvq.kvq_encode_fp8(x[:, 512:], codes[:, 512:], s1)
    torch.cuda.synchronize()
    oc0, os0 = orc.encode_fp8(rows.c)
    oc1, os1 = orc.encode_fp8(rows.k_rope)
    assert np.array_equal(codes.cpu().numpy(), np.concatenate([oc0, oc1], 1))
    assert np.array_equal(bits(s0.cpu().numpy()), bits(os0))
    assert np.array_equal(bits(s1.cpu().numpy()), bits(os1))


def test_fp8_encode_full_sparse_workload(kvq, orc):
    """T = 131072 rows (the long-context workload), every byte."""
    rows = W.unit_rows(131072, seed=0)
    for x in (rows.c, rows.k_rope):
        codes, scales = gpu_fp8(kvq, x)
        oc, os_ = orc.encode_fp8(x)
        assert np.array_equal(codes, oc)
        assert np.array_equal(bits(scales), bits(os_))


def test_fp8_encode_rows_zero_is_noop(kvq):
    x = torch.zeros(0, 512, device="cuda")
    kvq.kvq_encode_fp8(x, torch.zeros(0, 512, dtype=torch.uint8, device="cuda"),
                       torch.zeros(0, device="cuda"))


# ---------------------------------------------------------------------------- TQ4 ------

def gpu_tq4(kvq, x, signs):
    xd = dev(x)
    R, D = x.shape
    packed = torch.full((R, D // 2), 0xCD, dtype=torch.uint8, device="cuda")
    rad = torch.full((R,), -1.0, dtype=torch.float32, device="cuda")
    kvq.kvq_encode_tq4(xd, dev(signs), packed, rad)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), rad.cpu().numpy()


def test_tq4_codebook_matches_oracle(kvq, orc):
    cb, thr = kvq.kvq_tq4_codebook()
    _, ocb, othr, _ = orc.tq4_codebook()
    assert np.array_equal(bits(cb), bits(ocb)) and np.array_equal(bits(thr), bits(othr))


def test_tq4_encode_full_workload(kvq, orc):
    """T = 32768 N(0,1) rows of the 4-bit tier, every byte and radius bit pattern."""
    rows = W.unit_rows(32768, seed=0)
    signs = W.sign_bits(0)
    p, r = gpu_tq4(kvq, rows.c, signs)
    op, orad = orc.encode_tq4(rows.c, signs)
    assert np.array_equal(bits(r), bits(orad))
    assert np.array_equal(p, op)


@pytest.mark.parametrize("dim", [64, 128, 256, 512, 1024])
def test_tq4_encode_dims_and_edges(kvq, orc, dim):
    g = np.random.default_rng(dim)
    x = (g.standard_normal((45, dim)) * np.exp(g.uniform(-8, 5, (45, 1)))).astype(np.float32)
    x[3] = 0.0                                             # inert row
    x[4] = 1.0                                             # rotates onto one axis
    x[5, :] = 0.0
    x[5, 7] = -3.0                                         # a signed unit vector
    x[6] = np.tile(np.float32([1.5, -1.5]), dim // 2)      # tie-heavy row
    signs = g.integers(0, 2 ** 32, dim // 32, dtype=np.uint64).astype(np.uint32)
    p, r = gpu_tq4(kvq, x, signs)
    op, orad = orc.encode_tq4(x, signs)
    assert np.array_equal(bits(r), bits(orad))
    assert np.array_equal(p, op)


def test_codecs_on_the_pinned_boundary_cases(kvq, orc):
    """The hand-built inputs that fix the oracle's readings, through the CUDA encoders:
    fp8 elements that are 41 x an exact e4m3 midpoint under a scale of exactly 41 (the
    division x / scale decides them), and rotated rows (all signs +1, x = e_0 + e_1)
    whose odd elements land exactly on the middle threshold 0 (an exact hit goes up)."""
    x = np.zeros((2, 512), np.float32)
    x[0, :8] = [448 * 41, 1.6875 * 41, 31 * 41, 432 * 41, -1.6875 * 41, 0.2109375 * 41, -31 * 41, 0]
    x[1, 0] = x[1, 1] = 1.0
    codes, scales = gpu_fp8(kvq, x)
    oc, os_ = orc.encode_fp8(x)
    assert np.array_equal(codes, oc) and np.array_equal(bits(scales), bits(os_))
    assert list(codes[0, :8]) == [0x7E, 0x3E, 0x60, 0x7E, 0xBE, 0x26, 0xE0, 0x00]
    signs = np.zeros(16, np.uint32)
    p, r = gpu_tq4(kvq, x[1:], signs)
    op, orad = orc.encode_tq4(x[1:], signs)
    assert np.array_equal(p, op) and np.array_equal(bits(r), bits(orad))
    assert np.all(p[0] == 0x8C)
    for b in (3, 6):
        packed = torch.full((1, 64 * b), 0xCD, dtype=torch.uint8, device="cuda")
        rad = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        kvq.kvq_encode_tq(dev(x[1:]), dev(signs), b, packed, rad)
        torch.cuda.synchronize()
        ref, ref_r = orc.encode_tq(x[1:], signs, b)
        assert np.array_equal(packed.cpu().numpy(), ref)
        assert np.array_equal(bits(rad.cpu().numpy()), bits(ref_r))


def test_tq4_refuses_non_pow2(kvq):
    x = torch.zeros(4, 384, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_encode_tq4(x, torch.zeros(12, dtype=torch.int32, device="cuda"),
                           torch.zeros(4, 192, dtype=torch.uint8, device="cuda"),
                           torch.zeros(4, device="cuda"))
    assert e.value.status == 2


# ---------------------------------------------------------------------------- q4_0 -----

def run_q4(kvq, wl, n_heads, sentinel=(0xA5, 0x5A)):
    kp = torch.full((wl.n_cells, n_heads, 144), sentinel[0], dtype=torch.uint8, device="cuda")
    vp = torch.full((wl.n_cells, n_heads, 144), sentinel[1], dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos0, table = dev(wl.pos0), dev(wl.page_table)
    kvq.kvq_append_q4(dev(wl.k), dev(wl.v), pos0, table, wl.page_size, wl.n_cells, kp, vp, st)
    n_seq, n_tok = wl.k.shape[:2]
    gk = torch.empty(n_seq, n_tok, n_heads, 256, dtype=torch.int16, device="cuda")
    gv = torch.empty_like(gk)
    kvq.kvq_gather_q4(kp, pos0, n_tok, table, wl.page_size, wl.n_cells, gk, st)
    kvq.kvq_gather_q4(vp, pos0, n_tok, table, wl.page_size, wl.n_cells, gv, st)
    torch.cuda.synchronize()
    return (kp.cpu().numpy(), vp.cpu().numpy(), gk.cpu().numpy().view(np.uint16),
            gv.cpu().numpy().view(np.uint16), int(st.item()))


def oracle_q4(orc, wl, n_heads, sentinel=(0xA5, 0x5A)):
    ok = np.full((wl.n_cells, n_heads, 144), sentinel[0], np.uint8)
    ov = np.full((wl.n_cells, n_heads, 144), sentinel[1], np.uint8)
    orc.append_q4(wl.k, wl.v, wl.pos0, wl.page_table, wl.page_size, wl.n_cells, ok, ov)
    n_tok = wl.k.shape[1]
    gk = orc.gather_q4(ok, wl.pos0, n_tok, wl.page_table, wl.page_size, wl.n_cells, n_heads)
    gv = orc.gather_q4(ov, wl.pos0, n_tok, wl.page_table, wl.page_size, wl.n_cells, n_heads)
    return ok, ov, gk, gv


def test_q4_small_page_crossing(kvq, orc):
    """A permuted table, a start 8 cells before a page end (one dispatch crosses pages),
    spare pages that must keep the sentinel, amplitude classes {1e-3, 1, 40}."""
    wl = W.q4_paged(n_seq=3, n_tok=17, n_heads=8, page_size=64, seed=5, spare_pages=3)
    kp, vp, gk, gv, st = run_q4(kvq, wl, 8)
    ok, ov, ogk, ogv = oracle_q4(orc, wl, 8)
    assert st == 0
    assert np.array_equal(kp, ok) and np.array_equal(vp, ov)
    assert np.array_equal(gk, ogk) and np.array_equal(gv, ogv)


def test_q4_tie_and_zero_blocks(kvq, orc):
    wl = W.q4_paged(n_seq=1, n_tok=6, n_heads=2, page_size=4, pos0=2, seed=6, spare_pages=1)
    hd = 256
    # rows chosen so that the ROTATED blocks hit the tie rule: the Hadamard transform
    # of e_0 * v is v/16 everywhere (all-equal blocks); of zero is zero (all-zero)
    wl.k[0, 0, 0] = 0.0
    wl.k[0, 1, 0] = 0.0
    wl.k[0, 1, 0, 0] = 3.0
    wl.k[0, 2, 1] = 0.0
    wl.k[0, 2, 1, 0] = -3.0
    wl.v[0, 3, 0] = 0.0
    wl.v[0, 3, 0, :2] = [2.0, -2.0]                   # blocks {v, -v, ...} after rotation
    kp, vp, gk, gv, _ = run_q4(kvq, wl, 2)
    ok, ov, ogk, ogv = oracle_q4(orc, wl, 2)
    assert np.array_equal(kp, ok) and np.array_equal(vp, ov)
    assert np.array_equal(gk, ogk) and np.array_equal(gv, ogv)
    cell = wl.page_table[0, (wl.pos0[0] + 0) // 4] * 4 + (wl.pos0[0] + 0) % 4
    assert bytes(kp[cell, 0, :18]) == bytes([0x00, 0x80] + [0x88] * 16)


def test_q4_bad_page_flagged(kvq, orc):
    wl = W.q4_paged(n_seq=2, n_tok=5, n_heads=1, page_size=4, seed=7)
    wl.page_table[1, :] = wl.n_cells            # page id outside the pool
    kp, vp, gk, gv, st = run_q4(kvq, wl, 1, sentinel=(0, 0))
    assert st & kvq.DEV_BAD_PAGE


@pytest.mark.slow
def test_q4_full_paged_workload(kvq, orc):
    """16 sequences x 8192 tokens x 8 heads, K and V: every pool byte and every
    gathered binary16."""
    wl = W.q4_paged(seed=0)
    kp, vp, gk, gv, st = run_q4(kvq, wl, 8)
    ok, ov, ogk, ogv = oracle_q4(orc, wl, 8)
    assert st == 0
    assert np.array_equal(kp, ok) and np.array_equal(vp, ov)
    assert np.array_equal(gk, ogk) and np.array_equal(gv, ogv)


# ------------------------------------------------------------------------- row gather --

@pytest.mark.parametrize("fmt", [1, 2])
def test_gather_rows_byte_exact(kvq, orc, fmt):
    T = 3000
    rows = W.unit_rows(T, seed=8)
    if fmt == 1:
        lat, ls = orc.encode_fp8(rows.c)
    else:
        lat, ls = orc.encode_tq4(rows.c, W.sign_bits(8))
    rope, rs = orc.encode_fp8(rows.k_rope)
    src = dict(lat=dev(lat), lat_scale=dev(ls), rope=dev(rope), rope_scale=dev(rs))
    idx = W.sparse_indices(T, 257, 1, seed=8)[0]
    idx[3] = T + 4                                          # out of range -> zeros + flag
    dst = {k: torch.full((257,) + v.shape[1:], 7, dtype=v.dtype, device="cuda") for k, v in src.items()}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_gather_rows(fmt, src, T, dev(idx), dst, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & kvq.DEV_BAD_INDEX
    good = np.arange(257) != 3
    for k, host in (("lat", lat), ("lat_scale", ls), ("rope", rope), ("rope_scale", rs)):
        got = dst[k].cpu().numpy()
        assert np.array_equal(got[good], host[idx[good]])
        assert not got[3].any()


# ------------------------------------------------------- append-time MLA row encode ------

@pytest.mark.parametrize("fmt,b", [(1, 8), (5, 3), (2, 4), (4, 6)], ids=["fp8", "tq3", "tq4", "tq6"])
@pytest.mark.parametrize("T", [1, 7, 1000])
def test_encode_mla_rows_match_oracle(kvq, orc, fmt, b, T):
    """kvq_encode_mla (latent in the tier, rope key in fp8, one launch) against the
    oracle's encoders: every code byte and scale bit pattern; magnitudes log-uniform
    1e-3..40 with a zero row."""
    rows = W.magnitude_rows(T, seed=90 + T, lo=1e-3, hi=40.0)
    rows.c[0] = 0.0
    signs = W.sign_bits(90)
    lw = 512 * b // 8
    lat = torch.full((T, lw), 0xAB, dtype=torch.uint8, device="cuda")
    ls = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
    rope = torch.full((T, 64), 0xAB, dtype=torch.uint8, device="cuda")
    rs = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
    kvq.kvq_encode_mla(dev(rows.c), dev(rows.k_rope), fmt, dev(signs), lat, ls, rope, rs)
    torch.cuda.synchronize()
    ref_lat, ref_ls = orc.encode_fp8(rows.c) if b == 8 else orc.encode_tq(rows.c, signs, b)
    ref_rope, ref_rs = orc.encode_fp8(rows.k_rope)
    assert np.array_equal(lat.cpu().numpy(), ref_lat)
    assert np.array_equal(bits(ls.cpu().numpy()), bits(ref_ls))
    assert np.array_equal(rope.cpu().numpy(), ref_rope)
    assert np.array_equal(bits(rs.cpu().numpy()), bits(ref_rs))


@pytest.mark.parametrize("fmt,b", [(1, 8), (2, 4)], ids=["fp8", "tq4"])
def test_encode_mla_strided_and_unaligned(kvq, orc, fmt, b):
    """Row strides wider than the rows (the one-launch form), and inputs 4 bytes off a
    16-byte boundary (the two-kernel fallback), into rows of wider code planes; the
    bytes past each row stay untouched."""
    T = 33
    rows = W.magnitude_rows(T, seed=97, lo=1e-2, hi=10.0)
    signs = W.sign_bits(97)
    lw = 512 * b // 8
    ref_lat, ref_ls = orc.encode_fp8(rows.c) if b == 8 else orc.encode_tq(rows.c, signs, b)
    ref_rope, ref_rs = orc.encode_fp8(rows.k_rope)
    for off in (0, 1):                                   # floats of offset
        cbuf = torch.zeros(T, 520 + off, dtype=torch.float32, device="cuda")
        cbuf[:, off:off + 512] = dev(rows.c)
        rbuf = torch.zeros(T, 72 + off, dtype=torch.float32, device="cuda")
        rbuf[:, off:off + 64] = dev(rows.k_rope)
        lat = torch.full((T, lw + 16), 0xAB, dtype=torch.uint8, device="cuda")
        ls = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
        rope = torch.full((T, 80), 0xAB, dtype=torch.uint8, device="cuda")
        rs = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
        kvq.kvq_encode_mla(cbuf[:, off:off + 512], rbuf[:, off:off + 64], fmt, dev(signs),
                           lat[:, :lw], ls, rope[:, :64], rs)
        torch.cuda.synchronize()
        got_lat, got_rope = lat.cpu().numpy(), rope.cpu().numpy()
        assert np.array_equal(got_lat[:, :lw], ref_lat)
        assert np.all(got_lat[:, lw:] == 0xAB)
        assert np.array_equal(bits(ls.cpu().numpy()), bits(ref_ls))
        assert np.array_equal(got_rope[:, :64], ref_rope)
        assert np.all(got_rope[:, 64:] == 0xAB)
        assert np.array_equal(bits(rs.cpu().numpy()), bits(ref_rs))
