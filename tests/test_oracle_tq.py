"""Pins of the oracle's rotated tiers at other widths: TQ-b with b = 3 and 6 bits
(colibri PR #399: the TurboQuant tier's KV_TQ=6 setting, the "quality-parity choice",
and a 3-bit setting named in the persistence messages), the same codec as TQ4 (randomized
Hadamard rotation, N(0,1) Lloyd-Max codebook of 2^b levels scaled by radius/sqrt(n)) with
the codes packed as a little-endian bit stream.  The pins: the Lloyd-Max fixed point in
40-digit arithmetic, the published 8-level quantizer, the distortion against its closed
form and the high-resolution (Panter-Dite) limit, brute-force nearest centroids, an
independent unpacking of the bit stream, b = 4 reproducing the TQ4 bytes, and the
attention over TQ-b rows restated in the rotated domain."""
import math

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
from scipy.stats import norm

import workloads as W

TAU = 1.0 / math.sqrt(192.0)


def _signs(signs, n=512):
    return np.array([-1.0 if (signs[i // 32] >> (i % 32)) & 1 else 1.0 for i in range(n)])


def _unpack(packed, bits, n):
    """Codes of TQ-b rows from their bytes: bit b*i + j of the row is bit j of code i,
    bit 0 being the low bit of byte 0 (numpy's little-endian bit order)."""
    b = np.unpackbits(packed, axis=-1, bitorder="little")[..., : n * bits]
    b = b.reshape(packed.shape[0], n, bits).astype(np.int64)
    return (b << np.arange(bits)).sum(-1)


@pytest.mark.parametrize("bits", [3, 4, 6])
def test_codebook_is_lloyd_max_fixed_point(orc, bits):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    lloyd, cb, thr, _ = orc.tq_codebook(bits)
    L = 1 << bits
    assert lloyd.shape == (L,) and np.all(np.diff(lloyd) > 0)
    assert np.allclose(lloyd, -lloyd[::-1], atol=1e-13)
    t = [mp.mpf("-inf")] + [(mp.mpf(lloyd[k]) + mp.mpf(lloyd[k + 1])) / 2 for k in range(L - 1)] \
        + [mp.mpf("inf")]
    worst = 0
    for k in range(L):
        pa = 0 if k == 0 else mp.npdf(t[k])
        pb = 0 if k == L - 1 else mp.npdf(t[k + 1])
        worst = max(worst, abs((pa - pb) / (mp.ncdf(t[k + 1]) - mp.ncdf(t[k])) - mp.mpf(lloyd[k])))
    assert worst < 1e-12
    # stored centroids: the binary16 roundings; thresholds: their midpoints (exact)
    assert np.array_equal(cb, lloyd.astype(np.float16).astype(np.float32))
    assert np.array_equal(thr, (cb[:-1] + cb[1:]) / np.float32(2))


def test_eight_level_quantizer_is_the_published_one(orc):
    """The N(0,1) Lloyd-Max quantizer with 8 levels: outputs 0.2451, 0.7560, 1.344,
    2.152 and mean squared error 0.03455 (the classic table of optimum quantizers)."""
    lloyd, cb, thr, _ = orc.tq_codebook(3)
    assert np.allclose(lloyd[4:], [0.2451, 0.7560, 1.344, 2.152], atol=6e-4)
    t = np.concatenate([[-np.inf], (lloyd[:-1] + lloyd[1:]) / 2, [np.inf]])
    mse = sum(scipy.integrate.quad(lambda x, c=lloyd[k]: (x - c) ** 2 * norm.pdf(x),
                                   t[k], t[k + 1], epsabs=1e-13)[0] for k in range(8))
    assert abs(mse - 0.03455) < 5e-5


@pytest.mark.parametrize("bits", [3, 4, 6])
def test_distortion_against_high_resolution_limit(orc, bits):
    """MSE of the stored codebook by numerical integration, compared with the
    Panter-Dite limit (sqrt(3) pi / 2) 4^-b, which Lloyd-Max approaches from below."""
    _, cb, thr, _ = orc.tq_codebook(bits)
    t = np.concatenate([[-np.inf], thr.astype(np.float64), [np.inf]])
    mse = sum(scipy.integrate.quad(lambda x, c=float(cb[k]): (x - c) ** 2 * norm.pdf(x),
                                   t[k], t[k + 1], epsabs=1e-14)[0] for k in range(1 << bits))
    pd = math.sqrt(3.0) * math.pi / 2.0 * 4.0 ** (-bits)
    lo = {3: 0.80, 4: 0.88, 6: 0.95}[bits]
    assert lo * pd < mse < pd


@pytest.mark.parametrize("bits", [3, 6])
def test_codes_are_nearest_centroid_and_bit_packed(orc, bits):
    """u = y/sigma recomputed in fp64 with scipy's Hadamard matrix: each code (read back
    with numpy's bit unpacking) is the nearest centroid except within rounding distance
    of a midpoint."""
    rows = W.unit_rows(T=64, seed=13 + bits)
    signs = W.sign_bits(13 + bits)
    packed, radius = orc.encode_tq(rows.c, signs, bits)
    assert packed.shape == (64, 512 * bits // 8)
    _, cb, thr, _ = orc.tq_codebook(bits)
    Hm = scipy.linalg.hadamard(512).astype(np.float64)
    y = (Hm @ (_signs(signs)[:, None] * rows.c.T.astype(np.float64))).T / math.sqrt(512)
    u = y / (np.linalg.norm(y, axis=1, keepdims=True) / math.sqrt(512))
    codes = _unpack(packed, bits, 512)
    nearest = np.argmin(np.abs(u[..., None] - cb[None, None, :]), axis=-1)
    close = np.min(np.abs(u[..., None] - thr[None, None, :]), axis=-1) < 1e-5
    assert np.all((codes == nearest) | close)
    assert np.mean(close) < 1e-3


def test_four_bits_reproduce_tq4(orc):
    rows = W.unit_rows(T=40, seed=21)
    signs = W.sign_bits(21)
    p4, r4 = orc.encode_tq4(rows.c, signs)
    p, r = orc.encode_tq(rows.c, signs, 4)
    assert np.array_equal(p, p4) and np.array_equal(r, r4)
    assert np.array_equal(orc.tq_codebook(4)[1], orc.tq4_codebook()[1])


@pytest.mark.parametrize("bits,lo,hi", [(3, 0.178, 0.194), (6, 0.0243, 0.0265)])
def test_rel_l2_and_radius(orc, bits, lo, hi):
    """Reconstruction rel-L2 on N(0,1) rows is the square root of the quantizer's
    distortion (0.03455 -> 0.186 at 3 bits; ~6.4e-4 -> ~0.025 at 6 bits); the radius
    is the row norm; every code is used about as often as its Gaussian cell mass."""
    rows = W.unit_rows(T=2000, seed=30 + bits)
    signs = W.sign_bits(30 + bits)
    packed, radius = orc.encode_tq(rows.c, signs, bits)
    norms = np.linalg.norm(rows.c.astype(np.float64), axis=1)
    assert np.max(np.abs(radius - norms) / norms) < 1e-6
    xhat, _ = orc.decode_tq(packed, radius, signs, 512, bits)
    rel = np.sqrt(np.mean((np.linalg.norm(xhat - rows.c, axis=1) / norms) ** 2))
    assert lo < rel < hi
    _, cb, thr, _ = orc.tq_codebook(bits)
    t = np.concatenate([[-np.inf], thr, [np.inf]])
    hist = np.bincount(_unpack(packed, bits, 512).ravel(), minlength=1 << bits) / (2000 * 512)
    assert np.allclose(hist, norm.cdf(t[1:]) - norm.cdf(t[:-1]), atol=3e-3)


@pytest.mark.parametrize("bits", [3, 6])
def test_inert_rows_and_refusals(orc, bits):
    x = np.zeros((3, 256), np.float32)
    x[1, 5] = -1.5
    packed, radius = orc.encode_tq(x, W.sign_bits(0), bits)
    assert radius[0] == 0 and not packed[0].any() and radius[2] == 0 and not packed[2].any()
    assert radius[1] == np.float32(1.5)
    with pytest.raises(ValueError):
        orc.encode_tq(np.ones((1, 384), np.float32), np.zeros(16, np.uint32), bits)
    with pytest.raises(ValueError):
        orc.encode_tq(np.ones((1, 64), np.float32), np.zeros(16, np.uint32), 5)


@pytest.mark.parametrize("bits,fmt", [(3, 5), (6, 4)])
def test_attention_over_tq_rows_matches_rotated_domain(orc, bits, fmt):
    """The oracle attends over fully dequantised TQ-b rows; the rotated-domain
    restatement (rot(q) . yhat for the score, unrot of the weighted sum) agrees."""
    T = 40
    rows = W.unit_rows(T, seed=40 + bits)
    signs = W.sign_bits(40 + bits)
    lat, rad = orc.encode_tq(rows.c, signs, bits)
    rope, rs = orc.encode_fp8(rows.k_rope)
    cache = dict(lat=lat, lat_scale=rad, rope=rope, rope_scale=rs)
    q = W.queries(1, 1, 2, seed=40 + bits)
    out, lse, bad = orc.mla_decode(seq_len=[T], seq_fmt=[fmt], q_lat=q.q_lat, q_rope=q.q_rope,
                                   sm_scale=TAU, tq4=cache, signs=signs)
    assert not bad
    _, yhat = orc.decode_tq(lat, rad, signs, 512, bits)
    kr = orc.decode_fp8(rope, rs)
    Hm = scipy.linalg.hadamard(512) / math.sqrt(512)
    s = _signs(signs)
    for h in range(2):
        rq = Hm @ (s * q.q_lat[0, 0, h])
        sc = float(np.float32(TAU)) * (yhat @ rq + kr @ q.q_rope[0, 0, h].astype(np.float64))
        p = np.exp(sc - sc.max())
        assert lse[0, 0, h] == pytest.approx(sc.max() + math.log(p.sum()), abs=1e-12)
        ref = s * (Hm @ ((p / p.sum()) @ yhat))
        assert np.allclose(out[0, 0, h], ref, atol=1e-12)
