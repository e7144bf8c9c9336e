"""Pins of the oracle's codecs against what the pages and the mathematics fix.

fp8 (colibri PR #399, Summary / Commit 1): per-row scale amax/448, RNE codes.
TQ4 (colibri PR #399, "Why rotated-int4 for the 4-bit tier"): randomized Hadamard
  rotation, 16-level N(0,1) Lloyd-Max codebook scaled by radius/sqrt(n), rel-L2 ~0.096,
  radius invariant under the rotation, rotated-domain consumer identities (the TQ4
  rebase comment), non-power-of-two refusal (the rebase note).
q4_0 (Strata PR #2533, kv_q4.metal port and fixture commits): orthonormal FWHT256,
  tie rule, all-zero group bits 0x8000 / 0x88, code step max|x|/8.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import scipy.integrate
from scipy.stats import norm

import workloads as W

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")


# ------------------------------------------------------------------------ fp8 ----------

def _e4m3_table():
    import torch
    v = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    return v.to(torch.float64).numpy()


def test_fp8_encode_is_nearest_code(orc):
    """Brute force: every code is the nearest table value to x/scale, ties to even
    mantissa, saturating at 448."""
    rows = W.fp8_tiny_rows(T=96, seed=11)
    x = np.concatenate([rows.c[:, :128], rows.k_rope], axis=1)
    codes, scales = orc.encode_fp8(x)
    table = _e4m3_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])])
    tv = table[finite]
    for r in range(x.shape[0]):
        amax = np.max(np.abs(x[r]))
        if amax == 0:
            assert scales[r] == 0 and not codes[r].any()
            continue
        assert scales[r] == np.float32(amax) / np.float32(448.0)
        u = (x[r] / scales[r]).astype(np.float32).astype(np.float64)
        for i in range(x.shape[1]):
            dist = np.abs(tv - u[i])
            best = finite[dist == dist.min()]
            val = table[codes[r, i]]
            assert abs(val - u[i]) == dist.min() or abs(u[i]) >= 448
            if len(set(table[best])) > 1:       # a true tie between two values
                assert codes[r, i] & 1 == 0
        # the row maximum always lands on +-448
        j = int(np.argmax(np.abs(x[r])))
        assert codes[r, j] & 0x7F == 0x7E


def test_fp8_divides_by_the_scale(orc):
    """The codes come from x / scale (one IEEE division), not x * (1 / scale).

    With amax = 448 * 41 the scale is exactly 41, and every x below is 41 times an
    exact midpoint m between an odd e4m3 code and the even code above it, so x / 41 = m
    exactly and round-to-nearest-even picks the even (upper) code.  fp32(1/41) is below
    1/41 by about 2^-24.4 relative, so x * fp32(1/41) falls just under m and would pick
    the odd (lower) code: the two readings disagree on every such element.
      m = 1.6875 (between 1.625 = 0x3D and 1.75 = 0x3E)  -> 0x3E
      m = 31     (between 30 = 0x5F and 32 = 0x60)        -> 0x60
      m = 432    (between 416 = 0x7D and 448 = 0x7E)      -> 0x7E
      m = 0.2109375 (between 0x25 and 0x26)               -> 0x26
    """
    amax = np.float32(448 * 41)
    x = np.zeros((1, 16), np.float32)
    x[0, :8] = [amax, 1.6875 * 41, 31 * 41, 432 * 41, -1.6875 * 41, 0.2109375 * 41, -31 * 41, 0]
    codes, scales = orc.encode_fp8(x)
    assert scales[0] == np.float32(41.0)
    assert list(codes[0, :8]) == [0x7E, 0x3E, 0x60, 0x7E, 0xBE, 0x26, 0xE0, 0x00]
    # the reading it rules out gives the odd neighbours
    inv = np.float32(1.0) / np.float32(41.0)
    assert np.float32(x[0, 1]) * inv < np.float32(1.6875)


def test_fp8_zero_rows_and_scales(orc):
    rows = W.fp8_tiny_rows(T=1024, seed=0)
    codes, scales = orc.encode_fp8(rows.c)
    for t in (0, 511, 1023, 300):
        assert scales[t] == 0.0 and not codes[t].any()
    rc, rs = orc.encode_fp8(rows.k_rope)
    assert rs[300] > 0 and rs[0] == 0
    # reconstruction error within half a code step (relative 2^-4 of the value's binade)
    dec = orc.decode_fp8(codes, scales)
    nz = scales > 0
    err = np.abs(dec[nz] - rows.c[nz])
    assert np.all(err <= np.abs(rows.c[nz]) * 2 ** -4 + scales[nz][:, None] * 2 ** -10 + 1e-30)


# ------------------------------------------------------------------------ TQ4 ----------

def test_codebook_is_lloyd_max_fixed_point(orc):
    lloyd, cb, thr, iters = orc.tq4_codebook()
    assert iters <= 20000
    # symmetric
    assert np.allclose(lloyd, -lloyd[::-1], atol=1e-13)
    # centroid condition E[X | cell] in closed form, with thresholds at midpoints
    t = np.concatenate([[-np.inf], (lloyd[:-1] + lloyd[1:]) / 2, [np.inf]])
    cond = (norm.pdf(t[:-1]) - norm.pdf(t[1:])) / (norm.cdf(t[1:]) - norm.cdf(t[:-1]))
    assert np.max(np.abs(cond - lloyd)) < 1e-12
    # the stored centroids are the binary16 roundings; thresholds their midpoints
    assert np.array_equal(cb, lloyd.astype(np.float16).astype(np.float32))
    assert np.array_equal(thr, (cb[:-1] + cb[1:]) / np.float32(2))
    assert np.max(np.abs(cb - lloyd) / np.abs(lloyd)) < 5e-4
    # published positive half (4 significant digits)
    assert np.allclose(lloyd[8:], [0.1284, 0.3881, 0.6568, 0.9423, 1.256, 1.618, 2.069, 2.733],
                       atol=6e-4)


def test_codebook_distortion_closed_form(orc):
    lloyd, cb, thr, _ = orc.tq4_codebook()
    t = np.concatenate([[-np.inf], thr.astype(np.float64), [np.inf]])
    mse = 0.0
    for k in range(16):
        f = lambda x, c=float(cb[k]): (x - c) ** 2 * norm.pdf(x)
        mse += scipy.integrate.quad(f, t[k], t[k + 1], epsabs=1e-13)[0]
    assert abs(mse - 0.009501) < 2e-5
    assert 0.093 < math.sqrt(mse) < 0.100


@pytest.mark.parametrize("n", [8, 64, 256, 512])
def test_fwht_matches_sylvester_hadamard(orc, n):
    g = np.random.default_rng(n)
    x = g.integers(-50, 50, n).astype(np.float64)
    Hm = scipy.linalg.hadamard(n)
    assert np.array_equal(orc.fwht_f64(x), Hm @ x)
    assert np.array_equal(orc.fwht_f64(orc.fwht_f64(x)), n * x)      # H H = n I
    xf = g.standard_normal(n).astype(np.float32)
    assert np.allclose(orc.fwht_f32(xf), Hm @ xf.astype(np.float64), rtol=0, atol=1e-5 * n)


def test_tq4_scale_constant_is_correctly_rounded(orc):
    """A unit vector e_0 rotates to c * (+-1, ..., +-1) with c = fp32(1/sqrt(512))."""
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    exact = Fraction(str(Decimal(1) / Decimal(512).sqrt()))
    c0 = np.float32(float(exact))
    cands = [np.nextafter(c0, np.float32(0)), c0, np.nextafter(c0, np.float32(1))]
    c = min(cands, key=lambda v: abs(Fraction(float(v)) - exact))
    assert np.array([c], np.float32).view(np.uint32)[0] == 0x3D3504F3
    # e_0 rotates to y_i = c for every i (no sign flips); the radius is then the pinned
    # reduction: 32 partial sums of 16 fused c*c steps (exact in fp64, one rounding
    # each), a butterfly of fp32 additions, an IEEE square root.
    x = np.zeros((1, 512), np.float32)
    x[0, 0] = 1.0
    packed, radius = orc.encode_tq4(x, np.zeros(16, np.uint32))
    acc = np.float32(0)
    for _ in range(16):
        acc = np.float32(float(c) * float(c) + float(acc))
    part = np.full(32, acc, np.float32)
    for o in (16, 8, 4, 2, 1):
        part = (part + part[np.arange(32) ^ o]).astype(np.float32)
    assert radius[0] == np.sqrt(part[0])


def test_tq4_radius_invariance_and_rel_l2(orc):
    rows = W.unit_rows(T=4000, seed=2)
    signs = W.sign_bits(2)
    packed, radius = orc.encode_tq4(rows.c, signs)
    norms = np.linalg.norm(rows.c.astype(np.float64), axis=1)
    assert np.max(np.abs(radius - norms) / norms) < 1e-6
    xhat, yhat = orc.decode_tq4(packed, radius, signs, 512)
    rel = np.linalg.norm(xhat - rows.c, axis=1) / norms
    assert 0.093 < np.sqrt(np.mean(rel ** 2)) < 0.100          # the page: ~0.096
    # every code is used, roughly as the Gaussian cell masses say
    codes = np.stack([packed & 15, packed >> 4], -1).ravel()
    hist = np.bincount(codes, minlength=16) / codes.size
    _, cb, thr, _ = orc.tq4_codebook()
    t = np.concatenate([[-np.inf], thr, [np.inf]])
    assert np.allclose(hist, norm.cdf(t[1:]) - norm.cdf(t[:-1]), atol=3e-3)


def test_tq4_codes_are_nearest_centroid(orc):
    """Rotated coordinate u = y/sigma recomputed in fp64 with scipy's Hadamard matrix;
    the code is the nearest centroid except within rounding distance of a midpoint."""
    rows = W.unit_rows(T=64, seed=3)
    signs = W.sign_bits(3)
    packed, radius = orc.encode_tq4(rows.c, signs)
    _, cb, thr, _ = orc.tq4_codebook()
    Hm = scipy.linalg.hadamard(512).astype(np.float64)
    s = np.array([-1.0 if (signs[i // 32] >> (i % 32)) & 1 else 1.0 for i in range(512)])
    y = (Hm @ (s[:, None] * rows.c.T.astype(np.float64))).T / math.sqrt(512)
    u = y / (np.linalg.norm(y, axis=1, keepdims=True) / math.sqrt(512))
    codes = np.stack([packed & 15, packed >> 4], -1).reshape(64, 512)
    nearest = np.argmin(np.abs(u[..., None] - cb[None, None, :]), axis=-1)
    close = np.min(np.abs(u[..., None] - thr[None, None, :]), axis=-1) < 1e-5
    assert np.all((codes == nearest) | close)
    assert np.mean(close) < 1e-3


def test_tq4_rotated_domain_identities(orc):
    """q . xhat == rot(q) . yhat and sum_t w_t xhat_t == unrot(sum_t w_t yhat_t), with
    rot(q) = (1/sqrt n) H (s (.) q) (the native TQ4 consumer's identities)."""
    rows = W.unit_rows(T=32, seed=4)
    signs = W.sign_bits(4)
    packed, radius = orc.encode_tq4(rows.c, signs)
    xhat, yhat = orc.decode_tq4(packed, radius, signs, 512)
    Hm = scipy.linalg.hadamard(512).astype(np.float64) / math.sqrt(512)
    s = np.array([-1.0 if (signs[i // 32] >> (i % 32)) & 1 else 1.0 for i in range(512)])
    q = np.random.default_rng(4).standard_normal(512)
    rq = Hm @ (s * q)
    assert np.allclose(xhat @ q, yhat @ rq, rtol=0, atol=1e-12 * np.abs(xhat).sum(1).max())
    w = np.random.default_rng(5).random(32)
    unrot = s * (Hm @ (w @ yhat))
    assert np.allclose(w @ xhat, unrot, rtol=0, atol=1e-12)


def test_rotated_tiers_exact_threshold_hit_goes_up(orc):
    """code = #{k : u >= t_k}: a value exactly on a threshold takes the upper code.

    The middle threshold of every symmetric codebook is exactly 0.  With all signs +1
    and x = e_0 + e_1, the first FWHT stage gives (2, 0) and the later stages copy that
    pattern, so y_i = 2c for even i and exactly 0 for odd i: every odd element sits on
    the middle threshold and must take code L/2 (the reading u > t_k would give L/2 - 1).
    For TQ4 the even elements have u = 2c / (32c * c) = sqrt(2), between t_11 = 1.0992
    and t_12 = 1.4370, so code 12: every packed byte is 0x8C."""
    x = np.zeros((1, 512), np.float32)
    x[0, 0] = x[0, 1] = 1.0
    signs = np.zeros(16, np.uint32)
    lloyd, cb, thr, _ = orc.tq4_codebook()
    assert thr[7] == 0.0 and thr[11] < math.sqrt(2) < thr[12]
    packed, radius = orc.encode_tq4(x, signs)
    assert np.all(packed[0] == 0x8C)
    for bits in (3, 6):
        L = 1 << bits
        cbb, thb = orc.tq_codebook(bits)[1:3]
        assert thb[L // 2 - 1] == 0.0
        pk, _ = orc.encode_tq(x, signs, bits)
        stream = np.unpackbits(pk[0], bitorder="little")
        codes = stream.reshape(512, bits) @ (1 << np.arange(bits))
        assert np.all(codes[1::2] == L // 2)


def test_tq4_inert_rows_and_refusal(orc):
    x = np.zeros((3, 512), np.float32)
    x[1, 7] = 2.5
    packed, radius = orc.encode_tq4(x, W.sign_bits(0))
    assert radius[0] == 0 and not packed[0].any()
    assert radius[2] == 0 and not packed[2].any()
    assert radius[1] == np.float32(2.5)
    for bad in (500, 384, 96, 513):
        with pytest.raises(ValueError):
            orc.encode_tq4(np.ones((1, bad), np.float32), np.zeros(32, np.uint32))
        with pytest.raises(ValueError):
            orc.decode_tq4(np.zeros((1, bad // 2), np.uint8), np.ones(1, np.float32),
                           np.zeros(32, np.uint32), bad)


# ----------------------------------------------------------------------- q4_0 ----------

def _read_golden(name):
    import os
    lines = [l.split("#")[0].strip() for l in open(os.path.join(GOLDEN, name))]
    return bytes.fromhex("".join(l for l in lines if l))


def test_q4_all_zero_group_golden(orc):
    out = orc.q4_block(np.zeros(32, np.float32))
    assert bytes(out) == _read_golden("q4_all_zero_block.hex")
    # a zero row through the whole append: every block the same 18 bytes
    z = orc.fwht256_q4(np.zeros(256, np.float32))
    assert not z.any()


def test_q4_tie_rule(orc):
    v = np.float32(1.5)
    # {v, -v, v, -v, ...}: the tie resolves to +v, so d = v / -8 < 0
    blk = np.array([v, -v] * 16, np.float32)
    out = orc.q4_block(blk)
    d = np.frombuffer(bytes(out[:2]), np.float16)[0]
    assert d == np.float16(-v / 8)
    # one +v among -v: still +v
    blk = np.full(32, -v, np.float32)
    blk[19] = v
    d = np.frombuffer(bytes(orc.q4_block(blk)[:2]), np.float16)[0]
    assert d == np.float16(-v / 8)
    # all equal -v: mval = -v, d = +v/8, every element codes to 0
    out = orc.q4_block(np.full(32, -v, np.float32))
    assert np.frombuffer(bytes(out[:2]), np.float16)[0] == np.float16(v / 8)
    assert all(b == 0x00 for b in out[2:])
    # all equal +v: mval = +v, d = -v/8, every element codes to 0 as well
    out = orc.q4_block(np.full(32, v, np.float32))
    assert all(b == 0x00 for b in out[2:])
    # x = -mval lands on 16 and is clamped to 15
    blk = np.zeros(32, np.float32)
    blk[0], blk[17] = v, -v + np.float32(0.25)   # |.| smaller: +v is the maximum
    blk[5] = -v + np.float32(1e-3)
    out = orc.q4_block(blk)
    assert out[2] & 15 == 0                       # element 0 (the maximum) -> 0
    assert out[2 + 5] & 15 in (15,)               # ~ -mval -> clamped 15


def test_q4_dequant_error_bound(orc):
    """Round-to-nearest codes: away from the clamp, |(q - 8) d_f16 - z| is at most half a
    step |d| (the +8.5 offset rounds z/d + 8 half up), plus the binary16 rounding of d
    (|q - 8| <= 8 steps of relative 2^-11) and the fp32 reciprocal (2^-20 of a step).  A
    codeword without the half offset (floor) errs by up to a whole step and fails."""
    g = np.random.default_rng(8)
    n_checked = 0
    for amp in (1e-3, 1.0, 40.0):
        for _ in range(40):
            z = (g.standard_normal(32) * amp).astype(np.float32)
            out = orc.q4_block(z)
            d16 = float(np.frombuffer(bytes(out[:2]), np.float16)[0])
            q = np.array([(out[2 + j] & 15) if j < 16 else (out[2 + j - 16] >> 4) for j in range(32)],
                         np.int32)
            mval = z[np.argmax(np.abs(z))]
            d = abs(float(mval) / 8.0)
            clamped = (q == 15) & (z.astype(np.float64) / -(float(mval) / 8.0) >= 7.5)
            deq = (q - 8) * d16
            err = np.abs(deq - z.astype(np.float64))[~clamped]
            assert np.all(err <= d * (0.5 + 8 * 2.0 ** -11 + 2.0 ** -20)), (amp, err.max() / d)
            # the code step is max|x|/8 (the page): even a clamped element is within a step
            assert np.max(np.abs(deq - z)) <= np.max(np.abs(z)) / 8 * (1 + 2 ** -9) + 1e-30
            n_checked += int((~clamped).sum())
    assert n_checked > 3000


def test_q4_codeword_rounds_half_up(orc):
    """q = trunc(fma(z, id, 8.5)) on a block with d = 1 (mval = -8, id = 1): z + 8.5 is
    exact, so each code is z + 8 rounded half up, clamped to [0, 15].  Codes written out:
      j   z               z + 8.5       code      j   z        z + 8.5   code
      0   -8 (mval)       0.5           0         16   2.5     11        11
      1   0.5             9             9         17  -2.5     6         6
      2   0.5 - 2^-20     9 - 2^-20     8         18   4.5     13        13
      3   -0.5            8             8         19  -4.5     4         4
      4   -0.5 - 2^-20    8 - 2^-20     7         20   0.75    9.25      9
      5   1.5             10            10        21  -0.75    7.75      7
      6   -1.5            7             7         22   5.5     14        14
      7   6.5             15            15        23  -5.5     3         3
      8   7               15.5          15        24   6       14.5      14
      9   7.5             16 -> clamp   15        25  -6       2.5       2
      10  -7.5            1             1         26   2       10.5      10
      11  -7.5 - 2^-20    1 - 2^-20     0         27  -2       6.5       6
      12  3.25            11.75         11        28   1       9.5       9
      13  -3.25           5.25          5         29  -1       7.5       7
      14  0               8.5           8         30   0.25    8.75      8
      15  -0              8.5           8         31  -0.25    8.25      8
    d = 1.0 is binary16 0x3C00 (bytes 00 3C); byte 2 + j = q_j | q_(j+16) << 4."""
    e = 2.0 ** -20
    z = np.array([-8, 0.5, 0.5 - e, -0.5, -0.5 - e, 1.5, -1.5, 6.5, 7, 7.5, -7.5, -7.5 - e, 3.25, -3.25,
                  0.0, -0.0, 2.5, -2.5, 4.5, -4.5, 0.75, -0.75, 5.5, -5.5, 6, -6, 2, -2, 1, -1,
                  0.25, -0.25], np.float32)
    assert z[2] != 0.5 and z[4] != -0.5 and z[11] != -7.5
    q = [0, 9, 8, 8, 7, 10, 7, 15, 15, 15, 1, 0, 11, 5, 8, 8,
         11, 6, 13, 4, 9, 7, 14, 3, 14, 2, 10, 6, 9, 7, 8, 8]
    expect = bytes([0x00, 0x3C] + [q[j] | (q[j + 16] << 4) for j in range(16)])
    assert bytes(orc.q4_block(z)) == expect


def test_q4_reciprocal_uses_the_fp32_scale(orc):
    """id = 1/d from the fp32 d, before d is rounded to binary16 for storage.
    mval = -(8 + 2^-9) gives d = 1 + 2^-12 (exact in fp32), stored as binary16 1.0
    (0x3C00: 2^-12 is below half a binary16 ulp).  With the fp32 d, id = 1 - 2^-12 + ..., so
      z = 0.5: 8.5 + 0.49988 = 8.99988 -> 8   (the binary16 d would give 9)
      z = 4.5: 8.5 + 4.49890 = 12.9989 -> 12  (the binary16 d would give 13)
      z = -0.5: 8.00012 -> 8;  z = mval: 0.5 -> 0;  z = 0: 8."""
    z = np.zeros(32, np.float32)
    z[0] = -(8.0 + 2.0 ** -9)
    z[1], z[2], z[3] = 0.5, 4.5, -0.5
    assert np.float32(z[0] / -8.0) == np.float32(1 + 2.0 ** -12)
    q = [0, 8, 12, 8] + [8] * 28
    expect = bytes([0x00, 0x3C] + [q[j] | (q[j + 16] << 4) for j in range(16)])
    assert bytes(orc.q4_block(z)) == expect


def test_fwht256_orthonormal(orc):
    g = np.random.default_rng(9)
    x = g.standard_normal(256).astype(np.float32)
    z = orc.fwht256_q4(x)
    Hm = scipy.linalg.hadamard(256).astype(np.float64) / 16
    assert np.allclose(z, Hm @ x, atol=1e-5)
    assert np.allclose(orc.fwht256_q4(z), x, atol=1e-5)       # self-inverse
    assert abs(np.linalg.norm(z) - np.linalg.norm(x)) < 1e-4


def test_q4_append_placement_and_gather(orc):
    """Small paged workload with a permuted table and a page-crossing start: every
    (sequence, token, head) row lands at the cell the page table names (placement
    recomputed here), untouched cells keep the sentinel, gather returns
    f16((q - 8) * d) per element (numpy's binary16 conversion)."""
    wl = W.q4_paged(n_seq=3, n_tok=21, n_heads=2, page_size=8, seed=4, spare_pages=2)
    k_pool = np.full((wl.n_cells, 2, 144), 0xA5, np.uint8)
    v_pool = np.full((wl.n_cells, 2, 144), 0x5A, np.uint8)
    orc.append_q4(wl.k, wl.v, wl.pos0, wl.page_table, wl.page_size, wl.n_cells, k_pool, v_pool)
    touched = np.zeros(wl.n_cells, bool)
    for s in range(3):
        for t in range(21):
            pos = int(wl.pos0[s]) + t
            cell = wl.page_table[s, pos // 8] * 8 + pos % 8
            touched[cell] = True
            for h in range(2):
                for pool, src in ((k_pool, wl.k), (v_pool, wl.v)):
                    z = orc.fwht256_q4(src[s, t, h])
                    exp = np.concatenate([orc.q4_block(z[32 * b: 32 * b + 32]) for b in range(8)])
                    assert np.array_equal(pool[cell, h], exp)
    assert np.all(k_pool[~touched] == 0xA5) and np.all(v_pool[~touched] == 0x5A)
    out = orc.gather_q4(k_pool, wl.pos0, 21, wl.page_table, wl.page_size, wl.n_cells, 2)
    for s, t, h in [(0, 0, 0), (1, 7, 1), (2, 20, 0), (2, 9, 1)]:
        pos = int(wl.pos0[s]) + t
        cell = wl.page_table[s, pos // 8] * 8 + pos % 8
        blk = k_pool[cell, h].reshape(8, 18)
        d = blk[:, :2].copy().view(np.float16).astype(np.float32)[:, 0]
        lo, hi = blk[:, 2:] & 15, blk[:, 2:] >> 4
        q = np.concatenate([lo, hi], axis=1).astype(np.float32)
        exp = ((q - 8) * d[:, None]).astype(np.float16).view(np.uint16).ravel()
        assert np.array_equal(out[s, t, h], exp)
