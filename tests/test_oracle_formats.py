"""Pins of the oracle's number formats against library conversions and the format
definitions (e4m3: colibri PR #399, KV8 rebase note on the fp8 value grid; binary16:
Strata PR #2533, the software fp16 round-to-nearest-even of the q4 scale)."""
import numpy as np
import pytest
import torch


def _torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_table_matches_library(orc):
    ref = _torch_e4m3_values()
    for c in range(256):
        if c & 0x7F == 0x7F:
            assert np.isnan(ref[c])               # the library's NaN pattern ...
            assert orc.e4m3_value(c) == 0.0       # ... reads back as 0 on the page
            continue
        assert orc.e4m3_value(c) == ref[c], hex(c)


def test_e4m3_exhaustive_roundtrip(orc):
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        v = orc.e4m3_value(c)
        got = orc.e4m3_rne(np.float32(v if c != 0x80 else -0.0))
        assert got == c, (hex(c), v, hex(got))


def test_e4m3_midpoints_round_to_even(orc):
    ref = _torch_e4m3_values()
    pos = [c for c in range(0x7F)]                # 0x00 .. 0x7E, increasing values
    for a, b in zip(pos[:-1], pos[1:]):
        va, vb = ref[a], ref[b]
        mid = np.float32((va + vb) / 2)           # 5 significant bits: exact in fp32
        assert float(mid) == (va + vb) / 2
        even = a if (a & 1) == 0 else b
        assert orc.e4m3_rne(mid) == even, (hex(a), hex(b))
        assert orc.e4m3_rne(-mid) == even | 0x80
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1e9))
        assert orc.e4m3_rne(below) == a
        assert orc.e4m3_rne(above) == b
    # library conversion agrees on in-range values (it is RNE there)
    g = np.random.default_rng(5)
    x = (g.standard_normal(20000) * np.exp(g.uniform(-9, 6, 20000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([orc.e4m3_rne(v) for v in x], np.uint8)
    assert np.array_equal(lib, mine)


def test_e4m3_saturation_and_underflow(orc):
    for v in (448.0, 448.0001, 463.9, 464.0, 480.0, 1e6, 3.0e38):
        assert orc.e4m3_rne(np.float32(v)) == 0x7E
        assert orc.e4m3_rne(np.float32(-v)) == 0xFE
    tiny = 2.0 ** -10                              # half the smallest subnormal
    assert orc.e4m3_rne(np.float32(tiny)) == 0x00  # tie to even -> zero
    assert orc.e4m3_rne(np.float32(-tiny)) == 0x80  # sign kept
    assert orc.e4m3_rne(np.nextafter(np.float32(tiny), np.float32(1))) == 0x01
    assert orc.e4m3_rne(np.float32(1e-30)) == 0x00
    assert orc.e4m3_rne(np.float32(-1e-30)) == 0x80


def test_f16_all_patterns(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = h.view(np.float16).astype(np.float64)
    for i in range(0, 65536, 1):
        if np.isnan(vals[i]):
            continue
        assert orc.f16_value(i) == vals[i]
        assert orc.f16_rne(vals[i]) == i or (vals[i] == 0 and orc.f16_rne(vals[i]) == i)


def test_f16_rne_random_and_midpoints(orc):
    g = np.random.default_rng(3)
    x = g.standard_normal(30000) * np.exp(g.uniform(-25, 12, 30000))
    lib = x.astype(np.float16).view(np.uint16)      # numpy converts double -> half RNE
    mine = np.array([orc.f16_rne(float(v)) for v in x], np.uint16)
    assert np.array_equal(lib, mine)
    # exact midpoints between adjacent binary16 values (fp32 inputs, as the q4 scale)
    hs = np.arange(0, 0x7BFF, 37, dtype=np.uint16)
    a = hs.view(np.float16).astype(np.float64)
    b = (hs + 1).view(np.float16).astype(np.float64)
    mids = (a + b) / 2
    for hv, m in zip(hs, mids):
        even = int(hv) if int(hv) % 2 == 0 else int(hv) + 1
        assert orc.f16_rne(m) == even
    assert orc.f16_rne(65520.0) == 0x7C00
    assert orc.f16_rne(65519.99) == 0x7BFF
    assert orc.f16_rne(-0.0) == 0x8000
