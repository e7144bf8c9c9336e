"""CPU oracle of the quantized MLA KV-cache path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` may import this package.  The product package never
does, and this package never imports the product package: the two share no code.

The arithmetic lives in ``kvq_oracle.c`` (plain C, one thread, fp64 where the method
leaves precision open).  This module compiles it with gcc and wraps each routine for
numpy arrays.  Citations of the pages are in the C file, next to each routine.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_HDR = os.path.join(_HERE, "kvq_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkvq_oracle.so")

FMT_FP8 = 1
FMT_TQ4 = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fp contraction, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> C.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


_p = C.c_void_p
_i32, _i64, _f32 = C.c_int32, C.c_int64, C.c_float


class OrcMla(C.Structure):
    _fields_ = [
        ("n_seq", _i32), ("n_q", _i32), ("n_heads", _i32), ("d_lat", _i32), ("d_rope", _i32),
        ("causal", _i32),
        ("seq_len", _p), ("seq_fmt", _p), ("block_table", _p),
        ("max_pages", _i32), ("page_size", _i32), ("seq_stride_rows", _i64),
        ("fp8_lat", _p), ("fp8_lat_scale", _p), ("fp8_rope", _p), ("fp8_rope_scale", _p),
        ("tq4_lat", _p), ("tq4_radius", _p), ("tq4_rope", _p), ("tq4_rope_scale", _p),
        ("tq4_signs", _p),
        ("q_lat", _p), ("q_rope", _p), ("idx", _p), ("top_k", _i32), ("sm_scale", _f32),
        ("n_split", _i32), ("head_lo", _i32), ("head_hi", _i32),
        ("seq_sel", _p), ("n_sel", _i32),
    ]


def _declare(L: C.CDLL) -> None:
    L.orc_e4m3_value.restype = C.c_double
    L.orc_e4m3_value.argtypes = [C.c_uint8]
    L.orc_e4m3_rne.restype = C.c_uint8
    L.orc_e4m3_rne.argtypes = [C.c_float]
    L.orc_f16_rne.restype = C.c_uint16
    L.orc_f16_rne.argtypes = [C.c_double]
    L.orc_f16_value.restype = C.c_double
    L.orc_f16_value.argtypes = [C.c_uint16]
    L.orc_encode_fp8.restype = None
    L.orc_encode_fp8.argtypes = [_p, _i64, C.c_int, _i64, _p, _i64, _p]
    L.orc_decode_fp8.restype = None
    L.orc_decode_fp8.argtypes = [_p, _i64, C.c_int, _i64, _p, _p]
    L.orc_tq4_codebook.restype = C.c_int
    L.orc_tq4_codebook.argtypes = [_p, _p, _p, _p]
    L.orc_fwht_f32.restype = None
    L.orc_fwht_f32.argtypes = [_p, C.c_int]
    L.orc_fwht_f64.restype = None
    L.orc_fwht_f64.argtypes = [_p, C.c_int]
    L.orc_encode_tq4.restype = C.c_int
    L.orc_encode_tq4.argtypes = [_p, _i64, C.c_int, _i64, _p, _p, _i64, _p]
    L.orc_decode_tq4.restype = C.c_int
    L.orc_decode_tq4.argtypes = [_p, _i64, C.c_int, _i64, _p, _p, _p, _p]
    L.orc_tq_codebook.restype = C.c_int
    L.orc_tq_codebook.argtypes = [C.c_int, _p, _p, _p, _p]
    L.orc_encode_tq.restype = C.c_int
    L.orc_encode_tq.argtypes = [C.c_int, _p, _i64, C.c_int, _i64, _p, _p, _i64, _p]
    L.orc_decode_tq.restype = C.c_int
    L.orc_decode_tq.argtypes = [C.c_int, _p, _i64, C.c_int, _i64, _p, _p, _p, _p]
    L.orc_fwht256_q4.restype = None
    L.orc_fwht256_q4.argtypes = [_p, _p]
    L.orc_q4_block.restype = None
    L.orc_q4_block.argtypes = [_p, _p]
    L.orc_append_q4.restype = C.c_int
    L.orc_append_q4.argtypes = [_p, _p, C.c_int, _p, C.c_int, C.c_int, C.c_int, _p, C.c_int,
                                C.c_int, _i64, _p, _p]
    L.orc_gather_q4.restype = C.c_int
    L.orc_gather_q4.argtypes = [_p, C.c_int, _p, C.c_int, C.c_int, C.c_int, _p, C.c_int,
                                C.c_int, _i64, _p]
    L.orc_mla_decode.restype = C.c_int
    L.orc_project_rows.argtypes = [_p, _i64, C.c_int, _p, C.c_int, _i64, _p]
    L.orc_project_rows.restype = None
    L.orc_project_append_q4.argtypes = [_p, C.c_int, _p, C.c_int, C.c_int, _p, _p, C.c_int,
                                        C.c_int, _p, C.c_int, C.c_int, _i64, _p, _p]
    L.orc_mla_decode.argtypes = [C.POINTER(OrcMla), _p, _p, _p]
    L.orc_q4_decode.argtypes = [C.c_int, C.c_int, C.c_int, _p, _p, C.c_int, C.c_int, _i64, _p, _p,
                                _p, _p, C.c_double, _p, C.c_int, _p, _p, _p]
    L.orc_q4_decode.restype = C.c_int


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --- number formats -----------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def e4m3_rne(v: float) -> int:
    return lib().orc_e4m3_rne(float(v))


def f16_rne(v: float) -> int:
    return lib().orc_f16_rne(float(v))


def f16_value(h: int) -> float:
    return lib().orc_f16_value(int(h))


# --- fp8 ------------------------------------------------------------------------------

def encode_fp8(x: np.ndarray):
    """rows [R][dim] fp32 -> (codes u8 [R][dim], scales f32 [R])."""
    x = _c(x, np.float32)
    R, D = x.shape
    codes = np.empty((R, D), np.uint8)
    scales = np.empty(R, np.float32)
    lib().orc_encode_fp8(_ptr(x), R, D, D, _ptr(codes), D, _ptr(scales))
    return codes, scales


def decode_fp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    R, D = codes.shape
    out = np.empty((R, D), np.float64)
    lib().orc_decode_fp8(_ptr(codes), R, D, D, _ptr(scales), _ptr(out))
    return out


# --- TQ4 ------------------------------------------------------------------------------

def tq4_codebook():
    """(lloyd fp64 [16], centroids f32 [16] (binary16 values), thresholds f32 [15], iters)."""
    lloyd = np.empty(16, np.float64)
    cb = np.empty(16, np.float32)
    thr = np.empty(15, np.float32)
    it = C.c_int(0)
    lib().orc_tq4_codebook(_ptr(lloyd), _ptr(cb), _ptr(thr), C.addressof(it))
    return lloyd, cb, thr, it.value


def fwht_f32(w: np.ndarray) -> np.ndarray:
    w = _c(w, np.float32).copy()
    lib().orc_fwht_f32(_ptr(w), w.shape[-1])
    return w


def fwht_f64(w: np.ndarray) -> np.ndarray:
    w = _c(w, np.float64).copy()
    lib().orc_fwht_f64(_ptr(w), w.shape[-1])
    return w


def encode_tq4(x: np.ndarray, sign_bits: np.ndarray):
    """rows [R][n] fp32 -> (packed u8 [R][n/2], radius f32 [R]); raises for non-pow2 n."""
    x = _c(x, np.float32)
    sb = _c(sign_bits, np.uint32)
    R, D = x.shape
    packed = np.empty((R, D // 2), np.uint8)
    radius = np.empty(R, np.float32)
    rc = lib().orc_encode_tq4(_ptr(x), R, D, D, _ptr(sb), _ptr(packed), D // 2, _ptr(radius))
    if rc != 0:
        raise ValueError(f"oracle TQ4 encode refused dim={D} (rc={rc})")
    return packed, radius


def decode_tq4(packed: np.ndarray, radius: np.ndarray, sign_bits: np.ndarray, dim: int):
    """-> (xhat fp64 [R][dim] in the original basis, yhat fp64 [R][dim] rotated)."""
    packed = _c(packed, np.uint8)
    radius = _c(radius, np.float32)
    sb = _c(sign_bits, np.uint32)
    R = packed.shape[0]
    xhat = np.empty((R, dim), np.float64)
    yhat = np.empty((R, dim), np.float64)
    rc = lib().orc_decode_tq4(_ptr(packed), R, dim, dim // 2, _ptr(radius), _ptr(sb),
                              _ptr(xhat), _ptr(yhat))
    if rc != 0:
        raise ValueError(f"oracle TQ4 decode refused dim={dim}")
    return xhat, yhat


# --- TQ-b (b = 3, 4, 6) ---------------------------------------------------------------

TQ_FMT = {3: 5, 4: 2, 6: 4}        # library / oracle format code of each width


def tq_codebook(bits: int):
    """(lloyd fp64 [2^b], centroids f32 [2^b] (binary16 values), thresholds f32 [2^b - 1],
    iterations)."""
    L = 1 << bits
    lloyd = np.empty(L, np.float64)
    cb = np.empty(L, np.float32)
    thr = np.empty(L - 1, np.float32)
    it = C.c_int(0)
    if lib().orc_tq_codebook(bits, _ptr(lloyd), _ptr(cb), _ptr(thr), C.addressof(it)) != 0:
        raise ValueError(f"oracle TQ codebook refused bits={bits}")
    return lloyd, cb, thr, it.value


def encode_tq(x: np.ndarray, sign_bits: np.ndarray, bits: int):
    """rows [R][n] fp32 -> (packed u8 [R][n*b/8], radius f32 [R])."""
    x = _c(x, np.float32)
    sb = _c(sign_bits, np.uint32)
    R, D = x.shape
    rb = D * bits // 8
    packed = np.empty((R, rb), np.uint8)
    radius = np.empty(R, np.float32)
    rc = lib().orc_encode_tq(bits, _ptr(x), R, D, D, _ptr(sb), _ptr(packed), rb, _ptr(radius))
    if rc != 0:
        raise ValueError(f"oracle TQ encode refused dim={D} bits={bits} (rc={rc})")
    return packed, radius


def decode_tq(packed: np.ndarray, radius: np.ndarray, sign_bits: np.ndarray, dim: int, bits: int):
    """-> (xhat fp64 [R][dim] in the original basis, yhat fp64 [R][dim] rotated)."""
    packed = _c(packed, np.uint8)
    radius = _c(radius, np.float32)
    sb = _c(sign_bits, np.uint32)
    R = packed.shape[0]
    xhat = np.empty((R, dim), np.float64)
    yhat = np.empty((R, dim), np.float64)
    rc = lib().orc_decode_tq(bits, _ptr(packed), R, dim, dim * bits // 8, _ptr(radius), _ptr(sb),
                             _ptr(xhat), _ptr(yhat))
    if rc != 0:
        raise ValueError(f"oracle TQ decode refused dim={dim} bits={bits}")
    return xhat, yhat


# --- q4_0 -----------------------------------------------------------------------------

def fwht256_q4(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    z = np.empty(256, np.float32)
    lib().orc_fwht256_q4(_ptr(x), _ptr(z))
    return z


def q4_block(z: np.ndarray) -> np.ndarray:
    z = _c(z, np.float32)
    out = np.empty(18, np.uint8)
    lib().orc_q4_block(_ptr(z), _ptr(out))
    return out


def append_q4(k, v, pos0, page_table, page_size, n_cells, k_pool, v_pool):
    """k, v [n_seq][n_tok][n_heads][256] fp32; pools [n_cells][n_heads][144] u8 (in place)."""
    k = _c(k, np.float32)
    v = _c(v, np.float32)
    pos0 = _c(pos0, np.int32)
    pt = _c(page_table, np.int32)
    n_seq, n_tok, n_heads, hd = k.shape
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    rc = lib().orc_append_q4(_ptr(k), _ptr(v), n_seq, _ptr(pos0), n_tok, n_heads, hd, _ptr(pt),
                             pt.shape[1], page_size, n_cells, _ptr(k_pool), _ptr(v_pool))
    if rc != 0:
        raise ValueError(f"oracle q4 append refused (rc={rc})")


def project_rows(h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """h [rows][d_model] fp32; w [d_model][n_out] fp32, or uint16 bfloat16 patterns ->
    y [rows][n_out] fp32 in the library's fixed summation order."""
    h = _c(h, np.float32)
    bf16 = w.dtype == np.uint16
    w = _c(w, np.uint16 if bf16 else np.float32)
    rows, d_model = h.shape
    n_out = w.shape[1]
    assert w.shape[0] == d_model
    y = np.empty((rows, n_out), np.float32)
    lib().orc_project_rows(_ptr(h), rows, d_model, _ptr(w), int(bf16), n_out, _ptr(y))
    return y


def project_append_q4(h, w_k, w_v, pos0, page_table, page_size, n_cells, k_pool, v_pool):
    """h [n_seq][n_tok][d_model] fp32; w_k, w_v [d_model][n_heads * 256] fp32 or uint16
    bfloat16 patterns; pools [n_cells][n_heads][144] u8 (in place)."""
    h = _c(h, np.float32)
    bf16 = w_k.dtype == np.uint16
    w_k = _c(w_k, np.uint16 if bf16 else np.float32)
    w_v = _c(w_v, np.uint16 if bf16 else np.float32)
    pos0 = _c(pos0, np.int32)
    pt = _c(page_table, np.int32)
    n_seq, n_tok, d_model = h.shape
    n_heads = w_k.shape[1] // 256
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    rc = lib().orc_project_append_q4(_ptr(h), n_seq, _ptr(pos0), n_tok, d_model, _ptr(w_k),
                                     _ptr(w_v), int(bf16), n_heads, _ptr(pt), pt.shape[1],
                                     page_size, n_cells, _ptr(k_pool), _ptr(v_pool))
    if rc != 0:
        raise ValueError(f"oracle projected q4 append refused (rc={rc})")


def gather_q4(pool, pos0, n_tok, page_table, page_size, n_cells, n_heads) -> np.ndarray:
    """-> binary16 bit patterns u16 [n_seq][n_tok][n_heads][256]."""
    pool = _c(pool, np.uint8)
    pos0 = _c(pos0, np.int32)
    pt = _c(page_table, np.int32)
    n_seq = pos0.shape[0]
    out = np.empty((n_seq, n_tok, n_heads, 256), np.uint16)
    rc = lib().orc_gather_q4(_ptr(pool), n_seq, _ptr(pos0), n_tok, n_heads, 256, _ptr(pt),
                             pt.shape[1], page_size, n_cells, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle q4 gather refused (rc={rc})")
    return out


def q4_decode(*, seq_len, page_table, page_size, n_cells, k_pool, v_pool, q, n_kv, sm_scale,
              gate=None, seq_sel=None):
    """q4_0 paged GQA decode attention in fp64: q [n_seq][n_qh][256] fp32 (unrotated),
    pools [n_cells][n_kv][144] u8, optional gate [n_seq][n_qh][256] fp32.
    -> (out [n_seq][n_qh][256] f64, lse [n_seq][n_qh] f64, bad_page flag)."""
    seq_len = _c(seq_len, np.int32)
    pt = _c(page_table, np.int32)
    q = _c(q, np.float32)
    n_seq, n_qh, hd = q.shape
    assert hd == 256
    k_pool = _c(k_pool, np.uint8)
    v_pool = _c(v_pool, np.uint8)
    g = None if gate is None else _c(gate, np.float32)
    sel = None if seq_sel is None else _c(seq_sel, np.int32)
    out = np.zeros((n_seq, n_qh, 256), np.float64)
    lse = np.full((n_seq, n_qh), np.nan, np.float64)
    bad = np.zeros(1, np.uint32)
    rc = lib().orc_q4_decode(n_seq, n_qh, n_kv, _ptr(seq_len), _ptr(pt), pt.shape[1], page_size,
                             n_cells, _ptr(k_pool), _ptr(v_pool), _ptr(q),
                             None if g is None else _ptr(g), float(sm_scale),
                             None if sel is None else _ptr(sel), 0 if sel is None else len(sel),
                             _ptr(out), _ptr(lse), _ptr(bad))
    if rc != 0:
        raise ValueError(f"oracle q4 decode refused (rc={rc})")
    return out, lse, int(bad[0])


# --- MLA decode -----------------------------------------------------------------------

def mla_abs_terms(*, lat_rows, rope_rows, q_lat, q_rope, sm_scale):
    """The sum of the absolute values of the terms of each output element of one
    sequence's decode (colibri PR #399: out = sum_t softmax(s)_t c_t), the denominator of
    the Σ|terms|-relative error: A[q][h][d] = sum_t p_t |c_{t,d}|, with p the softmax of
    s_t = sm_scale (q_lat . c_t + q_rope . k_rope_t), in fp64 over the dequantized rows
    lat_rows [T][512] and rope_rows [T][64] (every row admissible).  |out_d| <= A_d,
    with equality when every c_{t,d} >= 0."""
    lat = np.asarray(lat_rows, np.float64)
    rope = np.asarray(rope_rows, np.float64)
    tau = float(np.float32(sm_scale))
    s = tau * (np.asarray(q_lat, np.float64) @ lat.T + np.asarray(q_rope, np.float64) @ rope.T)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    return p @ np.abs(lat)


def mla_decode(*, seq_len, seq_fmt, q_lat, q_rope, sm_scale, causal=False,
               block_table=None, page_size=0, seq_stride_rows=0,
               fp8=None, tq4=None, signs=None, idx=None, n_split=0,
               heads=None, seq_sel=None):
    """fp64 absorbed-MLA decode.

    fp8 / tq4: dicts with keys lat, lat_scale (radius for tq4), rope, rope_scale.
    q_lat [n_seq][n_q][H][512], q_rope [n_seq][n_q][H][64].
    Returns (out fp64 [n_seq][n_q][H][512], lse fp64 [n_seq][n_q][H], bad_index flag);
    entries outside `heads` / `seq_sel` are NaN.
    """
    q_lat = _c(q_lat, np.float32)
    q_rope = _c(q_rope, np.float32)
    n_seq, n_q, H, DL = q_lat.shape
    DR = q_rope.shape[-1]
    seq_len = _c(seq_len, np.int32)
    seq_fmt = _c(seq_fmt, np.int32)
    keep = [q_lat, q_rope, seq_len, seq_fmt]
    p = OrcMla()
    p.n_seq, p.n_q, p.n_heads, p.d_lat, p.d_rope = n_seq, n_q, H, DL, DR
    p.causal = int(bool(causal))
    p.seq_len, p.seq_fmt = _ptr(seq_len), _ptr(seq_fmt)
    if block_table is not None:
        bt = _c(block_table, np.int32)
        keep.append(bt)
        p.block_table, p.max_pages, p.page_size = _ptr(bt), bt.shape[1], page_size
    p.seq_stride_rows = seq_stride_rows
    for name, tier in (("fp8", fp8), ("tq4", tq4)):
        if tier is None:
            continue
        lat = _c(tier["lat"], np.uint8)
        ls = _c(tier["lat_scale"], np.float32)
        rope = _c(tier["rope"], np.uint8)
        rs = _c(tier["rope_scale"], np.float32)
        keep += [lat, ls, rope, rs]
        if name == "fp8":
            p.fp8_lat, p.fp8_lat_scale, p.fp8_rope, p.fp8_rope_scale = map(_ptr, (lat, ls, rope, rs))
        else:
            p.tq4_lat, p.tq4_radius, p.tq4_rope, p.tq4_rope_scale = map(_ptr, (lat, ls, rope, rs))
    if signs is not None:
        sg = _c(signs, np.uint32)
        keep.append(sg)
        p.tq4_signs = _ptr(sg)
    if idx is not None:
        ix = _c(idx, np.int32)
        keep.append(ix)
        p.idx, p.top_k = _ptr(ix), ix.shape[-1]
    p.q_lat, p.q_rope = _ptr(q_lat), _ptr(q_rope)
    p.sm_scale = float(sm_scale)
    p.n_split = int(n_split)
    h0, h1 = (0, H) if heads is None else heads
    p.head_lo, p.head_hi = h0, h1
    if seq_sel is not None:
        ss = _c(seq_sel, np.int32)
        keep.append(ss)
        p.seq_sel, p.n_sel = _ptr(ss), ss.shape[0]
    out = np.full((n_seq, n_q, H, DL), np.nan, np.float64)
    lse = np.full((n_seq, n_q, H), np.nan, np.float64)
    bad = C.c_uint32(0)
    lib().orc_mla_decode(C.byref(p), _ptr(out), _ptr(lse), C.addressof(bad))
    del keep
    return out, lse, bool(bad.value)
