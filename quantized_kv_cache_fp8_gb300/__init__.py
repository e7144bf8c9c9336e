"""Quantized MLA KV cache on GB300 — Python binding of the C ABI ``libkvq``.

Each function here has the name of the C entry point it wraps and only marshals its
arguments (torch tensors -> device pointers, the current CUDA stream): every step of
the path runs in the CUDA kernels of ``libkvq.so``.  There is no fallback: if the
library is missing or fails to load, importing :func:`lib` raises.

Layouts and semantics are documented once, in ``include/kvq.h``.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

__all__ = [
    "KvqError", "lib", "kvq_version", "kvq_tq4_codebook", "kvq_set_fault",
    "kvq_encode_fp8", "kvq_encode_tq4", "kvq_append_q4", "kvq_project_append_q4",
    "kvq_gather_q4", "kvq_gather_rows", "WEIGHT_F32", "WEIGHT_BF16",
    "kvq_mla_decode", "kvq_mla_decode_workspace", "kvq_mla_decode_noalloc", "kvq_mla_decode_kernel",
    "MlaCache",
    "MlaProblem", "Q4Problem", "make_q4_problem", "kvq_q4_decode", "kvq_q4_decode_workspace",
    "FMT_FP8", "FMT_TQ4", "FMT_Q4_0", "FMT_TQ6", "FMT_TQ3", "TQ_FMT", "kvq_encode_tq", "kvq_encode_mla",
    "kvq_tq_codebook", "DEV_BAD_INDEX", "DEV_BAD_PAGE", "DEV_TIMEOUT",
    "DEV_BAD_FORMAT",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkvq.so")

FMT_FP8, FMT_TQ4, FMT_Q4_0, FMT_TQ6, FMT_TQ3 = 1, 2, 3, 4, 5
WEIGHT_F32, WEIGHT_BF16 = 0, 1
TQ_FMT = {3: FMT_TQ3, 4: FMT_TQ4, 6: FMT_TQ6}     # rotated tier of each code width
IMPL_AUTO, IMPL_SIMT, IMPL_TC, IMPL_MMA, IMPL_TC16, IMPL_TCF8 = 0, 1, 2, 3, 4, 5
IMPL_BY_FMT = 6   # kvq_mla_decode_kernel only: fp8 sequences on IMPL_TCF8, TQ4 ones on IMPL_TC
DEV_BAD_INDEX, DEV_BAD_PAGE, DEV_TIMEOUT, DEV_BAD_FORMAT = 1, 2, 4, 8
STATUS = {0: "KVQ_OK", 1: "KVQ_EINVAL", 2: "KVQ_ENOTPOW2", 3: "KVQ_EFORMAT", 4: "KVQ_EALIGN",
          5: "KVQ_EWORKSPACE", 6: "KVQ_ECUDA", 7: "KVQ_EFAULT_INJECTED", 8: "KVQ_EMISMATCH",
          9: "KVQ_EIO"}

# every symbol include/kvq.h declares
EXPORTS = ["kvq_version", "kvq_status_string", "kvq_last_error", "kvq_set_fault",
           "kvq_set_wait_limit_ns",
           "kvq_tq4_codebook", "kvq_tq_codebook", "kvq_encode_fp8", "kvq_encode_tq4",
           "kvq_encode_tq", "kvq_encode_mla", "kvq_append_q4", "kvq_project_append_q4",
           "kvq_gather", "kvq_mla_decode_workspace", "kvq_mla_decode_kernel", "kvq_mla_decode",
           "kvq_mla_decode_noalloc", "kvq_q4_decode_workspace", "kvq_q4_decode",
           "kvq_cache_probe", "kvq_cache_save", "kvq_cache_save_f32", "kvq_cache_append",
           "kvq_cache_load_workspace", "kvq_cache_load"]


class KvqError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status


_p = C.c_void_p
_i32, _i64, _f32 = C.c_int32, C.c_int64, C.c_float


class MlaCache(C.Structure):
    _fields_ = [("lat", _p), ("lat_scale", _p), ("rope", _p), ("rope_scale", _p),
                ("n_rows", _i64)]


class GatherDesc(C.Structure):
    _fields_ = [("format", _i32),
                ("q4_pool", _p), ("n_seq", _i32), ("n_tok", _i32), ("n_heads", _i32),
                ("head_dim", _i32), ("pos0", _p), ("n_cells", _i64), ("q4_out", _p),
                ("page_table", _p), ("max_pages", _i32), ("page_size", _i32),
                ("mla_src", MlaCache), ("mla_src_rows", _i64), ("idx", _p), ("n_idx", _i64),
                ("dst_lat", _p), ("dst_lat_scale", _p), ("dst_rope", _p),
                ("dst_rope_scale", _p), ("dev_status", _p)]


class MlaProblem(C.Structure):
    _fields_ = [("n_seq", _i32), ("n_q", _i32), ("n_heads", _i32), ("d_lat", _i32),
                ("d_rope", _i32), ("causal", _i32), ("max_seq_len", _i32),
                ("seq_len", _p), ("seq_fmt", _p), ("fmt", _i32), ("block_table", _p),
                ("max_pages", _i32), ("page_size", _i32), ("seq_stride_rows", _i64),
                ("fp8", MlaCache), ("tq4", MlaCache), ("tq4_signs", _p),
                ("q_lat", _p), ("q_rope", _p), ("idx", _p), ("top_k", _i32),
                ("sm_scale", _f32), ("split_rows", _i32), ("impl", _i32),
                ("overlap_prior", _i32)]


class Q4Problem(C.Structure):
    _fields_ = [("n_seq", _i32), ("n_qh", _i32), ("n_kv", _i32), ("head_dim", _i32),
                ("seq_len", _p), ("max_seq_len", _i32), ("page_table", _p),
                ("max_pages", _i32), ("page_size", _i32), ("n_cells", _i64),
                ("k_pool", _p), ("v_pool", _p), ("q", _p), ("gate", _p),
                ("sm_scale", _f32), ("split_rows", _i32)]


class CacheInfo(C.Structure):
    _fields_ = [("format", _i32), ("codec", _i32), ("bits", _i32), ("d_lat", _i32),
                ("d_rope", _i32), ("n_rows", _i64), ("record_bytes", _i64),
                ("trailing_bytes", _i64)]


_lock = threading.Lock()
_lib = None


def lib() -> C.CDLL:
    """Load libkvq.so (built by ``__graft_entry__.build()``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libkvq.so not built ({LIB_PATH}); run __graft_entry__.build()")
            L = C.CDLL(LIB_PATH)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    L.kvq_version.restype = C.c_int
    L.kvq_status_string.restype = C.c_char_p
    L.kvq_status_string.argtypes = [C.c_int]
    L.kvq_last_error.restype = C.c_char_p
    L.kvq_set_fault.restype = C.c_int
    L.kvq_set_fault.argtypes = [C.c_char_p]
    L.kvq_set_wait_limit_ns.restype = C.c_int
    L.kvq_set_wait_limit_ns.argtypes = [C.c_uint64]
    L.kvq_tq4_codebook.restype = C.c_int
    L.kvq_tq4_codebook.argtypes = [_p, _p]
    L.kvq_encode_fp8.restype = C.c_int
    L.kvq_encode_fp8.argtypes = [_p, _i64, C.c_int, _i64, _p, _i64, _p, _p]
    L.kvq_tq_codebook.restype = C.c_int
    L.kvq_tq_codebook.argtypes = [C.c_int, _p, _p]
    L.kvq_encode_tq.restype = C.c_int
    L.kvq_encode_tq.argtypes = [_p, _i64, C.c_int, _i64, C.c_int, _p, _p, _i64, _p, _p]
    L.kvq_encode_mla.restype = C.c_int
    L.kvq_encode_mla.argtypes = [_p, _i64, _p, _i64, _i64, C.c_int, _p, _p, _i64, _p, _p, _i64, _p, _p]
    L.kvq_encode_tq4.restype = C.c_int
    L.kvq_encode_tq4.argtypes = [_p, _i64, C.c_int, _i64, _p, _p, _i64, _p, _p]
    L.kvq_append_q4.restype = C.c_int
    L.kvq_append_q4.argtypes = [_p, _p, C.c_int, _p, C.c_int, C.c_int, C.c_int, _p, C.c_int,
                                C.c_int, _i64, _p, _p, _p, _p]
    L.kvq_project_append_q4.restype = C.c_int
    L.kvq_project_append_q4.argtypes = [_p, C.c_int, _p, C.c_int, C.c_int, _p, _p, C.c_int,
                                        C.c_int, C.c_int, _p, C.c_int, C.c_int, _i64, _p, _p,
                                        _p, _p]
    L.kvq_gather.restype = C.c_int
    L.kvq_gather.argtypes = [C.POINTER(GatherDesc), _p]
    L.kvq_mla_decode_workspace.restype = C.c_size_t
    L.kvq_mla_decode_workspace.argtypes = [C.POINTER(MlaProblem)]
    L.kvq_mla_decode_kernel.restype = C.c_int
    L.kvq_mla_decode_kernel.argtypes = [C.POINTER(MlaProblem)]
    L.kvq_mla_decode.restype = C.c_int
    L.kvq_mla_decode.argtypes = [C.POINTER(MlaProblem), _p, _p, _p, C.c_size_t, _p, _p]
    L.kvq_mla_decode_noalloc.restype = C.c_int
    L.kvq_mla_decode_noalloc.argtypes = [C.POINTER(MlaProblem), _p, _p, _p, _p]
    L.kvq_cache_probe.restype = C.c_int
    L.kvq_cache_probe.argtypes = [C.c_char_p, C.POINTER(CacheInfo)]
    L.kvq_cache_save.restype = C.c_int
    L.kvq_cache_save.argtypes = [C.c_char_p, C.c_int32, C.POINTER(MlaCache), _p, _i64, _p]
    L.kvq_cache_save_f32.restype = C.c_int
    L.kvq_cache_save_f32.argtypes = [C.c_char_p, _p, _p, _i64, _p]
    L.kvq_cache_append.restype = C.c_int
    L.kvq_cache_append.argtypes = [C.c_char_p, C.c_int32, C.POINTER(MlaCache), _i64, _i64, _p]
    L.kvq_cache_load_workspace.restype = C.c_size_t
    L.kvq_cache_load_workspace.argtypes = []
    L.kvq_cache_load.restype = C.c_int
    L.kvq_cache_load.argtypes = [C.c_char_p, C.c_int32, _p, C.POINTER(MlaCache), _i64,
                                 C.POINTER(_i64), _p, C.c_size_t, _p]
    L.kvq_q4_decode_workspace.restype = C.c_size_t
    L.kvq_q4_decode_workspace.argtypes = [C.POINTER(Q4Problem)]
    L.kvq_q4_decode.restype = C.c_int
    L.kvq_q4_decode.argtypes = [C.POINTER(Q4Problem), _p, _p, _p, C.c_size_t, _p, _p]


def _check(status: int):
    if status != 0:
        raise KvqError(status, lib().kvq_last_error().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream
    import torch
    return torch.cuda.current_stream().cuda_stream


# ---------------------------------------------------------------------------------------

def kvq_version() -> int:
    return lib().kvq_version()


def kvq_set_fault(spec: str | None) -> None:
    _check(lib().kvq_set_fault(None if spec is None else spec.encode()))


def kvq_tq4_codebook():
    import numpy as np
    cb = np.empty(16, np.float32)
    thr = np.empty(15, np.float32)
    _check(lib().kvq_tq4_codebook(cb.ctypes.data, thr.ctypes.data))
    return cb, thr


def kvq_tq_codebook(bits: int):
    import numpy as np
    L = 1 << bits
    cb = np.empty(L, np.float32)
    thr = np.empty(L - 1, np.float32)
    _check(lib().kvq_tq_codebook(bits, cb.ctypes.data, thr.ctypes.data))
    return cb, thr


def kvq_encode_fp8(x, codes, scales, stream=None) -> None:
    """x fp32 [rows][>=dim] -> codes u8 [rows][>=dim], scales fp32 [rows]; dim = codes
    columns used = x.shape[1] unless x is a strided view."""
    rows, dim = x.shape
    _check(lib().kvq_encode_fp8(_ptr(x), rows, dim, x.stride(0), _ptr(codes), codes.stride(0),
                                _ptr(scales), _stream(stream)))


def kvq_encode_tq4(x, sign_bits, packed, radius, stream=None) -> None:
    rows, dim = x.shape
    _check(lib().kvq_encode_tq4(_ptr(x), rows, dim, x.stride(0), _ptr(sign_bits), _ptr(packed),
                                packed.stride(0), _ptr(radius), _stream(stream)))


def kvq_encode_tq(x, sign_bits, bits, packed, radius, stream=None) -> None:
    """Rotated-tier encode at 3, 4 or 6 bits: packed u8 [rows][>= dim*bits/8]."""
    rows, dim = x.shape
    _check(lib().kvq_encode_tq(_ptr(x), rows, dim, x.stride(0), int(bits), _ptr(sign_bits),
                               _ptr(packed), packed.stride(0), _ptr(radius), _stream(stream)))


def kvq_encode_mla(c_lat, k_rope, fmt, sign_bits, lat, lat_scale, rope, rope_scale, stream=None) -> None:
    """Append-time encode of MLA rows: latent c_lat fp32 [rows][512] into the tier `fmt`
    (lat u8 [rows][>= 512 * bits / 8], lat_scale fp32 [rows]) and rope key k_rope fp32
    [rows][64] into fp8 (rope u8 [rows][>= 64], rope_scale fp32 [rows]), in one call."""
    rows = c_lat.shape[0]
    _check(lib().kvq_encode_mla(_ptr(c_lat), c_lat.stride(0), _ptr(k_rope), k_rope.stride(0), rows,
                                int(fmt), _ptr(sign_bits), _ptr(lat), lat.stride(0), _ptr(lat_scale),
                                _ptr(rope), rope.stride(0), _ptr(rope_scale), _stream(stream)))


def kvq_append_q4(k, v, pos0, page_table, page_size, n_cells, k_pool, v_pool,
                  dev_status=None, stream=None) -> None:
    n_seq, n_tok, n_heads, hd = k.shape
    _check(lib().kvq_append_q4(_ptr(k), _ptr(v), n_seq, _ptr(pos0), n_tok, n_heads, hd,
                               _ptr(page_table), page_table.shape[1], page_size, n_cells,
                               _ptr(k_pool), _ptr(v_pool), _ptr(dev_status), _stream(stream)))


def kvq_project_append_q4(h, w_k, w_v, pos0, page_table, page_size, n_cells, k_pool, v_pool,
                          dev_status=None, stream=None) -> None:
    """h fp32 [n_seq][n_tok][d_model]; w_k, w_v [d_model][n_heads * 256] float32 or
    bfloat16 tensors; the projected rows are appended as kvq_append_q4 appends k, v."""
    n_seq, n_tok, d_model = h.shape
    w_type = WEIGHT_BF16 if str(w_k.dtype).endswith("bfloat16") else WEIGHT_F32
    n_heads = w_k.shape[1] // 256
    if tuple(w_k.shape) != (d_model, n_heads * 256) or tuple(w_v.shape) != tuple(w_k.shape) \
            or w_v.dtype != w_k.dtype:
        raise ValueError("w_k, w_v must both be [d_model][n_heads * 256] of one dtype")
    _check(lib().kvq_project_append_q4(_ptr(h), n_seq, _ptr(pos0), n_tok, d_model, _ptr(w_k),
                                       _ptr(w_v), w_type, n_heads, 256, _ptr(page_table),
                                       page_table.shape[1], page_size, n_cells, _ptr(k_pool),
                                       _ptr(v_pool), _ptr(dev_status), _stream(stream)))


def kvq_gather_q4(pool, pos0, n_tok, page_table, page_size, n_cells, out, dev_status=None,
                  stream=None) -> None:
    """q4_0 mode of kvq_gather: out u16/fp16 [n_seq][n_tok][n_heads][256]."""
    d = GatherDesc()
    d.format = FMT_Q4_0
    d.q4_pool, d.n_seq, d.n_tok = _ptr(pool), pos0.shape[0], n_tok
    d.n_heads, d.head_dim = out.shape[2], out.shape[3]
    d.pos0, d.n_cells, d.q4_out = _ptr(pos0), n_cells, _ptr(out)
    d.page_table, d.max_pages, d.page_size = _ptr(page_table), page_table.shape[-1], page_size
    d.dev_status = _ptr(dev_status)
    _check(lib().kvq_gather(C.byref(d), _stream(stream)))


def kvq_gather_rows(fmt, src: dict, src_rows, idx, dst: dict, page_table=None, page_size=0,
                    dev_status=None, stream=None) -> None:
    """fp8 / TQ4 mode of kvq_gather: copy rows idx of `src` planes into `dst` planes."""
    d = GatherDesc()
    d.format = fmt
    d.mla_src = MlaCache(_ptr(src["lat"]), _ptr(src["lat_scale"]), _ptr(src["rope"]),
                         _ptr(src["rope_scale"]), src["lat"].shape[0])
    d.mla_src_rows = src_rows
    d.idx, d.n_idx = _ptr(idx), idx.numel()
    if page_table is not None:
        d.page_table, d.max_pages, d.page_size = _ptr(page_table), page_table.shape[-1], page_size
    d.dst_lat, d.dst_lat_scale = _ptr(dst["lat"]), _ptr(dst["lat_scale"])
    d.dst_rope, d.dst_rope_scale = _ptr(dst["rope"]), _ptr(dst["rope_scale"])
    d.dev_status = _ptr(dev_status)
    _check(lib().kvq_gather(C.byref(d), _stream(stream)))


def _cache(planes):
    if planes is None:
        return MlaCache()
    return MlaCache(_ptr(planes["lat"]), _ptr(planes["lat_scale"]), _ptr(planes["rope"]),
                    _ptr(planes["rope_scale"]), planes["lat"].shape[0])


def make_problem(*, seq_len, q_lat, q_rope, sm_scale, max_seq_len, fmt=FMT_FP8, seq_fmt=None,
                 causal=False, block_table=None, page_size=0, seq_stride_rows=0, fp8=None,
                 tq4=None, signs=None, idx=None, split_rows=0, impl=0,
                 overlap_prior=0) -> MlaProblem:
    """Fill a kvq_mla_problem from torch tensors.  The returned object holds a reference
    to every tensor whose device pointer it carries, so the memory stays allocated (and
    is not handed to a later allocation) for as long as the problem is alive."""
    n_seq, n_q, H, DL = q_lat.shape
    p = MlaProblem()
    p.n_seq, p.n_q, p.n_heads, p.d_lat, p.d_rope = n_seq, n_q, H, DL, q_rope.shape[-1]
    p.causal, p.max_seq_len = int(bool(causal)), int(max_seq_len)
    p.seq_len, p.seq_fmt, p.fmt = _ptr(seq_len), _ptr(seq_fmt), fmt
    if block_table is not None:
        p.block_table, p.max_pages, p.page_size = _ptr(block_table), block_table.shape[-1], page_size
    p.seq_stride_rows = seq_stride_rows
    p.fp8, p.tq4, p.tq4_signs = _cache(fp8), _cache(tq4), _ptr(signs)
    p.q_lat, p.q_rope = _ptr(q_lat), _ptr(q_rope)
    if idx is not None:
        p.idx, p.top_k = _ptr(idx), idx.shape[-1]
    p.sm_scale, p.split_rows, p.impl = float(sm_scale), int(split_rows), int(impl)
    p.overlap_prior = int(overlap_prior)
    p._keep = [seq_len, seq_fmt, block_table, fp8, tq4, signs, q_lat, q_rope, idx]
    return p


def kvq_mla_decode_workspace(p: MlaProblem) -> int:
    return lib().kvq_mla_decode_workspace(C.byref(p))


def kvq_mla_decode_kernel(p: MlaProblem) -> int:
    """The kernel kvq_mla_decode runs for p: IMPL_SIMT, IMPL_TC, IMPL_MMA, IMPL_TC16, IMPL_TCF8
    or IMPL_BY_FMT (a batch of per-sequence formats split by tier)."""
    r = lib().kvq_mla_decode_kernel(C.byref(p))
    if r < 0:
        _check(-r)
    return r


def kvq_mla_decode(p: MlaProblem, out, lse=None, workspace=None, dev_status=None,
                   stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kvq_mla_decode(C.byref(p), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                _ptr(dev_status), _stream(stream)))


def kvq_mla_decode_noalloc(p: MlaProblem, out, lse=None, dev_status=None, stream=None) -> None:
    """kvq_mla_decode with the library's fixed scratch array instead of a workspace, for
    callers that cannot allocate device memory (see include/kvq.h)."""
    _check(lib().kvq_mla_decode_noalloc(C.byref(p), _ptr(out), _ptr(lse), _ptr(dev_status),
                                        _stream(stream)))


def make_q4_problem(*, seq_len, page_table, page_size, k_pool, v_pool, q, sm_scale,
                    max_seq_len, gate=None, split_rows=0) -> Q4Problem:
    """Fill a kvq_q4_problem from torch tensors: pools [n_cells, n_kv, 144] uint8, q (and
    gate) [n_seq, n_qh, 256] fp32, page_table [n_seq, max_pages] int32.  The returned
    object keeps a reference to every tensor whose pointer it carries."""
    n_seq, n_qh, hd = q.shape
    p = Q4Problem()
    p.n_seq, p.n_qh, p.n_kv, p.head_dim = n_seq, n_qh, k_pool.shape[1], hd
    p.seq_len, p.max_seq_len = _ptr(seq_len), int(max_seq_len)
    p.page_table, p.max_pages, p.page_size = _ptr(page_table), page_table.shape[-1], int(page_size)
    p.n_cells = k_pool.shape[0]
    p.k_pool, p.v_pool, p.q, p.gate = _ptr(k_pool), _ptr(v_pool), _ptr(q), _ptr(gate)
    p.sm_scale, p.split_rows = float(sm_scale), int(split_rows)
    p._keep = [seq_len, page_table, k_pool, v_pool, q, gate]
    return p


def kvq_q4_decode_workspace(p: Q4Problem) -> int:
    return lib().kvq_q4_decode_workspace(C.byref(p))


def kvq_q4_decode(p: Q4Problem, out, lse=None, workspace=None, dev_status=None,
                  stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kvq_q4_decode(C.byref(p), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                               _ptr(dev_status), _stream(stream)))


# --- cache files ------------------------------------------------------------------------

def kvq_cache_probe(path) -> CacheInfo:
    info = CacheInfo()
    _check(lib().kvq_cache_probe(os.fsencode(path), C.byref(info)))
    return info


def kvq_cache_save(path, fmt, planes: dict, rows, signs=None, stream=None) -> None:
    """planes: dict of device tensors lat, lat_scale, rope, rope_scale (a quantized tier)."""
    c = _cache(planes)
    _check(lib().kvq_cache_save(os.fsencode(path), int(fmt), C.byref(c), _ptr(signs), int(rows),
                                _stream(stream)))


def kvq_cache_save_f32(path, lat, rope, stream=None) -> None:
    _check(lib().kvq_cache_save_f32(os.fsencode(path), _ptr(lat), _ptr(rope), lat.shape[0],
                                    _stream(stream)))


def kvq_cache_append(path, fmt, planes: dict, row0, rows, stream=None) -> None:
    c = _cache(planes)
    _check(lib().kvq_cache_append(os.fsencode(path), int(fmt), C.byref(c), int(row0), int(rows),
                                  _stream(stream)))


def kvq_cache_load_workspace() -> int:
    return lib().kvq_cache_load_workspace()


def kvq_cache_load(path, fmt, planes: dict, signs=None, workspace=None, stream=None) -> int:
    """Load `path` under `fmt` into the device planes (their row count is the capacity);
    returns the rows loaded."""
    c = _cache(planes)
    n = _i64(0)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kvq_cache_load(os.fsencode(path), int(fmt), _ptr(signs), C.byref(c), c.n_rows,
                                C.byref(n), _ptr(workspace), ws_bytes, _stream(stream)))
    return n.value
