"""Test infrastructure: a plain-Python restatement of the cache file layout and its load
rules, for checking the library's kvq_cache_* calls byte for byte.  Only tests and the
benchmark's baseline use it.

Rules (colibri PR #399, Commit 1: ".coli_kv v2 ... quantize-on-upgrade from v1,
reject-on-mismatch, self-heal"; Commit 6: the magic encodes the tier, a header word
carries codec << 8 | bits; the review thread: a cache written under one mode must be
refused under another, and containers whose byte counts do not add up are refused).
The byte layout is the library's own (kvq.h): 16 little-endian u32 header words, the
rotation signs for rotated tiers, then row-interleaved records.
"""
import struct

import numpy as np

F32, FP8, TQ4, TQ6, TQ3 = 0, 1, 2, 4, 5
BITS = {TQ3: 3, TQ4: 4, TQ6: 6}
MAGIC = {F32: b"KVQ1", FP8: b"KVQ2", TQ3: b"KVQ3", TQ4: b"KVQ3", TQ6: b"KVQ3"}
D_LAT, D_ROPE = 512, 64


class Mismatch(Exception):
    """The file holds another mode: refused, never misread."""


class BadFile(Exception):
    """Not a cache file of this layout, or its byte counts do not add up."""


def lat_bytes(fmt):
    return D_LAT * 4 if fmt == F32 else D_LAT if fmt == FP8 else D_LAT * BITS[fmt] // 8


def record_bytes(fmt):
    return (D_LAT + D_ROPE) * 4 if fmt == F32 else lat_bytes(fmt) + 4 + D_ROPE + 4


def codec_bits(fmt):
    return 32 if fmt == F32 else 8 if fmt == FP8 else (1 << 8) | BITS[fmt]


def header(fmt, n_rows):
    words = [struct.unpack("<I", MAGIC[fmt])[0], 1, D_LAT, D_ROPE, n_rows & 0xFFFFFFFF,
             n_rows >> 32, fmt, codec_bits(fmt), record_bytes(fmt)] + [0] * 7
    return struct.pack("<16I", *words)


def records(fmt, planes, rows=None):
    """Row-interleaved records of the planes (numpy): lat | lat_scale | rope | rope_scale."""
    lat = np.ascontiguousarray(planes["lat"]).view(np.uint8).reshape(len(planes["lat"]), -1)
    n = lat.shape[0] if rows is None else rows
    parts = [lat[:n],
             np.ascontiguousarray(planes["lat_scale"][:n], np.float32).view(np.uint8).reshape(n, 4),
             np.ascontiguousarray(planes["rope"][:n]).view(np.uint8).reshape(n, -1),
             np.ascontiguousarray(planes["rope_scale"][:n], np.float32).view(np.uint8).reshape(n, 4)]
    return np.concatenate(parts, axis=1).tobytes()


def file_bytes(fmt, planes, signs=None, rows=None):
    n = len(planes["lat"]) if rows is None else rows
    body = header(fmt, n)
    if fmt in BITS:
        body += np.ascontiguousarray(signs, np.uint32).astype("<u4").tobytes()
    return body + records(fmt, planes, n)


def f32_file_bytes(lat, rope):
    lat = np.ascontiguousarray(lat, np.float32)
    rope = np.ascontiguousarray(rope, np.float32)
    rec = np.concatenate([lat.view(np.uint8), rope.view(np.uint8)], axis=1).tobytes()
    return header(F32, lat.shape[0]) + rec


def read(path):
    """-> dict(format, codec, bits, n_rows, trailing, signs, planes) or raises BadFile."""
    data = open(path, "rb").read()
    if len(data) < 64:
        raise BadFile("shorter than a header")
    w = struct.unpack("<16I", data[:64])
    fmt = w[6]
    if fmt not in MAGIC or data[:4] != MAGIC[fmt] or w[1] != 1 or w[2] != D_LAT or w[3] != D_ROPE \
            or w[7] != codec_bits(fmt) or w[8] != record_bytes(fmt) or any(w[9:]):
        raise BadFile("not a cache file of this layout")
    off = 64
    signs = None
    if fmt in BITS:
        if len(data) < off + 64:
            raise BadFile("rotation signs missing")
        signs = np.frombuffer(data[off:off + 64], "<u4").astype(np.uint32)
        off += 64
    n = w[4] | (w[5] << 32)
    rb = record_bytes(fmt)
    if len(data) < off + n * rb:
        raise BadFile("fewer bytes than the header counts")
    rec = np.frombuffer(data[off:off + n * rb], np.uint8).reshape(n, rb)
    if fmt == F32:
        planes = dict(lat=rec[:, :D_LAT * 4].copy().view("<f4").reshape(n, D_LAT),
                      rope=rec[:, D_LAT * 4:].copy().view("<f4").reshape(n, D_ROPE))
    else:
        lb = lat_bytes(fmt)
        planes = dict(lat=rec[:, :lb].copy(),
                      lat_scale=rec[:, lb:lb + 4].copy().view("<f4").reshape(n),
                      rope=rec[:, lb + 4:lb + 4 + D_ROPE].copy(),
                      rope_scale=rec[:, lb + 4 + D_ROPE:].copy().view("<f4").reshape(n))
    return dict(format=fmt, codec=w[7] >> 8, bits=w[7] & 0xFF, n_rows=n,
                trailing=len(data) - off - n * rb, signs=signs, planes=planes)


def load_as(path, fmt, signs=None):
    """The planes a load under `fmt` must produce: the file's own records when it holds
    `fmt` (rotated: with the same signs), the oracle encoders' output for an fp32 file,
    Mismatch for anything else."""
    import oracle
    f = read(path)
    if f["format"] == F32:
        p = f["planes"]
        if fmt == FP8:
            lat, ls = oracle.encode_fp8(p["lat"])
        else:
            lat, ls = oracle.encode_tq(p["lat"], signs, BITS[fmt])
        rope, rs = oracle.encode_fp8(p["rope"])
        return dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs)
    if f["format"] != fmt:
        raise Mismatch(f"file holds format {f['format']}, not {fmt}")
    if fmt in BITS and not np.array_equal(f["signs"], np.asarray(signs, np.uint32)):
        raise Mismatch("rotated with other signs")
    return f["planes"]


def append_bytes(path, fmt, planes, row0, rows):
    """The file an append of rows [row0, row0 + rows) must leave: the bytes after the
    header's complete records are cut, the new records follow, the count is updated."""
    f = read(path)
    if f["format"] != fmt:
        raise Mismatch(f"file holds format {f['format']}, not {fmt}")
    data = open(path, "rb").read()
    keep = len(data) - f["trailing"]
    part = {k: v[row0:row0 + rows] for k, v in planes.items()}
    out = bytearray(data[:keep]) + records(fmt, part, rows)
    out[:64] = header(fmt, f["n_rows"] + rows)
    return bytes(out)

