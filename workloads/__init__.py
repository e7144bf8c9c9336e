"""Seeded synthetic inputs for the quantized MLA KV-cache path.

This module holds only random draws (numpy PCG64 through ``default_rng``) and plain
shape bookkeeping: none of the method's arithmetic.  It is the one module both the
CUDA path's tests/bench and the oracle consume, so that both sides see identical
bytes.  Every recipe restates one of the five workloads of the method's evaluation:

  fp8_tiny      T=1024 latent+rope rows, magnitudes log-uniform [1e-3, 40], a few
                all-zero rows; H=16 single query.
  tq4           T=32768 N(0,1) rows, a 512-bit rotation sign vector; H=64.
  q4_paged      16 sequences x 8192 tokens of K and V, 8 heads x 256, amplitudes
                {1e-3, 1, 40} per row, page size 64, permuted page table, pos0 = 56.
  sparse        T=131072 fp8 rows, H=128, 2048 unique indices per query.
  ragged        32 sequences, lengths U{1024..65536}, 4 queries each, H=64, half
                fp8 and half TQ4, magnitudes log-uniform [1e-2, 10], page size 64.

Sizes can be scaled down (the parity tests run the same recipes at sizes the oracle
finishes in seconds).  The rotation sign vector is a random input of the TQ4 codec:
it is drawn here and passed to both sides as data.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D_LAT = 512
D_ROPE = 64
SM_SCALE = np.float32(1.0 / math.sqrt(192.0))   # softmax scale tau of every workload


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def normal(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(shape, dtype=np.float32)


def log_uniform(g: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    return np.exp(g.uniform(math.log(lo), math.log(hi), n)).astype(np.float32)


def sign_bits(seed: int, n: int = D_LAT) -> np.ndarray:
    """n random bits (1 marks a -1 sign), packed LSB-first into uint32 words."""
    bits = rng(seed + 7919).integers(0, 2, n).astype(np.uint64)
    # bit i lives in word i // 32 at position i % 32
    words = np.zeros(n // 32, np.uint64)
    for i in range(n):
        words[i // 32] |= bits[i] << np.uint64(i % 32)
    return words.astype(np.uint32)


@dataclass
class MlaRows:
    """fp32 latent rows c [T][512] and rope keys k_rope [T][64]."""
    c: np.ndarray
    k_rope: np.ndarray


@dataclass
class Queries:
    q_lat: np.ndarray    # [n_seq][n_q][H][512]
    q_rope: np.ndarray   # [n_seq][n_q][H][64]


def fp8_tiny_rows(T: int = 1024, seed: int = 0) -> MlaRows:
    """Rows N(0,1) scaled per row by a magnitude log-uniform in [1e-3, 40] (one draw per
    row, applied to c and k_rope); rows 0, T/2-1 and T-1 all zero, row 300 zero in c
    only (when T > 300)."""
    g = rng(seed)
    mag = log_uniform(g, T, 1e-3, 40.0)
    c = normal(g, (T, D_LAT)) * mag[:, None]
    kr = normal(g, (T, D_ROPE)) * mag[:, None]
    for t in {0, T // 2 - 1, T - 1}:
        if 0 <= t < T:
            c[t] = 0.0
            kr[t] = 0.0
    if T > 300:
        c[300] = 0.0
    return MlaRows(c, kr)


def unit_rows(T: int, seed: int) -> MlaRows:
    """Rows N(0,1), no magnitude scaling."""
    g = rng(seed)
    return MlaRows(normal(g, (T, D_LAT)), normal(g, (T, D_ROPE)))


def magnitude_rows(T: int, seed: int, lo: float, hi: float) -> MlaRows:
    """Rows N(0,1) times a per-row magnitude log-uniform in [lo, hi]."""
    g = rng(seed)
    mag = log_uniform(g, T, lo, hi)
    return MlaRows(normal(g, (T, D_LAT)) * mag[:, None], normal(g, (T, D_ROPE)) * mag[:, None])


def queries(n_seq: int, n_q: int, H: int, seed: int) -> Queries:
    g = rng(seed + 104729)
    return Queries(normal(g, (n_seq, n_q, H, D_LAT)), normal(g, (n_seq, n_q, H, D_ROPE)))


def sparse_indices(T: int, k: int, n: int, seed: int) -> np.ndarray:
    """n lists of k unique row indices drawn uniformly without replacement from [0, T)."""
    g = rng(seed + 1299709)
    return np.stack([g.choice(T, size=k, replace=False) for _ in range(n)]).astype(np.int32)


def planted_codes(shape, frac: float, seed: int):
    """A mask of about `frac` of the entries of `shape` and, for each entry, one of the
    two e4m3 bytes S.1111.111 (0x7F, 0xFF) that no encoder writes, for planting into
    an encoded cache."""
    g = rng(seed + 15485863)
    mask = g.random(shape) < frac
    return mask, np.where(g.random(shape) < 0.5, 0x7F, 0xFF).astype(np.uint8)


@dataclass
class Q4Workload:
    k: np.ndarray            # [n_seq][n_tok][n_heads][256] fp32
    v: np.ndarray
    pos0: np.ndarray         # [n_seq] int32
    page_table: np.ndarray   # [n_seq][max_pages] int32
    page_size: int
    n_cells: int


def q4_paged(n_seq: int = 16, n_tok: int = 8192, n_heads: int = 8, page_size: int = 64,
             pos0: int | None = None, seed: int = 0, spare_pages: int = 0) -> Q4Workload:
    """K and V rows N(0,1) times an amplitude drawn uniformly from {1e-3, 1, 40} per
    (sequence, token, K/V, head) row; the page table is a permutation of all page ids."""
    if pos0 is None:
        pos0 = page_size - 8
    g = rng(seed)
    amp_choices = np.array([1e-3, 1.0, 40.0], np.float32)
    k = normal(g, (n_seq, n_tok, n_heads, 256))
    k *= amp_choices[g.integers(0, 3, (n_seq, n_tok, n_heads))][..., None]
    v = normal(g, (n_seq, n_tok, n_heads, 256))
    v *= amp_choices[g.integers(0, 3, (n_seq, n_tok, n_heads))][..., None]
    max_pages = (pos0 + n_tok + page_size - 1) // page_size
    n_pages = n_seq * max_pages + spare_pages
    perm = g.permutation(n_pages).astype(np.int32)
    table = perm[: n_seq * max_pages].reshape(n_seq, max_pages)
    return Q4Workload(k, v, np.full(n_seq, pos0, np.int32), table, page_size, n_pages * page_size)


def projection_inputs(n_seq: int, n_tok: int, d_model: int, n_heads: int, seed: int,
                      bf16: bool = False):
    """Hidden rows h [n_seq][n_tok][d_model] (N(0,1) times a per-token amplitude drawn
    from {1e-3, 1, 40}) and K/V projection weights [d_model][n_heads * 256], N(0, 1/d_model)
    so that projected rows are of the order of h.  With bf16 the weights are bfloat16 bit
    patterns (uint16): the upper halves of the fp32 draws."""
    g = rng(seed + 13)
    amp_choices = np.array([1e-3, 1.0, 40.0], np.float32)
    h = normal(g, (n_seq, n_tok, d_model))
    h *= amp_choices[g.integers(0, 3, (n_seq, n_tok))][..., None]
    sd = np.float32(1.0 / np.sqrt(d_model))
    w_k = normal(g, (d_model, n_heads * 256)) * sd
    w_v = normal(g, (d_model, n_heads * 256)) * sd
    if bf16:
        w_k = (w_k.view(np.uint32) >> 16).astype(np.uint16)
        w_v = (w_v.view(np.uint32) >> 16).astype(np.uint16)
    return h, w_k, w_v


def paged_table(n_seq: int, n_tok: int, page_size: int, pos0: int, seed: int):
    """(pos0 [n_seq], page table [n_seq][max_pages], n_cells) for appending n_tok tokens
    per sequence from position pos0: the table is a seeded permutation of all page ids."""
    g = rng(seed + 7)
    max_pages = (pos0 + n_tok + page_size - 1) // page_size
    perm = g.permutation(n_seq * max_pages).astype(np.int32)
    return np.full(n_seq, pos0, np.int32), perm.reshape(n_seq, max_pages), n_seq * max_pages * page_size


@dataclass
class RaggedWorkload:
    seq_len: np.ndarray       # [n_seq] int32
    seq_fmt: np.ndarray       # [n_seq] int32 (1 = fp8, 2 = TQ4)
    page_size: int
    block_table: np.ndarray   # [n_seq][max_pages] int32 page ids within the seq's tier pool
    pool_pages: dict          # fmt -> number of pages in that tier's pool
    rows: dict                # fmt -> MlaRows laid out by POOL row (page-permuted)
    queries: Queries
    signs: np.ndarray
    n_q: int
    H: int


def ragged_layout(n_seq: int = 32, len_lo: int = 1024, len_hi: int = 65536, page_size: int = 64,
                  seed: int = 0):
    """The shape of the ragged batch without its rows, for timing runs that generate the
    rows on the device: (L [n_seq], fmt [n_seq], block table, pages per tier)."""
    g = rng(seed + 11)
    L = g.integers(len_lo, len_hi + 1, n_seq).astype(np.int32)
    fmt = np.where(np.arange(n_seq) < n_seq // 2, 1, 2).astype(np.int32)
    pages = (L + page_size - 1) // page_size
    table = np.full((n_seq, int(pages.max())), -1, np.int32)
    pool_pages = {}
    for f in (1, 2):
        seqs = np.nonzero(fmt == f)[0]
        total = int(pages[seqs].sum())
        pool_pages[f] = total
        perm = g.permutation(total).astype(np.int32)
        o = 0
        for s in seqs:
            table[s, : pages[s]] = perm[o: o + pages[s]]
            o += pages[s]
    return L, fmt, table, pool_pages


def ragged(n_seq: int = 32, n_q: int = 4, H: int = 64, len_lo: int = 1024,
           len_hi: int = 65536, page_size: int = 64, seed: int = 0,
           mag: tuple = (1e-2, 10.0)) -> RaggedWorkload:
    """Sequence i holds L_i ~ U{len_lo..len_hi} rows; sequences [0, n/2) use the fp8
    tier and [n/2, n) the TQ4 tier; each tier has its own pool of pages, handed out to
    its sequences in a seeded random order.  Pool rows are generated directly (the
    values of a row do not depend on where its page sits)."""
    g = rng(seed)
    L = g.integers(len_lo, len_hi + 1, n_seq).astype(np.int32)
    fmt = np.where(np.arange(n_seq) < n_seq // 2, 1, 2).astype(np.int32)
    pages = (L + page_size - 1) // page_size
    max_pages = int(pages.max())
    table = np.full((n_seq, max_pages), -1, np.int32)
    pool_pages = {}
    rows = {}
    for f in (1, 2):
        seqs = np.nonzero(fmt == f)[0]
        total = int(pages[seqs].sum())
        pool_pages[f] = total
        perm = g.permutation(total).astype(np.int32)
        o = 0
        for s in seqs:
            table[s, : pages[s]] = perm[o: o + pages[s]]
            o += pages[s]
        n_rows = total * page_size
        m = log_uniform(g, n_rows, *mag)
        rows[f] = MlaRows(normal(g, (n_rows, D_LAT)) * m[:, None],
                          normal(g, (n_rows, D_ROPE)) * m[:, None])
    return RaggedWorkload(L, fmt, page_size, table, pool_pages, rows,
                          queries(n_seq, n_q, H, seed), sign_bits(seed), n_q, H)
