"""GPU parity of the split-T absorbed-MLA decode against the fp64 oracle: every output
row (query, head) within 1e-4 * max|out| of that row, lse within 1e-4 absolute.
The caches are encoded by the oracle and uploaded, so this file tests the decode
alone (the encoders are pinned byte-exact in test_parity_codecs.py)."""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
TOL = 1e-4
IMPLS = pytest.mark.parametrize("impl", [1, 2, 3, 4, 5],
                                ids=["cudacore", "tcgen05", "mma", "tcgen05x16", "tcgen05f8"])


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_fp8_gb300 as k
    return k


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def encode(orc, rows, fmt, signs=None):
    if fmt == 1:
        lat, ls = orc.encode_fp8(rows.c)
    else:
        lat, ls = orc.encode_tq4(rows.c, signs)
    rope, rs = orc.encode_fp8(rows.k_rope)
    return dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs)


def run_gpu(kvq, *, cache_fmt, caches, seq_len, q, sm_scale=W.SM_SCALE, signs=None,
            seq_fmt=None, idx=None, causal=False, block_table=None, page_size=0,
            seq_stride_rows=0, split_rows=0, max_seq_len=None, impl=0, kernel=None):
    if impl == 5 and (cache_fmt != 1 or seq_fmt is not None):
        pytest.skip("impl 5 reads problems of fp8 rows only")
    dcaches = {f: {k: dev(v) for k, v in c.items()} for f, c in caches.items()}
    n_seq, n_q, H, _ = q.q_lat.shape
    p = kvq.make_problem(
        seq_len=dev(np.asarray(seq_len, np.int32)), q_lat=dev(q.q_lat), q_rope=dev(q.q_rope),
        sm_scale=sm_scale, max_seq_len=max(seq_len) if max_seq_len is None else max_seq_len,
        fmt=cache_fmt, seq_fmt=None if seq_fmt is None else dev(np.asarray(seq_fmt, np.int32)),
        causal=causal, block_table=None if block_table is None else dev(block_table),
        page_size=page_size, seq_stride_rows=seq_stride_rows, fp8=dcaches.get(1),
        tq4=dcaches.get(2), signs=None if signs is None else dev(signs),
        idx=None if idx is None else dev(idx), split_rows=split_rows, impl=impl)
    keep = (dcaches, p)
    if kernel is not None:
        assert kvq.kvq_mla_decode_kernel(p) == kernel
    ws = torch.empty(max(1, kvq.kvq_mla_decode_workspace(p)), dtype=torch.uint8, device="cuda")
    out = torch.full((n_seq, n_q, H, 512), np.nan, dtype=torch.float32, device="cuda")
    lse = torch.full((n_seq, n_q, H), np.nan, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_mla_decode(p, out, lse, ws, st)
    torch.cuda.synchronize()
    del keep
    return out.cpu().numpy(), lse.cpu().numpy(), int(st.item())


def check(out, lse, ref, ref_lse, sel=None):
    if sel is not None:
        out, lse, ref, ref_lse = out[sel], lse[sel], ref[sel], ref_lse[sel]
    assert not np.isnan(out).any()
    err = np.abs(out - ref).max(axis=-1)
    bar = TOL * np.abs(ref).max(axis=-1)
    empty = np.isneginf(ref_lse)
    assert np.all(out[empty] == 0) and np.all(np.isneginf(lse[empty]))
    ok = empty | (err <= bar)
    assert ok.all(), f"worst err/max|out| = {np.max(err[~empty] / np.abs(ref[~empty]).max(-1)):.3e}"
    # lse is a log of a sum of exponentials of scores as large as ~|lse|; fp32 score
    # accumulation leaves a relative error of a few 1e-7 of that magnitude
    assert np.allclose(lse[~empty], ref_lse[~empty], rtol=2e-6, atol=1e-4)
    scale = np.maximum(np.abs(ref[~empty]).max(-1), np.finfo(np.float64).tiny)
    return float(np.max(err[~empty] / scale)) if (~empty).any() else 0.0


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("T,split", [(1, 0), (17, 0), (63, 32), (65, 32), (1024, 0), (1000, 96)])
@IMPLS
def test_decode_tiny_shapes(kvq, orc, impl, fmt, T, split):
    rows = W.fp8_tiny_rows(T, seed=T) if fmt == 1 else W.unit_rows(T, seed=T)
    signs = W.sign_bits(T)
    cache = encode(orc, rows, fmt, signs)
    q = W.queries(1, 1, 16, seed=T)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=fmt, caches={fmt: cache}, seq_len=[T], q=q,
                           signs=signs, split_rows=split)
    kw = dict(fp8=cache) if fmt == 1 else dict(tq4=cache, signs=signs)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[fmt], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, **kw)
    assert st == 0
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_fp8_tiny_workload(kvq, orc, impl):
    """T=1024 fp8 rows with magnitudes log-uniform in [1e-3, 40] and zero rows, H=16."""
    rows = W.fp8_tiny_rows(1024, seed=0)
    cache = encode(orc, rows, 1)
    q = W.queries(1, 1, 16, seed=0)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=[1024], q=q)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[1024], seq_fmt=[1], q_lat=q.q_lat,
                                     q_rope=q.q_rope, sm_scale=W.SM_SCALE, fp8=cache)
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_fp8_unwritten_pattern_reads_zero(kvq, orc, impl):
    """The e4m3 pattern S.1111.111, which the encoder never writes, reads back as 0 in
    the latent and the rope parts alike (planted into about 5% of the codes)."""
    T = 700
    rows = W.unit_rows(T, seed=5)
    cache = encode(orc, rows, 1)
    for i, key in enumerate(("lat", "rope")):
        mask, val = W.planted_codes(cache[key].shape, 0.05, seed=5 + i)
        cache[key] = np.where(mask, val, cache[key])
    q = W.queries(1, 1, 16, seed=5)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=[T], q=q)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[1], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, fp8=cache)
    assert st == 0
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_tq4_workload(kvq, orc, impl):
    """T=32768 N(0,1) rows of the 4-bit tier, H=64 (every head)."""
    T = 32768
    rows = W.unit_rows(T, seed=0)
    signs = W.sign_bits(0)
    cache = encode(orc, rows, 2, signs)
    q = W.queries(1, 1, 64, seed=0)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=2, caches={2: cache}, seq_len=[T], q=q, signs=signs)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[2], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, tq4=cache, signs=signs)
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_sparse_workload(kvq, orc, impl):
    """T=131072 fp8 rows, H=128, 2048 unique indices per query; plus the dense variant
    on a sample of heads."""
    T = 131072
    rows = W.unit_rows(T, seed=0)
    cache = encode(orc, rows, 1)
    q = W.queries(1, 1, 128, seed=0)
    idx = W.sparse_indices(T, 2048, 1, seed=0)[None]
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=[T], q=q, idx=idx)
    ref, ref_lse, bad = orc.mla_decode(seq_len=[T], seq_fmt=[1], q_lat=q.q_lat, q_rope=q.q_rope,
                                       sm_scale=W.SM_SCALE, fp8=cache, idx=idx)
    assert st == 0 and not bad
    check(out, lse, ref, ref_lse)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=[T], q=q)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[1], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, fp8=cache, heads=(0, 8))
    check(out, lse, ref, ref_lse, sel=(slice(None), slice(None), slice(0, 8)))


@IMPLS
def test_decode_ragged_mixed_small(kvq, orc, impl):
    """Ragged, paged, mixed tiers, 4 causal queries per sequence; lengths include 0,
    1 and a sequence shorter than n_q."""
    wl = W.ragged(n_seq=6, n_q=4, H=8, len_lo=1, len_hi=700, page_size=64, seed=3)
    wl.seq_len[0] = 0
    wl.seq_len[1] = 1
    wl.seq_len[4] = 3
    caches = {f: encode(orc, wl.rows[f], f, wl.signs) for f in (1, 2)}
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches=caches, seq_len=wl.seq_len, q=wl.queries,
                           signs=wl.signs, seq_fmt=wl.seq_fmt, causal=True,
                           block_table=wl.block_table, page_size=wl.page_size, split_rows=64)
    ref, ref_lse, _ = orc.mla_decode(seq_len=wl.seq_len, seq_fmt=wl.seq_fmt, q_lat=wl.queries.q_lat,
                                     q_rope=wl.queries.q_rope, sm_scale=W.SM_SCALE, causal=True,
                                     block_table=wl.block_table, page_size=wl.page_size,
                                     fp8=caches[1], tq4=caches[2], signs=wl.signs)
    assert st == 0
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_fp8_paged_causal_batch(kvq, orc, impl):
    """fp8 rows only, paged (page size 64, seeded permuted table), 4 causal queries per
    sequence, 20 heads (a full and a partial group of 16); lengths 0, 1, 3, 650, 1300."""
    L = np.array([0, 1, 3, 650, 1300], np.int32)
    ps, n_q, H = 64, 4, 20
    pages = (L + ps - 1) // ps
    total = int(pages.sum())
    perm = np.random.default_rng(41).permutation(total).astype(np.int32)
    table = np.full((len(L), int(pages.max())), -1, np.int32)
    o = 0
    for i, n in enumerate(pages):
        table[i, :n] = perm[o:o + n]
        o += n
    rows = W.magnitude_rows(total * ps, seed=41, lo=1e-2, hi=10.0)
    cache = encode(orc, rows, 1)
    q = W.queries(len(L), n_q, H, seed=41)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=L, q=q, causal=True,
                           block_table=table, page_size=ps)
    ref, ref_lse, _ = orc.mla_decode(seq_len=L, seq_fmt=np.ones(len(L), np.int32), q_lat=q.q_lat,
                                     q_rope=q.q_rope, sm_scale=W.SM_SCALE, causal=True, block_table=table,
                                     page_size=ps, fp8=cache)
    assert st == 0
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_fp8_strided_sequences(kvq, orc, impl):
    """fp8 rows only, three sequences in one pool at a stride of 2048 rows (contiguous:
    the TMA path), lengths 2048, 1500 and 777, 2 causal queries, 16 heads."""
    L = np.array([2048, 1500, 777], np.int32)
    stride, n_q, H = 2048, 2, 16
    rows = W.magnitude_rows(stride * len(L), seed=43, lo=1e-3, hi=40.0)
    cache = encode(orc, rows, 1)
    q = W.queries(len(L), n_q, H, seed=43)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=L, q=q, causal=True,
                           seq_stride_rows=stride)
    ref, ref_lse, _ = orc.mla_decode(seq_len=L, seq_fmt=np.ones(len(L), np.int32), q_lat=q.q_lat,
                                     q_rope=q.q_rope, sm_scale=W.SM_SCALE, causal=True, seq_stride_rows=stride,
                                     fp8=cache)
    assert st == 0
    check(out, lse, ref, ref_lse)


@pytest.mark.slow
@IMPLS
def test_decode_ragged_workload(kvq, orc, impl):
    """The full ragged batch (32 sequences, lengths U{1024..65536}, 4 causal queries,
    H=64, 16 fp8 + 16 TQ4 sequences, page size 64); the oracle checks 8 heads of 4
    sequences (two of each tier)."""
    wl = W.ragged(seed=0)
    caches = {f: encode(orc, wl.rows[f], f, wl.signs) for f in (1, 2)}
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches=caches, seq_len=wl.seq_len, q=wl.queries,
                           signs=wl.signs, seq_fmt=wl.seq_fmt, causal=True,
                           block_table=wl.block_table, page_size=wl.page_size)
    sel = np.array([0, 7, 16, 31], np.int32)
    ref, ref_lse, _ = orc.mla_decode(seq_len=wl.seq_len, seq_fmt=wl.seq_fmt, q_lat=wl.queries.q_lat,
                                     q_rope=wl.queries.q_rope, sm_scale=W.SM_SCALE, causal=True,
                                     block_table=wl.block_table, page_size=wl.page_size,
                                     fp8=caches[1], tq4=caches[2], signs=wl.signs, seq_sel=sel,
                                     heads=(0, 8))
    assert st == 0
    check(out[sel][:, :, :8], lse[sel][:, :, :8], ref[sel][:, :, :8], ref_lse[sel][:, :, :8])


@pytest.mark.parametrize("fmt", [1, 2])
@IMPLS
def test_decode_partial_head_block_multi_tile(kvq, orc, impl, fmt):
    """H=20 (one full block of 16 heads and one of 4), 2 causal queries, splits of 640
    rows (5 tiles of 128, so the staging ring wraps) over T=2900 (a ragged last tile)."""
    T = 2900
    rows = W.magnitude_rows(T, seed=40 + fmt, lo=1e-2, hi=10.0)
    signs = W.sign_bits(40)
    cache = encode(orc, rows, fmt, signs)
    q = W.queries(1, 2, 20, seed=40)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=fmt, caches={fmt: cache}, seq_len=[T], q=q,
                           signs=signs, causal=True, split_rows=640)
    kw = dict(fp8=cache) if fmt == 1 else dict(tq4=cache, signs=signs)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[fmt], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, causal=True, **kw)
    assert st == 0
    check(out, lse, ref, ref_lse)


@pytest.mark.parametrize("fmt", [1, 2])
@IMPLS
def test_decode_sixteen_heads_long(kvq, orc, impl, fmt):
    """T=131072 rows, H=16, one query: the HBM-bound decode points, library splits."""
    T = 131072
    rows = W.unit_rows(T, seed=50)
    signs = W.sign_bits(50)
    cache = encode(orc, rows, fmt, signs)
    q = W.queries(1, 1, 16, seed=50)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=fmt, caches={fmt: cache}, seq_len=[T], q=q,
                           signs=signs)
    kw = dict(fp8=cache) if fmt == 1 else dict(tq4=cache, signs=signs)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[fmt], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, **kw)
    assert st == 0
    check(out, lse, ref, ref_lse)


@pytest.mark.parametrize("fmt", [1, 2])
@IMPLS
def test_decode_rows_past_the_pool(kvq, orc, impl, fmt):
    """A contiguous cache whose pool ends inside the sequence (300 rows, seq_len 500): the
    rows past the pool are skipped and flagged as bad pages, so the result is the
    attention over the 300 rows that exist."""
    T, L = 300, 500
    rows = W.unit_rows(T, seed=45 + fmt)
    signs = W.sign_bits(45)
    cache = encode(orc, rows, fmt, signs)
    q = W.queries(1, 1, 16, seed=45)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=fmt, caches={fmt: cache}, seq_len=[L], q=q,
                           signs=signs)
    kw = dict(fp8=cache) if fmt == 1 else dict(tq4=cache, signs=signs)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[fmt], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, **kw)
    assert st & kvq.DEV_BAD_PAGE
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_mixed_tiers_many_splits(kvq, orc, impl):
    """A seq_fmt batch of an fp8 and a TQ4 sequence (T=3000 each) in splits of 32 rows:
    94 splits, so the combine runs in its four-quarter grid, the fp8 rows summed by
    four 128-dim CTAs and the TQ4 rows (unrotated over all 512 dims) by one."""
    T = 3000
    rows = W.magnitude_rows(2 * T, seed=48, lo=1e-2, hi=10.0)    # sequence i: pool rows i*T ..
    signs = W.sign_bits(48)
    caches = {1: encode(orc, rows, 1), 2: encode(orc, rows, 2, signs)}
    q = W.queries(2, 1, 8, seed=48)
    kw = dict(seq_len=[T, T], q=q, signs=signs, seq_fmt=[1, 2], seq_stride_rows=T, split_rows=32)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches=caches, **kw)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T, T], seq_fmt=[1, 2], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, seq_stride_rows=T, fp8=caches[1],
                                     tq4=caches[2], signs=signs)
    assert st == 0
    check(out, lse, ref, ref_lse)


@pytest.mark.gpu
def test_decode_mixed_batch_split_by_tier(kvq, orc):
    """The library's choice for a seq_fmt batch with enough work: its fp8 sequences on the
    e4m3 kernel and its TQ4 sequences on the 32-head kernel, into one set of partials.
    A paged causal ragged batch (lengths 0, 1, 3 and U{500..3000}, 4 queries, 16 heads)
    and an fp8 + TQ4 pair in splits of 32 rows (157 splits)."""
    wl = W.ragged(n_seq=8, n_q=4, H=16, len_lo=500, len_hi=3000, page_size=64, seed=5)
    wl.seq_len[0] = 0
    wl.seq_len[1] = 1
    wl.seq_len[5] = 3
    caches = {f: encode(orc, wl.rows[f], f, wl.signs) for f in (1, 2)}
    kw = dict(cache_fmt=1, caches=caches, seq_len=wl.seq_len, q=wl.queries, signs=wl.signs,
              seq_fmt=wl.seq_fmt, causal=True, block_table=wl.block_table, page_size=wl.page_size)
    out, lse, st = run_gpu(kvq, impl=0, kernel=kvq.IMPL_BY_FMT, **kw)
    ref, ref_lse, _ = orc.mla_decode(seq_len=wl.seq_len, seq_fmt=wl.seq_fmt, q_lat=wl.queries.q_lat,
                                     q_rope=wl.queries.q_rope, sm_scale=W.SM_SCALE, causal=True,
                                     block_table=wl.block_table, page_size=wl.page_size,
                                     fp8=caches[1], tq4=caches[2], signs=wl.signs)
    assert st == 0
    check(out, lse, ref, ref_lse)

    T = 5000
    rows = W.magnitude_rows(2 * T, seed=49, lo=1e-2, hi=10.0)
    signs = W.sign_bits(49)
    caches = {1: encode(orc, rows, 1), 2: encode(orc, rows, 2, signs)}
    q = W.queries(2, 1, 16, seed=49)
    kw = dict(seq_len=[T, T], q=q, signs=signs, seq_fmt=[2, 1], seq_stride_rows=T, split_rows=32)
    out, lse, st = run_gpu(kvq, impl=0, kernel=kvq.IMPL_BY_FMT, cache_fmt=1, caches=caches, **kw)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T, T], seq_fmt=[2, 1], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, seq_stride_rows=T, fp8=caches[1],
                                     tq4=caches[2], signs=signs)
    assert st == 0
    check(out, lse, ref, ref_lse)


@pytest.mark.gpu
@pytest.mark.slow
def test_decode_ragged_workload_split_by_tier(kvq, orc):
    """The full ragged batch under the library's choice (fp8 sequences on the e4m3
    kernel, TQ4 ones on the 32-head kernel); the oracle checks 8 heads of 4 sequences."""
    wl = W.ragged(seed=0)
    caches = {f: encode(orc, wl.rows[f], f, wl.signs) for f in (1, 2)}
    out, lse, st = run_gpu(kvq, impl=0, kernel=kvq.IMPL_BY_FMT, cache_fmt=1, caches=caches,
                           seq_len=wl.seq_len, q=wl.queries, signs=wl.signs, seq_fmt=wl.seq_fmt,
                           causal=True, block_table=wl.block_table, page_size=wl.page_size)
    sel = np.array([0, 7, 16, 31], np.int32)
    ref, ref_lse, _ = orc.mla_decode(seq_len=wl.seq_len, seq_fmt=wl.seq_fmt, q_lat=wl.queries.q_lat,
                                     q_rope=wl.queries.q_rope, sm_scale=W.SM_SCALE, causal=True,
                                     block_table=wl.block_table, page_size=wl.page_size,
                                     fp8=caches[1], tq4=caches[2], signs=wl.signs, seq_sel=sel,
                                     heads=(0, 8))
    assert st == 0
    check(out[sel][:, :, :8], lse[sel][:, :, :8], ref[sel][:, :, :8], ref_lse[sel][:, :, :8])


@pytest.mark.parametrize("fmt", [1, 2])
@IMPLS
def test_decode_sum_abs_terms_error(kvq, orc, impl, fmt):
    """The error of every output element relative to the sum of the absolute values of
    its terms, sum_t p_t |c_t,d| (the dot-product tolerance form), on the fp8 tiny
    workload (magnitudes 1e-3..40, zero rows) and on T=4096 N(0,1) rows of the 4-bit
    tier, H=16.  Measured on GB300: 1.7e-5 to 3.5e-5 (fp8; the fp32 CUDA-core kernel
    included, so it is the fp32 rounding of logits of magnitude ~10^2, which moves each
    p_t by ~|s|·2^-23) and 5e-7 to 1.2e-6 (TQ4); the bound is 1e-4."""
    T = 1024 if fmt == 1 else 4096
    rows = W.fp8_tiny_rows(T, seed=0) if fmt == 1 else W.unit_rows(T, seed=0)
    signs = W.sign_bits(0)
    cache = encode(orc, rows, fmt, signs)
    q = W.queries(1, 1, 16, seed=0)
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=fmt, caches={fmt: cache}, seq_len=[T], q=q,
                           signs=signs)
    kw = dict(fp8=cache) if fmt == 1 else dict(tq4=cache, signs=signs)
    ref, _, _ = orc.mla_decode(seq_len=[T], seq_fmt=[fmt], q_lat=q.q_lat, q_rope=q.q_rope,
                               sm_scale=W.SM_SCALE, **kw)
    if fmt == 1:
        c = orc.decode_fp8(cache["lat"], cache["lat_scale"])
    else:
        c, _ = orc.decode_tq4(cache["lat"], cache["lat_scale"], signs, 512)
    kr = orc.decode_fp8(cache["rope"], cache["rope_scale"])
    A = orc.mla_abs_terms(lat_rows=c, rope_rows=kr, q_lat=q.q_lat[0], q_rope=q.q_rope[0],
                          sm_scale=W.SM_SCALE)
    err = np.abs(out[0] - ref[0])
    nz = A > 0
    assert st == 0 and np.all(err[~nz] == 0)
    worst = float((err[nz] / A[nz]).max())
    print(f"sum|terms|-relative error, fmt {fmt}, impl {impl}: {worst:.3e}")
    assert worst <= 1e-4


@IMPLS
def test_decode_bad_index_and_sparse_causal(kvq, orc, impl):
    T, NQ = 500, 3
    rows = W.unit_rows(T, seed=9)
    cache = encode(orc, rows, 1)
    q = W.queries(1, NQ, 4, seed=9)
    idx = W.sparse_indices(T, 100, NQ, seed=9)[None]
    idx[0, 1, 5] = T + 10
    idx[0, 2, 0] = -3
    out, lse, st = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=[T], q=q, idx=idx,
                           causal=True, split_rows=32)
    ref, ref_lse, bad = orc.mla_decode(seq_len=[T], seq_fmt=[1], q_lat=q.q_lat, q_rope=q.q_rope,
                                       sm_scale=W.SM_SCALE, fp8=cache, idx=idx, causal=True)
    assert bad and st & kvq.DEV_BAD_INDEX
    check(out, lse, ref, ref_lse)


@IMPLS
def test_decode_split_invariance(kvq, orc, impl):
    """Different split sizes give results within the same bar of the oracle."""
    T = 5000
    rows = W.magnitude_rows(T, seed=10, lo=1e-2, hi=10)
    cache = encode(orc, rows, 1)
    q = W.queries(1, 2, 8, seed=10)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[1], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, fp8=cache)
    for split in (32, 64, 4992, 5000, 8192):
        out, lse, _ = run_gpu(kvq, impl=impl, cache_fmt=1, caches={1: cache}, seq_len=[T], q=q,
                              split_rows=split)
        check(out, lse, ref, ref_lse)


def test_decode_host_errors(kvq):
    rows = torch.zeros(10, 512, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(10, device="cuda")
    cache = dict(lat=rows, lat_scale=sc, rope=rows[:, :64].contiguous(), rope_scale=sc)
    ql = torch.zeros(1, 1, 4, 512, device="cuda")
    qr = torch.zeros(1, 1, 4, 64, device="cuda")
    p = kvq.make_problem(seq_len=torch.tensor([10], dtype=torch.int32, device="cuda"), q_lat=ql,
                         q_rope=qr, sm_scale=0.1, max_seq_len=10, fmt=kvq.FMT_FP8, fp8=cache)
    out = torch.zeros(1, 1, 4, 512, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_mla_decode(p, out, None, None)
    assert e.value.status == 5                       # workspace missing
    ws = torch.empty(kvq.kvq_mla_decode_workspace(p), dtype=torch.uint8, device="cuda")
    kvq.kvq_set_fault("kvq_mla_decode:6")
    try:
        out.fill_(7.0)
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_mla_decode(p, out, None, ws)
        assert e.value.status == 6
        torch.cuda.synchronize()
        assert torch.all(out == 7.0)                 # nothing launched, nothing written
    finally:
        kvq.kvq_set_fault(None)
    kvq.kvq_mla_decode(p, out, None, ws)
    torch.cuda.synchronize()
    assert torch.all(out == 0.0)                     # equal (zero) scores: the mean of zeros


@pytest.mark.gpu
@pytest.mark.parametrize("rewrite_q", [False, True])
def test_decode_overlap_prior_back_to_back(kvq, orc, rewrite_q):
    """overlap_prior = 1 on the e4m3 kernel: three fp8 problems (distinct caches, one
    workspace) decoded back to back, five times over, inside a CUDA graph, so that each
    decode may start during the combine before it.  Every output equals the oracle.  With
    rewrite_q a device copy writes each call's queries just before the call (a kernel that
    does not let dependents launch early, so the decode still reads them after it)."""
    T, H = 16384, 16
    probs, refs, keep = [], [], []
    for i in range(3):
        rows = W.unit_rows(T, seed=70 + i)
        cache = encode(orc, rows, 1)
        q = W.queries(1, 1, H, seed=70 + i)
        dc = {k: dev(v) for k, v in cache.items()}
        ql, qr = dev(q.q_lat), dev(q.q_rope)
        ql_dst, qr_dst = (torch.empty_like(ql), torch.empty_like(qr)) if rewrite_q else (ql, qr)
        p = kvq.make_problem(seq_len=dev(np.array([T], np.int32)), q_lat=ql_dst, q_rope=qr_dst,
                             sm_scale=W.SM_SCALE, max_seq_len=T, fmt=1, fp8=dc, impl=5,
                             overlap_prior=1)
        assert kvq.kvq_mla_decode_kernel(p) == kvq.IMPL_TCF8
        ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[1], q_lat=q.q_lat, q_rope=q.q_rope,
                                         sm_scale=W.SM_SCALE, fp8=cache)
        probs.append(p)
        refs.append((ref, ref_lse))
        keep.append((dc, ql, qr, ql_dst, qr_dst))
    ws = torch.empty(max(kvq.kvq_mla_decode_workspace(p) for p in probs), dtype=torch.uint8, device="cuda")
    outs = [torch.full((1, 1, H, 512), np.nan, device="cuda") for _ in probs]
    lses = [torch.full((1, 1, H), np.nan, device="cuda") for _ in probs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def calls():
        for (p, o, l, k) in zip(probs, outs, lses, keep):
            if rewrite_q:
                k[3].copy_(k[1])
                k[4].copy_(k[2])
            kvq.kvq_mla_decode(p, o, l, ws, st)

    calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(5):
            calls()
    for o, l in zip(outs, lses):
        o.fill_(np.nan)
        l.fill_(np.nan)
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for o, l, (ref, ref_lse) in zip(outs, lses, refs):
        check(o.cpu().numpy(), l.cpu().numpy(), ref, ref_lse)
