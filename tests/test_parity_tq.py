"""GPU parity of the rotated tiers at 3 and 6 bits (colibri PR #399: KV_TQ=6 and a
3-bit setting beside the 4-bit tier): every encoded byte and radius bit equal to the
oracle's (kvq_encode_tq), the decode over 3- and 6-bit rows (the CUDA-core kernel and
the 16-head tcgen05 kernel) within 1e-4 * max|out| of the fp64 oracle, and the row
gather byte for byte."""
import numpy as np
import pytest
import torch

import workloads as W
from test_parity_decode import check, run_gpu

pytestmark = pytest.mark.gpu
FMT = {3: 5, 6: 4}


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_fp8_gb300 as k
    return k


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_encode(kvq, x, signs, bits, ldp=None):
    R, D = x.shape
    rb = D * bits // 8
    ldp = rb if ldp is None else ldp
    packed = torch.full((R, ldp), 0xA5, dtype=torch.uint8, device="cuda")
    radius = torch.full((R,), -1.0, dtype=torch.float32, device="cuda")
    kvq.kvq_encode_tq(dev(x), dev(signs), bits, packed, radius)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), radius.cpu().numpy()


@pytest.mark.parametrize("bits", [3, 6])
@pytest.mark.parametrize("dim", [64, 128, 256, 512, 1024])
def test_encode_byte_exact(kvq, orc, bits, dim):
    g = W.rng(dim + bits)
    x = W.normal(g, (257, dim)) * W.log_uniform(g, 257, 1e-3, 40.0)[:, None].astype(np.float32)
    x[5] = 0.0                                              # inert row
    x[9, :] = 0.0
    x[9, 3] = 1.0                                           # one nonzero element
    signs = W.sign_bits(dim + bits, n=max(dim, 32))
    packed, radius = gpu_encode(kvq, x, signs, bits)
    ref, ref_r = orc.encode_tq(x, signs, bits)
    assert np.array_equal(radius.view(np.uint32), ref_r.view(np.uint32))
    assert np.array_equal(packed, ref)


@pytest.mark.parametrize("bits", [3, 6])
def test_encode_strided_leaves_padding(kvq, orc, bits):
    g = W.rng(50 + bits)
    full = W.normal(g, (100, 640))
    x = full[:, :512]                                       # ldx 640
    signs = W.sign_bits(50 + bits)
    rb = 512 * bits // 8
    xd = dev(full)[:, :512]
    packed = torch.full((100, rb + 32), 0xA5, dtype=torch.uint8, device="cuda")
    radius = torch.empty(100, dtype=torch.float32, device="cuda")
    kvq.kvq_encode_tq(xd, dev(signs), bits, packed, radius)
    torch.cuda.synchronize()
    p = packed.cpu().numpy()
    ref, ref_r = orc.encode_tq(x, signs, bits)
    assert np.array_equal(p[:, :rb], ref) and np.all(p[:, rb:] == 0xA5)
    assert np.array_equal(radius.cpu().numpy().view(np.uint32), ref_r.view(np.uint32))


@pytest.mark.slow
def test_encode_full_workload_six_bits(kvq, orc):
    """The 4-bit tier's workload (T=32768 N(0,1) rows of 512) at 6 bits."""
    rows = W.unit_rows(32768, seed=0)
    signs = W.sign_bits(0)
    packed, radius = gpu_encode(kvq, rows.c, signs, 6)
    ref, ref_r = orc.encode_tq(rows.c, signs, 6)
    assert np.array_equal(packed, ref)
    assert np.array_equal(radius.view(np.uint32), ref_r.view(np.uint32))


def encode_cache(orc, rows, signs, bits):
    lat, rad = orc.encode_tq(rows.c, signs, bits)
    rope, rs = orc.encode_fp8(rows.k_rope)
    return dict(lat=lat, lat_scale=rad, rope=rope, rope_scale=rs)


@pytest.mark.parametrize("impl", [1, 4], ids=["cudacore", "tcgen05x16"])
@pytest.mark.parametrize("bits", [3, 6])
@pytest.mark.parametrize("T,split", [(1, 0), (17, 0), (65, 32), (1000, 96), (4096, 0), (20000, 0)])
def test_decode_over_tq_rows(kvq, orc, bits, T, split, impl):
    rows = W.magnitude_rows(T, seed=T + bits, lo=1e-2, hi=10.0)
    signs = W.sign_bits(T + bits)
    cache = encode_cache(orc, rows, signs, bits)
    q = W.queries(1, 1, 16, seed=T)
    out, lse, st = run_gpu(kvq, cache_fmt=FMT[bits], caches={2: cache}, seq_len=[T], q=q,
                           signs=signs, split_rows=split, impl=impl)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T], seq_fmt=[FMT[bits]], q_lat=q.q_lat,
                                     q_rope=q.q_rope, sm_scale=W.SM_SCALE, tq4=cache, signs=signs)
    assert st == 0
    check(out, lse, ref, ref_lse)


@pytest.mark.parametrize("impl", [1, 4], ids=["cudacore", "tcgen05x16"])
@pytest.mark.parametrize("bits", [3, 6])
def test_decode_paged_causal_multi_query(kvq, orc, bits, impl):
    """Two sequences through a permuted block table (pages of 16), 3 causal queries."""
    lengths = [150, 47]
    rows = W.unit_rows(320, seed=60 + bits)
    signs = W.sign_bits(60 + bits)
    cache = encode_cache(orc, rows, signs, bits)
    table = np.random.default_rng(60).permutation(20).astype(np.int32).reshape(2, 10)
    q = W.queries(2, 3, 8, seed=60)
    kw = dict(seq_len=lengths, q=q, signs=signs, block_table=table, page_size=16, causal=True)
    out, lse, st = run_gpu(kvq, cache_fmt=FMT[bits], caches={2: cache}, impl=impl, **kw)
    ref, ref_lse, _ = orc.mla_decode(seq_len=lengths, seq_fmt=[FMT[bits]] * 2, q_lat=q.q_lat,
                                     q_rope=q.q_rope, sm_scale=W.SM_SCALE, causal=True,
                                     block_table=table, page_size=16, tq4=cache, signs=signs)
    assert st == 0
    check(out, lse, ref, ref_lse)


def test_mixed_batch_tensor_core_flags_six_bit_sequences(kvq, orc):
    """A seq_fmt batch of an fp8 and a 6-bit sequence: the CUDA-core kernel reads both;
    the two tensor-core kernels read the fp8 one and flag the other (out 0, lse -inf)."""
    T = 300
    rows = W.unit_rows(2 * T, seed=70)                     # sequence i: pool rows i*T ..
    signs = W.sign_bits(70)
    c8 = dict(zip(("lat", "lat_scale"), orc.encode_fp8(rows.c)))
    c8["rope"], c8["rope_scale"] = orc.encode_fp8(rows.k_rope)
    c6 = encode_cache(orc, rows, signs, 6)
    q = W.queries(2, 1, 16, seed=70)
    kw = dict(cache_fmt=1, caches={1: c8, 2: c6}, seq_len=[T, T], q=q, signs=signs,
              seq_fmt=[1, 4], seq_stride_rows=T)
    ref, ref_lse, _ = orc.mla_decode(seq_len=[T, T], seq_fmt=[1, 4], q_lat=q.q_lat, q_rope=q.q_rope,
                                     sm_scale=W.SM_SCALE, seq_stride_rows=T, fp8=c8, tq4=c6,
                                     signs=signs)
    out, lse, st = run_gpu(kvq, impl=1, **kw)
    assert st == 0
    check(out, lse, ref, ref_lse)
    for impl in (2, 3, 4):
        out2, lse2, st2 = run_gpu(kvq, impl=impl, **kw)
        assert st2 & kvq.DEV_BAD_FORMAT
        check(out2[:1], lse2[:1], ref[:1], ref_lse[:1])
        assert np.all(out2[1] == 0) and np.all(np.isneginf(lse2[1]))


@pytest.mark.parametrize("bits", [3, 6])
def test_gather_rows_byte_exact(kvq, orc, bits):
    T = 2000
    rows = W.unit_rows(T, seed=80 + bits)
    lat, ls = orc.encode_tq(rows.c, W.sign_bits(80), bits)
    rope, rs = orc.encode_fp8(rows.k_rope)
    src = dict(lat=dev(lat), lat_scale=dev(ls), rope=dev(rope), rope_scale=dev(rs))
    idx = W.sparse_indices(T, 129, 1, seed=80)[0]
    dst = {k: torch.full((129,) + v.shape[1:], 7, dtype=v.dtype, device="cuda") for k, v in src.items()}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_gather_rows(FMT[bits], src, T, dev(idx), dst, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for k, host in (("lat", lat), ("lat_scale", ls), ("rope", rope), ("rope_scale", rs)):
        assert np.array_equal(dst[k].cpu().numpy(), host[idx])
