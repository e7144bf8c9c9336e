"""kvq_mla_decode_noalloc: the decode for callers that cannot allocate device memory
(an allocator or memory pool that owns the device, a loop that must not enter the
allocator, an embedding handed only pre-placed buffers).  Its scratch is a fixed device
array inside the library, so it takes no workspace.  Checked through the C ABI against
kvq_mla_decode with a caller workspace, on different problems called one after the other
(each call reuses the array the one before left behind), and directly against the oracle
on one of them.

This file is named to be collected last; it must pass on its own in a fresh process as
well as after every other test."""
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


def problem(kvq, orc, fmt, T, H, n_q, seed):
    rows = W.magnitude_rows(T, seed=seed, lo=1e-2, hi=10.0)
    signs = W.sign_bits(seed)
    if fmt == kvq.FMT_FP8:
        lat, ls = orc.encode_fp8(rows.c)
    else:
        lat, ls = orc.encode_tq4(rows.c, signs)
    rope, rs = orc.encode_fp8(rows.k_rope)
    cache = {k: dev(v) for k, v in dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs).items()}
    q = W.queries(1, n_q, H, seed=seed)
    kw = dict(fp8=cache) if fmt == kvq.FMT_FP8 else dict(tq4=cache, signs=dev(signs))
    p = kvq.make_problem(seq_len=dev(np.array([T], np.int32)), q_lat=dev(q.q_lat),
                         q_rope=dev(q.q_rope), sm_scale=W.SM_SCALE, max_seq_len=T, fmt=fmt,
                         causal=n_q > 1, **kw)
    host = dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs)
    ref = lambda: orc.mla_decode(seq_len=np.array([T], np.int32), seq_fmt=np.array([fmt], np.int32),
                                 q_lat=q.q_lat, q_rope=q.q_rope, sm_scale=W.SM_SCALE, causal=n_q > 1,
                                 **(dict(fp8=host) if fmt == kvq.FMT_FP8 else dict(tq4=host, signs=signs)))
    return p, ref


def decode_both(kvq, p, with_lse=True):
    shape = (p.n_seq, p.n_q, p.n_heads)
    ws = torch.empty(kvq.kvq_mla_decode_workspace(p), dtype=torch.uint8, device="cuda")
    out_ref = torch.full(shape + (512,), np.nan, device="cuda")
    lse_ref = torch.full(shape, np.nan, device="cuda")
    kvq.kvq_mla_decode(p, out_ref, lse_ref, ws)
    out = torch.full(shape + (512,), np.nan, device="cuda")
    lse = torch.full(shape, np.nan, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_mla_decode_noalloc(p, out, lse if with_lse else None, st)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), lse.cpu().numpy(), out_ref.cpu().numpy(), lse_ref.cpu().numpy(),
            int(st.item()))


def test_noalloc_matches_workspace_decode_twice(kvq, orc):
    # calls in a row, different problems, kernels and scratch footprints: the 32-head
    # tcgen05 kernel (TQ4, 64 heads), the e4m3 kernel (fp8, 16 heads, 3 causal queries,
    # also checked against the oracle), the warp-level MMA kernel (fp8, forced) and the
    # CUDA-core kernel (TQ4 forced to impl 1, no lse output)
    for fmt, T, H, n_q, seed, impl in ((kvq.FMT_TQ4, 32768, 64, 1, 0, 0), (kvq.FMT_FP8, 5000, 16, 3, 1, 0),
                                       (kvq.FMT_FP8, 3000, 16, 1, 3, 3), (kvq.FMT_TQ4, 3000, 8, 1, 2, 1)):
        p, ref = problem(kvq, orc, fmt, T, H, n_q, seed)
        p.impl = impl
        with_lse = impl != 1
        out, lse, out_ref, lse_ref, st = decode_both(kvq, p, with_lse)
        assert st == 0
        assert not np.isnan(out).any()
        err = np.abs(out - out_ref).max(axis=-1)
        assert np.all(err <= 1e-4 * np.abs(out_ref).max(axis=-1))
        if with_lse:
            assert not np.isnan(lse).any()
            assert np.allclose(lse, lse_ref, rtol=2e-6, atol=1e-4)
        else:
            assert np.isnan(lse).all()                  # lse=None: nothing written there
        if fmt == kvq.FMT_FP8 and n_q == 3:
            # the fixed-array call on its own against the fp64 oracle
            o_ref, l_ref, _ = ref()
            o_ref = o_ref.reshape(out.shape)
            assert np.all(np.abs(out - o_ref).max(axis=-1) <= 1e-4 * np.abs(o_ref).max(axis=-1))
            assert np.allclose(lse, l_ref.reshape(lse.shape), rtol=2e-6, atol=1e-4)


def test_noalloc_against_the_oracle(kvq, orc):
    """The allocation-free decode checked directly against the fp64 oracle at one size
    (fp8, T = 777, 16 heads): within 1e-4 of max|out| per (query, head) row."""
    T, H, seed = 777, 16, 5
    rows = W.magnitude_rows(T, seed=seed, lo=1e-2, hi=10.0)
    lat, ls = orc.encode_fp8(rows.c)
    rope, rs = orc.encode_fp8(rows.k_rope)
    q = W.queries(1, 1, H, seed=seed)
    cache = {k: dev(v) for k, v in dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs).items()}
    p = kvq.make_problem(seq_len=dev(np.array([T], np.int32)), q_lat=dev(q.q_lat),
                         q_rope=dev(q.q_rope), sm_scale=W.SM_SCALE, max_seq_len=T,
                         fmt=kvq.FMT_FP8, fp8=cache)
    out = torch.full((1, 1, H, 512), np.nan, device="cuda")
    lse = torch.full((1, 1, H), np.nan, device="cuda")
    kvq.kvq_mla_decode_noalloc(p, out, lse)
    torch.cuda.synchronize()
    ref, ref_lse, _ = orc.mla_decode(seq_len=np.array([T], np.int32), seq_fmt=np.array([orc.FMT_FP8], np.int32),
                                     q_lat=q.q_lat, q_rope=q.q_rope, sm_scale=W.SM_SCALE,
                                     fp8=dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs))
    o = out.cpu().numpy().reshape(H, 512)
    r = ref.reshape(H, 512)
    assert np.all(np.abs(o - r).max(axis=-1) <= 1e-4 * np.abs(r).max(axis=-1))
    assert np.allclose(lse.cpu().numpy().ravel(), ref_lse.ravel(), rtol=2e-6, atol=1e-4)


def test_noalloc_rejects_problems_beyond_its_scratch(kvq):
    """A problem needing more than the fixed 64 MiB is refused before any launch."""
    H, n_q, n_seq, T = 128, 4, 64, 65536
    z = lambda *s: torch.zeros(*s, device="cuda")
    planes = dict(lat=torch.zeros(16, 512, dtype=torch.uint8, device="cuda"), lat_scale=z(16),
                  rope=torch.zeros(16, 64, dtype=torch.uint8, device="cuda"), rope_scale=z(16))
    p = kvq.make_problem(seq_len=torch.full((n_seq,), T, dtype=torch.int32, device="cuda"),
                         q_lat=z(n_seq, n_q, H, 512), q_rope=z(n_seq, n_q, H, 64), sm_scale=0.1,
                         max_seq_len=T, fmt=kvq.FMT_FP8, fp8=planes, seq_stride_rows=T)
    assert kvq.kvq_mla_decode_workspace(p) > (64 << 20)
    out = torch.full((n_seq, n_q, H, 512), 7.0, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_mla_decode_noalloc(p, out)
    assert e.value.status == 5
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
