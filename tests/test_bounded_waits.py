"""The failure path of the tensor-core decode kernels, made to happen without a fault.

Every wait in the pipelines of the tcgen05 kernels is bounded by %globaltimer.  With the
limit cut to 200 ns (kvq_set_wait_limit_ns) the waits for copies and for the other
warps' hand-overs, which take microseconds on a problem of this size, give up.  The call
must still return, set KVQ_DEV_TIMEOUT, and leave no output row that reads as a result
(an aborted CTA poisons its partial, so each row it feeds is NaN; a row whose CTAs all
finished must equal the oracle).  With the
default limit restored the next call on the same buffers must match the oracle again,
which shows that the aborted CTAs freed their tensor memory and left the context usable.
"""
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


@pytest.mark.parametrize("impl", [2, 4, 5], ids=["tcgen05", "tcgen05x16", "tcgen05f8"])
@pytest.mark.parametrize("fmt", [1, 2])
def test_waits_give_up_then_recover(kvq, orc, impl, fmt):
    if impl == 5 and fmt != 1:
        pytest.skip("impl 5 reads fp8 rows only")
    T, H = 32768, 32
    rows = W.magnitude_rows(T, seed=21, lo=1e-2, hi=10.0)
    signs = W.sign_bits(21)
    if fmt == 1:
        lat, ls = orc.encode_fp8(rows.c)
    else:
        lat, ls = orc.encode_tq4(rows.c, signs)
    rope, rs = orc.encode_fp8(rows.k_rope)
    host = dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs)
    cache = {k: dev(v) for k, v in host.items()}
    q = W.queries(1, 1, H, seed=21)
    kw = dict(fp8=cache) if fmt == 1 else dict(tq4=cache, signs=dev(signs))
    p = kvq.make_problem(seq_len=dev(np.array([T], np.int32)), q_lat=dev(q.q_lat),
                         q_rope=dev(q.q_rope), sm_scale=W.SM_SCALE, max_seq_len=T, fmt=fmt,
                         impl=impl, **kw)
    assert kvq.kvq_mla_decode_kernel(p) == impl
    ws = torch.empty(kvq.kvq_mla_decode_workspace(p), dtype=torch.uint8, device="cuda")
    ref, ref_lse, _ = orc.mla_decode(seq_len=np.array([T], np.int32), seq_fmt=np.array([fmt], np.int32),
                                     q_lat=q.q_lat, q_rope=q.q_rope, sm_scale=W.SM_SCALE,
                                     **(dict(fp8=host) if fmt == 1 else dict(tq4=host, signs=signs)))
    ref = ref.reshape(H, 512)
    tol = 1e-4 * np.abs(ref).max(axis=-1)

    out = torch.full((1, 1, H, 512), 7.0, device="cuda")
    lse = torch.full((1, 1, H), 7.0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert kvq.lib().kvq_set_wait_limit_ns(200) == 0
    try:
        kvq.kvq_mla_decode(p, out, lse, ws, dev_status=st)
        torch.cuda.synchronize()
    finally:
        assert kvq.lib().kvq_set_wait_limit_ns(0) == 0
    assert st.item() & kvq.DEV_TIMEOUT
    o = out.cpu().numpy().reshape(H, 512)
    aborted = np.isnan(o).all(axis=-1)
    assert aborted.any()
    # a row is either poisoned whole or a correct result: never a wrong finite value
    assert not np.isnan(o[~aborted]).any()
    assert np.all(np.abs(o[~aborted] - ref[~aborted]).max(axis=-1) <= tol[~aborted])
    assert np.isnan(lse.cpu().numpy().ravel()[aborted]).all()

    # the default limit again: the same call completes and matches the oracle
    st.zero_()
    out.fill_(7.0)
    kvq.kvq_mla_decode(p, out, lse, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = out.cpu().numpy().reshape(H, 512)
    assert np.all(np.abs(o - ref).max(axis=-1) <= tol)
    assert np.allclose(lse.cpu().numpy().ravel(), ref_lse.ravel(), rtol=2e-6, atol=1e-4)
