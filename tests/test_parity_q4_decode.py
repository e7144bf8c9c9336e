"""GPU parity of the q4_0 paged GQA decode attention (Strata PR #2533, qsa decode commit)
against the fp64 oracle over the same stored pools: every output row (sequence, query
head) within 1e-4 * max|out| of that row, lse within 1e-4 absolute (plus a few 1e-7
relative), the bad-page flag raised exactly when the oracle raises it.  The pools are
written by the oracle's q4_0 append from seeded rows of the q4_0 paged workload
(N(0,1) times amplitude classes {1e-3, 1, 40}, permuted page table)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-4
SCALE = 1.0 / 16.0


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_fp8_gb300 as k
    return k


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def make_case(orc, n_seq, n_qh, n_kv, lengths, seed, page_size=16, spare_pages=0):
    """Pools written by the oracle's append of max(lengths) tokens per sequence from
    position 0; a sequence of length L reads its first L positions."""
    n_tok = max(max(lengths), 1)
    wl = W.q4_paged(n_seq=n_seq, n_tok=n_tok, n_heads=n_kv, page_size=page_size, pos0=0,
                    seed=seed, spare_pages=spare_pages)
    kp = np.zeros((wl.n_cells, n_kv, 144), np.uint8)
    vp = np.zeros((wl.n_cells, n_kv, 144), np.uint8)
    orc.append_q4(wl.k, wl.v, wl.pos0, wl.page_table, page_size, wl.n_cells, kp, vp)
    g = W.rng(seed + 101)
    q = W.normal(g, (n_seq, n_qh, 256))
    gate = W.normal(g, (n_seq, n_qh, 256)) * 3.0
    return dict(seq_len=np.asarray(lengths, np.int32), page_table=wl.page_table,
                page_size=page_size, n_cells=wl.n_cells, k_pool=kp, v_pool=vp, q=q,
                n_kv=n_kv), gate


def run_gpu(kvq, case, gate=None, split_rows=0, max_seq_len=None, with_lse=True,
            sm_scale=SCALE):
    n_seq, n_qh, _ = case["q"].shape
    if max_seq_len is None:
        max_seq_len = int(case["seq_len"].max()) if n_seq else 0
    t = dict(seq_len=dev(case["seq_len"]), page_table=dev(case["page_table"]),
             k_pool=dev(case["k_pool"]), v_pool=dev(case["v_pool"]), q=dev(case["q"]),
             gate=None if gate is None else dev(gate))
    p = kvq.make_q4_problem(page_size=case["page_size"], sm_scale=sm_scale,
                            max_seq_len=max_seq_len, split_rows=split_rows, **t)
    ws = torch.empty(max(kvq.kvq_q4_decode_workspace(p), 1), dtype=torch.uint8, device="cuda")
    out = torch.full((n_seq, n_qh, 256), np.nan, dtype=torch.float32, device="cuda")
    lse = torch.full((n_seq, n_qh), np.nan, dtype=torch.float32, device="cuda") if with_lse else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_q4_decode(p, out, lse, ws, st)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), None if lse is None else lse.cpu().numpy(), int(st.item()))


def check(out, lse, ref, ref_lse, sel=None):
    if sel is not None:
        out, ref, ref_lse = out[sel], ref[sel], ref_lse[sel]
        lse = None if lse is None else lse[sel]
    assert not np.isnan(out).any()
    empty = np.isneginf(ref_lse)
    assert np.all(out[empty] == 0)
    err = np.abs(out - ref).max(axis=-1)
    bar = TOL * np.abs(ref).max(axis=-1)
    ok = empty | (err <= bar)
    scale = np.maximum(np.abs(ref[~empty]).max(-1), np.finfo(np.float64).tiny)
    worst = float(np.max(err[~empty] / scale)) if (~empty).any() else 0.0
    assert ok.all(), f"worst err/max|out| = {worst:.3e}"
    if lse is not None:
        assert np.all(np.isneginf(lse[empty]))
        assert np.allclose(lse[~empty], ref_lse[~empty], rtol=2e-6, atol=1e-4)
    return worst


@pytest.mark.parametrize("n_qh,n_kv", [(2, 2), (4, 2), (8, 2), (16, 2), (16, 8)])
@pytest.mark.parametrize("split", [0, 32])
def test_ratios_ragged_lengths(kvq, orc, n_qh, n_kv, split):
    """Group ratios 1, 2, 4, 8 (8: two warps per KV head); lengths 0 (empty), 1, one
    short of and one past two 16-position tiles, page-crossing, several splits with a
    ragged tail."""
    lengths = [0, 1, 31, 33, 70, 200]
    case, gate = make_case(orc, len(lengths), n_qh, n_kv, lengths, seed=n_qh * 10 + n_kv)
    for gt in (None, gate):
        ref, ref_lse, bad = orc.q4_decode(sm_scale=SCALE, gate=gt, **case)
        out, lse, st = run_gpu(kvq, case, gate=gt, split_rows=split)
        assert bad == 0 and st == 0
        check(out, lse, ref, ref_lse)


@pytest.mark.parametrize("split", [16, 40, 64, 1000])
def test_split_sizes(kvq, orc, split):
    """The LSE combine over 1 to 19 splits, split sizes that are and are not multiples of
    the 16-position tile a warp takes per step."""
    lengths = [300, 129, 5]
    case, gate = make_case(orc, 3, 8, 2, lengths, seed=77, page_size=32)
    ref, ref_lse, _ = orc.q4_decode(sm_scale=SCALE, gate=gate, **case)
    out, lse, st = run_gpu(kvq, case, gate=gate, split_rows=split)
    assert st == 0
    check(out, lse, ref, ref_lse)


def test_without_lse_and_other_scale(kvq, orc):
    case, _ = make_case(orc, 2, 4, 1, [40, 90], seed=5)
    ref, ref_lse, _ = orc.q4_decode(sm_scale=0.3, **case)
    out, lse, st = run_gpu(kvq, case, with_lse=False, sm_scale=0.3)
    assert lse is None and st == 0
    check(out, None, ref, ref_lse)


def test_bad_pages_skipped_and_flagged(kvq, orc):
    """A missing page (-1), a page id past the pool, and a length past the page table:
    those positions are skipped, KVQ_DEV_BAD_PAGE is raised, the rest matches."""
    lengths = [64, 64, 64]
    case, gate = make_case(orc, 3, 8, 4, lengths, seed=9, page_size=16)
    table = case["page_table"].copy()
    table[0, 1] = -1
    table[1, 3] = case["n_cells"] // 16 + 5
    case["page_table"] = table
    ref, ref_lse, bad = orc.q4_decode(sm_scale=SCALE, gate=gate, **case)
    assert bad == 1
    out, lse, st = run_gpu(kvq, case, gate=gate, split_rows=32)
    assert st & kvq.DEV_BAD_PAGE
    check(out, lse, ref, ref_lse)
    # the third sequence alone is clean
    out2, lse2, st2 = run_gpu(kvq, dict(case, seq_len=np.array([0, 0, 64], np.int32)), gate=gate)
    assert st2 == 0
    # a length past the table (4 pages of 16 = 64 positions) flags too
    case3 = dict(case, seq_len=np.array([0, 0, 80], np.int32))
    ref3, ref3_lse, bad3 = orc.q4_decode(sm_scale=SCALE, **case3)
    out3, lse3, st3 = run_gpu(kvq, case3)
    assert bad3 == 1 and st3 & kvq.DEV_BAD_PAGE
    check(out3, lse3, ref3, ref3_lse)


def test_all_positions_bad_gives_empty_row(kvq, orc):
    case, _ = make_case(orc, 2, 4, 2, [20, 20], seed=13, page_size=16)
    table = case["page_table"].copy()
    table[0, :] = -1
    case["page_table"] = table
    ref, ref_lse, bad = orc.q4_decode(sm_scale=SCALE, **case)
    out, lse, st = run_gpu(kvq, case)
    assert bad == 1 and st & kvq.DEV_BAD_PAGE
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    check(out, lse, ref, ref_lse)


def test_seq_len_clamped_to_max(kvq, orc):
    """seq_len beyond the host bound max_seq_len reads only max_seq_len positions."""
    case, _ = make_case(orc, 2, 4, 2, [50, 50], seed=17)
    out, lse, st = run_gpu(kvq, dict(case, seq_len=np.array([50, 50], np.int32)),
                           max_seq_len=30, split_rows=16)
    ref, ref_lse, _ = orc.q4_decode(sm_scale=SCALE, **dict(case, seq_len=np.array([30, 30], np.int32)))
    assert st == 0
    check(out, lse, ref, ref_lse)


def test_empty_batch(kvq):
    case = dict(seq_len=np.zeros(0, np.int32), page_table=np.zeros((0, 1), np.int32),
                page_size=16, n_cells=16, k_pool=np.zeros((16, 2, 144), np.uint8),
                v_pool=np.zeros((16, 2, 144), np.uint8), q=np.zeros((0, 4, 256), np.float32),
                n_kv=2)
    out, lse, st = run_gpu(kvq, case, max_seq_len=0)
    assert out.shape == (0, 4, 256) and st == 0


@pytest.mark.slow
def test_full_paged_workload_sampled(kvq, orc):
    """16 sequences x 8192 positions, 8 KV heads and 16 query heads (2 per KV head),
    page_size 64, permuted table, gated; the launch the timing run uses (library-chosen
    splits).  Three sequences are checked against the oracle row by row; every row is
    finite with a finite lse."""
    wl = W.q4_paged(n_seq=16, n_tok=8192, n_heads=8, page_size=64, pos0=0, seed=0)
    kp = np.zeros((wl.n_cells, 8, 144), np.uint8)
    vp = np.zeros((wl.n_cells, 8, 144), np.uint8)
    orc.append_q4(wl.k, wl.v, wl.pos0, wl.page_table, 64, wl.n_cells, kp, vp)
    del wl.k, wl.v
    g = W.rng(1234)
    q = W.normal(g, (16, 16, 256))
    gate = W.normal(g, (16, 16, 256))
    case = dict(seq_len=np.full(16, 8192, np.int32), page_table=wl.page_table, page_size=64,
                n_cells=wl.n_cells, k_pool=kp, v_pool=vp, q=q, n_kv=8)
    out, lse, st = run_gpu(kvq, case, gate=gate)
    assert st == 0
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    sel = np.array([0, 7, 15], np.int32)
    ref, ref_lse, bad = orc.q4_decode(sm_scale=SCALE, gate=gate, seq_sel=sel, **case)
    assert bad == 0
    check(out, lse, ref, ref_lse, sel=sel)
