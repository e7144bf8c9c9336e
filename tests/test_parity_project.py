"""GPU parity of the projection-fused q4_0 append (kvq_project_append_q4): every pool byte
equals the oracle's, which projects in the same fixed fp32 order and then appends."""
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


def weights_dev(w):
    if w.dtype == np.uint16:
        return dev(w.view(np.int16)).view(torch.bfloat16)
    return dev(w)


def run_both(kvq, orc, n_seq, n_tok, d_model, n_heads, bf16, page_size=16, pos0=11, seed=0,
             sentinel=(0xC3, 0x3C)):
    h, w_k, w_v = W.projection_inputs(n_seq, n_tok, d_model, n_heads, seed=seed, bf16=bf16)
    p0, table, n_cells = W.paged_table(n_seq, n_tok, page_size, pos0, seed=seed)
    n_cells += 2 * page_size                             # spare cells keep the sentinel
    kp = torch.full((n_cells, n_heads, 144), sentinel[0], dtype=torch.uint8, device="cuda")
    vp = torch.full((n_cells, n_heads, 144), sentinel[1], dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_project_append_q4(dev(h), weights_dev(w_k), weights_dev(w_v), dev(p0), dev(table),
                              page_size, n_cells, kp, vp, st)
    torch.cuda.synchronize()
    ok = np.full((n_cells, n_heads, 144), sentinel[0], np.uint8)
    ov = np.full((n_cells, n_heads, 144), sentinel[1], np.uint8)
    orc.project_append_q4(h, w_k, w_v, p0, table, page_size, n_cells, ok, ov)
    return kp.cpu().numpy(), vp.cpu().numpy(), ok, ov, int(st.item())


@pytest.mark.parametrize("n_seq,n_tok", [(1, 1), (1, 3), (2, 3), (2, 5), (3, 13)])
@pytest.mark.parametrize("bf16", [False, True])
def test_project_append_matches_oracle(kvq, orc, n_seq, n_tok, bf16):
    """1, 2, 3 or 4 token pairs in a group, groups of 8 with a ragged last one, pages
    crossed, K and V of 8 heads."""
    kp, vp, ok, ov, st = run_both(kvq, orc, n_seq, n_tok, 1024, 8, bf16, seed=n_seq * 10 + n_tok)
    assert st == 0
    assert np.array_equal(kp, ok) and np.array_equal(vp, ov)


@pytest.mark.parametrize("d_model", [4, 60, 1000, 4096])
def test_project_append_widths(kvq, orc, d_model):
    """Chunks that are short or empty (d_model < 64, not a multiple of 64) and a full
    4096-wide hidden row."""
    kp, vp, ok, ov, st = run_both(kvq, orc, 2, 9, d_model, 2, d_model % 8 == 0, seed=d_model)
    assert st == 0
    assert np.array_equal(kp, ok) and np.array_equal(vp, ov)


def test_project_append_identity_is_plain_append(kvq, orc):
    """Identity K weights and permutation V weights: the fused producer writes the bytes
    kvq_append_q4 writes for h and its permuted columns."""
    g = np.random.default_rng(5)
    n_seq, n_tok, n_heads = 2, 7, 2
    h = (g.standard_normal((n_seq, n_tok, 512)) * 3).astype(np.float32)
    eye = np.eye(512, dtype=np.float32)
    perm = g.permutation(512)
    p0, table, n_cells = W.paged_table(n_seq, n_tok, 8, 3, seed=5)
    kp = torch.zeros((n_cells, n_heads, 144), dtype=torch.uint8, device="cuda")
    vp = torch.zeros_like(kp)
    kvq.kvq_project_append_q4(dev(h), dev(eye), dev(eye[:, perm]), dev(p0), dev(table), 8,
                              n_cells, kp, vp)
    ak = torch.zeros_like(kp)
    av = torch.zeros_like(kp)
    kvq.kvq_append_q4(dev(h.reshape(n_seq, n_tok, n_heads, 256)),
                      dev(h[..., perm].reshape(n_seq, n_tok, n_heads, 256)), dev(p0), dev(table),
                      8, n_cells, ak, av)
    torch.cuda.synchronize()
    assert torch.equal(kp, ak) and torch.equal(vp, av)


def test_project_append_bad_page(kvq, orc):
    """A sequence whose page ids fall outside the pool: its tokens are skipped (their
    cells keep the sentinel) and KVQ_DEV_BAD_PAGE is set; the other sequence is exact."""
    n_seq, n_tok, d_model, n_heads, ps = 2, 6, 256, 1, 4
    h, w_k, w_v = W.projection_inputs(n_seq, n_tok, d_model, n_heads, seed=9)
    p0, table, n_cells = W.paged_table(n_seq, n_tok, ps, 1, seed=9)
    good = table.copy()
    table[1, :] = n_cells // ps + 5
    kp = torch.full((n_cells, n_heads, 144), 0x77, dtype=torch.uint8, device="cuda")
    vp = torch.full_like(kp, 0x77)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_project_append_q4(dev(h), dev(w_k), dev(w_v), dev(p0), dev(table), ps, n_cells, kp, vp, st)
    torch.cuda.synchronize()
    assert int(st.item()) & kvq.DEV_BAD_PAGE
    ok = np.full((n_cells, n_heads, 144), 0x77, np.uint8)
    ov = np.full_like(ok, 0x77)
    orc.project_append_q4(h[:1], w_k, w_v, p0[:1], good[:1], ps, n_cells, ok, ov)
    assert np.array_equal(kp.cpu().numpy(), ok) and np.array_equal(vp.cpu().numpy(), ov)


@pytest.mark.slow
def test_project_append_decode_step_workload(kvq, orc):
    """The bench's producer workload: 16 sequences x 1 new token, d_model 4096, 8 KV heads,
    bfloat16 weights; every pool byte."""
    kp, vp, ok, ov, st = run_both(kvq, orc, 16, 1, 4096, 8, True, page_size=64, pos0=8191, seed=21)
    assert st == 0
    assert np.array_equal(kp, ok) and np.array_equal(vp, ov)
