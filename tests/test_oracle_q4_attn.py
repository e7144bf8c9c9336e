"""Pins of the oracle's q4_0 paged decode attention (Strata PR #2533, qsa decode commit):
the oracle works in the rotated domain (rotated q, rows as stored, output rotated back,
then gated); these tests restate the same attention in the plain domain with a library
Hadamard matrix and check the two agree, plus closed forms and the degenerate cases."""
import numpy as np
import pytest
import scipy.linalg

import workloads as W

SCALE = 1.0 / 16.0                      # 1 / sqrt(256)


def dequant_rows(pool, cells, kvh):
    """Decode [n][144]-byte q4_0 rows from bytes (nibble - 8) * fp16 d, in the plain
    byte order of the format (independent of the oracle's code)."""
    rows = pool[cells, kvh]                                  # [n][144]
    out = np.empty((rows.shape[0], 256), np.float64)
    for b in range(8):
        blk = rows[:, 18 * b: 18 * b + 18]
        d = blk[:, 0:2].copy().view(np.float16).astype(np.float32)[:, 0]
        qs = blk[:, 2:18]
        codes = np.concatenate([qs & 15, qs >> 4], axis=1).astype(np.float32)   # j, j + 16
        out[:, 32 * b: 32 * b + 32] = ((codes - 8.0) * d[:, None]).astype(np.float64)
    return out


def make_case(orc, n_seq, n_qh, n_kv, lengths, seed, page_size=16):
    wl_pos0, table, n_cells = W.paged_table(n_seq, max(lengths), page_size, 0, seed=seed)
    g = W.rng(seed + 3)
    k = W.normal(g, (n_seq, max(lengths), n_kv, 256)) * 2.0
    v = W.normal(g, (n_seq, max(lengths), n_kv, 256))
    k_pool = np.zeros((n_cells, n_kv, 144), np.uint8)
    v_pool = np.zeros((n_cells, n_kv, 144), np.uint8)
    orc.append_q4(k, v, wl_pos0, table, page_size, n_cells, k_pool, v_pool)
    q = W.normal(g, (n_seq, n_qh, 256))
    gate = W.normal(g, (n_seq, n_qh, 256))
    return dict(seq_len=np.asarray(lengths, np.int32), page_table=table, page_size=page_size,
                n_cells=n_cells, k_pool=k_pool, v_pool=v_pool, q=q, n_kv=n_kv), gate


def plain_attention(case, gate, gate_first=False):
    """softmax(scale q.k) v with unrotated rows (rows as stored are H x / 16)."""
    H = scipy.linalg.hadamard(256).astype(np.float64) / 16.0
    q, table, ps = case["q"], case["page_table"], case["page_size"]
    n_seq, n_qh, _ = q.shape
    grp = n_qh // case["n_kv"]
    out = np.zeros((n_seq, n_qh, 256))
    lse = np.full((n_seq, n_qh), -np.inf)
    for s in range(n_seq):
        L = int(case["seq_len"][s])
        if L == 0:
            continue
        cells = np.array([table[s, t // ps] * ps + t % ps for t in range(L)])
        for h in range(n_qh):
            kr = dequant_rows(case["k_pool"], cells, h // grp) @ H     # rows back to plain
            vr = dequant_rows(case["v_pool"], cells, h // grp) @ H
            sc = SCALE * (kr @ q[s, h].astype(np.float64))
            m = sc.max()
            p = np.exp(sc - m)
            o = p @ vr / p.sum()
            lse[s, h] = m + np.log(p.sum())
            if gate is not None:
                sig = 1.0 / (1.0 + np.exp(-gate[s, h].astype(np.float64)))
                # the wrong placement gates the rotated row and rotates afterwards
                o = (((o @ H) * sig) @ H) if gate_first else o * sig
            out[s, h] = o
    return out, lse


@pytest.mark.parametrize("n_qh,n_kv", [(4, 2), (8, 2), (3, 3)])
def test_rotated_domain_equals_plain_domain(orc, n_qh, n_kv):
    case, gate = make_case(orc, 3, n_qh, n_kv, [1, 37, 70], seed=n_qh)
    for gt in (None, gate):
        out, lse, bad = orc.q4_decode(sm_scale=SCALE, gate=gt, **case)
        ref, ref_lse = plain_attention(case, gt)
        assert bad == 0
        assert np.max(np.abs(out - ref)) <= 1e-12 * np.max(np.abs(ref))
        assert np.allclose(lse, ref_lse, rtol=1e-13, atol=1e-13)


def test_gate_after_rotation_is_discriminated(orc):
    case, gate = make_case(orc, 1, 4, 2, [50], seed=9)
    out, _, _ = orc.q4_decode(sm_scale=SCALE, gate=gate, **case)
    wrong, _ = plain_attention(case, gate, gate_first=True)
    assert np.max(np.abs(out - wrong)) > 1e-2 * np.max(np.abs(out))


def test_single_row_and_uniform_scores(orc):
    case, gate = make_case(orc, 2, 4, 2, [1, 40], seed=4)
    H = scipy.linalg.hadamard(256).astype(np.float64) / 16.0
    out, lse, _ = orc.q4_decode(sm_scale=SCALE, **case)
    cell0 = case["page_table"][0, 0] * case["page_size"]
    for h in range(4):                                   # one row: out = that V row
        v0 = dequant_rows(case["v_pool"], np.array([cell0]), h // 2)[0] @ H
        assert np.allclose(out[0, h], v0, rtol=0, atol=1e-14 * np.abs(v0).max())
    case["q"] = np.zeros_like(case["q"])                 # q = 0: the mean of the V rows
    out, lse, _ = orc.q4_decode(sm_scale=SCALE, **case)
    cells = np.array([case["page_table"][1, t // 16] * 16 + t % 16 for t in range(40)])
    for h in range(4):
        mean = dequant_rows(case["v_pool"], cells, h // 2).mean(0) @ H
        assert np.allclose(out[1, h], mean, rtol=0, atol=1e-13 * np.abs(mean).max())
        assert lse[1, h] == pytest.approx(np.log(40.0), abs=1e-13)


def test_empty_sequence_and_missing_page(orc):
    case, _ = make_case(orc, 2, 2, 1, [0, 40], seed=6)
    out, lse, bad = orc.q4_decode(sm_scale=SCALE, **case)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0])) and bad == 0
    ref, _, _ = orc.q4_decode(sm_scale=SCALE, **dict(case, seq_len=np.array([0, 32], np.int32)))
    case["page_table"] = case["page_table"].copy()
    case["page_table"][1, 2] = -1                        # rows 32..39 have no page
    out2, _, bad2 = orc.q4_decode(sm_scale=SCALE, **case)
    assert bad2 == 1
    assert np.array_equal(out2[1], ref[1])               # those rows are simply absent
