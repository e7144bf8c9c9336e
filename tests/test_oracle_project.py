"""Pins of the oracle's projection producer (orc_project_rows / orc_project_append_q4).

The pages leave the arithmetic of the K/V projection to the model; the library fixes a
summation order so that the rotated q4_0 codes of its fused producer can be compared
byte for byte.  What is pinned here is independent of that order: exact results where
every partial sum is exact, identity and permutation weights, bfloat16 widening, and the
fp32 error bound against an fp64 product."""
import numpy as np
import pytest

import workloads as W


def test_exact_integer_products(orc):
    """Small integers: every product and partial sum is an integer below 2^24, so any
    order gives the exact value.  A dropped, doubled or transposed term fails."""
    g = np.random.default_rng(1)
    for d_model, n_out in [(8, 5), (100, 33), (256, 64), (1028, 17)]:
        h = g.integers(-8, 9, (3, d_model)).astype(np.float32)
        w = g.integers(-8, 9, (d_model, n_out)).astype(np.float32)
        y = orc.project_rows(h, w)
        ref = h.astype(np.int64) @ w.astype(np.int64)
        assert np.array_equal(y, ref.astype(np.float32)), d_model


def test_identity_and_permutation_weights(orc):
    """Identity weights return h bit for bit (every other term is an exact zero), a
    permutation returns the permuted row; so the fused append equals the plain append of
    those rows."""
    g = np.random.default_rng(2)
    h = (g.standard_normal((2, 3, 512)) * 7).astype(np.float32)
    eye = np.eye(512, dtype=np.float32)
    perm = g.permutation(512)
    pmat = eye[:, perm]                                  # column c selects h[perm[c]]
    assert np.array_equal(orc.project_rows(h.reshape(-1, 512), eye), h.reshape(-1, 512))
    assert np.array_equal(orc.project_rows(h.reshape(-1, 512), pmat), h.reshape(-1, 512)[:, perm])

    pos0, table, n_cells = W.paged_table(2, 3, 4, 2, seed=3)
    fk = np.full((n_cells, 2, 144), 0x11, np.uint8)
    fv = np.full((n_cells, 2, 144), 0x22, np.uint8)
    orc.project_append_q4(h, eye, pmat, pos0, table, 4, n_cells, fk, fv)
    pk = np.full_like(fk, 0x11)
    pv = np.full_like(fv, 0x22)
    orc.append_q4(h.reshape(2, 3, 2, 256), h[..., perm].reshape(2, 3, 2, 256), pos0, table, 4,
                  n_cells, pk, pv)
    assert np.array_equal(fk, pk) and np.array_equal(fv, pv)


def test_bfloat16_weights_widen_exactly(orc):
    h, w_k, _ = W.projection_inputs(1, 4, 256, 1, seed=4, bf16=True)
    widened = (w_k.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(orc.project_rows(h.reshape(-1, 256), w_k),
                          orc.project_rows(h.reshape(-1, 256), widened))


@pytest.mark.parametrize("d_model", [4, 60, 1000, 4096])
def test_error_bound_against_fp64(orc, d_model):
    """A chain of at most L fmas and six pairwise levels: |y - exact| <=
    (L + 6) u sum |h w| (u = 2^-24, first order).  One dropped term of this data would
    exceed the bound by orders of magnitude."""
    h, w, _ = W.projection_inputs(1, 5, d_model, 1, seed=d_model)
    h2 = h.reshape(-1, d_model)
    y = orc.project_rows(h2, w).astype(np.float64)
    exact = h2.astype(np.float64) @ w.astype(np.float64)
    mag = np.abs(h2.astype(np.float64)) @ np.abs(w.astype(np.float64))
    L = 4 * ((d_model + 255) // 256)
    bound = (L + 6) * 2.0 ** -24 * mag * (1 + 1e-6)
    assert np.all(np.abs(y - exact) <= bound)
    # the bound is tight enough to catch a missing term
    k = d_model // 2
    dropped = exact - h2[:, k:k + 1].astype(np.float64) * w[k:k + 1, :].astype(np.float64)
    assert np.mean(np.abs(dropped - exact) > bound) > 0.5
