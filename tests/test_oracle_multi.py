"""Pins for the multi-query and selected-query oracles (CPU only).

"Fast Attention Residuals", section "Multi-query AttnRes": M queries read the
same sources, each with its own weights and full-width output; selected
reads take a per-token query from an [E, R] bank by id.  The oracles compose
the single-query oracle (itself pinned in test_oracle.py); what the
composition adds -- which query feeds which output, how gradients of shared
sources and of bank rows are summed -- is pinned here by central finite
differences in float64, closed forms (a zero query reads the plain mean, one
source reads itself) and index invariances (permuting queries or bank rows).
"""
import numpy as np
import pytest

from oracle import attnres_oracle
from oracle.multi import attnres_multi_oracle, attnres_selected_oracle

EPS = 2.0 ** -23


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _loss_multi(v, Q, dy, ko):
    out = attnres_multi_oracle(v, Q, key_offset=ko, precision="f64", nthreads=1)
    return float(np.sum(out["y"] * dy))


@pytest.mark.parametrize("R,ko", [(6, 0), (3, 3), (3, 1)])
def test_multi_finite_differences(R, ko):
    rng = np.random.default_rng(7 + R + ko)
    S, N, D, M = 3, 2, 6, 3
    v = _rand(rng, S, N, D)
    Q = _rand(rng, M, R)
    dy = _rand(rng, M, N, D)
    out = attnres_multi_oracle(v, Q, dy=dy, key_offset=ko, precision="f64", nthreads=1)
    h = 1e-6
    num_dv = np.zeros_like(v)
    for idx in np.ndindex(*v.shape):
        vp, vm = v.copy(), v.copy()
        vp[idx] += h
        vm[idx] -= h
        num_dv[idx] = (_loss_multi(vp, Q, dy, ko) - _loss_multi(vm, Q, dy, ko)) / (2 * h)
    num_dq = np.zeros_like(Q)
    for idx in np.ndindex(*Q.shape):
        Qp, Qm = Q.copy(), Q.copy()
        Qp[idx] += h
        Qm[idx] -= h
        num_dq[idx] = (_loss_multi(v, Qp, dy, ko) - _loss_multi(v, Qm, dy, ko)) / (2 * h)
    np.testing.assert_allclose(out["dvalues"], num_dv, rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(out["dq"], num_dq, rtol=1e-7, atol=1e-8)


def test_multi_zero_query_reads_the_mean_and_one_source_reads_itself():
    rng = np.random.default_rng(3)
    v = _rand(rng, 4, 5, 8)
    Q = _rand(rng, 3, 8)
    Q[1] = 0.0
    out = attnres_multi_oracle(v, Q, key_offset=0, precision="f64", nthreads=1)
    np.testing.assert_allclose(out["alpha"][:, 1], 0.25, rtol=1e-15)
    np.testing.assert_allclose(out["y"][1], np.mean(v, axis=0), rtol=1e-13, atol=1e-15)
    one = attnres_multi_oracle(v[:1], Q, dy=_rand(rng, 3, 5, 8), key_offset=0, precision="f64",
                               nthreads=1)
    for m in range(3):
        np.testing.assert_array_equal(one["y"][m], v[0])
    np.testing.assert_array_equal(one["dq"], 0.0)


def test_multi_query_permutation_permutes_outputs_and_gradients():
    rng = np.random.default_rng(11)
    v = _rand(rng, 5, 4, 8)
    Q = _rand(rng, 4, 4)
    dy = _rand(rng, 4, 4, 8)
    perm = np.array([2, 0, 3, 1])
    a = attnres_multi_oracle(v, Q, dy=dy, key_offset=4, precision="f64", nthreads=1)
    b = attnres_multi_oracle(v, Q[perm], dy=dy[perm], key_offset=4, precision="f64", nthreads=1)
    np.testing.assert_array_equal(b["y"], a["y"][perm])
    np.testing.assert_array_equal(b["alpha"], a["alpha"][:, perm])
    np.testing.assert_array_equal(b["dq"], a["dq"][perm])
    np.testing.assert_allclose(b["dvalues"], a["dvalues"], rtol=1e-12, atol=1e-14)
    # rstd does not depend on the query
    np.testing.assert_array_equal(a["rstd"], b["rstd"])


def test_multi_one_query_equals_single():
    rng = np.random.default_rng(5)
    v = _rand(rng, 3, 6, 16)
    q = _rand(rng, 8)
    dy = _rand(rng, 6, 16)
    single = attnres_oracle(v, q, dy=dy, key_offset=8, precision="f64", nthreads=1)
    multi = attnres_multi_oracle(v, q[None], dy=dy[None], key_offset=8, precision="f64", nthreads=1)
    np.testing.assert_array_equal(multi["y"][0], single["y"])
    np.testing.assert_array_equal(multi["dq"][0], single["dq"])
    np.testing.assert_array_equal(multi["dvalues"], single["dvalues"])


def _loss_sel(v, B, ids, dy, ko):
    out = attnres_selected_oracle(v, B, ids, key_offset=ko, precision="f64", nthreads=1)
    return float(np.sum(out["y"] * dy))


def test_selected_finite_differences():
    rng = np.random.default_rng(17)
    S, N, D, R, E, K = 3, 4, 6, 3, 3, 2
    v = _rand(rng, S, N, D)
    B = _rand(rng, E, R)
    ids = np.array([[0, 2], [2, 2], [1, 0], [0, 0]])
    dy = _rand(rng, N, K, D)
    out = attnres_selected_oracle(v, B, ids, dy=dy, key_offset=3, precision="f64", nthreads=1)
    h = 1e-6
    num_db = np.zeros_like(B)
    for idx in np.ndindex(*B.shape):
        Bp, Bm = B.copy(), B.copy()
        Bp[idx] += h
        Bm[idx] -= h
        num_db[idx] = (_loss_sel(v, Bp, ids, dy, 3) - _loss_sel(v, Bm, ids, dy, 3)) / (2 * h)
    num_dv = np.zeros_like(v)
    for idx in np.ndindex(*v.shape):
        vp, vm = v.copy(), v.copy()
        vp[idx] += h
        vm[idx] -= h
        num_dv[idx] = (_loss_sel(vp, B, ids, dy, 3) - _loss_sel(vm, B, ids, dy, 3)) / (2 * h)
    np.testing.assert_allclose(out["dbank"], num_db, rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(out["dvalues"], num_dv, rtol=1e-7, atol=1e-8)


def test_selected_constant_ids_equal_multi_and_unused_rows_get_zero():
    rng = np.random.default_rng(23)
    v = _rand(rng, 4, 5, 8)
    B = _rand(rng, 4, 8)
    ids = np.tile(np.array([[3, 1]]), (5, 1))
    dy = _rand(rng, 5, 2, 8)
    sel = attnres_selected_oracle(v, B, ids, dy=dy, key_offset=0, precision="f64", nthreads=1)
    mul = attnres_multi_oracle(v, B[[3, 1]], dy=np.transpose(dy, (1, 0, 2)), key_offset=0,
                               precision="f64", nthreads=1)
    np.testing.assert_allclose(sel["y"], np.transpose(mul["y"], (1, 0, 2)), rtol=1e-15)
    np.testing.assert_allclose(sel["dbank"][[3, 1]], mul["dq"], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(sel["dbank"][[0, 2]], 0.0)
    np.testing.assert_allclose(sel["dvalues"], mul["dvalues"], rtol=1e-12, atol=1e-14)


def test_selected_bank_permutation_invariance():
    rng = np.random.default_rng(29)
    v = _rand(rng, 3, 6, 8)
    B = _rand(rng, 5, 4)
    ids = rng.integers(0, 5, size=(6, 3))
    dy = _rand(rng, 6, 3, 8)
    perm = np.array([4, 2, 0, 1, 3])          # new row i holds old row perm[i]
    inv = np.argsort(perm)
    a = attnres_selected_oracle(v, B, ids, dy=dy, key_offset=4, precision="f64", nthreads=1)
    b = attnres_selected_oracle(v, B[perm], inv[ids], dy=dy, key_offset=4, precision="f64",
                                nthreads=1)
    np.testing.assert_array_equal(b["y"], a["y"])
    np.testing.assert_allclose(b["dbank"], a["dbank"][perm], rtol=1e-13, atol=1e-15)


def test_selected_rejects_out_of_range_ids():
    v = np.zeros((2, 3, 8))
    with pytest.raises(ValueError):
        attnres_selected_oracle(v, np.zeros((2, 8)), np.array([[0], [2], [1]]), precision="f64")
