"""Pins for the FP64 oracle (CPU only).

The pages print no worked numeric example for AttnRes, so the oracle is pinned
by things other than itself:
  * hand-derived closed forms on a two-source, two-channel case (forward and
    backward, including the RMSNorm-backward term that cancels there);
  * special cases that reduce to library routines (one source, identical
    sources, zero query -> numpy mean, zero rows -> the eps floor);
  * invariances the equation implies (positive rescaling of one source, scale
    invariance under output RMSNorm, Euler identities for homogeneous maps);
  * central finite differences in float64 for every gradient;
  * gradients from torch.autograd on an independent float64 restatement.
Equation: "Fast Attention Residuals", section "Equation"; defaults eps=2^-23,
scale=1 from its Quickstart signature.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attnres_oracle

EPS = 2.0 ** -23


def run64(v, q, **kw):
    return attnres_oracle(np.asarray(v, np.float64), np.asarray(q, np.float64),
                          precision="f64", nthreads=1, **kw)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------
X = math.log(3.0) / 2.0


def two_source_case(eps):
    # v0 = [1, 1], v1 = [3, -3], q = [x, -x], one token, R = D = 2.
    v = np.array([[[1.0, 1.0]], [[3.0, -3.0]]])
    q = np.array([X, -X])
    return v, q


def test_closed_form_forward_exact_eps():
    v, q = two_source_case(EPS)
    out = run64(v, q, eps=EPS)
    # key RMS: mean(t^2) = 1 and 9
    r0 = 1.0 / math.sqrt(1.0 + EPS)
    r1 = 1.0 / math.sqrt(9.0 + EPS)
    z1 = r1 * (3.0 * X + 3.0 * X)      # z0 = r0 * (x - x) = 0
    a1 = 1.0 / (1.0 + math.exp(-z1))
    a0 = 1.0 - a1
    np.testing.assert_allclose(out["rstd"][0], [r0, r1], rtol=1e-15)
    np.testing.assert_allclose(out["logit"][0], [0.0, z1], atol=1e-15)
    np.testing.assert_allclose(out["alpha"][0], [a0, a1], rtol=1e-14)
    np.testing.assert_allclose(out["y"][0], [a0 * 1 + a1 * 3, a0 * 1 - a1 * 3], rtol=1e-14)


def test_closed_form_forward_backward_no_eps():
    # With eps = 0: z = [0, ln 3], alpha = [1/4, 3/4], y = [5/2, -2].
    v, q = two_source_case(0.0)
    dy = np.array([[1.0, 0.0]])
    out = run64(v, q, eps=0.0, dy=dy)
    np.testing.assert_allclose(out["alpha"][0], [0.25, 0.75], rtol=1e-15)
    np.testing.assert_allclose(out["y"][0], [2.5, -2.0], rtol=1e-15)
    # Backward by hand: do = dy; da = [1, 3]; delta = 5/2; dz = [-3/8, 3/8].
    # k0 = [1, 1], k1 = [1, -1];  dq = sum_s dz_s k_s = [0, -3/4].
    np.testing.assert_allclose(out["dq"], [0.0, -0.75], atol=1e-15)
    # dt0 = r0 dz0 (q - 0 * k0) = -3/8 [x, -x]
    # dt1 = r1 dz1 (q - (ln3 / 2) k1) = 0 because ln3/2 = x  (the (z/R) k term)
    dv = out["dvalues"][:, 0, :]
    np.testing.assert_allclose(dv[0], [0.25 - 3 * X / 8, 3 * X / 8], rtol=1e-14)
    np.testing.assert_allclose(dv[1], [0.75, 0.0], atol=1e-15)


def test_closed_form_key_offset_and_out_norm():
    # Pad the two-source case to D = 4 with non-key channels; key in the final
    # two channels (the page's placement) or the first two.
    base_v, q = two_source_case(0.0)
    pad = np.array([[[2.0, -1.0]], [[4.0, 0.5]]])
    for ko in (0, 2):
        v = np.concatenate([base_v, pad], axis=2) if ko == 0 else np.concatenate([pad, base_v], axis=2)
        w = np.array([2.0, 0.5, 1.0, -1.0])
        out = run64(v, q, eps=0.0, key_offset=ko)
        np.testing.assert_allclose(out["alpha"][0], [0.25, 0.75], rtol=1e-15)
        o = 0.25 * v[0, 0] + 0.75 * v[1, 0]
        np.testing.assert_allclose(out["y"][0], o, rtol=1e-15)
        on = run64(v, q, eps=0.0, key_offset=ko, w_o=w)
        rho = 1.0 / math.sqrt(float(np.mean(o * o)))
        np.testing.assert_allclose(on["o_rstd"][0], rho, rtol=1e-15)
        np.testing.assert_allclose(on["y"][0], rho * o * w, rtol=1e-14)


def test_single_source_is_identity():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((1, 5, 16))
    q = rng.standard_normal(16)
    dy = rng.standard_normal((5, 16))
    out = run64(v, q, dy=dy)
    assert np.array_equal(out["y"], v[0])
    assert np.array_equal(out["alpha"], np.ones((5, 1)))
    assert np.array_equal(out["dq"], np.zeros(16))
    assert np.array_equal(out["dvalues"][0], dy)


def test_identical_sources():
    rng = np.random.default_rng(2)
    row = rng.standard_normal((1, 3, 24))
    v = np.repeat(row, 6, axis=0)
    q = rng.standard_normal(24)
    dy = rng.standard_normal((3, 24))
    out = run64(v, q, dy=dy)
    np.testing.assert_allclose(out["alpha"], np.full((3, 6), 1 / 6), rtol=1e-15)
    np.testing.assert_allclose(out["y"], row[0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out["dq"], 0.0, atol=1e-13)
    # dz = 0, so every source gets alpha * dy
    for s in range(6):
        np.testing.assert_allclose(out["dvalues"][s], dy / 6, rtol=1e-12, atol=1e-14)


def test_zero_query_gives_mean():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((7, 4, 32))
    out = run64(v, np.zeros(32))
    np.testing.assert_allclose(out["alpha"], np.full((4, 7), 1 / 7), rtol=1e-15)
    np.testing.assert_allclose(out["y"], v.mean(axis=0), rtol=1e-13, atol=1e-15)


def test_zero_row_eps_floor():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((3, 2, 8))
    v[1, 0, :] = 0.0
    q = rng.standard_normal(8)
    out = run64(v, q)
    assert out["rstd"][0, 1] == pytest.approx(2.0 ** 11.5, rel=1e-15)
    assert out["logit"][0, 1] == 0.0
    assert np.all(np.isfinite(out["y"]))


def test_all_zero_token_uniform_and_zero_read():
    v = np.zeros((5, 1, 16))
    q = np.random.default_rng(5).standard_normal(16)
    out = run64(v, q, dy=np.ones((1, 16)))
    np.testing.assert_allclose(out["alpha"], np.full((1, 5), 0.2), rtol=1e-15)
    assert np.array_equal(out["y"], np.zeros((1, 16)))


def test_positive_rescaling_leaves_routing():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((4, 6, 32))
    q = rng.standard_normal(32) / math.sqrt(32)
    base = run64(v, q)
    v2 = v.copy()
    v2[2] *= 4.0
    scaled = run64(v2, q)
    # k_s is unchanged up to eps: |dz| <= |z| * eps / mean(t^2) ~ 1e-7
    np.testing.assert_allclose(scaled["alpha"], base["alpha"], atol=1e-6)
    np.testing.assert_allclose(scaled["rstd"][:, 2], base["rstd"][:, 2] / 4.0, rtol=1e-6)


def test_out_norm_scale_invariance():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((5, 3, 64))
    q = rng.standard_normal(64) / 8
    w = 1 + 0.1 * rng.standard_normal(64)
    a = run64(v, q, w_o=w)
    b = run64(8.0 * v, q, w_o=w)
    np.testing.assert_allclose(b["y"], a["y"], rtol=1e-6, atol=1e-7)


def test_euler_identities():
    # Without out-norm and with eps -> 0, y is 1-homogeneous in the sources
    # jointly:  sum_s <dv_s, v_s> = <dy, y>.  With out-norm it is 0-homogeneous:
    # sum_s <dv_s, v_s> = 0.
    rng = np.random.default_rng(8)
    v = rng.standard_normal((4, 3, 16))
    q = rng.standard_normal(16)
    dy = rng.standard_normal((3, 16))
    out = run64(v, q, dy=dy, eps=0.0)
    lhs = float(np.sum(out["dvalues"] * v))
    assert lhs == pytest.approx(float(np.sum(dy * out["y"])), rel=1e-12)
    w = 1 + 0.1 * rng.standard_normal(16)
    on = run64(v, q, dy=dy, eps=0.0, w_o=w)
    assert abs(float(np.sum(on["dvalues"] * v))) < 1e-12
    # w_o enters linearly: <dw_o, w_o> = <dy, y>
    assert float(np.dot(on["dw_o"], w)) == pytest.approx(float(np.sum(dy * on["y"])), rel=1e-12)


# --------------------------------------------------------------------------
# Finite differences (float64, central)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("S,N,D,R,ko,outn", [
    (1, 2, 8, 8, 0, False),
    (3, 2, 8, 8, 0, True),
    (4, 3, 16, 8, 0, False),
    (4, 3, 16, 8, 8, True),
    (2, 1, 12, 4, 5, True),
])
def test_finite_differences(S, N, D, R, ko, outn):
    rng = np.random.default_rng(100 + S * 7 + D + ko)
    v = rng.standard_normal((S, N, D))
    q = rng.standard_normal(R)
    w = 1 + 0.3 * rng.standard_normal(D) if outn else None
    dy = rng.standard_normal((N, D))
    out = run64(v, q, w_o=w, dy=dy, key_offset=ko)

    def loss(vv, qq, ww):
        r = run64(vv, qq, w_o=ww, key_offset=ko)
        return float(np.sum(r["y"] * dy))

    h = 1e-6
    fd_v = np.zeros_like(v)
    for idx in np.ndindex(v.shape):
        vp = v.copy(); vp[idx] += h
        vm = v.copy(); vm[idx] -= h
        fd_v[idx] = (loss(vp, q, w) - loss(vm, q, w)) / (2 * h)
    np.testing.assert_allclose(out["dvalues"], fd_v, rtol=1e-6, atol=1e-7)
    fd_q = np.zeros_like(q)
    for j in range(R):
        qp = q.copy(); qp[j] += h
        qm = q.copy(); qm[j] -= h
        fd_q[j] = (loss(v, qp, w) - loss(v, qm, w)) / (2 * h)
    np.testing.assert_allclose(out["dq"], fd_q, rtol=1e-6, atol=1e-7)
    if outn:
        fd_w = np.zeros_like(w)
        for j in range(D):
            wp = w.copy(); wp[j] += h
            wm = w.copy(); wm[j] -= h
            fd_w[j] = (loss(v, q, wp) - loss(v, q, wm)) / (2 * h)
        np.testing.assert_allclose(out["dw_o"], fd_w, rtol=1e-6, atol=1e-7)


# --------------------------------------------------------------------------
# Independent float64 autograd derivation of the gradients
# --------------------------------------------------------------------------
def autograd_reference(v, q, w, dy, ko, eps, scale):
    vt = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    wt = None if w is None else torch.tensor(w, dtype=torch.float64, requires_grad=True)
    R = qt.shape[0]
    key = vt[..., ko:ko + R]
    k = key * torch.rsqrt(key.pow(2).mean(-1, keepdim=True) + eps)
    logits = scale * (k * qt).sum(-1)          # [S, N]
    p = torch.softmax(logits, dim=0)
    o = (p.unsqueeze(-1) * vt).sum(0)
    if wt is not None:
        o = o * torch.rsqrt(o.pow(2).mean(-1, keepdim=True) + eps) * wt
    (o * torch.tensor(dy)).sum().backward()
    return o.detach().numpy(), vt.grad.numpy(), qt.grad.numpy(), (None if wt is None else wt.grad.numpy())


@pytest.mark.parametrize("S,N,D,R,ko,outn,scale", [
    (8, 2, 64, 64, 0, False, 1.0),
    (5, 4, 64, 16, 48, True, 0.7),
    (9, 3, 32, 8, 0, True, 1.0),
])
def test_against_float64_autograd(S, N, D, R, ko, outn, scale):
    rng = np.random.default_rng(S * 31 + D)
    v = rng.standard_normal((S, N, D)) * rng.uniform(0.5, 2.0, (S, 1, 1))
    q = rng.standard_normal(R)
    w = 1 + 0.1 * rng.standard_normal(D) if outn else None
    dy = rng.standard_normal((N, D))
    y_ref, gv, gq, gw = autograd_reference(v, q, w, dy, ko, EPS, scale)
    out = run64(v, q, w_o=w, dy=dy, key_offset=ko, scale=scale)
    np.testing.assert_allclose(out["y"], y_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out["dvalues"], gv, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["dq"], gq, rtol=1e-10, atol=1e-12)
    if outn:
        np.testing.assert_allclose(out["dw_o"], gw, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------
# Entry points agree; threading does not change results
# --------------------------------------------------------------------------
def test_bf16_entry_matches_f64_entry_and_threads():
    from attention_residuals_gb300.workloads import make_random
    wl = make_random(6, 37, 64, 32, key_offset=16, out_norm=True, seed=9)
    a = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=16, nthreads=1)
    b = attnres_oracle(wl.values.double().numpy(), wl.q.double().numpy(), w_o=wl.w_o.double().numpy(),
                       dy=wl.dy.double().numpy(), key_offset=16, nthreads=5, precision="f64")
    for k in ("y", "alpha", "rstd", "logit", "o_rstd", "dvalues"):
        assert np.array_equal(a[k], b[k]), k
    np.testing.assert_allclose(a["dq"], b["dq"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a["dw_o"], b["dw_o"], rtol=1e-13, atol=1e-15)


def test_rejects_bad_arguments():
    v = np.zeros((2, 1, 8))
    with pytest.raises(ValueError):
        run64(v, np.zeros(9))                       # R > D
    with pytest.raises(ValueError):
        run64(v, np.zeros(4), key_offset=5)         # key slice past D
