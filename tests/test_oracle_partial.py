"""Pins for the fused block-partial read oracle (CPU only).

"Fast Attention Residuals", section "Full and Block schedules": the caller
sums the partial block before the read; the fused read forms that sum
itself.  Pinned here against things other than the oracle: PyTorch's own
bf16 tensor add (the rounding the unfused caller would get), the two-step
unfused computation, central finite differences in float64 for every
gradient including the extra gradient reaching the new partial sum, and the
read being independent of how the partial sum is split.
"""
import numpy as np
import pytest
import torch

from oracle import attnres_oracle
from oracle.partial import (attnres_partial_oracle, bf16_bits_from_f32, bits_to_f64,
                            partial_sum_bits)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_rounding_matches_torch_bf16_add():
    g = torch.Generator().manual_seed(0)
    a = (torch.randn(4096, generator=g) * torch.logspace(-8, 8, 4096)).to(torch.bfloat16)
    b = (torch.randn(4096, generator=g) * 3).to(torch.bfloat16)
    a[:8] = torch.tensor([0.0, -0.0, 1.0, 1.0, 3.0e38, -3.0e38, 1e-40, 2.0]).to(torch.bfloat16)
    b[:8] = torch.tensor([0.0, 0.0, 2.0 ** -8, 3 * 2.0 ** -9, 3.0e38, 1.0, 1e-40, -2.0]).to(torch.bfloat16)
    np.testing.assert_array_equal(partial_sum_bits(a, b), _bits(a + b))


def test_rne_ties_to_even_and_nan():
    # 1 + 2^-8 lies half way between bf16 neighbours 1 and 1 + 2^-7: ties go to even (1)
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, np.nan, -0.0], np.float32)
    bits = bf16_bits_from_f32(x)
    np.testing.assert_array_equal(bits_to_f64(bits[:2]), [1.0, 1.0 + 2.0 ** -6])
    assert bits[2] == 0x7FC0 and bits[3] == 0x8000


def test_equals_unfused_two_step():
    g = torch.Generator().manual_seed(1)
    S1, N, D, R = 4, 7, 64, 32
    comp = torch.randn(S1, N, D, generator=g).to(torch.bfloat16)
    part = torch.randn(N, D, generator=g).to(torch.bfloat16)
    delta = torch.randn(N, D, generator=g).to(torch.bfloat16)
    q = (torch.randn(R, generator=g) / R ** 0.5).to(torch.bfloat16)
    dy = torch.randn(N, D, generator=g).to(torch.bfloat16)
    gp = torch.randn(N, D, generator=g).to(torch.bfloat16)
    fused = attnres_partial_oracle(comp, part, delta, q, dy=dy, g_partial=gp, key_offset=0)
    pn = part + delta                       # the caller's bf16 add
    unf = attnres_oracle(torch.cat([comp, pn[None]]), q, dy=dy, key_offset=0)
    np.testing.assert_array_equal(fused["y"], unf["y"])
    np.testing.assert_array_equal(fused["partial_new"], pn.double().numpy())
    np.testing.assert_array_equal(fused["d_completed"], unf["dvalues"][:-1])
    np.testing.assert_array_equal(fused["d_partial"], unf["dvalues"][-1] + gp.double().numpy())


@pytest.mark.parametrize("out_norm", [False, True])
def test_finite_differences(out_norm):
    rng = np.random.default_rng(5)
    S1, N, D, R = 2, 2, 6, 3
    comp, part, delta = rng.standard_normal((S1, N, D)), rng.standard_normal((N, D)), rng.standard_normal((N, D))
    q = rng.standard_normal(R)
    w = 1 + 0.1 * rng.standard_normal(D) if out_norm else None
    dy = rng.standard_normal((N, D))
    gp = rng.standard_normal((N, D))

    def loss(c, p, d):
        r = attnres_partial_oracle(c, p, d, q, w_o=w, key_offset=3, precision="f64", nthreads=1)
        return float(np.sum(r["y"] * dy) + np.sum(r["partial_new"] * gp))

    out = attnres_partial_oracle(comp, part, delta, q, w_o=w, dy=dy, g_partial=gp, key_offset=3,
                                 precision="f64", nthreads=1)
    h = 1e-6
    for name, arr, ref in (("part", part, out["d_partial"]), ("delta", delta, out["d_partial"]),
                           ("comp", comp, out["d_completed"])):
        num = np.zeros_like(arr)
        for idx in np.ndindex(*arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = {"part": (comp, ap, delta), "delta": (comp, part, ap), "comp": (ap, part, delta)}[name]
            args_m = {"part": (comp, am, delta), "delta": (comp, part, am), "comp": (am, part, delta)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(ref, num, rtol=1e-7, atol=1e-8, err_msg=name)


def test_split_of_the_partial_sum_does_not_matter_in_f64():
    rng = np.random.default_rng(9)
    comp = rng.standard_normal((3, 4, 8))
    total = rng.standard_normal((4, 8))
    d1 = rng.standard_normal((4, 8))
    q = rng.standard_normal(8)
    a = attnres_partial_oracle(comp, total - d1, d1, q, key_offset=0, precision="f64", nthreads=1)
    b = attnres_partial_oracle(comp, total, np.zeros_like(total), q, key_offset=0, precision="f64", nthreads=1)
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-13, atol=1e-14)
