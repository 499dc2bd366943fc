"""The parity checker itself, on the CPU: what the GPU tests call a pass.

The round-to-nearest-even bf16 copy of the oracle's own FP64 gradient (the
best any bf16 kernel can return) must pass every check, and mistakes planted
in oracle results must fail:
  * one 16-byte vector of one dvalues row replaced by its neighbour (an
    indexing slip that moves the whole-tensor norm far less than 2e-3);
  * one token's gradient computed with the wrong logit scale (a `scale`
    dropped on one code path);
  * a reduced gradient rounded toward zero instead of to nearest even.
"""
import numpy as np
import pytest

from attention_residuals_gb300.workloads import make_random
from oracle import attnres_oracle
from parity_utils import (GRAD_REL_L2, bf16_rne, check_dvalues, check_vec_grad, grad_elem_err,
                          rel_l2)


@pytest.fixture(scope="module")
def case():
    wl = make_random(6, 211, 2048, 512, key_offset=1536, out_norm=True, seed=5, scale=2.5, eps=1e-2)
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=wl.key_offset,
                         eps=wl.eps, scale=wl.scale)
    return wl, ref


def test_rounded_oracle_passes(case):
    wl, ref = case
    errs = {}
    check_dvalues(bf16_rne(ref["dvalues"]), ref["dvalues"], errs)
    import torch
    for key, n in (("dq", wl.R), ("dw_o", wl.D)):
        f32 = torch.tensor(ref[key], dtype=torch.float32)
        check_vec_grad(f32.to(torch.bfloat16), f32, ref[key], errs, key=key)
    assert errs["dvalues_elem"] <= 1.0 and errs["dvalues"] <= GRAD_REL_L2


def test_one_shifted_vector_fails_per_entry_only(case):
    wl, ref = case
    dv = bf16_rne(ref["dvalues"]).copy()
    s, n, c = 3, 117, 40  # 16-byte vector 40 of row (3, 117) takes vector 41's values
    dv[s, n, 8 * c:8 * c + 8] = dv[s, n, 8 * c + 8:8 * c + 16]
    assert rel_l2(dv, ref["dvalues"]) <= GRAD_REL_L2  # the norm alone does not see it
    assert grad_elem_err(dv, ref["dvalues"]) > 1.0
    with pytest.raises(AssertionError):
        check_dvalues(dv, ref["dvalues"], {})


def test_wrong_scale_on_one_token_fails(case):
    wl, ref = case
    n = 77
    wrong = attnres_oracle(wl.values[:, n:n + 1], wl.q, w_o=wl.w_o, dy=wl.dy[n:n + 1],
                           key_offset=wl.key_offset, eps=wl.eps, scale=1.0)
    dv = bf16_rne(ref["dvalues"]).copy()
    dv[:, n] = bf16_rne(wrong["dvalues"][:, 0])
    with pytest.raises(AssertionError):
        check_dvalues(dv, ref["dvalues"], {})


def test_rounding_toward_zero_fails(case):
    import torch
    wl, ref = case
    f32 = np.asarray(ref["dq"], np.float32)
    bits = f32.view(np.uint32) & np.uint32(0xFFFF0000)  # truncation: round toward zero
    trunc = torch.from_numpy(bits.view(np.float32).copy()).to(torch.bfloat16)
    assert not np.array_equal(trunc.float().numpy(), bf16_rne(f32))
    with pytest.raises(AssertionError):
        check_vec_grad(trunc, torch.from_numpy(f32), ref["dq"], {})
