"""Comparison helpers for GPU-vs-oracle parity (tolerances written here).

Tolerances (per the operator's accuracy contract):
  * forward output y (bf16): per-element relative error <= 1e-2, with the
    denominator floored at 1e-3 * the row's RMS so that entries that cancel
    to ~0 in exact arithmetic do not divide by ~0;
  * alpha (fp32): absolute error <= 1e-4;
  * dvalues, dq, dw_o: relative L2 error over the whole tensor <= 2e-3.
    dq and dw_o come in FP32 and bf16; the bound applies to the FP32 copy
    and the bf16 copy must be its exact round-to-nearest-even (bf16 rounding
    alone can move a short vector by more than 2e-3); a vector of 1024 or
    more entries is also held to 2e-3 in bf16 (rounding alone gives about
    1.1e-3 there);
  * dvalues, element by element as well: a whole-tensor norm cannot see one
    wrong 16-byte vector among millions, so every entry must satisfy
        |x - x*| <= 2^-8 |x*| + 2e-3 rms_row(x*) + 1e-5 rms(x*)
    where 2^-8 is bf16's unit roundoff (the most one round-to-nearest-even
    can move a value, relative), the row floor covers FP32 rounding and
    cancellation in the kernel's arithmetic, and the whole-tensor floor
    covers rows whose weights underflow in FP32 (a softmax weight below
    ~1e-38 is zero there and tiny, not zero, in FP64);
  * rstd, o_rstd (fp32): relative error <= 1e-4; logits: absolute error
    <= 1e-4 * max(1, |z|).
"""
import numpy as np
import torch

Y_REL = 1e-2
ALPHA_ABS = 1e-4
GRAD_REL_L2 = 2e-3
STAT_REL = 1e-4
ELEM_REL = 2.0 ** -8       # bf16 unit roundoff
ELEM_ROW_FLOOR = 2e-3      # x RMS of the row (last axis)
ELEM_ALL_FLOOR = 1e-5      # x RMS of the whole tensor
BF16_VEC_MIN = 1024        # vectors this long are held to GRAD_REL_L2 in bf16 too


def to_np(t):
    if isinstance(t, (list, tuple)):
        return np.stack([to_np(x) for x in t])
    return t.detach().float().cpu().numpy().astype(np.float64)


def y_rel_err(y, y_ref):
    y = np.asarray(y, np.float64).reshape(y_ref.shape)
    rms = np.sqrt(np.mean(y_ref ** 2, axis=-1, keepdims=True))
    denom = np.maximum(np.abs(y_ref), 1e-3 * rms)
    denom = np.where(denom > 0, denom, 1.0)
    return float(np.max(np.abs(y - y_ref) / denom)) if y_ref.size else 0.0


def rel_l2(x, ref):
    x = np.asarray(x, np.float64).reshape(ref.shape)
    n = np.linalg.norm(ref)
    if n == 0:
        return float(np.linalg.norm(x))
    return float(np.linalg.norm(x - ref) / n)


def grad_elem_err(x, ref):
    """Largest |x - x*| / (2^-8 |x*| + 2e-3 rms_row(x*) + 1e-5 rms(x*)) over
    all entries (rows along the last axis); <= 1 passes."""
    ref = np.asarray(ref, np.float64)
    x = np.asarray(x, np.float64).reshape(ref.shape)
    if ref.size == 0:
        return 0.0
    rms_row = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    rms_all = float(np.sqrt(np.mean(ref ** 2)))
    bound = ELEM_REL * np.abs(ref) + ELEM_ROW_FLOOR * rms_row + ELEM_ALL_FLOOR * rms_all
    bound = np.where(bound > 0, bound, np.finfo(np.float64).tiny)
    return float(np.max(np.abs(x - ref) / bound))


def check_dvalues(dv, ref, errs, tag="", key="dvalues"):
    """Whole-tensor rel-L2 <= 2e-3 and the per-entry bound of grad_elem_err."""
    ref = np.asarray(ref, np.float64)
    dv = np.asarray(dv, np.float64).reshape(ref.shape)
    errs[key] = rel_l2(dv, ref)
    errs[key + "_elem"] = grad_elem_err(dv, ref)
    assert errs[key] <= GRAD_REL_L2, (tag, key, errs)
    assert errs[key + "_elem"] <= 1.0, (tag, key + " (per entry)", errs)
    return errs


def check_vec_grad(bf16, f32, ref, errs, tag="", key="dq"):
    """A reduced gradient returned in bf16 and FP32: the FP32 copy within
    2e-3 (rel-L2), the bf16 copy its exact round-to-nearest-even, and the
    bf16 copy itself within 2e-3 when it has >= 1024 entries."""
    ref = np.asarray(ref, np.float64)
    b = to_np(bf16).reshape(ref.shape)
    f = to_np(f32).reshape(ref.shape)
    errs[key + "_f32"] = rel_l2(f, ref)
    errs[key + "_bf16"] = rel_l2(b, ref)
    assert errs[key + "_f32"] <= GRAD_REL_L2, (tag, key, errs)
    np.testing.assert_array_equal(b, bf16_rne(f), err_msg=f"{tag} {key}: bf16 is not RNE of the FP32 copy")
    if ref.size >= BF16_VEC_MIN:
        assert errs[key + "_bf16"] <= GRAD_REL_L2, (tag, key + " (bf16)", errs)
    return errs


def check_forward(fwd, ref, *, out_norm, tag=""):
    errs = {}
    errs["y"] = y_rel_err(to_np(fwd["y"]).reshape(ref["y"].shape), ref["y"])
    errs["alpha"] = float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"]))) if ref["alpha"].size else 0.0
    errs["rstd"] = float(np.max(np.abs(to_np(fwd["rstd"]) / ref["rstd"] - 1))) if ref["rstd"].size else 0.0
    z = ref["logit"]
    errs["logit"] = float(np.max(np.abs(to_np(fwd["logit"]) - z) / np.maximum(1, np.abs(z)))) if z.size else 0.0
    assert errs["y"] <= Y_REL, (tag, errs)
    assert errs["alpha"] <= ALPHA_ABS, (tag, errs)
    assert errs["rstd"] <= STAT_REL, (tag, errs)
    assert errs["logit"] <= STAT_REL, (tag, errs)
    if out_norm:
        errs["o_rstd"] = float(np.max(np.abs(to_np(fwd["o_rstd"]) / ref["o_rstd"] - 1)))
        assert errs["o_rstd"] <= STAT_REL, (tag, errs)
    return errs


def bf16_rne(x):
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def check_backward(bwd, ref, *, out_norm, tag=""):
    errs = {}
    check_dvalues(to_np(bwd["dvalues"]), ref["dvalues"], errs, tag)
    check_vec_grad(bwd["dq"], bwd["dq_f32"], ref["dq"], errs, tag, "dq")
    if out_norm:
        check_vec_grad(bwd["dw_o"], bwd["dw_o_f32"], ref["dw_o"], errs, tag, "dw_o")
    return errs


def cuda_copy(wl, device="cuda"):
    return (wl.values.to(device), wl.q.to(device),
            None if wl.w_o is None else wl.w_o.to(device), wl.dy.to(device))


def poison_like(t):
    if t.dtype == torch.bfloat16:
        return torch.full_like(t, float("nan"))
    return torch.full_like(t, float("nan"))
