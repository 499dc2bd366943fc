"""Comparison helpers for GPU-vs-oracle parity (tolerances written here).

Tolerances (per the operator's accuracy contract):
  * forward output y (bf16): per-element relative error <= 1e-2, with the
    denominator floored at 1e-3 * the row's RMS so that entries that cancel
    to ~0 in exact arithmetic do not divide by ~0;
  * alpha (fp32): absolute error <= 1e-4;
  * dvalues, dq, dw_o: relative L2 error over the whole tensor <= 2e-3.
    dq and dw_o come in FP32 and bf16; the bound applies to the FP32 copy
    and the bf16 copy must be its exact round-to-nearest-even (bf16 rounding
    alone can move a short vector by more than 2e-3);
  * rstd, o_rstd (fp32): relative error <= 1e-4; logits: absolute error
    <= 1e-4 * max(1, |z|).
"""
import numpy as np
import torch

Y_REL = 1e-2
ALPHA_ABS = 1e-4
GRAD_REL_L2 = 2e-3
STAT_REL = 1e-4


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
    dv = to_np(bwd["dvalues"]).reshape(ref["dvalues"].shape)
    errs["dvalues"] = rel_l2(dv, ref["dvalues"])
    errs["dq_f32"] = rel_l2(to_np(bwd["dq_f32"]), ref["dq"])
    errs["dq_bf16"] = rel_l2(to_np(bwd["dq"]), ref["dq"])
    for k in ("dvalues", "dq_f32"):
        assert errs[k] <= GRAD_REL_L2, (tag, k, errs)
    np.testing.assert_array_equal(to_np(bwd["dq"]), bf16_rne(to_np(bwd["dq_f32"])))
    if out_norm:
        errs["dw_o_f32"] = rel_l2(to_np(bwd["dw_o_f32"]), ref["dw_o"])
        errs["dw_o_bf16"] = rel_l2(to_np(bwd["dw_o"]), ref["dw_o"])
        assert errs["dw_o_f32"] <= GRAD_REL_L2, (tag, errs)
        np.testing.assert_array_equal(to_np(bwd["dw_o"]), bf16_rne(to_np(bwd["dw_o_f32"])))
    return errs


def cuda_copy(wl, device="cuda"):
    return (wl.values.to(device), wl.q.to(device),
            None if wl.w_o is None else wl.w_o.to(device), wl.dy.to(device))


def poison_like(t):
    if t.dtype == torch.bfloat16:
        return torch.full_like(t, float("nan"))
    return torch.full_like(t, float("nan"))
