"""FP64 oracle of the fused block-partial read (test infrastructure only: the
tests, the smoke check and the benchmark's CPU-baseline leg use it; the
product path never does).

"Fast Attention Residuals", section "Full and Block schedules": Block
supplies the embedding, the completed block sums and an optional current
partial sum; the caller sums the partial block before the read and passes it
as one ordinary (unaveraged) source.  The fused read takes the previous
partial sum and the newest writer output ("delta") instead of their sum:

    partial_new = partial + delta          (a bf16 tensor add: the FP32 sum
                                            rounded to bf16, nearest-even)
    y           = read(completed..., partial_new)   (section "Equation")

and returns partial_new with y.  Backward: partial and delta both feed
partial_new with unit weight, so each receives the read's gradient for the
partial_new source plus whatever gradient reaches partial_new from its later
uses (g_partial).

The read itself is the single-query FP64 oracle; this module only forms the
rounded sum and adds the gradients (in FP64).
"""
from __future__ import annotations

import numpy as np

from .oracle import _as_bits, attnres_oracle


def bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the
    uint16 bit patterns: add 0x7fff plus the lowest kept bit, then keep the
    top 16 bits.  NaNs keep a quiet-NaN pattern."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(x32, dtype=np.float32))
    return np.where(nan, np.uint16(0x7FC0), r)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def partial_sum_bits(partial, delta) -> np.ndarray:
    """partial + delta as a bf16 tensor add: each operand widened exactly to
    FP32, one FP32 add, one rounding to bf16."""
    a = bits_to_f64(_as_bits(partial)).astype(np.float32)
    b = bits_to_f64(_as_bits(delta)).astype(np.float32)
    with np.errstate(over="ignore"):  # overflow to infinity is the FP32 result
        return bf16_bits_from_f32(a + b)


def attnres_partial_oracle(completed, partial, delta, q, *, eps=2.0 ** -23, scale=1.0, w_o=None, dy=None,
                           g_partial=None, key_offset=None, nthreads=None, precision="bf16"):
    """Fused block-partial read.

    completed: packed [S-1, N, D] (S-1 >= 0 sources); partial, delta: [N, D];
    q: [R]; dy: [N, D] or None; g_partial: [N, D] gradient reaching
    partial_new from later uses, or None (zero).  precision "bf16" takes bf16
    bit patterns (torch bf16 tensors or uint16) and rounds partial_new to
    bf16; "f64" takes float64 arrays and adds exactly (for finite
    differences).
    Returns the single-query oracle's outputs for the sources
    (completed..., partial_new) plus partial_new (float64 values), and with
    dy: d_completed [S-1, N, D] and d_partial (= d_delta) [N, D].
    """
    if precision == "bf16":
        pn_bits = partial_sum_bits(partial, delta)
        comp = _as_bits(completed)
        N, D = pn_bits.shape
        comp = comp.reshape(-1, N, D)
        sources = np.concatenate([comp, pn_bits[None]], axis=0)
        pn = bits_to_f64(pn_bits)
        g = None if g_partial is None else bits_to_f64(_as_bits(g_partial))
    elif precision == "f64":
        pn = np.asarray(partial, np.float64) + np.asarray(delta, np.float64)
        N, D = pn.shape
        comp = np.asarray(completed, np.float64).reshape(-1, N, D)
        sources = np.concatenate([comp, pn[None]], axis=0)
        g = None if g_partial is None else np.asarray(g_partial, np.float64)
    else:
        raise ValueError(precision)
    r = attnres_oracle(sources, q, eps=eps, scale=scale, w_o=w_o, dy=dy, key_offset=key_offset,
                       nthreads=nthreads, precision=precision)
    r["partial_new"] = pn
    if dy is not None:
        dv = r.pop("dvalues")
        r["d_completed"] = dv[:-1]
        r["d_partial"] = dv[-1] + (0.0 if g is None else g)
    return r
