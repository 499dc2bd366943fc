"""FP64 oracle of the multi-query and selected-query reads (test
infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the product path never does).

"Fast Attention Residuals", section "Multi-query AttnRes": the same sources
are read with M queries [M, R] (1 <= M <= 16); each query has its own source
weights and its own full-width output.  Per query this is exactly the
single-query read of section "Equation", so the oracle is that definition
written out: one call of the single-query FP64 oracle per query.  The
sources' gradient is the sum over queries of each read's gradient (the
sources feed every read), each query's gradient comes from its own read.

The same section's `attnres_selected(sources, query_bank, ids)` takes an
[E, R] query bank and integer [..., K] ids and returns [..., K, D]: output
(n, k) is the single-query read of token n's sources with query
bank[ids[n, k]].  Its oracle calls the single-query oracle once per
(bank row, k) on the tokens that select that row; a bank row's gradient is
the sum of the gradients of every read that used it, and a row no token
selects gets a zero gradient.

All sums are in IEEE double; nothing here rounds.
"""
from __future__ import annotations

import numpy as np

from .oracle import _as_bits, attnres_oracle


def _rows(x, precision):
    if precision == "bf16":
        return _as_bits(x)
    return np.ascontiguousarray(x, dtype=np.float64)


def attnres_multi_oracle(values, queries, *, eps=2.0 ** -23, scale=1.0, dy=None,
                         key_offset=None, nthreads=None, precision="bf16", want_dvalues=True):
    """Multi-query read.

    values: packed [S, N, D]; queries: [M, R]; dy: [M, N, D] (query-major) or
    None.  Returns float64 arrays: y [M, N, D], alpha / logit [N, M, S],
    rstd [N, S], and with dy: dq [M, R], dvalues [S, N, D].
    """
    v = _rows(values, precision)
    Q = _rows(queries, precision)
    if Q.ndim != 2:
        raise ValueError("queries must be [M, R]")
    M = Q.shape[0]
    S, N, D = v.shape
    g = None if dy is None else _rows(dy, precision)
    if g is not None and g.shape != (M, N, D):
        raise ValueError("dy must be [M, N, D]")
    y = np.empty((M, N, D))
    alpha = np.empty((N, M, S))
    logit = np.empty((N, M, S))
    rstd = None
    dq = np.zeros((M, Q.shape[1])) if g is not None else None
    dv = np.zeros((S, N, D)) if (g is not None and want_dvalues) else None
    for m in range(M):
        r = attnres_oracle(v, Q[m], eps=eps, scale=scale, dy=None if g is None else g[m],
                           key_offset=key_offset, nthreads=nthreads, precision=precision,
                           want_dvalues=want_dvalues)
        y[m] = r["y"]
        alpha[:, m] = r["alpha"]
        logit[:, m] = r["logit"]
        rstd = r["rstd"]
        if g is not None:
            dq[m] = r["dq"]
            if dv is not None:
                dv += r["dvalues"]
    out = {"y": y, "alpha": alpha, "logit": logit, "rstd": rstd}
    if g is not None:
        out["dq"] = dq
        if dv is not None:
            out["dvalues"] = dv
    return out


def attnres_selected_oracle(values, bank, ids, *, eps=2.0 ** -23, scale=1.0, dy=None,
                            key_offset=None, nthreads=None, precision="bf16", want_dvalues=True):
    """Selected-query read.

    values: packed [S, N, D]; bank: [E, R]; ids: integer [N, K] with
    0 <= ids < E; dy: [N, K, D] or None.  Returns float64 arrays: y [N, K, D],
    alpha / logit [N, K, S], rstd [N, S], and with dy: dbank [E, R],
    dvalues [S, N, D].
    """
    v = _rows(values, precision)
    B = _rows(bank, precision)
    ids = np.asarray(ids)
    if ids.ndim != 2:
        raise ValueError("ids must be [N, K]")
    S, N, D = v.shape
    E, R = B.shape
    K = ids.shape[1]
    if ids.shape[0] != N or (ids.size and (ids.min() < 0 or ids.max() >= E)):
        raise ValueError("ids out of range")
    g = None if dy is None else _rows(dy, precision)
    if g is not None and g.shape != (N, K, D):
        raise ValueError("dy must be [N, K, D]")
    y = np.zeros((N, K, D))
    alpha = np.zeros((N, K, S))
    logit = np.zeros((N, K, S))
    rstd = np.zeros((N, S))
    dbank = np.zeros((E, R)) if g is not None else None
    dv = np.zeros((S, N, D)) if (g is not None and want_dvalues) else None
    for e in range(E):
        for k in range(K):
            tok = np.nonzero(ids[:, k] == e)[0]
            if tok.size == 0:
                continue
            r = attnres_oracle(np.ascontiguousarray(v[:, tok]), B[e], eps=eps, scale=scale,
                               dy=None if g is None else np.ascontiguousarray(g[tok, k]),
                               key_offset=key_offset, nthreads=nthreads, precision=precision,
                               want_dvalues=want_dvalues)
            y[tok, k] = r["y"]
            alpha[tok, k] = r["alpha"]
            logit[tok, k] = r["logit"]
            rstd[tok] = r["rstd"]
            if g is not None:
                dbank[e] += r["dq"]
                if dv is not None:
                    dv[:, tok] += r["dvalues"]
    out = {"y": y, "alpha": alpha, "logit": logit, "rstd": rstd}
    if g is not None:
        out["dbank"] = dbank
        if dv is not None:
            out["dvalues"] = dv
    return out
