"""Comparison metric between a device result and the fp64 oracle (test infrastructure).

Relative error of an element, e_i = |g_i - o_i| / max(|o_i|, s_i), where the
floor s_i is the rms of the row of `o` that holds element i (the last axis: a
token's output or gradient vector, one output row of one expert's weight
gradient).  A floor is needed because an element can be close to zero; a row is
one vector quantity whose components share a scale, whereas the rms of a whole
tensor mixes tokens and experts of very different magnitude (an expert with
one routed row next to one with hundreds).  The bound for bf16 operands with
fp32 accumulation is max e_i <= 2e-2 and mean e_i <= 3e-3 per tensor.  The
normwise error ||g - o|| / ||o|| and the tensor-wide-floor figures are reported
beside it.
"""
from __future__ import annotations

import numpy as np

MAX_REL = 2e-2
MEAN_REL = 3e-3


def rel_error(got, ref):
    g = np.asarray(got, dtype=np.float64)
    o = np.asarray(ref, dtype=np.float64)
    if o.size == 0:
        return dict(max=0.0, mean=0.0, norm=0.0, max_global=0.0)
    if o.ndim == 0:
        g, o = g.reshape(1), o.reshape(1)
    diff = np.abs(g - o)
    row = np.sqrt(np.mean(o * o, axis=-1, keepdims=True))
    tiny = np.finfo(np.float64).tiny
    e = diff / np.maximum(np.abs(o), np.maximum(row, tiny))
    # rows that are exactly zero in the reference: judge against the tensor's rms
    rms = float(np.sqrt(np.mean(o * o)))
    if o.ndim > 1:
        zero_rows = (row == 0).squeeze(-1)
        if np.any(zero_rows):
            e[zero_rows] = diff[zero_rows] / max(rms, tiny)
    eg = diff / np.maximum(np.abs(o), max(rms, tiny))
    nrm = float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-300))
    return dict(max=float(e.max()), mean=float(e.mean()), norm=nrm, max_global=float(eg.max()),
                mean_global=float(eg.mean()))


def compare(name, got, ref, max_rel=MAX_REL, mean_rel=MEAN_REL):
    """Raise AssertionError with the figures when the tolerance is exceeded; return the figures."""
    g = np.asarray(got, dtype=np.float64)
    if not np.all(np.isfinite(g)):
        raise AssertionError(f"{name}: non-finite values in device result")
    r = rel_error(g, ref)
    if r["max"] > max_rel or r["mean"] > mean_rel:
        raise AssertionError(f"{name}: max rel {r['max']:.3e} (<= {max_rel}), mean rel {r['mean']:.3e} "
                             f"(<= {mean_rel}), normwise {r['norm']:.3e}")
    return r
