"""Comparison metric between a device result and the fp64 oracle (test infrastructure).

Relative error of an element, e_i = |g_i - o_i| / max(|o_i|, s_i), where the
floor s_i is the rms of the row of `o` that holds element i (the last axis: a
token's output or gradient vector, one output row of one expert's weight
gradient).  A floor is needed because an element can be close to zero; a row is
one vector quantity whose components share a scale, whereas the rms of a whole
tensor mixes tokens and experts of very different magnitude (an expert with one
routed row next to one with hundreds).

A weight gradient is one parameter tensor per expert, and one row of it can be
arbitrarily small for a reason that fp32 arithmetic cannot resolve: with a single
routed token the row of neuron i is dh_i * x, and dh_i vanishes where h_i sits on
the root of silu' (h ~ -1.2785), where an fp32 evaluation keeps an absolute error
of the order of the fp32 rounding of h but no relative accuracy.  For weight
gradients (``param_axes=(-2, -1)``) the floor is therefore
max(row rms, 1e-3 * rms of that expert's whole matrix): the second term is an
absolute allowance tied to the parameter's own scale, far above fp32 rounding and
far below the scale of any row that carries signal.

The bound for bf16 operands with fp32 accumulation is max e_i <= 2e-2 and
mean e_i <= 3e-3 per tensor, and ``compare`` asserts it under two floors: the
row floor above and the tensor-wide floor, e_i = |g_i - o_i| / max(|o_i|, rms(o))
with the rms over the whole tensor (``max_global``, ``mean_global``).  A result
must meet both.  The normwise error ||g - o|| / ||o|| is reported beside them.
"""
from __future__ import annotations

import numpy as np

MAX_REL = 2e-2
MEAN_REL = 3e-3


PARAM_FRAC = 1e-3


def rel_error(got, ref, param_axes=None):
    g = np.asarray(got, dtype=np.float64)
    o = np.asarray(ref, dtype=np.float64)
    if o.size == 0:
        return dict(max=0.0, mean=0.0, norm=0.0, max_global=0.0, mean_global=0.0)
    if o.ndim == 0:
        g, o = g.reshape(1), o.reshape(1)
    diff = np.abs(g - o)
    floor = np.sqrt(np.mean(o * o, axis=-1, keepdims=True))
    if param_axes is not None and o.ndim > 1:
        axes = tuple(a % o.ndim for a in param_axes)
        floor = np.maximum(floor, PARAM_FRAC * np.sqrt(np.mean(o * o, axis=axes, keepdims=True)))
    tiny = np.finfo(np.float64).tiny
    e = diff / np.maximum(np.abs(o), np.maximum(floor, tiny))
    # rows that are exactly zero in the reference: judge against the tensor's rms
    rms = float(np.sqrt(np.mean(o * o)))
    zero = np.broadcast_to(floor == 0, o.shape)
    if o.ndim > 1 and np.any(zero):
        e = np.where(zero, diff / max(rms, tiny), e)
    eg = diff / np.maximum(np.abs(o), max(rms, tiny))
    nrm = float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-300))
    return dict(max=float(e.max()), mean=float(e.mean()), norm=nrm, max_global=float(eg.max()),
                mean_global=float(eg.mean()))


def compare(name, got, ref, max_rel=MAX_REL, mean_rel=MEAN_REL, param_axes=None):
    """Raise AssertionError with the figures when either floor exceeds the tolerance; return the figures."""
    g = np.asarray(got, dtype=np.float64)
    if not np.all(np.isfinite(g)):
        raise AssertionError(f"{name}: non-finite values in device result")
    r = rel_error(g, ref, param_axes)
    if r["max"] > max_rel or r["mean"] > mean_rel or r["max_global"] > max_rel or r["mean_global"] > mean_rel:
        raise AssertionError(f"{name}: row floor max rel {r['max']:.3e}, mean {r['mean']:.3e}; tensor floor max "
                             f"{r['max_global']:.3e}, mean {r['mean_global']:.3e} (bounds {max_rel}, {mean_rel}); "
                             f"normwise {r['norm']:.3e}")
    return r


# the axes of one expert's weight-gradient matrix (its parameter tensor)
WEIGHT_GRAD = (-2, -1)
