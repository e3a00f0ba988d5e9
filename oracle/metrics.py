"""Comparison metric between a device result and the fp64 oracle (test infrastructure).

Per element e_i = |g_i - o_i| / max(|o_i|, rms(o)), with rms over the whole
tensor, so that elements near zero are judged against the tensor's scale.
The bound for bf16 inputs with fp32 accumulation is max <= 2e-2, mean <= 3e-3.
"""
from __future__ import annotations

import numpy as np

MAX_REL = 2e-2
MEAN_REL = 3e-3


def rel_error(got, ref):
    g = np.asarray(got, dtype=np.float64).ravel()
    o = np.asarray(ref, dtype=np.float64).ravel()
    if o.size == 0:
        return dict(max=0.0, mean=0.0, norm=0.0)
    rms = float(np.sqrt(np.mean(o * o)))
    scale = np.maximum(np.abs(o), rms if rms > 0 else 1.0)
    e = np.abs(g - o) / scale
    nrm = float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-300))
    return dict(max=float(e.max()), mean=float(e.mean()), norm=nrm)


def compare(name, got, ref, max_rel=MAX_REL, mean_rel=MEAN_REL):
    """Raise AssertionError with the figures when the tolerance is exceeded; return the figures."""
    r = rel_error(got, ref)
    if not np.all(np.isfinite(np.asarray(got, dtype=np.float64))):
        raise AssertionError(f"{name}: non-finite values in device result")
    if r["max"] > max_rel or r["mean"] > mean_rel:
        raise AssertionError(f"{name}: max rel {r['max']:.3e} (<= {max_rel}), mean rel {r['mean']:.3e} "
                             f"(<= {mean_rel}), normwise {r['norm']:.3e}")
    return r
