"""Seeded synthetic inputs for the MoE expert layer.

This module is the single source of inputs for both the fp64 oracle and the
CUDA path.  It draws numbers and nothing else: no routing, no GEMM, no
activation of the method lives here.

Generator: counter-based splitmix64 + Box-Muller (definition in ``gen.c``),
rounded to bf16 with round-to-nearest-even.  Because each element is a pure
function of (seed, stream, index), slices (one expert's weights, a handful of
token rows) can be regenerated on their own.

Workloads follow the five configurations of the benchmark description:

* ``tiny``   T=64,    d=128,  E=8,   n=64,   K=2  forward only
* ``c2``     T=4096,  d=2048, E=128, n=512,  K=8  near-uniform load (~256 rows/expert)
* ``c3``     T=8192,  d=7168, E=256, n=2048, K=8  router bias ~N(0, 0.5)
* ``c4``     T=8192,  d=2880, E=128, n=2880, K=4  log-Zipf(s=1.2) prior b_e = -1.2 ln(e+1)
* ``c5``     T=32768, d=1536, E=512, n=256,  K=8  token rounding to M_tile=128 (``c5_plain`` without)
* ``c2_cap``, ``c2_cap_probs``  the c2 shape under the capacity (drop/pad) dispatch, capacity factor 1

Layouts (row-major, the pages' ``(E, out, in)`` stacking of nn.Linear weights):
X[T,d], W_r[d,E], W_gate[E,n,d], W_up[E,n,d], W_down[E,d,n], bias[E] fp32, dO[T,d].
Weights are drawn with standard deviation 1/sqrt(fan_in) (fan_in = d for W_r,
W_gate, W_up; n for W_down); X and dO with standard deviation 1.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile
from dataclasses import dataclass, replace

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "gen.c")
_SO = os.path.join(_DIR, "_gen.so")

# Stream ids, one per tensor.
S_X, S_WR, S_WGATE, S_WUP, S_WDOWN, S_BIAS, S_DO = 1, 2, 3, 4, 5, 6, 7

_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into _gen.so next to it (plain C, any host arch)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64, u64, dbl = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        lib.synth_normal_bf16.argtypes = [u16p, i64, u64, u64, i64, dbl, dbl]
        lib.synth_normal_f32.argtypes = [ctypes.POINTER(ctypes.c_float), i64, u64, u64, i64, dbl, dbl]
        lib.synth_int_bf16.argtypes = [u16p, i64, u64, u64, i64, ctypes.c_int32, ctypes.c_int32]
        lib.synth_uniform_f64.argtypes = [ctypes.POINTER(ctypes.c_double), i64, u64, u64, i64]
        lib.synth_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().synth_num_threads())


def normal_bf16(n: int, stream: int, offset: int = 0, mean: float = 0.0, std: float = 1.0,
                seed: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits (uint16) of N(mean, std^2) draws, elements [offset, offset+n) of a stream."""
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _load().synth_normal_bf16(out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), n, seed, stream,
                              offset, mean, std)
    return out


def normal_f32(n: int, stream: int, offset: int = 0, mean: float = 0.0, std: float = 1.0,
               seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n, seed, stream,
                             offset, mean, std)
    return out


def int_bf16(n: int, stream: int, lo: int, hi: int, offset: int = 0, seed: int = 0) -> np.ndarray:
    """bf16 bits of integers drawn uniformly from [lo, hi] (exact in bf16 for |v| <= 256)."""
    out = np.empty(n, dtype=np.uint16)
    _load().synth_int_bf16(out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), n, seed, stream,
                           offset, lo, hi)
    return out


def uniform_f64(n: int, stream: int, offset: int = 0, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform_f64(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n, seed, stream,
                              offset)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to float32 exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bits (nearest-even), the same rounding the generator uses."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    n: int
    K: int
    bias: str = "none"        # "none" | "normal" (std 0.5) | "zipf" (b_e = -1.2 ln(e+1))
    m_tile: int = 0           # token rounding multiple; 0 = plain top-K
    fwd_only: bool = False
    integer: bool = False     # integer-valued inputs (exact GEMMs and router logits)
    seed: int = 0
    capacity_factor: float = 0.0  # capacity (drop/pad) dispatch; 0 = ragged
    drop_policy: str = "position"

    @property
    def pairs(self) -> int:
        """T*K, the number of routed pairs before token rounding."""
        return self.T * self.K

    def flops_fwd_bwd(self, P: int | None = None) -> int:
        """Algorithmic expert flops: 6Pdn forward + 12Pdn backward."""
        P = self.pairs if P is None else P
        return (6 if self.fwd_only else 18) * P * self.d * self.n


WORKLOADS = {
    "tiny": Workload("tiny", 64, 128, 8, 64, 2, fwd_only=True),
    "c2": Workload("c2", 4096, 2048, 128, 512, 8),
    "c3": Workload("c3", 8192, 7168, 256, 2048, 8, bias="normal"),
    "c4": Workload("c4", 8192, 2880, 128, 2880, 4, bias="zipf"),
    "c5": Workload("c5", 32768, 1536, 512, 256, 8, m_tile=128),
    "c5_plain": Workload("c5_plain", 32768, 1536, 512, 256, 8),
    # the capacity (drop/pad) dispatch variant on the c2 shape
    "c2_cap": Workload("c2_cap", 4096, 2048, 128, 512, 8, capacity_factor=1.0),
    "c2_cap_probs": Workload("c2_cap_probs", 4096, 2048, 128, 512, 8, capacity_factor=1.0, drop_policy="probs"),
}


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of a workload with some sizes replaced (small parity cases of the same shape family)."""
    return replace(wl, **kw)


# ---------------------------------------------------------------- tensors


def _gen(wl: Workload, n: int, stream: int, offset: int, std: float, lo=-2, hi=2) -> np.ndarray:
    if wl.integer:
        return int_bf16(n, stream, lo, hi, offset=offset, seed=wl.seed)
    return normal_bf16(n, stream, offset=offset, std=std, seed=wl.seed)


def make_x(wl: Workload, rows: np.ndarray | None = None) -> np.ndarray:
    """X[T,d] bf16 bits; with ``rows`` only those token rows."""
    if rows is None:
        return _gen(wl, wl.T * wl.d, S_X, 0, 1.0).reshape(wl.T, wl.d)
    return np.stack([_gen(wl, wl.d, S_X, int(t) * wl.d, 1.0) for t in rows]) if len(rows) else \
        np.zeros((0, wl.d), np.uint16)


def make_dout(wl: Workload, rows: np.ndarray | None = None) -> np.ndarray:
    """Upstream gradient dO[T,d] bf16 bits, N(0,1)."""
    if rows is None:
        return _gen(wl, wl.T * wl.d, S_DO, 0, 1.0).reshape(wl.T, wl.d)
    return np.stack([_gen(wl, wl.d, S_DO, int(t) * wl.d, 1.0) for t in rows]) if len(rows) else \
        np.zeros((0, wl.d), np.uint16)


def make_router(wl: Workload) -> np.ndarray:
    """W_r[d,E] bf16 bits, std 1/sqrt(d)."""
    return _gen(wl, wl.d * wl.E, S_WR, 0, 1.0 / math.sqrt(wl.d)).reshape(wl.d, wl.E)


def make_bias(wl: Workload) -> np.ndarray | None:
    """Per-expert router bias (fp32) or None."""
    if wl.bias == "none":
        return None
    if wl.bias == "normal":
        return normal_f32(wl.E, S_BIAS, std=0.5, seed=wl.seed)
    if wl.bias == "zipf":
        return (-1.2 * np.log(np.arange(1, wl.E + 1, dtype=np.float64))).astype(np.float32)
    raise ValueError(wl.bias)


def make_w_gate(wl: Workload, experts=None) -> np.ndarray:
    """W_gate[E,n,d] (or the listed experts) bf16 bits, std 1/sqrt(d)."""
    return _expert_tensor(wl, S_WGATE, wl.n, wl.d, 1.0 / math.sqrt(wl.d), experts, lo=-1, hi=1)


def make_w_up(wl: Workload, experts=None) -> np.ndarray:
    return _expert_tensor(wl, S_WUP, wl.n, wl.d, 1.0 / math.sqrt(wl.d), experts, lo=-1, hi=1)


def make_w_down(wl: Workload, experts=None) -> np.ndarray:
    """W_down[E,d,n] bf16 bits, std 1/sqrt(n)."""
    return _expert_tensor(wl, S_WDOWN, wl.d, wl.n, 1.0 / math.sqrt(wl.n), experts, lo=-1, hi=1)


def _expert_tensor(wl, stream, rows, cols, std, experts, lo, hi):
    per = rows * cols
    if experts is None:
        return _gen(wl, wl.E * per, stream, 0, std, lo, hi).reshape(wl.E, rows, cols)
    experts = list(experts)
    out = np.empty((len(experts), rows, cols), np.uint16)
    for i, e in enumerate(experts):
        out[i] = _gen(wl, per, stream, int(e) * per, std, lo, hi).reshape(rows, cols)
    return out
