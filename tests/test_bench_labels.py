"""Host-side consistency of the benchmark's kernel accounting with the CUDA sources (CPU only): every grouped-GEMM
instantiation the library launches maps to a named label, and every label the library's profiling hook reports
has algorithmic work figures."""
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "varlen_grouped_gemm_gb300", "csrc")


def _enums():
    src = open(os.path.join(CSRC, "gemm.cuh")).read()
    vals = {}
    for body in re.findall(r"enum \w+ \{([^}]*)\}", src):
        for name, v in re.findall(r"(\w+)\s*=\s*(\d+)", body):
            vals[name] = int(v)
    return vals


def _instantiations():
    """Template arguments of every launch_grouped_gemm in the library's own sources (not the test exports)."""
    out = []
    for f in sorted(os.listdir(CSRC)):
        if f.endswith(".cu") and f != "gemm_test.cu":
            out += [(f, m) for m in re.findall(r"launch_grouped_gemm<([^>]*)>", open(os.path.join(CSRC, f)).read())]
    return out


def test_every_grouped_gemm_instantiation_has_a_label():
    import bench
    ev = _enums()
    insts = _instantiations()
    assert len(insts) > 20
    for f, args in insts:
        a = [x.strip() for x in args.split(",")]
        nums = [str(ev.get(x, x)) for x in a]
        name = f"void vgg::grouped_gemm_kernel<{', '.join(nums)}>(vgg::GemmParams, vgg::Maps)"
        label = bench._label_of(name)
        assert label in set(bench._GEMM_LABELS.values()) | set(bench._MX_GEMM_LABELS.values()), (f, args, label)


@pytest.mark.parametrize("wl", ["c2", "c5", "c2_cap"])
def test_every_profiled_label_has_work_figures(wl):
    import bench
    names = set()
    for f in os.listdir(CSRC):
        if f.endswith(".cu"):
            names |= set(re.findall(r'VGG_LAUNCH\("([a-z_0-9]+)"', open(os.path.join(CSRC, f)).read()))
    assert {"gate_up_swiglu", "dact_dswiglu_e4m3", "quantize_do_e4m3"} <= names
    w = synth.WORKLOADS[wl]
    work = bench.kernel_work(w, w.T * w.K)
    missing = sorted(names - set(work))
    assert not missing, missing
    for k in names:
        flops, nbytes, moved = work[k]
        assert flops >= 0 and (nbytes > 0 or k == "zero_tail") and moved >= nbytes, k


def test_roofline_follows_the_byte_model():
    """The roofline of the dominant kernel divides the byte model's algorithmic bytes (gathered rows counted
    once per token, bf16 activations) by the launch time: dW gate/up at c2 moves 2Td + 4Pn + 4End."""
    import bench
    w = synth.WORKLOADS["c2"]
    P = w.T * w.K
    work = bench.kernel_work(w, P)
    alg = 2 * w.T * w.d + 4 * P * w.n + 4 * w.E * w.n * w.d
    assert work["dw_gate_up"][1] == alg
    pk = {"hbm_gbs": 6682.8, "bf16_sus": 1737.5, "source": "measured"}
    r = bench.roofline("dw_gate_up", work, 0.1832 * 10, 10, pk)
    assert r["bound"] == "hbm" and abs(r["frac"] - alg / 0.1832e-3 / 1e9 / 6682.8) < 1e-12
    assert abs(r["frac"] - 0.507) < 0.002
