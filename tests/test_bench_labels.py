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


def _write_capture(path, launches, metrics):
    """An ncu --csv capture: one row per (launch, metric) in ncu's column layout."""
    import csv
    with open(path, "w", newline="") as f:
        w = csv.writer(f)
        w.writerow(["ID", "Process ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value"])
        for i, name in enumerate(launches):
            for m, v in metrics(i, name).items():
                w.writerow([str(i), "1", name, m, "byte", f"{v:,.0f}"])


_DW = "void vgg::grouped_gemm_kernel<256, 3, 4, 1, 2, 3, 1, 0, false, 1, 1>(vgg::GemmParams, vgg::Maps)"
_DW_MX = "void vgg::grouped_gemm_kernel<192, 4, 4, 1, 0, 0, 1, 0, false, 1, 8>(vgg::GemmParams, vgg::Maps)"
_GU = "void vgg::grouped_gemm_kernel<256, 4, 4, 1, 1, 1, 0, 1, false, 2, 0>(vgg::GemmParams, vgg::Maps)"
_GU_MX = "void vgg::grouped_gemm_kernel<192, 4, 4, 1, 1, 1, 0, 1, false, 2, 8>(vgg::GemmParams, vgg::Maps)"


def test_traffic_parser_alternates_weight_gradient_launches(tmp_path):
    """Two captured steps: the gate/up GEMM, the grouping's two kernels, then dW gate/up and dW down (one template);
    per-launch bytes average a GEMM over its launches and every other label over the steps, and the two
    weight-gradient launches of a step are told apart by their order (bf16 and block-scaled alike)."""
    import bench
    step = [_GU, "vgg::perm_hist_kernel(int)", "vgg::perm_scatter_kernel(int)", _DW, _DW, _DW_MX, _DW_MX]
    nbytes = {_GU: 700, "vgg::perm_hist_kernel(int)": 3, "vgg::perm_scatter_kernel(int)": 5, _DW: None, _DW_MX: None}
    dw_order = {3: 600, 4: 400, 5: 300, 6: 100, 10: 620, 11: 420, 12: 320, 13: 120}
    path = str(tmp_path / "traffic.csv")
    _write_capture(path, step + step + ["void at::vectorized_elementwise_kernel<4>(int)"],
                   lambda i, name: {"dram__bytes_read.sum": (dw_order[i] if nbytes.get(name, 1) is None
                                                             else nbytes.get(name, 9)) * 1e6,
                                    "dram__bytes_write.sum": 0})
    rec = bench.ncu_traffic(path, "c2")["bytes_per_launch"]
    assert rec["gate_up_swiglu"] == 700e6
    assert rec["permute"] == 8e6  # both grouping kernels of a step, per step
    assert rec["dw_gate_up"] == 610e6 and rec["dw_down"] == 410e6
    assert rec["dw_gate_up_mx"] == 310e6 and rec["dw_down_mx"] == 110e6
    assert set(rec) == {"gate_up_swiglu", "permute", "dw_gate_up", "dw_down", "dw_gate_up_mx", "dw_down_mx"}


def test_launch_summary_labels_block_scaled_kernels_apart(tmp_path):
    """The launch-list summary labels a block-scaled GEMM by its flag, not as the bf16 GEMM of the same modes, and
    lists kernels outside the library apart."""
    import bench
    path = str(tmp_path / "launches.csv")
    _write_capture(path, [_GU, _GU, _GU_MX, "void at::vectorized_elementwise_kernel<4>(int)"],
                   lambda i, name: {"gpu__time_duration.sum": 1000.0 * (i + 1)})
    md = bench.ncu_launch_summary(path)
    assert "| gate_up_swiglu | 2 | 3.0 | 50.0% |" in md
    assert "| gate_up_swiglu_mx | 1 | 3.0 | 50.0% |" in md
    assert "Other kernels in the capture" in md and "at::vectorized_elementwise_kernel" in md
