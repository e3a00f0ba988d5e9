#!/usr/bin/env python3
"""Benchmark of the MoE expert-layer hot path (forward + backward) on GB300.

One step = routing, grouping, the grouped GEMMs, the combine and the whole
backward (dX, router gradient, weight gradients) on one batch of synthetic
inputs already resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2] [--impl ours|reference]

Multi-GPU: the path is replicated per GPU (no collective on the data path);
`value` is the work of all ranks over the slowest rank's time ("weak").
The reference arm (--impl reference) times the fp64 CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import resource
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer fwd+bwd TFLOPS & tokens/s (1 GB300), % of dense BF16 peak"
PAGE_A100_TFLOPS_C2 = 18 * 4096 * 8 * 2048 * 512 / 13.14e-3 / 1e12  # grouped GEMM on one A100, c2 workload


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def workload_desc(wl):
    s = f"{wl.name}: T={wl.T} d={wl.d} E={wl.E} n={wl.n} K={wl.K}"
    if wl.bias != "none":
        s += f" bias={wl.bias}"
    if wl.m_tile:
        s += f" token_rounding M_tile={wl.m_tile}"
    if wl.capacity_factor:
        s += f" capacity_dispatch factor={wl.capacity_factor} policy={wl.drop_policy}"
    return s


# ------------------------------------------------------------------------ per-kernel algorithmic work


def kernel_work(wl, P, dW_bytes=2):
    """Per kernel label: (flops, algorithmic bytes, bytes this design moves) of one launch (bf16 = 2 B).

    Algorithmic bytes follow the hot path's byte model: weights read once per launch, a gathered operand
    counted once per unique token row (2Td), every cached activation (H, U, A, Yw, dH, dU, A', dXp) in bf16,
    written once and read once.  The moved bytes count what this design stores and reads instead: H and U in
    fp32 (8Pn instead of 4Pn), the expert-sorted copies of X and dO that the backward GEMMs read (2Pd each
    instead of 2Td) and the bf16 low parts of dH, dU and A' that the weight-gradient GEMMs read.  The grouping
    and the sorted copies (gather_rows) have no place in the byte model (the gathers belong inside the GEMMs'
    loads): their algorithmic bytes are the ones they would move if they were the whole job."""
    T, d, E, n, K = wl.T, wl.d, wl.E, wl.n, wl.K
    same = lambda f, b: (f, b, b)
    dWb = dW_bytes
    return {
        "router_logits": same(2 * T * d * E, 2 * T * d + 2 * d * E + 4 * T * E),
        "topk_softmax": same(0, 4 * T * E + 8 * T * K),
        "permute": same(0, 4 * T * K + 16 * P + (4 * T * E if wl.m_tile else 0)),
        "gate_up_swiglu": (4 * P * d * n, 2 * T * d + 4 * E * n * d + 6 * P * n, 2 * T * d + 4 * E * n * d + 10 * P * n),
        "gate_up_swiglu_e4m3": (4 * P * d * n, T * d + 4 * T + 2 * E * n * d + 8 * E * n + 6 * P * n,
                                T * d + 4 * T + 2 * E * n * d + 8 * E * n + 10 * P * n),
        "quantize_e4m3": same(0, 3 * T * d + 4 * T),
        # block-scaled form: codes of 1 byte plus one scale byte per 32 values
        "quantize_mx": same(0, 3 * T * d + T * d // 32),
        "mx_tile_scales": same(0, 2 * P * d // 32 + 4 * P),  # the gathered rows' scale bytes, read and re-laid
        "quantize_mx_weights": same(0, 3 * E * n * d + E * n * d // 32),  # one weight per launch (outside the step)
        "gate_up_swiglu_mx": (4 * P * d * n, T * d + T * d // 32 + 2 * E * n * d + 2 * E * n * d // 32 + 4 * P * n
                              + P * n + P * n // 32,
                              T * d + T * d // 32 + 2 * E * n * d + 2 * E * n * d // 32 + 8 * P * n + P * n
                              + P * n // 32),
        "down_scale_mx": same(2 * P * d * n, P * n + P * n // 32 + E * d * n + E * d * n // 32 + 2 * P * d),
        # the block-scaled backward: dO per token (gathered codes, counted once per token), W_down^T, H and U,
        # dH, dU, A' (bf16) and the [dH | dU] codes; the dX GEMM on those codes
        "dact_dswiglu_mx": (2 * P * d * n, T * d + T * d // 32 + E * d * n + E * d * n // 32 + 10 * P * n
                            + 2 * P * n + 2 * P * n // 32,
                            P * d + P * d // 32 + E * d * n + E * d * n // 32 + 8 * P * n + 12 * P * n
                            + 2 * P * n + 2 * P * n // 32),
        "dx_gemm_mx": same(4 * P * d * n, 2 * P * n + 2 * P * n // 32 + 2 * E * d * n + 2 * E * d * n // 32
                           + 2 * P * d),
        # block-scaled weight gradients: the four operands quantized along tokens in one launch (dH, dU, A' read
        # as bf16 in the byte model, high and low parts moved; X and dO gathered, counted once per token), then
        # the two varlen-K GEMMs on the codes and their scales (per-expert padding to 128 tokens not counted)
        "quantize_cols_mx": (0, 6 * P * n + 4 * T * d + (3 * n + 2 * d) * P * 33 // 32,
                             12 * P * n + 4 * P * d + (3 * n + 2 * d) * P * 33 // 32),
        "mx_stage_offsets": same(0, 8 * E),
        "dw_gate_up_mx": same(4 * P * d * n, (2 * n + d) * P * 33 // 32 + 2 * dWb * E * n * d),
        "dw_down_mx": same(2 * P * d * n, (n + d) * P * 33 // 32 + dWb * E * d * n),
        "down_scale": same(2 * P * d * n, 2 * P * n + 2 * E * d * n + 2 * P * d),
        "down_scale_e4m3": same(2 * P * d * n, P * n + 4 * P + E * d * n + 4 * E * d + 2 * P * d),
        "quantize_a_e4m3": same(0, 3 * P * n + 4 * P),
        "quantize_hu_e4m3": same(0, 6 * P * n + 4 * P),
        "dx_gemm_e4m3": same(4 * P * d * n, 2 * P * n + 4 * P + 2 * E * n * d + 4 * E * d + 2 * P * d),
        "quantize_do_e4m3": same(0, 3 * T * d + 4 * T),  # dO per token (the sorted-row form, cap < T: 3Pd + 4P)
        "dact_dswiglu_e4m3": (2 * P * d * n, T * d + 4 * T + E * d * n + 4 * E * n + 10 * P * n,
                              P * d + 4 * P + E * d * n + 4 * E * n + 8 * P * n + 12 * P * n),
        "combine": same(0, 2 * P * d + 2 * T * d),
        "gather_rows": same(0, 4 * T * d + 4 * P * d),  # (+ the padding's zero rows, at most 15 per expert)
        "pad_offsets": same(0, 8 * E),
        "zero_tail": same(0, 0),
        "dact_dswiglu": (2 * P * d * n, 2 * T * d + 2 * E * d * n + 10 * P * n,
                         2 * P * d + 2 * E * d * n + 8 * P * n + 12 * P * n),
        "dx_gemm": same(4 * P * d * n, 4 * P * n + 4 * E * n * d + 2 * P * d),
        "wr_transpose": same(0, 4 * d * E),
        "token_backward": same(2 * P * d, 2 * P * d + 2 * T * d + 8 * T * E),
        "dwr_gemm": same(4 * T * d * E, 2 * T * d + 4 * T * E + 4 * d * E),  # dlogits as two bf16 parts
        "dwr_reduce": same(0, 8 * d * E),
        "dw_gate_up": (4 * P * d * n, 2 * T * d + 4 * P * n + 2 * dWb * E * n * d,
                       2 * P * d + 8 * P * n + 2 * dWb * E * n * d),
        "dw_down": (2 * P * d * n, 2 * T * d + 2 * P * n + dWb * E * d * n, 2 * P * d + 4 * P * n + dWb * E * d * n),
    }


def roofline(name, work, ms_total, launches, pk, traffic=None):
    """The kernel against its binding resource: algorithmic flops or bytes per launch over its average
    launch time, as a fraction of the measured peak (sustained bf16 for a kernel timed inside the step)."""
    fl, by, mv = work[name]
    avg_ms = ms_total / max(launches, 1)
    t_tensor = fl / (pk["bf16_sus"] * 1e12)
    t_hbm = by / (pk["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = fl / (avg_ms * 1e-3) / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_sus"], "traffic": traffic,
                "peak_source": f"{pk['source']} (sustained bf16)", "avg_launch_ms": avg_ms,
                "hbm_gbs_of_algorithmic_bytes": by / (avg_ms * 1e-3) / 1e9, "algorithmic_bytes": by,
                "moved_bytes": mv}
    achieved = by / (avg_ms * 1e-3) / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": traffic, "peak_source": pk["source"],
            "avg_launch_ms": avg_ms, "tflops": fl / (avg_ms * 1e-3) / 1e12, "tensor_frac": fl / (avg_ms * 1e-3) / 1e12
            / pk["bf16_sus"], "algorithmic_bytes": by, "moved_bytes": mv,
            "moved_gbs": mv / (avg_ms * 1e-3) / 1e9}


def hbm_stages(wl, P, prof, steps, pk):
    """The memory-bound stages against the measured HBM bandwidth: the route + permute stage as one (router
    logits, top-K, grouping: 2Td + 2dE + 16P + 4TE bytes, plus 4TE for the full scores under Token Rounding),
    the combine (2Pd + 2Td), the backward's per-token reduction (token_backward: 2Pd + 2Td + 8TE) and the sorted
    copies (gather_rows: 4Td + 4Pd, bytes it moves)."""
    T, d, E = wl.T, wl.d, wl.E
    per_step = lambda *names: sum(prof[k][0] for k in names if k in prof) / max(steps, 1)
    stages = {
        "route_permute": (("router_logits", "topk_softmax", "permute"),
                          2 * T * d + 2 * d * E + 16 * P + 4 * T * E + (4 * T * E if wl.m_tile else 0)),
        "combine": (("combine",), 2 * P * d + 2 * T * d),
        "token_backward": (("token_backward",), 2 * P * d + 2 * T * d + 8 * T * E),
        "gather_rows": (("gather_rows",), 4 * T * d + 4 * P * d),
    }
    out = {}
    for name, (kernels, nbytes) in stages.items():
        ms = per_step(*kernels)
        if ms <= 0:
            continue
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"kernels": list(kernels), "bytes": nbytes, "ms_per_step": ms, "gbs": gbs,
                     "frac_of_hbm": gbs / pk["hbm_gbs"]}
    return out


def kernel_table(prof, work, steps, pk):
    """Per kernel label: time per step, share, TFLOP/s, GB/s of algorithmic and of moved bytes, bound."""
    kernels = {}
    tot = max(sum(v[0] for v in prof.values()), 1e-9)
    for k, (kms, kl) in sorted(prof.items(), key=lambda kv: -kv[1][0]):
        if kl == 0:  # a label of the context that this pass did not launch
            continue
        f2, b2, m2 = work.get(k, (0, 0, 0))
        a = max(kms / max(kl, 1), 1e-9)
        kernels[k] = {"ms_per_step": kms / steps, "share": kms / tot,
                      "tflops": f2 / (a * 1e-3) / 1e12 if f2 else None,
                      "gbs_of_algorithmic_bytes": b2 / (a * 1e-3) / 1e9 if b2 else None,
                      "gbs_of_moved_bytes": m2 / (a * 1e-3) / 1e9 if m2 else None,
                      "bound": ("tensor" if f2 / (pk["bf16_sus"] * 1e12) >= b2 / (pk["hbm_gbs"] * 1e9) else "hbm")}
    return kernels


def activation_memory(buf, base=0) -> dict:
    """Device bytes of the layer's state between forward and backward, under the caching rule of the
    SonicMoE page (cache only what the backward needs, no O(T K d) tensor such as Y or the gathered X): what
    the forward keeps for the backward (routing state and the fp32 H and U from which the backward recomputes
    A), the forward-only temporaries (A for the down projection, Yw for the combine), the workspace (the
    backward's scratch, including its expert-sorted copies of X and dO) and the peak allocation of this
    workload (inputs, weights and gradients included; bytes allocated before `base` excluded)."""
    import torch
    nb = lambda *ts: int(sum(t.numel() * t.element_size() for t in ts if t is not None))
    kept = nb(buf.H, buf.U, buf.logits, buf.scores, buf.topk_ids, buf.topk_w, buf.offsets, buf.sorted_tok,
              buf.sorted_w, buf.tok_ptr, buf.tok_pairs)
    T = buf.topk_ids.shape[0]
    return {"kept_for_backward_bytes": kept, "kept_bytes_per_token": kept / T, "cached_o_tkd_tensors": [],
            "forward_temporaries_bytes": nb(buf.A, buf.Yw), "workspace_bytes": nb(buf.ws),
            "peak_allocated_bytes": int(torch.cuda.max_memory_allocated()) - int(base)}


def source_hash() -> str:
    """Hash of the CUDA sources: a recorded ncu traffic figure is used only while it matches."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "varlen_grouped_gemm_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from an ncu capture (profiles/dram_traffic_<workload>.json), or None
    when the kernels have changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_hash") != source_hash():
        return None
    return rec.get("bytes_per_launch", {}).get(kernel)


# Template arguments of the grouped GEMM (BN, stages, epilogue warps, depth, A mode, B mode, grouping,
# epilogue, fp32 out) -> the label the library's profiling hook uses.
_GEMM_LABELS = {
    (1, 1, 0, 1): "gate_up_swiglu", (0, 0, 0, 2): "down_scale", (0, 3, 2, 0): "router_logits",
    (0, 2, 0, 3): "dact_dswiglu", (0, 2, 0, 0): "dx_gemm", (2, 3, 1, 0): "dw_tiled (gate/up, down)",
    (2, 3, 2, 0): "dwr_gemm", (2, 4, 1, 0): "dw_gather_b", (3, 3, 1, 0): "dw_gather_a",
    (1, 1, 0, 4): "gate_up_swiglu_e4m3", (0, 0, 0, 5): "down_scale_e4m3", (0, 0, 0, 6): "dx_gemm_e4m3",
    (0, 0, 0, 7): "dact_dswiglu_e4m3",
}
# the block-scaled form (template flag X_MX = 8)
_MX_GEMM_LABELS = {(1, 1, 0, 1): "gate_up_swiglu_mx", (0, 0, 0, 2): "down_scale_mx", (0, 0, 0, 3): "dact_dswiglu_mx",
                   (0, 0, 0, 0): "dx_gemm_mx", (0, 0, 1, 0): "dw_mx (gate/up, down)"}
_OTHER_LABELS = {
    "topk_softmax_kernel": "topk_softmax", "perm_hist_kernel": "permute", "perm_scan_kernel": "permute",
    "perm_scatter_kernel": "permute", "tr_select_kernel": "permute", "transpose_f32_kernel": "permute",
    "perm_escan_kernel": "permute", "cap_select_kernel": "permute", "slot_offsets_kernel": "permute",
    "perm_fused_kernel": "permute",
    "combine_kernel": "combine",
    "token_backward_kernel": "token_backward", "transpose_bf16_kernel": "wr_transpose",
    "splitk_reduce_kernel": "dwr_reduce", "gather_rows_bulk_kernel": "gather_rows",
    "zero_tail_rows_kernel": "zero_tail", "quantize_rows_e4m3_kernel": "quantize_e4m3",
    "pad_offsets_kernel": "pad_offsets", "quantize_rows_mx_kernel": "quantize_mx",
    "quantize_weight_mx_kernel": "quantize_mx_weights", "mx_tile_scales_kernel": "mx_tile_scales",
    "quantize_cols_mx_kernel": "quantize_cols_mx", "mx_stage_offsets_kernel": "mx_stage_offsets",
}


def _ncu_rows(csv_path):
    import csv
    rows, hdr = [], None
    with open(csv_path) as f:
        for r in csv.reader(f):
            if r and r[0] == "ID":
                hdr = r
            elif hdr and len(r) == len(hdr):
                rows.append(dict(zip(hdr, r)))
    return rows


def _label_of(name: str):
    import re
    m = re.search(r"grouped_gemm_kernel<([^>]*)>", name)
    if m:
        a = [x.strip() for x in m.group(1).split(",")]
        key = (int(a[4]), int(a[5]), int(a[6]), int(a[7]))
        if len(a) > 10 and a[10].isdigit() and int(a[10]) & 8:
            return _MX_GEMM_LABELS.get(key, "grouped_gemm " + m.group(1))
        return _GEMM_LABELS.get(key, "grouped_gemm " + m.group(1))
    for k, v in _OTHER_LABELS.items():
        if k in name:
            return v
    return None


def ncu_traffic(csv_path: str, workload: str) -> dict:
    """Per-launch DRAM bytes (read + write) of one step's kernels from an ncu metrics capture, keyed by
    the profiling hook's labels; the two weight-gradient launches come in the order gate/up, down."""
    per, order = {}, []
    for r in _ncu_rows(csv_path):
        key = (r["ID"], r["Kernel Name"])
        if key not in per:
            per[key] = {}
            order.append(key)
        per[key][r["Metric Name"]] = float(r["Metric Value"].replace(",", ""))
    out, launches, dw_seen = {}, {}, 0
    for key in order:
        label = _label_of(key[1])
        if label is None:
            continue
        if label.startswith("dw_tiled") or label.startswith("dw_mx"):  # every step: dW gate/up, then dW down
            sfx = "_mx" if label.startswith("dw_mx") else ""
            label = ("dw_gate_up" if dw_seen % 2 == 0 else "dw_down") + sfx
            dw_seen += 1
        m = per[key]
        b = m.get("dram__bytes_read.sum", 0.0) + m.get("dram__bytes_write.sum", 0.0)
        out[label] = out.get(label, 0.0) + b
        if "grouped_gemm_kernel" in key[1]:
            launches[label] = launches.get(label, 0) + 1
    # a GEMM label is averaged over its launches; every other label over the captured steps (one launch of
    # the gate/up GEMM per step), so that the grouping's kernels add up to one entry-point launch
    steps = max(launches.get("gate_up_swiglu", 1), 1)
    out = {k: v / (launches[k] if k in launches else steps) for k, v in out.items()}
    return {"workload": workload, "source_hash": source_hash(), "bytes_per_launch": out}


def ncu_launch_summary(csv_path: str) -> str:
    """Markdown table of an ncu `--metrics gpu__time_duration.sum --csv` launch list: per kernel of this
    library, its launches, total device time and share (other kernels, e.g. torch fills, are listed apart)."""
    import csv
    rows, hdr = [], None
    with open(csv_path) as f:
        for r in csv.reader(f):
            if r and r[0] == "ID":
                hdr = r
            elif hdr and len(r) == len(hdr):
                rows.append(dict(zip(hdr, r)))
    agg, other = {}, {}
    for r in rows:
        name = r["Kernel Name"]
        ns = float(r["Metric Value"].replace(",", ""))
        label = _label_of(name)  # the block-scaled GEMMs by their flag, the others by their modes
        tgt = agg if label else other
        key = label or name.split("(")[0][:60]
        c, t = tgt.get(key, (0, 0.0))
        tgt[key] = (c + 1, t + ns)
    total = sum(t for _, t in agg.values())
    out = ["| kernel | launches | total (us) | share of this library's time |", "|---|---|---|---|"]
    for k, (c, t) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        out.append(f"| {k} | {c} | {t / 1e3:.1f} | {100 * t / total:.1f}% |")
    out.append("")
    out.append("Other kernels in the capture (input setup, L2 flush): " +
               ", ".join(f"{k} x{c}" for k, (c, t) in sorted(other.items(), key=lambda kv: -kv[1][1])))
    return "\n".join(out)


# ------------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                maxs.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": float(np.median(sms)), "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------------ the oracle as CPU baseline


def oracle_sample(wl, budget_s: float, max_experts: int | None = None):
    """Time the fp64 oracle (forward + backward, loop over experts) on the first experts of the
    workload until `budget_s` of wall time is spent.  Returns flops done, seconds, experts, cores."""
    from oracle import moe_oracle as mo
    X = synth.make_x(wl)
    W_r = synth.make_router(wl)
    bias = synth.make_bias(wl)
    dO = synth.make_dout(wl)
    ru0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    L = mo.router_logits(X, W_r, bias)
    cap_c = mo.expert_capacity(wl.T, wl.E, wl.K, wl.capacity_factor) if wl.capacity_factor else 0
    routing = mo.route_discrete(L, wl.K, wl.m_tile, scores=mo.softmax(L).astype(np.float32) if wl.m_tile else None,
                                capacity=cap_c, policy=wl.drop_policy)
    w_full = mo.combine_weights(L, routing.topk_ids)
    Xf = mo.bf16_bits_to_f64(X)
    dOf = mo.bf16_bits_to_f64(dO)
    flops = 2 * wl.T * wl.d * wl.E
    experts = 0
    for e in range(wl.E):
        if max_experts is not None and experts >= max_experts:
            break
        if time.perf_counter() - t0 > budget_s and experts > 0:
            break
        rows = routing.rows_of(e)
        experts += 1
        if len(rows) == 0:
            continue
        Wg = synth.make_w_gate(wl, [e])[0]
        Wu = synth.make_w_up(wl, [e])[0]
        Wd = synth.make_w_down(wl, [e])[0]
        mo.expert_block_backward(Xf[rows], dOf[rows], w_full[rows, e], Wg, Wu, Wd)
        flops += 18 * len(rows) * wl.d * wl.n
    wall = time.perf_counter() - t0
    ru1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu = (ru1.ru_utime - ru0.ru_utime) + (ru1.ru_stime - ru0.ru_stime)
    return dict(flops=flops, seconds=wall, experts=experts, cores=round(cpu / max(wall, 1e-9), 1),
                host_cpus=os.cpu_count())


# ------------------------------------------------------------------------ replicas (N > 1)
# One process per GPU, each a full replica of the layer on its own batch (no data-path collective):
# the job's time is the slowest rank's and its throughput all ranks' work over that time.


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, ms_per_step: float) -> float:
    """Units per second of the whole job: every rank processed units_per_rank in the slowest rank's time."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    wl = synth.WORKLOADS[args.workload]
    # each step is a bounded sample so that the whole run stays near two minutes
    budget = min(8.0, max(0.5, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(wl, budget_s=0.5, max_experts=1)
    flops, secs, experts, cores = 0, 0.0, 0, 0.0
    for _ in range(args.steps):
        r = oracle_sample(wl, budget_s=budget)
        flops += r["flops"]
        secs += r["seconds"]
        experts = r["experts"]
        cores = r["cores"]
    value = flops / secs / 1e12
    sample = (f"fp64 oracle fwd+bwd (loop over experts) on the first {experts} of {wl.E} experts with all their "
              f"routed tokens, plus the full router, per step ({budget:.0f} s budget)")
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(wl)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "host_cpus": os.cpu_count()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------ our arm


def measure_e4m3(vgg, ctx, wl, X, W_r, bias, W_gate, W_up, W_down, dO, buf, flush, stream, steps, warmup, pk):
    """The e4m3 forms against bf16 on the same inputs, eager calls: the forward (e4m3 gate/up; also the e4m3
    down projection; also forward only), and a training step (e4m3 forward GEMMs, and the e4m3 dSwiGLU and dX GEMMs
    in the backward).  Weights are quantized once, outside the timed steps; activations inside every step.  Each
    arm is timed with CUDA events (L2 flushed between steps), then run again with the library's per-launch
    events for the per-kernel times."""
    import torch
    b8 = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16,
                              device=X.device, capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy,
                              e4m3=True)
    w8 = vgg.E4m3Weights.quantize(ctx, W_gate, W_up)
    w8d = vgg.E4m3Weights.quantize(ctx, W_gate, W_up, W_down, backward=True)
    bmx = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16,
                               device=X.device, capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy,
                               mx=True)
    wmx = vgg.MxWeights.quantize(ctx, W_gate, W_up, W_down, backward=True)

    def mx_step():
        vgg.forward_mx(ctx, X, W_r, bias, wmx, bmx)
        vgg.backward_mx(ctx, dO, X, W_r, W_gate, W_up, W_down, wmx, bmx)

    def mx_step_mx_dw():  # the weight gradients block-scaled too
        vgg.forward_mx(ctx, X, W_r, bias, wmx, bmx)
        vgg.backward_mx(ctx, dO, X, W_r, W_gate, W_up, W_down, wmx, bmx, dw=True)

    def e4m3_step():
        vgg.forward_e4m3(ctx, X, W_r, bias, w8d, None, b8)
        vgg.backward_e4m3(ctx, dO, X, W_r, W_gate, W_up, W_down, w8d, b8)

    runs = {"bf16": lambda: vgg.forward(ctx, X, W_r, bias, W_gate, W_up, W_down, buf),
            "e4m3": lambda: vgg.forward_e4m3(ctx, X, W_r, bias, w8, W_down, b8),
            # forward only (inference): H and U, kept for the backward, are not written
            "bf16_infer": lambda: vgg.forward(ctx, X, W_r, bias, W_gate, W_up, W_down, buf, cache=False),
            "e4m3_infer": lambda: vgg.forward_e4m3(ctx, X, W_r, bias, w8, W_down, b8, cache=False),
            # the e4m3 down projection as well
            "e4m3_down8": lambda: vgg.forward_e4m3(ctx, X, W_r, bias, w8d, None, b8),
            "e4m3_down8_infer": lambda: vgg.forward_e4m3(ctx, X, W_r, bias, w8d, None, b8, cache=False),
            # the block-scaled (1 x 32) form of both forward GEMMs, A quantized in the gate/up epilogue
            "mx": lambda: vgg.forward_mx(ctx, X, W_r, bias, wmx, bmx),
            "mx_infer": lambda: vgg.forward_mx(ctx, X, W_r, bias, wmx, bmx, cache=False),
            "mx_step": mx_step,
            "mx_step_mx_dw": mx_step_mx_dw,
            # training steps
            "bf16_step": lambda: vgg.forward_backward(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf),
            "e4m3_step": e4m3_step}
    out = {}
    for name, fn in runs.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        vgg.moe_profile_enable(ctx, True)
        vgg.moe_profile_read(ctx)
        for i in range(steps):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        prof = vgg.moe_profile_read(ctx)
        vgg.moe_profile_enable(ctx, False)
        out[name] = (ms, prof)
    rc, code = vgg.moe_get_error(ctx)
    if rc != 0:
        raise RuntimeError(f"device error in the e4m3 arms: status {rc}, code {code}")
    P = int(b8.P.item())
    fl = 4 * P * wl.d * wl.n
    per = lambda name, k: out[name][1][k][0] / out[name][1][k][1]
    t8, t16 = per("e4m3", "gate_up_swiglu_e4m3"), per("bf16", "gate_up_swiglu")
    qx = out["e4m3"][1].get("quantize_e4m3", (0.0, 1))
    peak8 = 2 * pk["bf16"]
    dn, dn16 = per("e4m3_down8", "down_scale_e4m3"), per("bf16", "down_scale")
    dx8, dx16 = per("e4m3_step", "dx_gemm_e4m3"), per("bf16_step", "dx_gemm")
    qa = out["e4m3_down8"][1].get("quantize_a_e4m3", (0.0, 1))
    qh = out["e4m3_step"][1].get("quantize_hu_e4m3", (0.0, 1))
    da8, da16 = per("e4m3_step", "dact_dswiglu_e4m3"), per("bf16_step", "dact_dswiglu")
    qd = out["e4m3_step"][1].get("quantize_do_e4m3", (0.0, 1))
    fl_dn = 2 * P * wl.d * wl.n
    step_fl = wl.flops_fwd_bwd(P)
    gmx, dmx = per("mx", "gate_up_swiglu_mx"), per("mx", "down_scale_mx")
    amx, xmx = per("mx_step", "dact_dswiglu_mx"), per("mx_step", "dx_gemm_mx")
    qmx = out["mx"][1].get("quantize_mx", (0.0, 1))
    wgmx, wdmx = per("mx_step_mx_dw", "dw_gate_up_mx"), per("mx_step_mx_dw", "dw_down_mx")
    qcmx = per("mx_step_mx_dw", "quantize_cols_mx")
    del b8, w8, w8d, bmx, wmx
    return {"forward_ms": out["e4m3"][0], "bf16_forward_ms": out["bf16"][0],
            "forward_e4m3_down_ms": out["e4m3_down8"][0],
            "bf16_forward_infer_ms": out["bf16_infer"][0], "forward_infer_ms": out["e4m3_infer"][0],
            "forward_e4m3_down_infer_ms": out["e4m3_down8_infer"][0],
            "train_step_ms": out["e4m3_step"][0], "bf16_train_step_ms": out["bf16_step"][0],
            "train_step_tflops": step_fl / (out["e4m3_step"][0] * 1e-3) / 1e12,
            "gate_up_ms": t8, "bf16_gate_up_ms": t16, "quantize_x_ms": qx[0] / max(qx[1], 1),
            "down_ms": dn, "bf16_down_ms": dn16, "quantize_a_ms": qa[0] / max(qa[1], 1),
            "dx_ms": dx8, "bf16_dx_ms": dx16, "quantize_hu_ms": qh[0] / max(qh[1], 1),
            "dact_ms": da8, "bf16_dact_ms": da16, "quantize_do_ms": qd[0] / max(qd[1], 1),
            "gate_up_tflops": fl / (t8 * 1e-3) / 1e12, "bf16_gate_up_tflops": fl / (t16 * 1e-3) / 1e12,
            "down_tflops": fl_dn / (dn * 1e-3) / 1e12, "dx_tflops": fl / (dx8 * 1e-3) / 1e12,
            "dact_tflops": fl_dn / (da8 * 1e-3) / 1e12,
            "gate_up_peak_tflops": peak8, "gate_up_frac": fl / (t8 * 1e-3) / 1e12 / peak8,
            "block_scaled": {
                "forward_ms": out["mx"][0], "forward_infer_ms": out["mx_infer"][0],
                "gate_up_ms": gmx, "down_ms": dmx, "quantize_x_ms": qmx[0] / max(qmx[1], 1),
                "gate_up_tflops": fl / (gmx * 1e-3) / 1e12, "down_tflops": fl_dn / (dmx * 1e-3) / 1e12,
                "gate_up_frac": fl / (gmx * 1e-3) / 1e12 / peak8,
                "train_step_ms": out["mx_step"][0],
                "train_step_tflops": step_fl / (out["mx_step"][0] * 1e-3) / 1e12,
                "dact_ms": amx, "dx_ms": xmx, "dact_tflops": fl_dn / (amx * 1e-3) / 1e12,
                "dx_tflops": fl / (xmx * 1e-3) / 1e12,
                "train_step_mx_dw_ms": out["mx_step_mx_dw"][0],
                "mx_dw_gate_up_ms": wgmx, "mx_dw_down_ms": wdmx, "mx_dw_quantize_cols_ms": qcmx,
                "mx_dw_tflops": (fl + fl_dn) / ((wgmx + wdmx) * 1e-3) / 1e12,
                "recipe": "e4m3 codes with one power-of-two (UE8M0) scale per 32 values along the reduction "
                          "dimension of every operand row (kind::mxf8f6f4 UMMA); A quantized in the gate/up "
                          "epilogue, [dH|dU] in the dSwiGLU epilogue; 192-column tiles; the weight gradients (on "
                          "dH, dU, A' rounded once to bf16) and the router stay bf16; train_step_mx_dw_ms: the "
                          "same step with block-scaled weight "
                          "gradients (operands in blocks of 32 tokens of one expert, one quantizing launch)"},
            "peak_source": f"{pk['source']} bf16 burst x 2 (nominal e4m3/bf16 dense ratio 4.5/2.25)",
            "recipe": "e4m3 operands with one fp32 scale per row: X per token, A, dO and [dH|dU] per pair, weights per "
                      "output channel of each GEMM; fp32 accumulation; dW (on dH, dU, A' rounded once to bf16) and the "
                      "router stay bf16",
            "steps": steps, "l2": "flushed between steps", "launch": "eager calls"}


def measure_workload(vgg, ctx, name, steps, warmup, pk, dev, flush, stream):
    """One more workload's step on its own inputs: ms, TFLOP/s, tokens/s, the dominant kernel against its
    roofline, per-kernel shares and activation memory.  X, W_r, the bias and dO come from the seeded
    generator (they decide the routing); the expert weights are drawn on the device (torch's generator,
    seed 0, standard deviation 1/sqrt(fan_in)), which keeps the set-up of the largest workloads short: the
    step's time does not depend on their values.  The step runs as one CUDA graph, L2 flushed between steps."""
    import torch
    wl = synth.WORKLOADS[name]
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    X, dO, W_r = to_dev(synth.make_x(wl)), to_dev(synth.make_dout(wl)), to_dev(synth.make_router(wl))
    bias_h = synth.make_bias(wl)
    bias = None if bias_h is None else torch.from_numpy(bias_h).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    draw = lambda shape, fan_in: torch.randn(shape, generator=g, device=dev, dtype=torch.bfloat16).mul_(fan_in ** -0.5)
    W_gate = draw((wl.E, wl.n, wl.d), wl.d)
    W_up = draw((wl.E, wl.n, wl.d), wl.d)
    W_down = draw((wl.E, wl.d, wl.n), wl.n)
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16,
                               device=dev, capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy)
    for _ in range(warmup):
        vgg.forward_backward(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf)
    graph = vgg.StepGraph(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf)
    graph.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        evs[i][0].record(stream)
        graph.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    vgg.moe_profile_enable(ctx, True)
    vgg.moe_profile_read(ctx)
    for i in range(steps):
        flush.zero_()
        vgg.forward_backward(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf)
    torch.cuda.synchronize()
    prof = vgg.moe_profile_read(ctx)
    vgg.moe_profile_enable(ctx, False)
    rc, code = vgg.moe_get_error(ctx)
    if rc != 0:
        raise RuntimeError(f"device error in workload {name}: status {rc}, code {code}")
    P = int(buf.P.item())
    counts = buf.counts.cpu().numpy()
    work = kernel_work(wl, P)
    dname, (dms, dl) = max(prof.items(), key=lambda kv: kv[1][0])
    flops = wl.flops_fwd_bwd(P)
    out = {"workload": workload_desc(wl), "ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12,
           "pct_of_peak_bf16": 100 * flops / (ms * 1e-3) / 1e12 / pk["bf16_sus"], "tokens_per_s": wl.T / (ms * 1e-3),
           "pairs": P, "empty_experts": int((counts == 0).sum()), "max_rows_per_expert": int(counts.max()),
           "roofline": roofline(dname, work, dms, dl, pk, recorded_traffic(wl.name, dname)),
           "hbm_stages": hbm_stages(wl, P, prof, steps, pk),
           "kernels": {k: {"ms_per_step": v["ms_per_step"], "share": round(v["share"], 4)}
                       for k, v in kernel_table(prof, work, steps, pk).items()},
           "activation_memory": activation_memory(buf, base), "steps": steps,
           "expert_weights": "drawn on the device (torch generator, seed 0)"}
    del graph, buf, X, dO, W_r, bias, W_gate, W_up, W_down
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import varlen_grouped_gemm_gb300 as vgg
    from varlen_grouped_gemm_gb300 import build as lib_build

    torch.cuda.set_device(local_rank)
    if not os.path.exists(vgg.LIB_PATH):
        lib_build.build()
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
    wl = synth.WORKLOADS[args.workload]
    pk = peaks()
    dev = torch.device("cuda", local_rank)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    X_h, dO_h = synth.make_x(wl), synth.make_dout(wl)
    X = to_dev(X_h)
    dO = to_dev(dO_h)
    W_r = to_dev(synth.make_router(wl))
    bias_h = synth.make_bias(wl)
    bias = None if bias_h is None else torch.from_numpy(bias_h).to(dev)
    W_gate = to_dev(synth.make_w_gate(wl))
    W_up = to_dev(synth.make_w_up(wl))
    W_down = to_dev(synth.make_w_down(wl))
    ctx = vgg.Context(local_rank)
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16,
                               device=dev, capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def eager_step():
        vgg.forward_backward(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf)

    for _ in range(args.warmup):
        eager_step()
    rc, code = vgg.moe_get_error(ctx)
    if rc != 0:
        raise RuntimeError(f"device error after warm-up: status {rc}, code {code}")
    P = int(buf.P.item())
    counts = buf.counts.cpu().numpy()
    # the step as a CUDA graph (the library's host work done once, at capture), unless --no-graph
    graph = None if args.no_graph else vgg.StepGraph(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf)
    step = graph.replay if graph is not None else eager_step

    # timed region: K steps, per-step events, L2 flushed between steps outside the events
    clocks = ClockSampler(local_rank)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # clock samples: a 0.5 s busy pre-roll of the same step right before the timed region, and the region
    clocks.start()
    t_end = time.perf_counter() + (0.0 if args.profile_run else 0.5)
    while time.perf_counter() < t_end:
        step()
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    rc, code = vgg.moe_get_error(ctx)
    if rc != 0:
        raise RuntimeError(f"device error in timed region: status {rc}, code {code}")
    # per-kernel times: the same K steps again, eager, with the library's per-launch events
    vgg.moe_profile_enable(ctx, True)
    vgg.moe_profile_read(ctx)
    for i in range(args.steps):
        flush.zero_()
        eager_step()
    torch.cuda.synchronize()
    prof = vgg.moe_profile_read(ctx)
    vgg.moe_profile_enable(ctx, False)
    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)
    ms = total_ms / args.steps
    flops = wl.flops_fwd_bwd(P)
    tflops = whole_job_rate(world, flops, ms) / 1e12
    tokens_s = whole_job_rate(world, wl.T, ms)

    # dominant kernel and its roofline: the binding resource of its algorithmic work
    work = kernel_work(wl, P)
    dname, (dms, dlaunch) = max(prof.items(), key=lambda kv: kv[1][0])
    roof = roofline(dname, work, dms, dlaunch, pk, recorded_traffic(wl.name, dname))
    kernels = kernel_table(prof, work, args.steps, pk)
    # the grouping's kernels: one cooperative launch per grouping (token rounding and the capacity dispatch
    # group twice, with a select kernel and a transpose or slot-offset kernel between)
    launches_per_label = {"permute": (4 if (wl.m_tile or wl.capacity_factor) else 1)}
    gpu_launches = int(sum(cnt * launches_per_label.get(k, 1) for k, (_, cnt) in prof.items()))

    # end to end through the public API with host buffers: H2D of X and dO, D2H of O and dX per step
    e2e = None
    if not args.no_e2e:
        X_pin = torch.from_numpy(X_h.view(np.int16)).view(torch.bfloat16).pin_memory()
        dO_pin = torch.from_numpy(dO_h.view(np.int16)).view(torch.bfloat16).pin_memory()
        O_pin = torch.empty((wl.T, wl.d), dtype=torch.bfloat16).pin_memory()
        dX_pin = torch.empty((wl.T, wl.d), dtype=torch.bfloat16).pin_memory()
        # serial: each step's copies and the step one after another on one stream, L2 flushed between steps
        ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            ee[i][0].record(stream)
            X.copy_(X_pin, non_blocking=True)
            dO.copy_(dO_pin, non_blocking=True)
            step()
            O_pin.copy_(buf.O, non_blocking=True)
            dX_pin.copy_(buf.dX, non_blocking=True)
            ee[i][1].record(stream)
        torch.cuda.synchronize()
        serial_ms = max_over_ranks(float(sum(a.elapsed_time(b) for a, b in ee)), dist, dev) / args.steps
        # pipelined, as a training loop with a prefetching loader runs it: two sets of device buffers; a copy
        # stream brings step i+1's inputs in and takes step i's results out while the compute stream runs
        # step i.  The copy stream is in order, so step i+1's inputs land in a slot only after the results of
        # step i-1 (the slot's previous user) were read out, and step i+1 starts only after its inputs landed.
        buf2 = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16,
                                    device=dev, capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy)
        slots = [(X, dO, buf), (torch.empty_like(X), torch.empty_like(dO), buf2)]
        cs = torch.cuda.Stream(device=dev)
        h2d = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        for _ in range(2):  # warm-up of the second buffer set
            vgg.forward_backward(ctx, slots[1][0], W_r, bias, W_gate, W_up, W_down, slots[1][1], buf2, stream)
        torch.cuda.synchronize()
        if graph is not None:
            graph2 = vgg.StepGraph(ctx, slots[1][0], W_r, bias, W_gate, W_up, W_down, slots[1][1], buf2)
            runs = [graph.replay, graph2.replay]
        else:
            runs = [lambda i=i: vgg.forward_backward(ctx, slots[i][0], W_r, bias, W_gate, W_up, W_down, slots[i][1],
                                                     slots[i][2], stream) for i in range(2)]
        if dist is not None:
            dist.barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(cs)
        with torch.cuda.stream(cs):
            X.copy_(X_pin, non_blocking=True)
            dO.copy_(dO_pin, non_blocking=True)
            h2d[0].record(cs)
        for i in range(args.steps):
            Xi, dOi, bi = slots[i % 2]
            stream.wait_event(h2d[i % 2])
            runs[i % 2]()
            done[i % 2].record(stream)
            with torch.cuda.stream(cs):
                if i + 1 < args.steps:
                    Xn, dOn, _ = slots[(i + 1) % 2]
                    Xn.copy_(X_pin, non_blocking=True)
                    dOn.copy_(dO_pin, non_blocking=True)
                    h2d[(i + 1) % 2].record(cs)
                cs.wait_event(done[i % 2])
                O_pin.copy_(bi.O, non_blocking=True)
                dX_pin.copy_(bi.dX, non_blocking=True)
        t1.record(cs)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(t0.elapsed_time(t1), dist, dev) / args.steps
        del buf2, slots, runs
        e2e = {"value": whole_job_rate(world, flops, e_ms) / 1e12, "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": 2 * 2 * wl.T * wl.d, "d2h_bytes_per_step": 2 * 2 * wl.T * wl.d,
               "mode": "pipelined: step i+1's H2D and step i's D2H on a copy stream during step i "
                       "(L2 not flushed; per-step working set larger than L2)",
               "serial_ms_per_step": serial_ms,
               "serial_value": whole_job_rate(world, flops, serial_ms) / 1e12}

    e4m3 = None
    if not args.no_e4m3:
        e4m3 = measure_e4m3(vgg, ctx, wl, X, W_r, bias, W_gate, W_up, W_down, dO, buf, flush, stream,
                            max(3, min(args.steps, 20)), max(3, args.warmup), pk)

    per_workload = None
    if world == 1 and args.per_workload:
        per_workload = {}
        for name in [w for w in args.per_workload.split(",") if w and w != wl.name]:
            per_workload[name] = measure_workload(vgg, ctx, name, max(3, min(args.steps, 10)), 3, pk, dev, flush,
                                                  stream)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        r = oracle_sample(wl, budget_s=float(os.environ.get("VGG_CPU_BASELINE_SECONDS", "15")))
        cpu = {"value": r["flops"] / r["seconds"] / 1e12, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd on the first {r['experts']} of {wl.E} experts with all their routed "
                         f"tokens, plus the full router ({r['seconds']:.1f} s)",
               "host_cpus": r["host_cpus"]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": tflops / world / PAGE_A100_TFLOPS_C2 if wl.name == "c2" else None,
            "dtype": "bf16", "data": "synthetic (seeded splitmix64 + Box-Muller, shapes of the workload)",
            "config": {"workload": workload_desc(wl), "pairs": P, "kept_pairs": int(counts.sum()),
                       "empty_experts": int((counts == 0).sum()),
                       "max_rows_per_expert": int(counts.max()), "dW_dtype": "bf16",
                       "l2": "flushed between steps (256 MB write, outside the per-step events)",
                       "launch": ("eager calls" if graph is None else
                                  f"the step's {gpu_launches // max(args.steps, 1)} launches as one CUDA graph"),
                       "clock_samples": "nvidia-smi every 50 ms over a 0.5 s busy pre-roll of the same step and the timed region",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "tokens_per_s": tokens_s, "pct_of_peak_bf16": 100 * tflops / world / pk["bf16_sus"],
            "peak_bf16_tflops": pk["bf16_sus"], "peak_source": pk["source"] + " sustained",
            "step_ms_min": min(step_ms), "step_ms_median": float(np.median(step_ms)),
            "roofline": roof, "hbm_stages": hbm_stages(wl, P, prof, args.steps, pk), "kernels": kernels,
            "gpu_launches": gpu_launches,
            "activation_memory": activation_memory(buf),
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clk, "e4m3_forward": e4m3,
            "per_workload": per_workload,
        }
        if wl.name == "c2":
            line["baseline_note"] = ("vs_baseline divides by the pages' grouped-GEMM figure for this workload "
                                     "(13.14 ms fwd+bwd = 47.1 TFLOP/s on one A100): context, another machine")
        print(json.dumps(line), flush=True)
    return 0


def run_mx_profile(args) -> int:
    """Two iterations of the block-scaled forward and backward (``--mx-dw``: the block-scaled weight gradients too)
    on the workload's seeded X, W_r, bias and dO, with expert weights drawn on the device as ``measure_workload``
    draws them: the program an ncu capture of the block-scaled kernels runs.  Prints one JSON line."""
    import torch
    import varlen_grouped_gemm_gb300 as vgg
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda:0")

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    X, dO, W_r = to_dev(synth.make_x(wl)), to_dev(synth.make_dout(wl)), to_dev(synth.make_router(wl))
    bias_h = synth.make_bias(wl)
    bias = None if bias_h is None else torch.from_numpy(bias_h).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    draw = lambda shape, fan_in: torch.randn(shape, generator=g, device=dev, dtype=torch.bfloat16).mul_(fan_in ** -0.5)
    W_gate, W_up, W_down = draw((wl.E, wl.n, wl.d), wl.d), draw((wl.E, wl.n, wl.d), wl.d), draw((wl.E, wl.d, wl.n), wl.n)
    ctx = vgg.Context(0)
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16,
                               device=dev, capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy, mx=True)
    w = vgg.MxWeights.quantize(ctx, W_gate, W_up, W_down, backward=True)
    for _ in range(2):
        vgg.forward_mx(ctx, X, W_r, bias, w, buf)
        vgg.backward_mx(ctx, dO, X, W_r, W_gate, W_up, W_down, w, buf, dw=args.mx_dw)
    torch.cuda.synchronize()
    rc, code = vgg.moe_get_error(ctx)
    if rc != 0:
        raise RuntimeError(f"device error in the block-scaled run: status {rc}, code {code}")
    print(json.dumps({"mx_profile_run": wl.name, "mx_dw": bool(args.mx_dw),
                      "device_gib": torch.cuda.max_memory_allocated(dev) / 2 ** 30}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="c2", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e4m3", action="store_true", help="skip the e4m3 gate/up forward measurement")
    ap.add_argument("--no-graph", action="store_true", help="time eager calls instead of the captured step graph")
    ap.add_argument("--per-workload", default="c3,c4,c5,c5_plain",
                    help="comma-separated further workloads timed after the main one (empty: none)")
    ap.add_argument("--ncu-summary", metavar="CSV", help="print a markdown summary of an ncu launch list and exit")
    ap.add_argument("--ncu-traffic", metavar="CSV", help="print per-kernel DRAM bytes of an ncu capture as JSON and exit")
    ap.add_argument("--mx-profile-run", action="store_true",
                    help="two iterations of the block-scaled forward and backward (for an ncu capture) and exit")
    ap.add_argument("--mx-dw", action="store_true", help="with --mx-profile-run: block-scaled weight gradients too")
    ap.add_argument("--profile-run", action="store_true",
                    help="for runs under ncu: no clock pre-roll, no end-to-end pass, no CPU baseline, no e4m3 forward, "
                         "eager launches")
    args = ap.parse_args()
    if args.profile_run:
        args.no_e2e = True
        args.no_cpu_baseline = True
        args.no_e4m3 = True
        args.no_graph = True
        args.per_workload = ""
    if args.ncu_summary:
        print(ncu_launch_summary(args.ncu_summary))
        return 0
    if args.ncu_traffic:
        print(json.dumps(ncu_traffic(args.ncu_traffic, args.workload), indent=1))
        return 0
    if args.mx_profile_run:
        return run_mx_profile(args)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
