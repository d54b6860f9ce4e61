"""Throughput of the fused CG tensor-product convolution (edges/s, forward + backward).

Headline workload (the JSON line's ``value``): the NequIP-like convolution --
10,000 nodes, 32 in-edges per node (320,000 edges), in1 = 32x(0e,1o,2e,3o),
SH l<=3, uvu with all 34 parity-allowed paths (l3 <= 3), FP32.  One step =
cgtp_conv_forward + cgtp_conv_backward over the whole graph (graph and plan are
built once, outside the timed region).

The same line carries ``per_config``: every other benchmark workload (tiny,
MACE-like FP32 and FP64, high-L batched, uvw radial with its peak device memory)
timed the same way, each with its own roofline.  ``--config`` times one workload
as the headline instead (tiny|nequip|mace|mace64|highl|uvw|uvw_edge|mixed|
nequip_bf16|nequip_sh).

Roofline model (FLOPs written out in ``model_flops``): FLOPs count the CG
nonzeros -- per edge and path 2 nnz(C) for C.Y, mul * 2 nnz_{m1,m3}(C) for the
contraction, mul * (2 l3 + 1) for the weight product, plus d_out per edge for
the receiver sum; backward = 3x forward; bytes = every input read once plus
every output written once.  Peaks are measured here: FP32 / FP64 FMA throughput
and L2 / HBM read bandwidth with the library's own measurement kernels
(cgtp_measure_fma / cgtp_measure_read), HBM copy bandwidth and bf16 tensor
throughput from MEASURED_PEAKS.json.

``e2e`` repeats the headline step through the public API with the step's
inputs copied from pinned host memory and every result copied back inside the
timed region (copies on their own streams, overlapping the neighbouring steps'
kernels); the measured pinned copy bandwidths are reported beside it.

``--impl reference`` times the oracle itself (the reference arm): the FP64
definition on every host core (one process per core, each over its own range
of receivers or samples), a bounded sample of the same full-size workload per
step.
"""

import argparse
import json
import math
import os
import platform
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CGTP-conv edges/s fwd and fwd+bwd (FP32/FP64); % of HBM/FLOP roofline"

CONFIGS = {
    "tiny": dict(name="tiny", dtype="float32"),
    "nequip": dict(name="nequip", dtype="float32"),
    "mace": dict(name="mace", dtype="float32"),
    "mace64": dict(name="mace", dtype="float64"),
    "highl": dict(name="highl", dtype="float32"),
    "uvw": dict(name="uvw", dtype="float32"),
    "uvw_edge": dict(name="uvw_edge", dtype="float32"),
    "mixed": dict(name="mixed", dtype="float32"),
    "nequip_bf16": dict(name="nequip", dtype="bfloat16"),
    "highl_bf16": dict(name="highl", dtype="bfloat16"),
    "uvw_edge_bf16": dict(name="uvw_edge", dtype="bfloat16"),
    "mixed_bf16": dict(name="mixed", dtype="bfloat16"),
    "nequip_sh": dict(name="nequip", dtype="float32", sh=True),
    "mixedmul": dict(name="mixedmul", dtype="float32"),
}
# the benchmark's five workloads besides the headline
PER_CONFIG = ["tiny", "mace", "mace64", "highl", "uvw"]
NODE_CHUNK = None                 # --node-chunk: node chunk of radial uvw plans (None: the plan's default)
L2_BYTES = 126 * 2 ** 20          # GB300 L2 (about 126 MiB usable)
FLUSH_BYTES = 512 * 2 ** 20       # buffer written between timed steps when flushing L2

WORKLOAD_NAMES = {
    "tiny": "tiny uvu conv (64 nodes, 512 edges, 8x(0e,1o), SH l<=1)",
    "nequip": "NequIP-like uvu conv (10k nodes x 32 in-edges, 32x(0e,1o,2e,3o), SH l<=3)",
    "mace": "MACE-like uvu conv (5k nodes, Poisson(40) in-degree, 128x(0e,1o,2e), SH l<=3)",
    "highl": "high-L batched TP (B=50k, 16x l=0..7, SH l<=7)",
    "uvw": "uvw radial conv (200k nodes x 32 in-edges, 64x(0e,1o,2e), K=8)",
    "uvw_edge": "uvw conv with per-edge weights (10k nodes x 32 in-edges, 16x(0e,1o,2e))",
    "mixed": "mixed uvu/uvw conv (10k nodes x 32 in-edges, 32x(0e,1o,2e), SH l<=2; "
             "0e outputs uvw with per-edge weights, 1o and 2e outputs uvu)",
    "mixedmul": "uvu conv with blocks of different multiplicity (10k nodes x 32 in-edges, "
                "32x0e+16x1o+16x2e, SH l<=2): the general kernels",
}


# ---------------------------------------------------------------------------
# peaks
# ---------------------------------------------------------------------------

def driver_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d.get("bf16_tflops", 1900.0), "src": "measured",
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0)}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "src": "fallback", "sm_max_mhz": 2070.0}


def _time_launches(fn, stream, reps):
    import torch
    best = None
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        work = fn()
        b.record(stream)
        b.synchronize()
        ms = a.elapsed_time(b)
        if best is None or ms < best[0]:
            best = (ms, work)
    return best


def measure_peaks(device):
    """FP32 (FFMA and paired FFMA2), FP64 FMA throughput and L2 / HBM read bandwidth,
    measured with the library's kernels on this GPU (best of 3 launches of ~20 ms each,
    after a calibration launch), with the SM clock sampled meanwhile."""
    import torch
    import clebsch_gordan_tensor_racah_gb300 as cg
    props = torch.cuda.get_device_properties(device)
    nsm = props.multi_processor_count
    stream = torch.cuda.current_stream(device)
    ctas = nsm * 8
    sink = torch.empty(ctas * 256 * 2, dtype=torch.float64, device=device)
    clocks = ClockSampler(device.index or 0)
    clocks.start()
    out = {"sms": nsm}
    for name, kind in (("fp32_ffma", cg.CGTP_MEASURE_FFMA), ("fp32_ffma2", cg.CGTP_MEASURE_FFMA2),
                       ("fp64_dfma", cg.CGTP_MEASURE_DFMA)):
        iters = 16
        while True:
            ms, fl = _time_launches(lambda: cg.measure_fma(kind, ctas, iters, sink, stream), stream, 1)
            if ms > 4.0 or iters >= 1 << 22:
                break
            iters *= 4
        iters = max(1, int(iters * 20.0 / max(ms, 1e-3)))
        ms, fl = _time_launches(lambda: cg.measure_fma(kind, ctas, iters, sink, stream), stream, 3)
        out[name + "_tflops"] = fl / (ms * 1e-3) / 1e12
    rsink = torch.empty(nsm * 4 * 256, dtype=torch.int32, device=device)
    rc = nsm * 4
    q = 4096 * rc
    l2buf = torch.ones((64 * 2 ** 20 // q) * q // 4, dtype=torch.int32, device=device)
    cg.measure_read(l2buf, 1, rc, rsink, stream)
    ms, nb = _time_launches(lambda: cg.measure_read(l2buf, 40, rc, rsink, stream), stream, 3)
    out["l2_read_gbs"] = nb / (ms * 1e-3) / 1e9
    del l2buf
    hbuf = torch.ones((4 * 2 ** 30 // q) * q // 4, dtype=torch.int32, device=device)
    ms, nb = _time_launches(lambda: cg.measure_read(hbuf, 1, rc, rsink, stream), stream, 3)
    out["hbm_read_gbs"] = nb / (ms * 1e-3) / 1e9
    del hbuf
    clk = clocks.stop() or {}
    out["sm_mhz_median"] = clk.get("sm_mhz")
    out["fp32_tflops"] = max(out["fp32_ffma_tflops"], out["fp32_ffma2_tflops"])
    out["fp64_tflops"] = out["fp64_dfma_tflops"]
    mhz = clk.get("sm_mhz") or 2070.0
    out["fp32_flops_per_clk_per_sm"] = out["fp32_tflops"] * 1e12 / (mhz * 1e6) / nsm
    out["fp64_flops_per_clk_per_sm"] = out["fp64_tflops"] * 1e12 / (mhz * 1e6) / nsm
    out["how"] = ("cgtp_measure_fma: 8 CTAs x 256 threads per SM, 16 independent FMA chains per thread; "
                  "cgtp_measure_read: 16-byte loads over 64 MiB (L2, 40 passes) and 4 GiB (HBM); best of 3")
    return out


def measure_link(device):
    """Pinned host<->device copy bandwidth (GB/s), one 512 MiB copy each way, best of 3."""
    import torch
    n = 512 * 2 ** 20
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=device)
    s = torch.cuda.current_stream(device)
    ms_h2d, _ = _time_launches(lambda: d.copy_(h, non_blocking=True), s, 3)
    ms_d2h, _ = _time_launches(lambda: h.copy_(d, non_blocking=True), s, 3)
    return {"h2d_gbs": n / (ms_h2d * 1e-3) / 1e9, "d2h_gbs": n / (ms_d2h * 1e-3) / 1e9}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def build_inputs(cfgkey, device, nodes=None):
    import torch
    import clebsch_gordan_tensor_racah_gb300 as cg
    from clebsch_gordan_tensor_racah_gb300 import workloads as wl
    c = CONFIGS[cfgkey]
    spec = dict(wl.SPECS[c["name"]])
    tdt = {"float64": torch.float64, "bfloat16": torch.bfloat16}.get(c["dtype"], torch.float32)
    mode = spec["mode"]
    if mode == "mixed":
        plan = cg.MixedPlan(spec["in1"], spec["in2"], spec["out"], spec["instructions"], spec["modes"], tdt)
        w_numel = (plan.wu_numel, plan.ww_numel)
    else:
        plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], mode, tdt,
                       radial_k=spec.get("K", 0) if mode == "uvw" else 0)
        if NODE_CHUNK and plan.radial_k:
            plan.set_node_chunk(NODE_CHUNK)
        w_numel = plan.w_numel
    over = {}
    if nodes:
        over["B" if spec["graph"] is None else "N"] = int(nodes)
    w = wl.make(c["name"], w_numel, seed=0, dtype="float32" if tdt == torch.bfloat16 else c["dtype"], **over)
    host = {k: v for k, v in w.items() if isinstance(v, np.ndarray)}
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in host.items()}
    if tdt == torch.bfloat16:   # features and weights stored as bfloat16 (FP32 arithmetic and outputs)
        dev = {k: (v.to(torch.bfloat16) if v.is_floating_point() else v) for k, v in dev.items()}
        host = {k: (dev[k].cpu() if dev[k].dtype == torch.bfloat16 else v) for k, v in host.items()}
    if c.get("sh"):   # raw edge vectors of random lengths instead of the harmonics
        rng = np.random.default_rng(7)
        r = rng.standard_normal((w["E"], 3)) * rng.uniform(0.5, 5.0, (w["E"], 1))
        host["rvec"] = r.astype(np.float32)
        del host["Y"]
        dev["rvec"] = torch.from_numpy(host["rvec"]).to(device)
        del dev["Y"]
    graph = None
    if "rowptr" in dev:
        graph = cg.Graph(dev["rowptr"], dev["col"], w["N"])
    return plan, graph, w, host, dev, spec, tdt


def step_fns(cfgkey, plan, graph, w, dev, tdt):
    """Returns (fwd, bwd, units, bytes_fwd, bytes_bwd, out_shape, inputs, outputs).

    bytes: every input read once plus every output written once (index arrays
    included).  inputs: the tensors one step reads (the e2e copy list);
    outputs(res): the result tensors of a step given bwd's return value."""
    import clebsch_gordan_tensor_racah_gb300 as cg
    es = 8 if tdt.__str__().endswith("64") else 4
    ei = 2 if tdt.__str__().endswith("bfloat16") else es   # input element size (outputs: es)
    if "rvec" in dev:   # edge-vector input: harmonics evaluated in the kernels
        N, E = w["N"], w["E"]
        x, rv, W = dev["x"], dev["rvec"], dev["W"]
        units = E
        idx = 4 * (N + 1 + E)
        nin = N * plan.d1 + 3 * E + W.numel()
        bf = es * (nin + N * plan.d_out) + idx
        bb = es * (2 * nin + N * plan.d_out + E * plan.d2) + idx + 8 * E

        def fwd(out, d=dev):
            return cg.cgtp_conv_forward_sh(plan, graph, d["x"], d["rvec"], d["W"], out=out)

        def bwd(g, outs, d=dev):
            return cg.cgtp_conv_backward_sh(plan, graph, g, d["x"], d["rvec"], d["W"])
        return fwd, bwd, units, bf, bb, (N, plan.d_out)
    if "Wu" in dev:   # mixed instruction list: two per-edge weight arrays
        N, E = w["N"], w["E"]
        x, Y, Wu, Ww = dev["x"], dev["Y"], dev["Wu"], dev["Ww"]
        units = E
        idx = 4 * (N + 1 + E)
        nin = N * plan.d1 + E * plan.d2 + Wu.numel() + Ww.numel()
        bf = ei * nin + es * N * plan.d_out + idx
        bb = ei * (nin + N * plan.d_out) + es * nin + idx + 8 * E
        ws, _ = plan.workspace(graph, x.device)
        import torch
        res = tuple(torch.empty(t.shape, dtype=plan.out_dtype, device=t.device) for t in (x, Y, Wu, Ww))

        def fwd(out, d=dev):
            return cg.cgtp_mixed_conv_forward(plan, graph, d["x"], d["Y"], d["Wu"], d["Ww"], out=out, workspace=ws)

        def bwd(g, outs, d=dev):
            return cg.cgtp_mixed_conv_backward(plan, graph, g, d["x"], d["Y"], d["Wu"], d["Ww"], workspace=ws,
                                               outs=res)
        return fwd, bwd, units, bf, bb, (N, plan.d_out)
    if "rowptr" in dev:
        N, E = w["N"], w["E"]
        WR = dev["W"] if "W" in dev else dev["R"]
        M = dev.get("M")
        units = E
        idx = 4 * (N + 1 + E)
        nin = N * plan.d1 + E * plan.d2 + WR.numel() + (M.numel() if M is not None else 0)
        bf = ei * nin + es * N * plan.d_out + idx
        bb = ei * (nin + N * plan.d_out) + es * nin + idx + 8 * E

        def fwd(out, d=dev):
            return cg.cgtp_conv_forward(plan, graph, d["x"], d["Y"], d["W"] if "W" in d else d["R"], d.get("M"),
                                        out=out)

        def bwd(g, outs, d=dev):
            return cg.cgtp_conv_backward(plan, graph, g, d["x"], d["Y"], d["W"] if "W" in d else d["R"],
                                         d.get("M"), outs=outs)
        out_shape = (N, plan.d_out)
    else:
        B = w["B"]
        units = B
        nin = B * (plan.d1 + plan.d2 + plan.w_numel)
        bf = ei * nin + es * B * plan.d_out                    # inputs read, output written
        bb = ei * (nin + B * plan.d_out) + es * nin            # inputs + gradient read, gradients written

        def fwd(out, d=dev):
            return cg.cgtp_forward(plan, d["x1"], d["x2"], d["W"], out=out)

        def bwd(g, outs, d=dev):
            return cg.cgtp_backward(plan, g, d["x1"], d["x2"], d["W"])
        out_shape = (B, plan.d_out)
    return fwd, bwd, units, bf, bb, out_shape


def launches_per_step(cfgkey, plan, w):
    """Kernels of this library one timed step (forward + backward) launches."""
    if plan.mode == "mixed":   # uvw and uvu forwards, fold; unfold, uvu and uvw backwards, two adds
        return 8
    if CONFIGS[cfgkey].get("sh"):   # forward, backward, per-edge chain rule to the edge vectors
        return 3
    if plan.mode == "uvw" and plan.radial_k > 0:
        return plan.launches_per_step(w["N"])
    return 2


def _cg_counts(l1, l2, l3):
    """(nnz of the real CG block, nnz of its (m1, m3) pattern): the number of terms of
    C.Y and of the contraction over m1 for one channel."""
    import clebsch_gordan_tensor_racah_gb300 as cg
    C = np.abs(cg.cgtp_real_cg_block(l1, l2, l3)) > 1e-12
    return int(C.sum()), int(C.any(axis=1).sum())


def model_flops(plan, n_nodes, units, graph=True):
    """Algorithmic FLOPs of one forward and one backward (FMA = 2), counting CG nonzeros.

    uvu, per edge (sample) and path, D3 = 2 l3 + 1:
        2 nnz(C)                       cy[m1,m3] = sum_m2 C[m1,m2,m3] Y[m2]
        mul * 2 nnz_{m1,m3}(C)         t[u,m3] = sum_m1 cy[m1,m3] x[u,m1]
        mul * D3                       the weight product W[u] t[u,m3]
      plus d_out per edge for the receiver sum (graphs only).
    uvw radial: the edge stage 2 nnz + mul1 * 2 nnz_{m1,m3} + 2 K mul1 D3 per edge and
      path (t, then S += R[e,k] t), and the node GEMM 2 K mul1 mul_out D3 per node and
      path.  uvw with per-edge weights: 2 nnz + mul1 * 2 nnz_{m1,m3} + 2 mul1 mul_out D3.
    Backward = 3 x forward.  Returns (fwd_cuda_core, fwd_tensor_core): the node GEMM of
    the radial uvw runs on the tensor cores, everything else on the FP32/FP64 pipes."""
    K = getattr(plan, "radial_k", 0)
    fe = fn = 0
    if plan.mode == "mixed":
        from clebsch_gordan_tensor_racah_gb300.workloads import irreps_terms
        a, b, o = (irreps_terms(s) for s in plan.irreps)
        for (i1, i2, io), m in zip(plan.instructions, plan.modes):
            (mul1, l1), (_, l2), (mul_out, l3) = a[i1], b[i2], o[io]
            nnz, nc = _cg_counts(l1, l2, l3)
            D3 = 2 * l3 + 1
            fe += 2 * nnz + mul1 * 2 * nc + (mul1 * D3 if m == "uvu" else 2 * mul1 * mul_out * D3)
        return (fe + plan.d_out) * units, 0.0
    for p in range(plan.n_paths):
        ints, _ = plan.path(p)
        l1, l2, l3, mul1, mul_out = ints[:5]
        nnz, nc = _cg_counts(l1, l2, l3)
        D3 = 2 * l3 + 1
        if plan.mode == "uvu":
            fe += 2 * nnz + mul1 * (2 * nc + D3)
        elif K == 0:
            fe += 2 * nnz + mul1 * 2 * nc + 2 * mul1 * mul_out * D3
        else:
            fe += 2 * nnz + mul1 * 2 * nc + 2 * K * mul1 * D3
            fn += 2 * K * mul1 * mul_out * D3
    agg = plan.d_out if (graph and plan.mode == "uvu") else 0
    return float((fe + agg) * units), float(fn * n_nodes)


def traffic_for(kname, cfgkey, algorithmic_bytes):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary
    (profiles/traffic.txt: kernel, workload, dram bytes per algorithmic byte measured on a
    smaller case of the same recipe); None when no capture matches this kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == kname and f[1] == cfgkey:
            return float(f[2]) * algorithmic_bytes
    return None


class ClockSampler:
    def __init__(self, index=0):
        self.samples, self.proc, self.thread = [], None, None
        self.index = index

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def rd():
            for line in self.proc.stdout:
                self.samples.append([s.strip() for s in line.split(",")])
        self.thread = threading.Thread(target=rd, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        rows = [r for r in self.samples if len(r) >= 9]
        if not rows:
            return None
        mhz = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(mhz)) if mhz else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# timing one workload
# ---------------------------------------------------------------------------

def time_steps(fwd, bwd, g, out, stream, steps, flush=None):
    """(fwd_ms, bwd_ms, step_ms): mean over `steps` steps, CUDA events on the launching
    stream.  With `flush` (a buffer larger than L2) the buffer is rewritten before every
    step, outside the events, so each step starts with a cold L2."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.add_(1)
        ev[i][0].record(stream)
        fwd(out)
        ev[i][1].record(stream)
        bwd(g, None)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    tf = [e[0].elapsed_time(e[1]) for e in ev]
    tb = [e[1].elapsed_time(e[2]) for e in ev]
    return float(np.mean(tf)), float(np.mean(tb)), float(np.mean(tf) + np.mean(tb))


def roofline_of(plan, w, units, bf, bb, fwd_ms, bwd_ms, tdt, pk, meas):
    """Per-direction roofline times and the step fraction (section-8(d) model)."""
    import torch
    graph = "N" in w
    n_nodes = w.get("N", w.get("B", 0))
    ff_cc, ff_tc = model_flops(plan, n_nodes, units, graph=graph)
    f64 = tdt == torch.float64
    alu = (meas["fp64_tflops"] if f64 else meas["fp32_tflops"]) * 1e12
    # tensor-core node GEMM of the radial uvw: kind::tf32 with three products per tile (3xTF32);
    # TF32 peak = measured bf16 peak x the nominal tf32/bf16 ratio (1.1 / 2.25)
    tc = pk["bf16_tflops"] * 1e12 * (1.1 / 2.25) / 3.0
    hbm = pk["hbm_gbs"] * 1e9

    def side(nbytes, f_cc, f_tc):
        t_mem = nbytes / hbm
        t_alu = f_cc / alu + f_tc / tc
        return max(t_mem, t_alu), ("hbm" if t_mem >= t_alu else ("alu" if f_tc == 0 else "alu+tensor"))
    rf, bound_f = side(bf, ff_cc, ff_tc)
    rb, bound_b = side(bb, 3 * ff_cc, 3 * ff_tc)
    return {"fwd_flops": ff_cc + ff_tc, "bwd_flops": 3 * (ff_cc + ff_tc), "fwd_tensor_flops": ff_tc,
            "fwd_bytes": int(bf), "bwd_bytes": int(bb),
            "fwd_roofline_ms": 1e3 * rf, "bwd_roofline_ms": 1e3 * rb, "fwd_bound": bound_f, "bwd_bound": bound_b,
            "fwd_frac": 1e3 * rf / fwd_ms, "bwd_frac": 1e3 * rb / bwd_ms,
            "step_frac": 1e3 * (rf + rb) / (fwd_ms + bwd_ms),
            "peaks_used": {"alu_tflops": alu / 1e12, "alu": "fp64 dfma" if f64 else "fp32 (max of ffma, ffma2)",
                           "tensor_tflops": tc / 1e12 if ff_tc else None, "hbm_gbs": hbm / 1e9}}


def run_config(cfgkey, device, steps, warmup, meas, pk, flush_l2=None, nodes=None):
    """Times one workload: warm-up, then `steps` timed steps; returns a dict (plus the
    objects the headline needs for e2e and the double backward)."""
    import torch
    if cfgkey == "uvw":
        torch.cuda.reset_peak_memory_stats(device)
    torch.cuda.synchronize()
    free0, total = torch.cuda.mem_get_info(device)
    plan, graph, w, host, dev, spec, tdt = build_inputs(cfgkey, device, nodes)
    torch.cuda.synchronize()
    fwd, bwd, units, bf, bb, out_shape = step_fns(cfgkey, plan, graph, w, dev, tdt)
    g = torch.randn(out_shape, dtype=tdt, device=device, generator=torch.Generator(device).manual_seed(1))
    out = torch.empty(out_shape, dtype=plan.out_dtype, device=device)
    stream = torch.cuda.current_stream(device)
    # inputs below L2 (tiny) are always timed cold; the others exceed L2 by themselves
    in_bytes = sum(t.numel() * t.element_size() for t in dev.values())
    flush = flush_l2 if flush_l2 is not None else (in_bytes < 2 * L2_BYTES)
    fbuf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device) if flush else None
    for _ in range(max(3, warmup)):
        fwd(out)
        bwd(g, None)
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index or 0)
    clocks.start()
    time.sleep(0.25)
    tf, tb, ts = time_steps(fwd, bwd, g, out, stream, steps, fbuf)
    clk = clocks.stop()
    free1, _ = torch.cuda.mem_get_info(device)
    r = {"workload": WORKLOAD_NAMES[CONFIGS[cfgkey]["name"]],
         "precision": {torch.float64: "f64", torch.bfloat16: "bf16 inputs, f32 arithmetic"}.get(tdt, "f32"),
         "units": int(units), "unit": "edges" if "N" in w else "samples", "steps": steps, "warmup": max(3, warmup),
         "fwd_ms": tf, "bwd_ms": tb, "step_ms": ts,
         "fwd_units_per_s": units / (tf * 1e-3), "fwd_bwd_units_per_s": units / (ts * 1e-3),
         "l2": ("L2 flushed before every timed step (512 MiB write)" if flush
                else f"inputs ({in_bytes / 1e9:.2f} GB) larger than L2, no flush"),
         "gpu_launches_per_step": launches_per_step(cfgkey, plan, w),
         "roofline": roofline_of(plan, w, units, bf, bb, tf, tb, tdt, pk, meas),
         "clocks": clk}
    if "N" in w:
        r.update(nodes=int(w["N"]), edges=int(w["E"]))
    else:
        r.update(batch=int(w["B"]))
    if cfgkey == "uvw":
        r["node_chunk"] = plan.node_chunk
        lib_bytes = plan.device_bytes() + graph.device_bytes()
        r["peak_memory"] = {
            "torch_peak_allocated_bytes": int(torch.cuda.max_memory_allocated(device)),
            "library_bytes": int(lib_bytes),
            "peak_device_bytes": int(torch.cuda.max_memory_allocated(device) + lib_bytes),
            "device_used_delta_bytes": int(free0 - free1),
            "how": "torch.cuda.max_memory_allocated (inputs, outputs, gradients) + the bytes the plan "
                   "and graph own (cgtp_plan_device_bytes, cgtp_graph_device_bytes)"}
    return r, (plan, graph, w, host, dev, tdt, fwd, bwd, g, out, out_shape, units, bf, bb)


def time_double_backward(plan, graph, w, dev, g, stream, units, roof):
    """Second derivatives (cgtp_conv_double_backward / cgtp_double_backward) with random
    cotangents, CUDA events on the launching stream, after warm-up.  It runs the
    forward and backward kernels once per operand (3 + 3 for uvu, 4 + 4 for uvw),
    so its roofline is that many forward and backward rooflines."""
    import torch
    import clebsch_gordan_tensor_racah_gb300 as cg
    gen = torch.Generator(g.device).manual_seed(2)
    if "Wu" in dev:
        c = {k: torch.randn(dev[k].shape, dtype=dev[k].dtype, device=g.device, generator=gen)
             for k in ("x", "Y", "Wu", "Ww")}
        ws, _ = plan.workspace(graph, g.device)

        def run():
            return cg.cgtp_mixed_conv_double_backward(plan, graph, g, dev["x"], dev["Y"], dev["Wu"], dev["Ww"],
                                                      c["x"], c["Y"], c["Wu"], c["Ww"], workspace=ws)
        n_op = 3
    elif "rowptr" in dev:
        keys = ["x", "Y", "W"] if "W" in dev else ["x", "Y", "R", "M"]
        c = {k: torch.randn(dev[k].shape, dtype=dev[k].dtype, device=g.device, generator=gen) for k in keys}
        WR = dev["W"] if "W" in dev else dev["R"]
        cWR = c["W"] if "W" in c else c["R"]

        def run():
            return cg.cgtp_conv_double_backward(plan, graph, g, dev["x"], dev["Y"], WR, c["x"], c["Y"], cWR,
                                                M=dev.get("M"), ggM=c.get("M"))
        n_op = len(keys)
    else:
        c = {k: torch.randn(dev[k].shape, dtype=dev[k].dtype, device=g.device, generator=gen)
             for k in ("x1", "x2", "W")}

        def run():
            return cg.cgtp_double_backward(plan, g, dev["x1"], dev["x2"], dev["W"], c["x1"], c["x2"], c["W"])
        n_op = 3
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    a.record(stream)
    for _ in range(reps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    rl = n_op * (roof["fwd_roofline_ms"] + roof["bwd_roofline_ms"])
    return {"ms": ms, "units_per_s": units / (ms / 1000.0), "launch_sequence": f"{n_op} forwards + {n_op} backwards + adds",
            "roofline_ms": rl, "frac": rl / ms}


def time_e2e(ctx, device, steps):
    """The headline step through the public API with host buffers: every step copies its
    inputs from pinned host memory and its results (output, gradients) back.  Copies run on
    their own streams with two device buffer sets, so step k's copies overlap steps k-1 and
    k+1's kernels; the timed region runs from the first copy to the last result on the host."""
    import torch
    plan, graph, w, host, dev, tdt, fwd, bwd, g, out, out_shape, units, bf, bb = ctx
    keys = [k for k in host if k not in ("rowptr", "col")]
    pin = {k: (v if isinstance(v, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(v))).pin_memory()
           for k, v in host.items() if k in keys}
    gh = g.cpu().pin_memory()
    sets = []
    for s in range(2):
        d = {k: (dev[k] if s == 0 else torch.empty_like(dev[k])) for k in keys}
        d.update({k: dev[k] for k in ("rowptr", "col") if k in dev})
        sets.append({"in": d, "g": g if s == 0 else torch.empty_like(g),
                     "out": out if s == 0 else torch.empty_like(out), "res": None,
                     "ev_in": torch.cuda.Event(), "ev_fwd": torch.cuda.Event(), "ev_bwd": torch.cuda.Event(),
                     "ev_out": torch.cuda.Event()})
    s_comp = torch.cuda.current_stream(device)
    s_h2d, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    out_h = [torch.empty(out_shape, dtype=plan.out_dtype).pin_memory() for _ in range(2)]
    res_h = [None, None]
    fwd_d, bwd_d = ctx[6], ctx[7]

    def launch(i, first):
        S = sets[i % 2]
        with torch.cuda.stream(s_h2d):
            if not first:
                s_h2d.wait_event(S["ev_bwd"])          # the previous step on this set has read its inputs
            for k in keys:
                S["in"][k].copy_(pin[k], non_blocking=True)
            S["g"].copy_(gh, non_blocking=True)
            S["ev_in"].record(s_h2d)
        s_comp.wait_event(S["ev_in"])
        if not first:
            s_comp.wait_event(S["ev_out"])             # its previous results have reached the host
        fwd_d(S["out"], d=S["in"])
        S["ev_fwd"].record(s_comp)
        r = bwd_d(S["g"], S["res"], d=S["in"])
        S["res"] = tuple(x for x in r)
        S["ev_bwd"].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(S["ev_fwd"])
            out_h[i % 2].copy_(S["out"], non_blocking=True)
            s_d2h.wait_event(S["ev_bwd"])
            if res_h[i % 2] is None:
                res_h[i % 2] = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in r if x is not None]
            for hb, x in zip(res_h[i % 2], [x for x in r if x is not None]):
                hb.copy_(x, non_blocking=True)
            S["ev_out"].record(s_d2h)
    # the step functions take an explicit input set (keyword d)
    for i in range(2):
        launch(i, True)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in pin.values()) + gh.numel() * gh.element_size()
    d2h = out_h[0].numel() * out_h[0].element_size() + sum(t.numel() * t.element_size() for t in res_h[0])
    k2 = max(4, steps // 2)
    t0 = time.perf_counter()
    for i in range(k2):
        launch(i, False)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / k2
    return {"value": units / e2e_s, "unit": "edges/s" if "N" in w else "samples/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": 1e3 * e2e_s,
            "how": "pinned host buffers; H2D and D2H copies on their own streams, two device buffer sets; "
                   "host wall clock from the first copy to the last result in host memory"}


# ---------------------------------------------------------------------------
# the oracle on the host cores (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

_W = {}


def _oracle_init(cfgkey, files, threads_env):
    os.environ.update(threads_env)
    _W["cfg"] = cfgkey
    _W["a"] = {k: np.load(f, mmap_mode="r") for k, f in files.items()}


def _oracle_work(lo, hi):
    """Forward + backward of the FP64 oracle over receivers (or samples) [lo, hi) of the
    full-size workload; returns (units processed, seconds)."""
    from clebsch_gordan_tensor_racah_gb300 import workloads as wl
    from oracle import conv as oconv, irreps as oirr
    c = CONFIGS[_W["cfg"]]
    spec = wl.SPECS[c["name"]]
    a = _W["a"]
    if "plan" not in _W:
        _W["plan"] = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], spec["mode"])
    p = _W["plan"]
    t0 = time.perf_counter()
    if spec["graph"] is None:
        x1, x2, W = (np.asarray(a[k][lo:hi]) for k in ("x1", "x2", "W"))
        out = oconv.tp_uvu_forward(p, x1, x2, W)
        oconv.tp_uvu_backward(p, out, x1, x2, W)
        return hi - lo, time.perf_counter() - t0
    rowptr = np.asarray(a["rowptr"])
    nodes = np.arange(lo, hi)
    edges = np.arange(rowptr[lo], rowptr[hi])
    if spec["mode"] == "uvu":
        out = oconv.conv_uvu_forward(p, a["x"], a["Y"], a["W"], rowptr, a["col"], nodes=nodes)
        g = np.zeros((rowptr.shape[0] - 1, p.d_out))
        g[lo:hi] = out
        oconv.conv_uvu_backward(p, g, a["x"], a["Y"], a["W"], rowptr, a["col"], edges=edges)
    else:
        out = oconv.conv_uvw_radial_forward(p, a["x"], a["Y"], a["R"], a["M"], rowptr, a["col"], nodes=nodes)
        g = np.zeros((rowptr.shape[0] - 1, p.d_out))
        g[lo:hi] = out
        oconv.conv_uvw_radial_backward(p, g, a["x"], a["Y"], a["R"], a["M"], rowptr, a["col"], edges=edges)
    return int(edges.size), time.perf_counter() - t0


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


class OracleTimer:
    """The FP64 oracle over the full-size workload on every host core: one spawned process
    per core (FP64 NumPy limited to one thread each), each taking its own range of receivers
    (or samples).  The workload is drawn once and shared read-only through .npy files."""

    def __init__(self, cfgkey, procs=None):
        import multiprocessing as mp
        from clebsch_gordan_tensor_racah_gb300 import workloads as wl
        from oracle import irreps as oirr
        c = CONFIGS[cfgkey]
        if c["name"] not in ("tiny", "nequip", "mace", "highl", "uvw"):
            raise ValueError(f"no oracle timing for {cfgkey}")
        spec = wl.SPECS[c["name"]]
        plan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], spec["mode"])
        w = wl.make(c["name"], plan.w_numel, seed=0, dtype=c["dtype"])
        self.tmp = tempfile.TemporaryDirectory(prefix="cgtp_oracle_")
        files = {}
        for k, v in w.items():
            if isinstance(v, np.ndarray):
                files[k] = os.path.join(self.tmp.name, k + ".npy")
                np.save(files[k], v)
        self.graph = spec["graph"] is not None
        self.n = int(w["N"] if self.graph else w["B"])
        self.rowptr = w.get("rowptr")
        self.procs = procs or os.cpu_count() or 1
        # one BLAS thread per process: the children read these when they import NumPy
        env = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        saved = {k: os.environ.get(k) for k in env}
        os.environ.update(env)
        try:
            self.pool = mp.get_context("spawn").Pool(self.procs, initializer=_oracle_init,
                                                     initargs=(cfgkey, files, env))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.cursor = 0
        self.pool.starmap(_oracle_work, [(0, 1)] * self.procs)   # imports and plan in every worker

    def step(self, per_proc):
        """One step: every process runs `per_proc` consecutive receivers (samples), the
        processes' ranges follow each other from the cursor (wrapping).  Returns
        (units, wall seconds)."""
        ranges = []
        for _ in range(self.procs):
            lo = self.cursor
            hi = min(self.n, lo + per_proc)
            ranges.append((lo, hi))
            self.cursor = 0 if hi >= self.n else hi
        t0 = time.perf_counter()
        res = self.pool.starmap(_oracle_work, ranges)
        return sum(u for u, _ in res), time.perf_counter() - t0

    def calibrate(self, target_s):
        """Receivers (samples) per process so that one step takes about target_s."""
        per = 1
        while True:
            u, dt = self.step(per)
            if dt > 0.3 * target_s or per >= self.n // self.procs:
                break
            per *= 4
        return max(1, min(self.n // self.procs, int(per * target_s / max(dt, 1e-3))))

    def close(self):
        self.pool.close()
        self.pool.join()
        self.tmp.cleanup()


def oracle_baseline(cfgkey, budget_s=15.0):
    """cpu_baseline of the headline line: the oracle on all host cores for about budget_s."""
    t = OracleTimer(cfgkey)
    try:
        per = t.calibrate(budget_s / 3)
        units = secs = 0.0
        n_steps = 0
        while secs < budget_s:
            u, dt = t.step(per)
            units += u
            secs += dt
            n_steps += 1
        unit = "edges" if t.graph else "samples"
        return {"value": units / secs, "unit": unit + "/s", "cores": t.procs, "kind": "oracle",
                "cpu": cpu_model(), "cpu_count": os.cpu_count(), "sampled": True,
                "sample": f"{n_steps} steps of {per} consecutive {'receivers' if t.graph else 'samples'} per "
                          f"process x {t.procs} processes of the full-size workload ({int(units)} {unit}, "
                          f"{secs:.1f} s), FP64 forward + backward"}
    finally:
        t.close()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cfgkey = args.config
    total = args.warmup + args.steps
    t = OracleTimer(cfgkey)
    try:
        per = t.calibrate(min(6.0, 100.0 / max(1, total)))
        for _ in range(args.warmup):
            t.step(per)
        units = secs = 0.0
        t_wall = time.perf_counter()
        for _ in range(args.steps):
            u, dt = t.step(per)
            units += u
            secs += dt
        wall = time.perf_counter() - t_wall
    finally:
        t.close()
    rate = units / secs
    unit = "edges/s" if t.graph else "samples/s"
    line = {"metric": METRIC, "value": rate, "unit": unit, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES[CONFIGS[cfgkey]["name"]],
                       "step": "FP64 oracle forward + backward over a sample of the full-size workload",
                       "sampled": True, "units_per_step": int(units / max(1, args.steps)),
                       "timed_wall_s": wall},
            "cpu_baseline": {"value": rate, "unit": unit, "cores": t.procs, "kind": "oracle",
                             "cpu": cpu_model(), "cpu_count": os.cpu_count(), "sampled": True,
                             "sample": f"{per} consecutive {'receivers' if t.graph else 'samples'} per process "
                                       f"x {t.procs} processes per step of the full-size workload"},
            "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# driver
# ---------------------------------------------------------------------------

def job_throughput(ms, units, world, device=None):
    """Whole-job throughput of N replicas (weak scaling: every rank processes its own
    `units`).  The step time is the slowest rank's (max over ranks, one all-reduce
    on the default process group when world > 1); value = world * units / time."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * units / (ms / 1000.0)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def headline_roofline(cfgkey, r, ctx, pk, meas):
    """The `roofline` object of the JSON line: the dominant kernel (the slower direction)
    against its binding peak; achieved = algorithmic bytes or FLOPs of one launch / its
    mean event-timed duration."""
    plan = ctx[0]
    ro = r["roofline"]
    dominant = "backward" if r["bwd_ms"] >= r["fwd_ms"] else "forward"
    d = "bwd" if dominant == "backward" else "fwd"
    ms = r[d + "_ms"]
    nbytes, flops = ro[d + "_bytes"], ro[d + "_flops"]
    if plan.mode == "uvu" and "N" not in ctx[2]:
        kname = {"fwd": "bt_forward_kernel", "bwd": "bt_backward_kernel"}[d]
    elif plan.mode == "uvu" and cfgkey == "mixedmul":   # blocks of different multiplicity: general kernels
        kname = {"fwd": "uvu_forward2_kernel", "bwd": "uvu_backward_kernel"}[d]
    elif plan.mode == "uvu":
        kname = {"fwd": "uvu_forward3_kernel", "bwd": "uvu_backward3_kernel"}[d]
    elif plan.mode == "mixed":
        kname = f"mixed {dominant} (uvu + per-edge uvw kernels)"
    elif plan.radial_k == 0:
        kname = {"fwd": "uvwe_fwd_kernel", "bwd": "uvwe_bwd_kernel"}[d]
    else:
        kname = f"uvw radial {dominant} (edge stage + tensor-core node GEMM)"
    if ro[d + "_bound"] == "hbm":
        ach = nbytes / (ms * 1e-3) / 1e9
        out = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
               "frac": ach / pk["hbm_gbs"], "peak_src": pk["src"] + " copy bandwidth (MEASURED_PEAKS.json)"}
    else:
        peak = ro["peaks_used"]["alu_tflops"]
        ach = flops / (ms * 1e-3) / 1e12
        out = {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
               "peak_src": "measured here: cgtp_measure_fma (" + ro["peaks_used"]["alu"] + ")"}
    out.update({"kernel": kname, "traffic": traffic_for(kname, cfgkey, nbytes),
                "algorithmic_bytes_per_launch": int(nbytes), "algorithmic_flops_per_launch": float(flops),
                "fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"], "fwd_roofline_ms": ro["fwd_roofline_ms"],
                "bwd_roofline_ms": ro["bwd_roofline_ms"], "step_frac": ro["step_frac"]})
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="nequip", choices=sorted(CONFIGS))
    ap.add_argument("--flush-l2", action="store_true",
                    help="rewrite a 512 MiB buffer before every timed step (cold L2) for every workload")
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-double-backward", action="store_true",
                    help="skip the (untimed-for-the-metric) second-derivative measurement")
    ap.add_argument("--node-chunk", type=int, default=None,
                    help="node chunk of radial uvw plans (cgtp_plan_set_node_chunk; default: the plan's)")
    ap.add_argument("--nodes", type=int, default=None,
                    help="smaller instance of the same recipe (nodes, or batch for highl)")
    ap.add_argument("--profile-run", action="store_true",
                    help="build, two warm-up steps and one step, no timing or JSON (for ncu captures)")
    ap.add_argument("--profile-double-backward", action="store_true",
                    help="with --profile-run: also one second-derivative call (its add kernels)")
    args = ap.parse_args()
    global NODE_CHUNK
    NODE_CHUNK = args.node_chunk
    if args.impl == "reference":
        return run_reference(args)

    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from __graft_entry__ import build
    if rank == 0:
        build()
    if world > 1:
        torch.distributed.barrier()
    build()

    if args.profile_run:
        plan, graph, w, host, dev, spec, tdt = build_inputs(args.config, device, args.nodes)
        fwd, bwd, units, bf, bb, out_shape = step_fns(args.config, plan, graph, w, dev, tdt)
        g = torch.randn(out_shape, dtype=tdt, device=device, generator=torch.Generator(device).manual_seed(1))
        out = torch.empty(out_shape, dtype=plan.out_dtype, device=device)
        for _ in range(3):
            fwd(out)
            bwd(g, None)
        if args.profile_double_backward:
            time_double_backward(plan, graph, w, dev, g, torch.cuda.current_stream(device), units,
                                 {"fwd_roofline_ms": 0.0, "bwd_roofline_ms": 0.0})
        torch.cuda.synchronize()
        print(f"profile run done: {args.config}, {units} units", flush=True)
        return

    pk = driver_peaks()
    meas = measure_peaks(device)
    flush = True if args.flush_l2 else None
    r, ctx = run_config(args.config, device, args.steps, args.warmup, meas, pk, flush, args.nodes)
    if world > 1:
        torch.distributed.barrier()
    ms, value = job_throughput(r["step_ms"], r["units"], world, device)
    clk = r.pop("clocks")
    unit = "edges/s" if r["unit"] == "edges" else "samples/s"
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": r["precision"], "data": "synthetic",
            "config": {"workload": r["workload"], "step": "conv forward + backward" if "nodes" in r
                       else "batched forward + backward", "l2": r["l2"],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       **({"nodes": r["nodes"], "edges": r["edges"]} if "nodes" in r else {"batch": r["batch"]})},
            "fwd_units_per_s": world * r["fwd_units_per_s"],
            "roofline": headline_roofline(args.config, r, ctx, pk, meas),
            "gpu_launches": r["gpu_launches_per_step"] * args.steps, "clocks": clk,
            "peaks": {**meas, "hbm_copy_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                      "driver_peaks": pk["src"]}}
    if not args.no_e2e:
        line["e2e"] = time_e2e(ctx, device, args.steps)
        line["e2e"]["link"] = measure_link(device)
        line["e2e"]["value"] *= world
    if not args.no_double_backward and ctx[5] != torch.bfloat16 and not CONFIGS[args.config].get("sh"):
        line["double_backward"] = time_double_backward(ctx[0], ctx[1], ctx[2], ctx[4], ctx[8],
                                                       torch.cuda.current_stream(device), r["units"], r["roofline"])
    line["per_workload_roofline"] = r["roofline"]
    del ctx
    torch.cuda.empty_cache()
    if not args.no_per_config and args.nodes is None:
        per = {}
        for k in PER_CONFIG:
            if k == args.config:
                continue
            steps = min(args.steps, 8) if k in ("uvw", "mace64") else args.steps
            rk, ck = run_config(k, device, steps, args.warmup, meas, pk, flush)
            del ck
            torch.cuda.empty_cache()
            per[k] = rk
        line["per_config"] = per
    if rank == 0 and not args.no_cpu_baseline and world == 1 and args.config in ("tiny", "nequip", "mace",
                                                                                   "highl", "uvw"):
        line["cpu_baseline"] = oracle_baseline(args.config)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
