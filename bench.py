"""Throughput of the fused CG tensor-product convolution (edges/s, forward + backward).

Default workload: the NequIP-like convolution -- 10,000 nodes, 32 in-edges per
node (320,000 edges), in1 = 32x(0e,1o,2e,3o), SH l<=3, uvu with all 34
parity-allowed paths (l3 <= 3), FP32.  One step = cgtp_conv_forward +
cgtp_conv_backward over the whole graph (the graph and plan are built once,
outside the timed region).  Other workloads: --config tiny|nequip|mace|mace64|highl|uvw.

Output: one JSON line (rank 0).  ``value`` is device-timed edges/s with inputs
resident in HBM; ``e2e`` repeats the step through the public API with the
step's inputs copied from pinned host memory and its results copied back inside
the timed region.  ``roofline`` describes the dominant kernel; ``cpu_baseline``
times the FP64 oracle on a bounded sample of the same workload.

``--impl reference`` times the oracle itself (the reference arm): host cores,
bounded sample, same metric and config.
"""

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CGTP-conv edges/s fwd and fwd+bwd (FP32/FP64); % of HBM/FLOP roofline"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "src": "measured", "sm_max_mhz": d.get("sm_max_mhz", 2070.0)}
    return {"hbm_gbs": 6800.0, "src": "fallback", "sm_max_mhz": 2070.0}


# FP32 / FP64 CUDA-core peaks from unit counts: 152 SMs x 128 FP32 lanes x 2 flop
# x clock; FP64 at the nominal 1.25 TFLOP/s of the part.
def alu_peak_tflops(dtype_name, mhz):
    if dtype_name == "f64":
        return 1.25
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


CONFIGS = {
    "tiny": dict(name="tiny", dtype="float32", over={}),
    "nequip": dict(name="nequip", dtype="float32", over={}),
    "mace": dict(name="mace", dtype="float32", over={}),
    "mace64": dict(name="mace", dtype="float64", over={}),
    "highl": dict(name="highl", dtype="float32", over={}),
    "nequip_bf16": dict(name="nequip", dtype="bfloat16", over={}),
    "nequip_sh": dict(name="nequip", dtype="float32", over={}, sh=True),
    "uvw_edge": dict(name="uvw_edge", dtype="float32", over={}),
    "mixed": dict(name="mixed", dtype="float32", over={}),
    "uvw": dict(name="uvw", dtype="float32", over={}),
}


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
        w_numel = plan.w_numel
    over = dict(c["over"])
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
    """Returns (fwd, bwd, units, bytes_fwd, bytes_bwd, flops_fwd, flops_bwd, out_shape)."""
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

        def fwd(out):
            return cg.cgtp_conv_forward_sh(plan, graph, x, rv, W, out=out)

        def bwd(g, outs):
            return cg.cgtp_conv_backward_sh(plan, graph, g, x, rv, W)
        return fwd, bwd, units, bf, bb, (N, plan.d_out)
    if "Wu" in dev:   # mixed instruction list: two per-edge weight arrays
        N, E = w["N"], w["E"]
        x, Y, Wu, Ww = dev["x"], dev["Y"], dev["Wu"], dev["Ww"]
        units = E
        idx = 4 * (N + 1 + E)
        nin = N * plan.d1 + E * plan.d2 + Wu.numel() + Ww.numel()
        bf = es * (nin + N * plan.d_out) + idx
        bb = es * (2 * nin + N * plan.d_out) + idx + 8 * E
        ws, _ = plan.workspace(graph, x.device)
        import torch
        res = (torch.empty_like(x), torch.empty_like(Y), torch.empty_like(Wu), torch.empty_like(Ww))

        def fwd(out):
            return cg.cgtp_mixed_conv_forward(plan, graph, x, Y, Wu, Ww, out=out, workspace=ws)

        def bwd(g, outs):
            return cg.cgtp_mixed_conv_backward(plan, graph, g, x, Y, Wu, Ww, workspace=ws, outs=res)
        return fwd, bwd, units, bf, bb, (N, plan.d_out)
    if "rowptr" in dev:
        N, E = w["N"], w["E"]
        x, Y = dev["x"], dev["Y"]
        WR = dev["W"] if "W" in dev else dev["R"]
        M = dev.get("M")
        units = E
        idx = 4 * (N + 1 + E)
        nin = N * plan.d1 + E * plan.d2 + WR.numel() + (M.numel() if M is not None else 0)
        bf = ei * nin + es * N * plan.d_out + idx
        bb = ei * (nin + N * plan.d_out) + es * nin + idx + 8 * E

        def fwd(out):
            return cg.cgtp_conv_forward(plan, graph, x, Y, WR, M, out=out)

        def bwd(g, outs):
            return cg.cgtp_conv_backward(plan, graph, g, x, Y, WR, M, outs=outs)
        out_shape = (N, plan.d_out)
    else:
        B = w["B"]
        x1, x2, W = dev["x1"], dev["x2"], dev["W"]
        units = B
        bf = es * (B * (plan.d1 + plan.d2 + plan.w_numel + plan.d_out))
        bb = es * (B * (2 * plan.d1 + 2 * plan.d2 + 2 * plan.w_numel + plan.d_out))

        def fwd(out):
            return cg.cgtp_forward(plan, x1, x2, W, out=out)

        def bwd(g, outs):
            return cg.cgtp_backward(plan, g, x1, x2, W)
        out_shape = (B, plan.d_out)
    return fwd, bwd, units, bf, bb, out_shape


def launches_per_step(cfgkey, plan, w):
    """Kernels of this library one timed step (forward + backward) launches."""
    if plan.mode == "mixed":   # uvw and uvu forwards, fold; unfold, uvu and uvw backwards, two adds
        return 8
    if CONFIGS[cfgkey].get("sh"):   # forward, backward, per-edge chain rule to the edge vectors
        return 3
    if plan.mode == "uvw" and plan.radial_k > 0:
        # per streamed node chunk: edge stage + node GEMM (forward); GEMM, edge stage,
        # two GEMMs and the split-K reduction (backward)
        v = int(os.environ.get("CGTP_UVW_CHUNK_NODES", "4096"))
        chunk = v if 1 <= v <= (1 << 20) else 4096
        return 7 * max(1, -(-w["N"] // chunk))
    return 2


def algorithmic_flops(plan, n_nodes, n_edges):
    """Algorithmic FLOPs of one forward and one backward launch (FMA = 2 flops).

    Per (edge, path) with D1 = 2l1+1, D3 = 2l3+1, NF = D1*D3 and nnz the CG
    nonzeros of the path:
      uvu forward : 2 nnz (cy = C.Y) + mul * (D1 + 2 NF)      (weight product, contraction)
      uvu backward: 4 nnz + mul * (6 NF + 3 D3)               (t, gW, w*g, gx, x (x) wg; C.Y and C.gc)
      uvw forward : 2 nnz + mul1 * 2 NF + 2 K mul1 D3 per edge, and the node GEMM
                    2 K mul1 mul_out D3 per node
      uvw backward: 4 nnz + 2 mul_out NF * 2 + 6 K mul_out D1 per edge, and three node
                    GEMMs (x M, M H, x^T H) of 2 K mul1 mul_out D1 each per node
    """
    fe = be = fn = bn = 0
    K = getattr(plan, "radial_k", 0)
    if plan.mode == "mixed":   # per instruction, with its own mode (the uvw ones with weights per edge)
        import clebsch_gordan_tensor_racah_gb300 as cg
        from clebsch_gordan_tensor_racah_gb300.workloads import irreps_terms
        a, b, o = (irreps_terms(s) for s in (plan.irreps[0], plan.irreps[1], plan.irreps[2]))
        for (i1, i2, io), m in zip(plan.instructions, plan.modes):
            (mul1, l1), (_, l2), (mul_out, l3) = a[i1], b[i2], o[io]
            D1, D3 = 2 * l1 + 1, 2 * l3 + 1
            NF, nnz = D1 * D3, int(np.count_nonzero(cg.cgtp_real_cg_block(l1, l2, l3)))
            if m == "uvu":
                fe += 2 * nnz + mul1 * (D1 + 2 * NF)
                be += 4 * nnz + mul1 * (6 * NF + 3 * D3)
            else:
                fe += 2 * nnz + mul1 * 2 * NF + 2 * mul1 * mul_out * D3
                be += 4 * nnz + mul1 * 4 * NF + 3 * 2 * mul1 * mul_out * D3 + 2 * mul1 * NF
        return fe * n_edges, be * n_edges
    for p in range(plan.n_paths):
        ints, C = plan.path(p)
        l1, l2, l3, mul1, mul_out = ints[:5]
        D1, D3 = 2 * l1 + 1, 2 * l3 + 1
        NF, nnz = D1 * D3, int(np.count_nonzero(C))
        if plan.mode == "uvu":
            fe += 2 * nnz + mul1 * (D1 + 2 * NF)
            be += 4 * nnz + mul1 * (6 * NF + 3 * D3)
        elif K == 0:   # weights per edge: t = C.x.Y, then the [u][w] matrix per edge
            fe += 2 * nnz + mul1 * 2 * NF + 2 * mul1 * mul_out * D3
            be += 4 * nnz + mul1 * 4 * NF + 3 * 2 * mul1 * mul_out * D3 + 2 * mul1 * NF
        else:
            fe += 2 * nnz + mul1 * 2 * NF + 2 * K * mul1 * D3
            fn += 2 * K * mul1 * mul_out * D3
            be += 4 * nnz + 4 * mul_out * NF + 6 * K * mul_out * D1
            bn += 3 * 2 * K * mul1 * mul_out * D1
    return fe * n_edges + fn * n_nodes, be * n_edges + bn * n_nodes


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


def time_oracle_sample(cfgkey, budget_s=8.0):
    """FP64 oracle on a bounded sample of the workload: (units/s, sample description)."""
    from clebsch_gordan_tensor_racah_gb300 import workloads as wl
    from oracle import conv as oconv, irreps as oirr
    c = CONFIGS[cfgkey]
    spec = wl.SPECS[c["name"]]
    if spec["mode"] == "mixed":
        lay = oconv.mixed_layout(spec["in1"], spec["in2"], spec["out"], spec["instructions"], spec["modes"])
        N = 60
        w = wl.make(c["name"], (lay[3], lay[4]), seed=0, dtype=c["dtype"], N=N)
        units, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            out = oconv.conv_mixed_forward(lay, w["x"], w["Y"], w["Wu"], w["Ww"], w["rowptr"], w["col"])
            oconv.conv_mixed_backward(lay, out, w["x"], w["Y"], w["Wu"], w["Ww"], w["rowptr"], w["col"])
            units += w["E"]
        dt = time.perf_counter() - t0
        return units / dt, f"{N}-node graph of the same recipe ({w['E']} edges), fwd+bwd repeated for {dt:.1f} s"
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], spec["mode"])
    if spec["graph"] is None:
        B = 64
        w = wl.make(c["name"], oplan.w_numel, seed=0, dtype=c["dtype"], B=B)
        units, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            out = oconv.tp_uvu_forward(oplan, w["x1"], w["x2"], w["W"])
            oconv.tp_uvu_backward(oplan, out, w["x1"], w["x2"], w["W"])
            units += B
        dt = time.perf_counter() - t0
        return units / dt, f"batches of {B} samples of the same recipe, fwd+bwd, {dt:.1f} s"
    # a smaller graph of the same recipe (same degree distribution and features)
    N = {"tiny": 64, "nequip": 120, "mace": 60, "uvw": 4, "uvw_edge": 120}[c["name"]]
    w = wl.make(c["name"], oplan.w_numel, seed=0, dtype="float32" if c["dtype"] == "bfloat16" else c["dtype"], N=N)
    units, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        if c.get("sh"):
            rv = np.random.default_rng(7).standard_normal((w["E"], 3))
            out = oconv.conv_uvu_forward_sh(oplan, w["x"], rv, w["W"], w["rowptr"], w["col"])
            oconv.conv_uvu_backward_sh(oplan, out, w["x"], rv, w["W"], w["rowptr"], w["col"])
        elif spec["mode"] == "uvu":
            out = oconv.conv_uvu_forward(oplan, w["x"], w["Y"], w["W"], w["rowptr"], w["col"])
            oconv.conv_uvu_backward(oplan, out, w["x"], w["Y"], w["W"], w["rowptr"], w["col"])
        elif "W" in w:
            out = oconv.conv_uvw_forward(oplan, w["x"], w["Y"], w["W"], w["rowptr"], w["col"])
            oconv.conv_uvw_backward(oplan, out, w["x"], w["Y"], w["W"], w["rowptr"], w["col"])
        else:
            out = oconv.conv_uvw_radial_forward(oplan, w["x"], w["Y"], w["R"], w["M"], w["rowptr"], w["col"])
            oconv.conv_uvw_radial_backward(oplan, out, w["x"], w["Y"], w["R"], w["M"], w["rowptr"], w["col"])
        units += w["E"]
    dt = time.perf_counter() - t0
    return units / dt, f"{N}-node graph of the same recipe ({w['E']} edges), fwd+bwd repeated for {dt:.1f} s"


def time_double_backward(plan, graph, w, dev, g, stream, units, roofline):
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
        n_op = 3   # x, Y and the weights (Wu, Ww) together: 3 forwards + 3 backwards of each single-mode plan
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
    roof = n_op * (roofline["fwd_roofline_ms"] + roofline["bwd_roofline_ms"])
    return {"ms": ms, "units_per_s": units / (ms / 1000.0), "launch_sequence": f"{n_op} forwards + {n_op} backwards + adds",
            "roofline_ms": roof, "frac": roof / ms}


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


def config_block(cfgkey, w, n_gpus):
    c = CONFIGS[cfgkey]
    spec = c["name"]
    d = {"workload": {"tiny": "tiny uvu conv (64 nodes, 512 edges)",
                      "nequip": "NequIP-like uvu conv (10k nodes x 32 in-edges, 32x(0e,1o,2e,3o), SH l<=3)",
                      "mace": "MACE-like uvu conv (5k nodes, Poisson(40) in-degree, 128x(0e,1o,2e), SH l<=3)",
                      "highl": "high-L batched TP (B=50k, 16x l=0..7, SH l<=7)",
                      "uvw": "uvw radial conv (200k nodes x 32 in-edges, 64x(0e,1o,2e), K=8)",
                      "uvw_edge": "uvw conv with per-edge weights (10k nodes x 32 in-edges, 16x(0e,1o,2e))",
                      "mixed": "mixed uvu/uvw conv (10k nodes x 32 in-edges, 32x(0e,1o,2e), SH l<=2; "
                               "0e outputs uvw with per-edge weights, 1o and 2e outputs uvu)"}[spec],
         "step": "conv forward + backward" if "N" in w else "batched forward + backward",
         "precision": "bfloat16 inputs, FP32 arithmetic and outputs" if c["dtype"] == "bfloat16" else c["dtype"],
         "edge_features": "raw edge vectors, harmonics evaluated in the kernels" if c.get("sh") else "harmonics Y",
         "l2": "inputs larger than L2 (no flush needed)",
         "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU"}
    if "N" in w:
        d.update(nodes=w["N"], edges=w["E"])
    else:
        d.update(batch=w["B"])
    return d


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cfgkey = args.config
    t_steps = []
    rate = None
    for i in range(args.warmup + args.steps):
        r, desc = time_oracle_sample(cfgkey, budget_s=max(2.0, 40.0 / max(1, args.warmup + args.steps)))
        if i >= args.warmup:
            t_steps.append(r)
    rate = float(np.median(t_steps))
    from clebsch_gordan_tensor_racah_gb300 import workloads as wl
    c = CONFIGS[cfgkey]
    units = wl.SPECS[c["name"]].get("N", 0) * wl.SPECS[c["name"]].get("deg", 0) or wl.SPECS[c["name"]].get("B") or 512
    line = {"metric": METRIC, "value": rate, "unit": "edges/s" if cfgkey != "highl" else "samples/s",
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * units / rate, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": config_block(cfgkey, {"N": 1, "E": 0} if cfgkey != "highl" else {"B": 1}, 1)["workload"]},
            "cpu_baseline": {"value": rate, "unit": "edges/s" if cfgkey != "highl" else "samples/s",
                             "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": rate, "unit": "edges/s" if cfgkey != "highl" else "samples/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="nequip", choices=sorted(CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-double-backward", action="store_true",
                    help="skip the (untimed-for-the-metric) second-derivative measurement")
    ap.add_argument("--nodes", type=int, default=None,
                    help="smaller instance of the same recipe (nodes, or batch for highl)")
    ap.add_argument("--profile-run", action="store_true",
                    help="build, two warm-up steps and one step, no timing or JSON (for ncu captures)")
    args = ap.parse_args()
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

    plan, graph, w, host, dev, spec, tdt = build_inputs(args.config, device, args.nodes)
    fwd, bwd, units, bf, bb, out_shape = step_fns(args.config, plan, graph, w, dev, tdt)
    g = torch.randn(out_shape, dtype=tdt, device=device, generator=torch.Generator(device).manual_seed(1))
    out = torch.empty(out_shape, dtype=plan.out_dtype, device=device)
    stream = torch.cuda.current_stream()

    def step():
        fwd(out)
        return bwd(g, None)

    if args.profile_run:
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        print(f"profile run done: {args.config}, {units} units", flush=True)
        return

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # per-kernel split (events on the launching stream)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    tf, tb = [], []
    for _ in range(3):
        ev[0].record(stream)
        fwd(out)
        ev[1].record(stream)
        bwd(g, None)
        ev[2].record(stream)
        torch.cuda.synchronize()
        tf.append(ev[0].elapsed_time(ev[1]))
        tb.append(ev[1].elapsed_time(ev[2]))
    # timed region
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fe = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    be = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e0.record(stream)
    for i in range(args.steps):
        fe[i].record(stream)
        fwd(out)
        be[i].record(stream)
        bwd(g, None)
    fe[args.steps].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    fwd_ms = float(np.mean([fe[i].elapsed_time(be[i]) for i in range(args.steps)]))
    bwd_ms = float(np.mean([be[i].elapsed_time(fe[i + 1]) for i in range(args.steps)]))
    ms, value = job_throughput(ms, units, world, device)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        pin = {k: (v if isinstance(v, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(v))).pin_memory()
               for k, v in host.items() if k not in ("rowptr", "col")}
        gh = g.cpu().pin_memory()
        out_h = torch.empty(out_shape, dtype=plan.out_dtype).pin_memory()
        res_h = None
        h2d = sum(t.numel() * t.element_size() for t in pin.values()) + gh.numel() * gh.element_size()

        def e2e_step():
            nonlocal res_h
            for k, t in pin.items():
                dev[k].copy_(t, non_blocking=True)
            g.copy_(gh, non_blocking=True)
            fwd(out)
            r = bwd(g, None)
            out_h.copy_(out, non_blocking=True)
            if res_h is None:
                res_h = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in r if x is not None]
            for hbuf, x in zip(res_h, [x for x in r if x is not None]):
                hbuf.copy_(x, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        d2h = out_h.numel() * out_h.element_size() + sum(t.numel() * t.element_size() for t in res_h)
        k2 = max(3, args.steps // 4)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k2):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / k2
        e2e = {"value": world * units / (e2e_ms / 1000.0), "unit": "edges/s" if "N" in w else "samples/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    pk = peaks()
    mhz = (clk or {}).get("sm_max_mhz") or pk["sm_max_mhz"]
    dt_name = "f64" if tdt == torch.float64 else "f32"
    alu_peak = alu_peak_tflops(dt_name, mhz)
    n_nodes = w.get("N", w.get("B", 0))
    ff, fb = algorithmic_flops(plan, n_nodes, units)
    dominant = "backward" if bwd_ms >= fwd_ms else "forward"
    dom_ms = bwd_ms if dominant == "backward" else fwd_ms
    dom_bytes = bb if dominant == "backward" else bf
    dom_flops = fb if dominant == "backward" else ff
    t_hbm = dom_bytes / (pk["hbm_gbs"] * 1e9)
    t_alu = dom_flops / (alu_peak * 1e12)
    kname = {("uvu", "forward"): "uvu_forward3_kernel", ("uvu", "backward"): "uvu_backward3_kernel",
             ("uvwe", "forward"): "uvwe_fwd_kernel", ("uvwe", "backward"): "uvwe_bwd_kernel",
             ("mixed", "forward"): "mixed forward (uvu_forward3_kernel + uvwe_fwd_kernel + fold)",
             ("mixed", "backward"): "mixed backward (uvu_backward3_kernel + uvwe_bwd_kernel + adds)",
             ("uvw", "forward"): "uvw forward (edge stage + node GEMM)",
             ("uvw", "backward"): "uvw backward (node GEMMs + edge stage)"}[
        ("uvwe" if plan.mode == "uvw" and plan.radial_k == 0 else plan.mode, dominant)]
    launches = launches_per_step(args.config, plan, w) * args.steps
    if "N" not in w:
        kname = {"forward": "bt_forward_kernel", "backward": "bt_backward_kernel"}[dominant]
    if t_hbm >= t_alu:
        achieved = dom_bytes / (dom_ms / 1000.0) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / pk["hbm_gbs"], "peak_src": pk["src"] + " (copy bandwidth)"}
    else:
        achieved = dom_flops / (dom_ms / 1000.0) / 1e12
        roofline = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                    "frac": achieved / alu_peak,
                    "peak_src": f"derived: 152 SMs x 128 FP32 lanes x 2 x {mhz:.0f} MHz" if dt_name == "f32"
                    else "nominal FP64 1.25 TFLOP/s"}
    roofline.update({"kernel": kname, "traffic": traffic_for(kname, args.config, dom_bytes),
                     "algorithmic_bytes_per_launch": int(dom_bytes), "algorithmic_flops_per_launch": int(dom_flops),
                     "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                     "fwd_roofline_ms": 1000 * max(bf / (pk["hbm_gbs"] * 1e9), ff / (alu_peak * 1e12)),
                     "bwd_roofline_ms": 1000 * max(bb / (pk["hbm_gbs"] * 1e9), fb / (alu_peak * 1e12))})
    roofline["step_frac"] = (roofline["fwd_roofline_ms"] + roofline["bwd_roofline_ms"]) / (fwd_ms + bwd_ms)
    line = {"metric": METRIC, "value": value, "unit": "edges/s" if "N" in w else "samples/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {torch.float64: "f64", torch.bfloat16: "bf16 inputs, f32 arithmetic"}.get(tdt, "f32"),
            "data": "synthetic",
            "config": config_block(args.config, w, world),
            "fwd_units_per_s": world * units / (fwd_ms / 1000.0),
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk}
    if not args.no_double_backward and tdt != torch.bfloat16 and not CONFIGS[args.config].get("sh"):
        line["double_backward"] = time_double_backward(plan, graph, w, dev, g, stream, units, roofline)
    if rank == 0 and not args.no_cpu_baseline:
        rate, desc = time_oracle_sample(args.config)
        line["cpu_baseline"] = {"value": rate, "unit": line["unit"], "cores": 1, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
