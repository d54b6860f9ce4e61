"""Full-size parity of the uvu workloads as bench.py times them.

At full size the oracle evaluates sampled outputs one by one: rows of out for
sampled receivers, gW / gY for sampled edges, gx for sampled senders (all their
out-edges), rows of the batched product; plus the homogeneity identities
<g,out> = <gx,x> = <gY,Y> = <gW,W> which hold at any size.
Tolerances: 1e-4 * max|ref| (FP32), 1e-10 * max|ref| (FP64) on the sampled rows;
the identities to 1e-4 (FP32) / 1e-9 (FP64) relative.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from clebsch_gordan_tensor_racah_gb300 import workloads as wl  # noqa: E402
from oracle import conv as oconv, graph as ograph, irreps as oirr  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = {np.dtype(np.float32): 1e-4, np.dtype(np.float64): 1e-10}


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def close(name, got, ref, tol):
    got = got.detach().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, np.float64)
    err, scale = np.abs(got - ref).max(), np.abs(ref).max()
    assert err <= tol * scale, f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


def homogeneity(g, out, pairs, tol):
    """<g, out> = <a, d out/d a . g> for every input a the output is linear in.

    Both sides are sums of many products of either sign that cancel heavily, so
    the rounding error is bounded relative to the sum of |products|, not to the
    cancelled result."""
    ref_terms = g.double() * out.double()
    ref, ref_abs = float(ref_terms.sum()), float(ref_terms.abs().sum())
    for nm, a, ga in pairs:
        terms = a.double() * ga.double()
        v, v_abs = float(terms.sum()), float(terms.abs().sum())
        assert abs(v - ref) <= tol * max(v_abs, ref_abs), (nm, v, ref, v_abs, ref_abs)


@pytest.mark.parametrize("name,dtype", [("nequip", np.float32), ("mace", np.float32), ("mace", np.float64)])
def test_conv_full_size_sampled(name, dtype):
    spec = wl.SPECS[name]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", tdt)
    w = wl.make(name, oplan.w_numel, seed=0, dtype=dtype)
    d = {k: T(v) for k, v in w.items() if isinstance(v, np.ndarray)}
    graph = cg.Graph(d["rowptr"], d["col"], w["N"])
    out = cg.cgtp_conv_forward(plan, graph, d["x"], d["Y"], d["W"])
    g = torch.randn(out.shape, dtype=tdt, device="cuda", generator=torch.Generator("cuda").manual_seed(3))
    gx, gY, gW, _ = cg.cgtp_conv_backward(plan, graph, g, d["x"], d["Y"], d["W"])
    tol = TOL[np.dtype(dtype)]
    rng = np.random.default_rng(5)
    N, E = w["N"], w["E"]
    deg = np.diff(w["rowptr"])
    # first and last rows, the longest and the shortest rows, random rows
    nodes = np.unique(np.concatenate([[0, N - 1, int(np.argmax(deg)), int(np.argmin(deg))], rng.integers(0, N, 14)]))
    ref = oconv.conv_uvu_forward(oplan, w["x"], w["Y"], w["W"], w["rowptr"], w["col"], nodes=nodes)
    close("out[sampled]", out[T(nodes)], ref, tol)
    gh = g.cpu().numpy()
    edges = np.unique(np.concatenate([[0, E - 1], rng.integers(0, E, 30)]))
    _, rgY, rgW = oconv.conv_uvu_backward(oplan, gh, w["x"], w["Y"], w["W"], w["rowptr"], w["col"], edges=edges)
    close("gY[sampled]", gY[T(edges)], rgY, tol)
    close("gW[sampled]", gW[T(edges)], rgW, tol)
    t_rowptr, t_eid, _ = ograph.transpose(w["rowptr"], w["col"], N)
    senders = np.unique(rng.integers(0, N, 6))
    sedges = np.concatenate([t_eid[t_rowptr[s]:t_rowptr[s + 1]] for s in senders])
    rgx, _, _ = oconv.conv_uvu_backward(oplan, gh, w["x"], w["Y"], w["W"], w["rowptr"], w["col"], edges=sedges)
    close("gx[sampled]", gx[T(senders)], rgx[senders], tol)
    itol = 1e-6 if dtype == np.float32 else 1e-13
    homogeneity(g, out, (("x", d["x"], gx), ("Y", d["Y"], gY), ("W", d["W"], gW)), itol)


def test_batched_high_l_full_size_sampled():
    spec = wl.SPECS["highl"]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", torch.float32)
    w = wl.make("highl", oplan.w_numel, seed=0)
    x1, x2, W = T(w["x1"]), T(w["x2"]), T(w["W"])
    out = cg.cgtp_forward(plan, x1, x2, W)
    rows = np.unique(np.concatenate([[0, w["B"] - 1], np.random.default_rng(2).integers(0, w["B"], 10)]))
    close("out[sampled]", out[T(rows)], oconv.tp_uvu_forward(oplan, w["x1"][rows], w["x2"][rows], w["W"][rows]), 1e-4)
    g = torch.randn(out.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(4))
    gx1, gx2, gW = cg.cgtp_backward(plan, g, x1, x2, W)
    r1, r2, rW = oconv.tp_uvu_backward(oplan, g[T(rows)].cpu().numpy(), w["x1"][rows], w["x2"][rows], w["W"][rows])
    close("gx1[sampled]", gx1[T(rows)], r1, 1e-4)
    close("gx2[sampled]", gx2[T(rows)], r2, 1e-4)
    close("gW[sampled]", gW[T(rows)], rW, 1e-4)
    homogeneity(g, out, (("x1", x1, gx1), ("x2", x2, gx2), ("W", W, gW)), 1e-6)
