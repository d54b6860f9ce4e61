"""Full-size parity of the per-edge-weight workloads as bench.py times them: uvw
with a weight matrix per edge and the mixed uvu/uvw instruction list (10,000
nodes x 32 in-edges each).

The oracle evaluates sampled outputs on sub-graphs that hold every edge the
sample depends on: all in-edges of sampled receivers (rows of out), the sampled
edges themselves (gY, gW rows), all out-edges of sampled senders (rows of gx).
The homogeneity identities <g,out> = <gx,x> = <gY,Y> = <gW,W> (mixed:
<gWu,Wu> + <gWw,Ww>) hold at any size.  Tolerances: 1e-4 * max|ref| on sampled
rows (FP32); identities to 1e-5 relative to the sum of |products|.

The sub-graph construction itself is checked on the CPU against the full oracle.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from clebsch_gordan_tensor_racah_gb300 import workloads as wl  # noqa: E402
from oracle import conv as oconv, graph as ograph, irreps as oirr  # noqa: E402


def sub_csr(rowptr, col, edges):
    """CSR of the CSR positions `edges` over the same nodes: (rowptr', col', sorted edges)."""
    edges = np.unique(np.asarray(edges, dtype=np.int64))
    N = len(rowptr) - 1
    dst = ograph.csr_dst(rowptr)[edges]
    rp = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))]).astype(np.int64)
    return rp, np.asarray(col, dtype=np.int64)[edges], edges


def in_edges(rowptr, nodes):
    return np.concatenate([np.arange(rowptr[n], rowptr[n + 1]) for n in nodes]).astype(np.int64)


def out_edges(rowptr, col, senders):
    t_rowptr, t_eid, _ = ograph.transpose(rowptr, col, len(rowptr) - 1)
    return np.concatenate([t_eid[t_rowptr[s]:t_rowptr[s + 1]] for s in senders]).astype(np.int64)


class Uvwe:
    """Oracle side of the per-edge uvw convolution on a sub-graph."""

    def __init__(self, spec):
        self.p = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvw")

    def fwd(self, x, Y, Ws, rp, cl):
        return oconv.conv_uvw_forward(self.p, x, Y, Ws[0], rp, cl)

    def bwd(self, g, x, Y, Ws, rp, cl):
        gx, gY, gW = oconv.conv_uvw_backward(self.p, g, x, Y, Ws[0], rp, cl)
        return gx, gY, (gW,)


class Mixed:
    def __init__(self, spec):
        self.lay = oconv.mixed_layout(spec["in1"], spec["in2"], spec["out"], spec["instructions"], spec["modes"])

    def fwd(self, x, Y, Ws, rp, cl):
        return oconv.conv_mixed_forward(self.lay, x, Y, Ws[0], Ws[1], rp, cl)

    def bwd(self, g, x, Y, Ws, rp, cl):
        gx, gY, gWu, gWw = oconv.conv_mixed_backward(self.lay, g, x, Y, Ws[0], Ws[1], rp, cl)
        return gx, gY, (gWu, gWw)


def sampled_refs(orc, g, x, Y, Ws, rowptr, col, nodes, edges, senders):
    """(out rows of nodes, (gY, gW...) rows of sorted edges, gx rows of senders)."""
    rp, cl, e = sub_csr(rowptr, col, in_edges(rowptr, nodes))
    out = orc.fwd(x, Y[e], [W[e] for W in Ws], rp, cl)[nodes]
    rp, cl, es = sub_csr(rowptr, col, edges)
    _, gY, gWs = orc.bwd(g, x, Y[es], [W[es] for W in Ws], rp, cl)
    rp, cl, e = sub_csr(rowptr, col, out_edges(rowptr, col, senders))
    gx = orc.bwd(g, x, Y[e], [W[e] for W in Ws], rp, cl)[0][senders]
    return out, es, (gY, gWs), gx


def test_sub_graph_sampling_matches_the_full_oracle():
    """CPU: the sampled references equal the full oracle's rows on a small graph of each recipe."""
    rng = np.random.default_rng(9)
    for name, orc_cls, ws_keys in (("uvw_edge", Uvwe, ("W",)), ("mixed", Mixed, ("Wu", "Ww"))):
        spec = wl.SPECS[name]
        orc = orc_cls(spec)
        w_numel = orc.p.w_numel if name == "uvw_edge" else (orc.lay[3], orc.lay[4])
        w = wl.make(name, w_numel, seed=1, dtype="float64", N=40, deg=6)
        Ws = [w[k] for k in ws_keys]
        N, E = w["N"], w["E"]
        g = rng.standard_normal((N, orc.fwd(w["x"], w["Y"], Ws, w["rowptr"], w["col"]).shape[1]))
        full_out = orc.fwd(w["x"], w["Y"], Ws, w["rowptr"], w["col"])
        full_gx, full_gY, full_gWs = orc.bwd(g, w["x"], w["Y"], Ws, w["rowptr"], w["col"])
        nodes = np.array([0, 7, 39])
        edges = np.array([E - 1, 3, 0, 17])
        senders = np.array([2, 39])
        out, es, (gY, gWs), gx = sampled_refs(orc, g, w["x"], w["Y"], Ws, w["rowptr"], w["col"], nodes, edges,
                                              senders)
        np.testing.assert_allclose(out, full_out[nodes], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(gY, full_gY[es], rtol=1e-12, atol=1e-12)
        for a, b in zip(gWs, full_gWs):
            np.testing.assert_allclose(a, b[es], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(gx, full_gx[senders], rtol=1e-12, atol=1e-12)


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def close(name, got, ref, tol=1e-4):
    got = got.detach().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, np.float64)
    err, scale = np.abs(got - ref).max(), np.abs(ref).max()
    assert err <= tol * scale, f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


def homogeneity(g, out, pairs, tol):
    """<g, out> = sum over the listed inputs a of <a, dL/da>, to tol relative to the sum of |products|."""
    ref_terms = g.double() * out.double()
    ref, ref_abs = float(ref_terms.sum()), float(ref_terms.abs().sum())
    for names, group in pairs:
        v = v_abs = 0.0
        for a, ga in group:
            terms = a.double() * ga.double()
            v, v_abs = v + float(terms.sum()), v_abs + float(terms.abs().sum())
            del terms
        assert abs(v - ref) <= tol * max(v_abs, ref_abs), (names, v, ref, v_abs, ref_abs)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["uvw_edge", "mixed"])
def test_per_edge_weights_full_size_sampled(name):
    spec = wl.SPECS[name]
    if name == "uvw_edge":
        orc = Uvwe(spec)
        plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvw", torch.float32, radial_k=0)
        w = wl.make(name, plan.w_numel, seed=0)
        keys = ("W",)
    else:
        orc = Mixed(spec)
        plan = cg.MixedPlan(spec["in1"], spec["in2"], spec["out"], spec["instructions"], spec["modes"],
                            torch.float32)
        w = wl.make(name, (plan.wu_numel, plan.ww_numel), seed=0)
        keys = ("Wu", "Ww")
    d = {k: T(v) for k, v in w.items() if isinstance(v, np.ndarray)}
    graph = cg.Graph(d["rowptr"], d["col"], w["N"])
    if name == "uvw_edge":
        out = cg.cgtp_conv_forward(plan, graph, d["x"], d["Y"], d["W"])
    else:
        out = cg.cgtp_mixed_conv_forward(plan, graph, d["x"], d["Y"], d["Wu"], d["Ww"])
    g = torch.randn(out.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(3))
    if name == "uvw_edge":
        gx, gY, gW, _ = cg.cgtp_conv_backward(plan, graph, g, d["x"], d["Y"], d["W"])
        gWs = (gW,)
    else:
        gx, gY, gWu, gWw = cg.cgtp_mixed_conv_backward(plan, graph, g, d["x"], d["Y"], d["Wu"], d["Ww"])
        gWs = (gWu, gWw)
    rng = np.random.default_rng(5)
    N, E = w["N"], w["E"]
    nodes = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 14)]))
    edges = np.concatenate([[0, E - 1], rng.integers(0, E, 30)])
    senders = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 4)]))
    Ws = [w[k] for k in keys]
    ref_out, es, (rgY, rgWs), rgx = sampled_refs(orc, g.cpu().numpy(), w["x"], w["Y"], Ws, w["rowptr"], w["col"],
                                                 nodes, edges, senders)
    close("out[sampled]", out[T(nodes)], ref_out)
    close("gY[sampled]", gY[T(es)], rgY)
    for k, a, b in zip(keys, gWs, rgWs):
        close(f"g{k}[sampled]", a[T(es)], b)
    close("gx[sampled]", gx[T(senders)], rgx)
    homogeneity(g, out, ((("x",), ((d["x"], gx),)), (("Y",), ((d["Y"], gY),)),
                         (keys, tuple((d[k], gw) for k, gw in zip(keys, gWs)))), 1e-5)
