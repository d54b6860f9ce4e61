"""GPU parity of the streamed uvw radial convolution (fully connected mixing,
W_e = R[e] @ M never formed) against the FP64 oracle, which forms W_e per edge.

Tolerance: max|err| <= 1e-4 * max|ref| per output tensor (FP32).  The node-chunk
size is lowered through cgtp_plan_set_node_chunk so several chunks (and a ragged
last chunk) are exercised on graphs the oracle evaluates in seconds; the full
200k-node workload is checked on sampled nodes, edges and gM entries plus the
homogeneity identities <g,out> = <gx,x> = <gY,Y> = <gR,R> = <gM,M>.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from clebsch_gordan_tensor_racah_gb300 import workloads as wl  # noqa: E402
from oracle import conv as oconv, graph as ograph, irreps as oirr  # noqa: E402

pytestmark = pytest.mark.gpu


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def close(name, got, ref, tol=1e-4):
    got = got.detach().cpu().numpy().astype(np.float64) if hasattr(got, "detach") else np.asarray(got)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
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


def make(N, chunk=None, seed=0, in1=None, out=None, in2=None):
    spec = dict(wl.SPECS["uvw"])
    if in1:
        spec.update(in1=in1, out=out, in2=in2)
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvw", torch.float32, radial_k=8)
    if chunk:
        plan.set_node_chunk(chunk)
        assert plan.node_chunk == chunk
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvw")
    over = dict(N=N)
    if in1:
        over.update(in1=in1, out=out, in2=in2, lmax_sh=max(int(t[0]) for t in in2.split("+")))
    w = wl.make("uvw", oplan.w_numel, seed=seed, **over)
    return plan, oplan, w


def run(plan, oplan, w, check_grad=True):
    d = {k: T(v) for k, v in w.items() if isinstance(v, np.ndarray)}
    graph = cg.Graph(d["rowptr"], d["col"], w["N"])
    out = cg.cgtp_conv_forward(plan, graph, d["x"], d["Y"], d["R"], d["M"])
    ref = oconv.conv_uvw_radial_forward(oplan, w["x"], w["Y"], w["R"], w["M"], w["rowptr"], w["col"])
    close("out", out, ref)
    if check_grad:
        g = np.random.default_rng(7).standard_normal(ref.shape).astype(np.float32)
        gx, gY, gR, gM = cg.cgtp_conv_backward(plan, graph, T(g), d["x"], d["Y"], d["R"], d["M"])
        rgx, rgY, rgR, rgM = oconv.conv_uvw_radial_backward(oplan, g, w["x"], w["Y"], w["R"], w["M"],
                                                            w["rowptr"], w["col"])
        close("gx", gx, rgx)
        close("gY", gY, rgY)
        close("gR", gR, rgR)
        close("gM", gM, rgM)


def test_uvw_small_single_chunk():
    plan, oplan, w = make(40)
    run(plan, oplan, w)


def test_uvw_several_chunks_ragged_tail():
    plan, oplan, w = make(70, chunk=16)
    run(plan, oplan, w)


def test_uvw_mixed_multiplicities():
    plan, oplan, w = make(30, chunk=8, in1="48x0e+40x1o+8x2e", out="24x0e+72x1o+16x2e", in2="0e+1o+2e")
    run(plan, oplan, w)


def test_uvw_full_size_sampled():
    """200,000 nodes x 32 in-edges, run as timed by bench.py (default chunking)."""
    plan, oplan, w = make(200_000)
    d = {k: T(v) for k, v in w.items() if isinstance(v, np.ndarray)}
    graph = cg.Graph(d["rowptr"], d["col"], w["N"])
    torch.cuda.reset_peak_memory_stats()
    out = cg.cgtp_conv_forward(plan, graph, d["x"], d["Y"], d["R"], d["M"])
    rng = np.random.default_rng(11)
    c = plan.node_chunk   # rows on both sides of the first chunk boundary
    nodes = np.concatenate([[0, 1, c - 1, c, c + 1, 199_999], rng.integers(0, 200_000, 10)])
    ref = oconv.conv_uvw_radial_forward(oplan, w["x"], w["Y"], w["R"], w["M"], w["rowptr"], w["col"], nodes=nodes)
    close("out[sampled]", out[torch.from_numpy(nodes).cuda()], ref)
    g = torch.randn(out.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(5))
    gx, gY, gR, gM = cg.cgtp_conv_backward(plan, graph, g, d["x"], d["Y"], d["R"], d["M"])
    gh = g.cpu().numpy()
    # sampled edges (gY, gR) and sampled senders (gx: all their out-edges)
    edges = rng.integers(0, w["E"], 12)
    _, rgY, rgR, _ = oconv.conv_uvw_radial_backward(oplan, gh, w["x"], w["Y"], w["R"], w["M"], w["rowptr"],
                                                    w["col"], edges=edges)
    close("gY[sampled]", gY[torch.from_numpy(edges).cuda()], rgY)
    close("gR[sampled]", gR[torch.from_numpy(edges).cuda()], rgR)
    t_rowptr, t_eid, _ = ograph.transpose(w["rowptr"], w["col"], w["N"])
    senders = np.array([3, c, 150_000])
    sedges = np.concatenate([t_eid[t_rowptr[s]:t_rowptr[s + 1]] for s in senders])
    rgx, _, _, _ = oconv.conv_uvw_radial_backward(oplan, gh, w["x"], w["Y"], w["R"], w["M"], w["rowptr"],
                                                  w["col"], edges=sedges)
    close("gx[sampled]", gx[torch.from_numpy(senders).cuda()], rgx[senders])
    # one whole (k, path) slice of gM, and sampled entries of other slices; every bound
    # scales with the oracle's slice, not with the GPU's own output
    gMh = gM.cpu().numpy()
    k, pi = 3, 5
    q = oplan.paths[pi]
    rsl = oconv.conv_uvw_radial_gM_slice(oplan, gh, w["x"], w["Y"], w["R"], w["rowptr"], w["col"], k, pi)
    close(f"gM[{k}][path {pi}]", gMh[k, q.woff:q.woff + q.mul1 * q.mul_out].reshape(q.mul1, q.mul_out), rsl)
    ent = [(0, 0, 0, 0), (7, 10, 63, 5), (5, 7, 2, 63)]
    rgm = oconv.conv_uvw_radial_gM_entries(oplan, gh, w["x"], w["Y"], w["R"], w["rowptr"], w["col"], ent)
    got = [gMh[kk, oplan.paths[p].woff + u * oplan.paths[p].mul_out + ww] for (kk, p, u, ww) in ent]
    assert np.abs(np.array(got) - rgm).max() <= 1e-4 * np.abs(rsl).max()
    # homogeneity: out is linear in each of x, Y, R and M
    homogeneity(g, out, (("x", d["x"], gx), ("Y", d["Y"], gY), ("R", d["R"], gR), ("M", d["M"], gM)), 1e-6)
    # bounded workspace: nothing edge-sized beyond inputs/outputs
    peak = torch.cuda.max_memory_allocated()
    assert peak < 12e9, peak
