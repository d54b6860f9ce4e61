"""GPU parity of the uvw convolution with a weight matrix per edge (radial_k = 0)
against the FP64 oracle: max|err| <= 1e-4 * max|ref| (FP32), <= 1e-10 * max|ref|
(FP64), for out, gx, gY, gW and the double backward.  Mixed multiplicities, empty
rows and a ragged graph are part of the recipe.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from oracle import conv as oconv, irreps as oirr  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = {np.float32: 1e-4, np.float64: 1e-10}


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def close(name, got, ref, dtype):
    got = got.cpu().numpy().astype(np.float64)
    err, scale = np.abs(got - ref).max(), np.abs(ref).max()
    assert err <= TOL[dtype] * scale, f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


def graph_of(rng, N, E):
    src = rng.integers(0, N, E)
    dst = rng.integers(0, N - 2, E)          # the last two receivers have no in-edges
    order = np.argsort(dst, kind="stable")
    rowptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))]).astype(np.int32)
    return rowptr, src[order].astype(np.int32)


@pytest.mark.parametrize("dtype,in1,out", [
    (np.float32, "16x0e+16x1o+16x2e", "16x0e+16x1o+16x2e"),
    (np.float64, "12x0e+5x1o+3x2e+2x3o", "7x0e+9x1o+4x2e+3x3o"),
])
def test_uvw_per_edge_weights(dtype, in1, out):
    rng = np.random.default_rng(12)
    in2 = "0e+1o+2e+3o"
    oplan = oirr.make_plan(in1, in2, out, "uvw")
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.Plan(in1, in2, out, "uvw", tdt, radial_k=0)
    assert plan.w_numel == oplan.w_numel
    N, E = 40, 300
    rowptr, col = graph_of(rng, N, E)
    x = rng.standard_normal((N, oplan.d1)).astype(dtype)
    Y = rng.standard_normal((E, oplan.d2)).astype(dtype)
    W = (rng.standard_normal((E, oplan.w_numel)) / 4).astype(dtype)
    graph = cg.Graph(T(rowptr), T(col), N)
    o = cg.cgtp_conv_forward(plan, graph, T(x), T(Y), T(W))
    close("out", o, oconv.conv_uvw_forward(oplan, x, Y, W, rowptr, col), dtype)
    g = rng.standard_normal((N, oplan.d_out)).astype(dtype)
    gx, gY, gW, gM = cg.cgtp_conv_backward(plan, graph, T(g), T(x), T(Y), T(W))
    assert gM is None
    for nm, a, b in zip(("gx", "gY", "gW"), (gx, gY, gW), oconv.conv_uvw_backward(oplan, g, x, Y, W, rowptr, col)):
        close(nm, a, b, dtype)
    c = [rng.standard_normal(a.shape).astype(dtype) for a in (x, Y, W)]
    got = cg.cgtp_conv_double_backward(plan, graph, T(g), T(x), T(Y), T(W), *(T(v) for v in c))
    ref = oconv.conv_uvw_double_backward(oplan, g, x, Y, W, *c, rowptr, col)
    for nm, a, b in zip(("d_gout", "d_x", "d_Y", "d_W"), got[:4], ref):
        close(nm, a, b, dtype)


def test_uvw_per_edge_two_plans_dense_rows():
    """A larger plan stays usable after a smaller one is created (the kernels'
    shared-memory limit is per kernel, not per plan), on rows of about 40 edges
    (five chunks of eight and a ragged tail per receiver)."""
    rng = np.random.default_rng(5)
    in2 = "0e+1o+2e+3o"
    big = ("16x0e+16x1o+16x2e+8x3o", "16x0e+16x1o+16x2e+8x3o")
    oplan = oirr.make_plan(big[0], in2, big[1], "uvw")
    plan = cg.Plan(big[0], in2, big[1], "uvw", torch.float32, radial_k=0)
    small = cg.Plan("2x0e", "0e", "2x0e", "uvw", torch.float32, radial_k=0)
    N, E = 12, 470
    rowptr, col = graph_of(rng, N, E)
    x = rng.standard_normal((N, oplan.d1)).astype(np.float32)
    Y = rng.standard_normal((E, oplan.d2)).astype(np.float32)
    W = (rng.standard_normal((E, oplan.w_numel)) / 4).astype(np.float32)
    graph = cg.Graph(T(rowptr), T(col), N)
    o = cg.cgtp_conv_forward(plan, graph, T(x), T(Y), T(W))
    close("out", o, oconv.conv_uvw_forward(oplan, x, Y, W, rowptr, col), np.float32)
    g = rng.standard_normal((N, oplan.d_out)).astype(np.float32)
    got = cg.cgtp_conv_backward(plan, graph, T(g), T(x), T(Y), T(W))
    for nm, a, b in zip(("gx", "gY", "gW"), got[:3], oconv.conv_uvw_backward(oplan, g, x, Y, W, rowptr, col)):
        close(nm, a, b, np.float32)
    del small
