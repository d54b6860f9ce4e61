"""GPU parity of the convolution with mixed uvu/uvw instruction lists against the
FP64 oracle: max|err| <= 1e-4 * max|ref| (FP32), <= 1e-10 * max|ref| (FP64), for
out, gx, gY, gWu, gWw and the double backward.  Ragged graphs with empty rows;
mixed lists, all-uvu and all-uvw lists; several instructions folding into the
same output block.
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
    assert got is not None, name
    got = got.cpu().numpy().astype(np.float64)
    err, scale = np.abs(got - ref).max(), np.abs(ref).max()
    assert err <= TOL[dtype] * scale, f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


def graph_of(rng, N, E):
    src = rng.integers(0, N, E)
    dst = rng.integers(0, N - 2, E)          # the last two receivers have no in-edges
    order = np.argsort(dst, kind="stable")
    rowptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))]).astype(np.int32)
    return rowptr, src[order].astype(np.int32)


def all_instructions(in1, in2, out):
    a, b, o = oirr.parse_irreps(in1), oirr.parse_irreps(in2), oirr.parse_irreps(out)
    ins = []
    for i1, (_, l1, p1) in enumerate(a):
        for i2, (_, l2, p2) in enumerate(b):
            for io, (_, l3, p3) in enumerate(o):
                if abs(l1 - l2) <= l3 <= l1 + l2 and p3 == p1 * p2:
                    ins.append((i1, i2, io))
    return ins


CASES = [
    # FP32, multiplicity 32 (the uvu part runs the baked kernels): scalar outputs fully
    # connected, the others channel-wise
    (np.float32, "32x0e+32x1o+32x2e", "0e+1o+2e", "32x0e+32x1o+32x2e", "l3==0"),
    # FP64, mixed multiplicities; uvw blocks change multiplicity
    (np.float64, "4x0e+4x1o+2x2e", "0e+1o+2e", "4x0e+4x1o+3x2e", "mul"),
    # degenerate lists
    (np.float32, "8x0e+8x1o", "0e+1o", "8x0e+8x1o", "uvu"),
    (np.float32, "8x0e+8x1o", "0e+1o", "8x0e+8x1o", "uvw"),
]


def modes_for(rule, ins, in1, out):
    a, o = oirr.parse_irreps(in1), oirr.parse_irreps(out)
    if rule in ("uvu", "uvw"):
        return [rule] * len(ins)
    if rule == "l3==0":
        return ["uvw" if o[io][1] == 0 else "uvu" for (_, _, io) in ins]
    return ["uvu" if a[i1][0] == o[io][0] and k % 2 == 0 else "uvw" for k, (i1, _, io) in enumerate(ins)]


@pytest.mark.parametrize("dtype,in1,in2,out,rule", CASES)
def test_mixed_conv_matches_oracle(dtype, in1, in2, out, rule):
    rng = np.random.default_rng(31)
    ins = all_instructions(in1, in2, out)
    modes = modes_for(rule, ins, in1, out)
    lay = oconv.mixed_layout(in1, in2, out, ins, modes)
    d1, d2, d_out, wu, ww, _ = lay
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.MixedPlan(in1, in2, out, ins, modes, tdt)
    assert (plan.d1, plan.d2, plan.d_out, plan.wu_numel, plan.ww_numel) == (d1, d2, d_out, wu, ww)
    N, E = 50, 420
    rowptr, col = graph_of(rng, N, E)
    x = rng.standard_normal((N, d1)).astype(dtype)
    Y = rng.standard_normal((E, d2)).astype(dtype)
    Wu = (rng.standard_normal((E, wu)) / 2).astype(dtype) if wu else None
    Ww = (rng.standard_normal((E, ww)) / 8).astype(dtype) if ww else None
    Wu0 = Wu if Wu is not None else np.zeros((E, 0))
    Ww0 = Ww if Ww is not None else np.zeros((E, 0))
    graph = cg.Graph(T(rowptr), T(col), N)
    tWu = T(Wu) if Wu is not None else None
    tWw = T(Ww) if Ww is not None else None
    o = cg.cgtp_mixed_conv_forward(plan, graph, T(x), T(Y), tWu, tWw)
    close("out", o, oconv.conv_mixed_forward(lay, x, Y, Wu0, Ww0, rowptr, col), dtype)
    g = rng.standard_normal((N, d_out)).astype(dtype)
    got = cg.cgtp_mixed_conv_backward(plan, graph, T(g), T(x), T(Y), tWu, tWw)
    ref = oconv.conv_mixed_backward(lay, g, x, Y, Wu0, Ww0, rowptr, col)
    for nm, a, b in zip(("gx", "gY", "gWu", "gWw"), got, ref):
        if b.size:
            close(nm, a, b, dtype)
    c = [rng.standard_normal(v.shape).astype(dtype) for v in (x, Y, Wu0, Ww0)]
    dd = cg.cgtp_mixed_conv_double_backward(plan, graph, T(g), T(x), T(Y), tWu, tWw, T(c[0]), T(c[1]),
                                            T(c[2]) if wu else None, T(c[3]) if ww else None)
    ref = oconv.conv_mixed_double_backward(lay, g, x, Y, Wu0, Ww0, *c, rowptr, col)
    for nm, a, b in zip(("d_gout", "d_x", "d_Y", "d_Wu", "d_Ww"), dd, ref):
        if b.size:
            close(nm, a, b, dtype)


def test_mixed_fold_of_several_uvu_instructions_into_one_block():
    """Three uvu instructions (0e x 0e, 1o x 1o, 2e x 2e -> 0e) fold into one block."""
    rng = np.random.default_rng(8)
    in1, in2, out = "8x0e+8x1o+8x2e", "0e+1o+2e", "8x0e+8x1o"
    ins = [(0, 0, 0), (1, 1, 0), (2, 2, 0), (0, 1, 1), (1, 0, 1), (2, 1, 1)]
    modes = ["uvu", "uvu", "uvu", "uvw", "uvu", "uvw"]
    lay = oconv.mixed_layout(in1, in2, out, ins, modes)
    plan = cg.MixedPlan(in1, in2, out, ins, modes, torch.float32)
    N, E = 30, 200
    rowptr, col = graph_of(rng, N, E)
    x = rng.standard_normal((N, lay[0])).astype(np.float32)
    Y = rng.standard_normal((E, lay[1])).astype(np.float32)
    Wu = rng.standard_normal((E, lay[3])).astype(np.float32)
    Ww = (rng.standard_normal((E, lay[4])) / 4).astype(np.float32)
    graph = cg.Graph(T(rowptr), T(col), N)
    o = cg.cgtp_mixed_conv_forward(plan, graph, T(x), T(Y), T(Wu), T(Ww))
    close("out", o, oconv.conv_mixed_forward(lay, x, Y, Wu, Ww, rowptr, col), np.float32)
    g = rng.standard_normal((N, lay[2])).astype(np.float32)
    got = cg.cgtp_mixed_conv_backward(plan, graph, T(g), T(x), T(Y), T(Wu), T(Ww))
    for nm, a, b in zip(("gx", "gY", "gWu", "gWw"), got, oconv.conv_mixed_backward(lay, g, x, Y, Wu, Ww, rowptr, col)):
        close(nm, a, b, np.float32)
