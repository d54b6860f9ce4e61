"""GPU parity of the bfloat16-input convolution and batched product (FP32
arithmetic and outputs).

The inputs x, Y, W and the output gradient are rounded to bfloat16 once; the
FP64 oracle consumes exactly those rounded values, so the only differences
left are FP32 rounding in the kernels: the FP32 bound applies,
max|err| <= 1e-4 * max|ref| per output tensor.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from clebsch_gordan_tensor_racah_gb300 import workloads as wl  # noqa: E402
from oracle import conv as oconv, irreps as oirr  # noqa: E402

pytestmark = pytest.mark.gpu


def close(name, got, ref):
    assert got.dtype == torch.float32, (name, got.dtype)
    got = got.cpu().numpy().astype(np.float64)
    err, scale = np.abs(got - ref).max(), np.abs(ref).max()
    assert err <= 1e-4 * scale, f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


@pytest.mark.parametrize("name,over", [("tiny", {}), ("nequip", dict(N=300)), ("mace", dict(N=150))])
def test_bf16_conv_fwd_bwd(name, over):
    spec = wl.SPECS[name]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    w = wl.make(name, oplan.w_numel, seed=9, **over)
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", torch.bfloat16)
    dev = torch.device("cuda")
    b = {k: torch.from_numpy(np.ascontiguousarray(w[k])).to(dev).to(torch.bfloat16) for k in ("x", "Y", "W")}
    h = {k: v.float().cpu().numpy().astype(np.float64) for k, v in b.items()}   # the exact bf16 values
    graph = cg.Graph(torch.from_numpy(w["rowptr"]).to(dev), torch.from_numpy(w["col"]).to(dev), w["N"])
    out = cg.cgtp_conv_forward(plan, graph, b["x"], b["Y"], b["W"])
    close("out", out, oconv.conv_uvu_forward(oplan, h["x"], h["Y"], h["W"], w["rowptr"], w["col"]))
    g = torch.randn(out.shape, device=dev, generator=torch.Generator(dev).manual_seed(3)).to(torch.bfloat16)
    gx, gY, gW, _ = cg.cgtp_conv_backward(plan, graph, g, b["x"], b["Y"], b["W"])
    r = oconv.conv_uvu_backward(oplan, g.float().cpu().numpy().astype(np.float64), h["x"], h["Y"], h["W"],
                                w["rowptr"], w["col"])
    for nm, a, ref in zip(("gx", "gY", "gW"), (gx, gY, gW), r):
        close(nm, a, ref)


def _batched_bf16(in1, in2, out, B, seed):
    """Batched product with bfloat16 inputs against the oracle on the same rounded values."""
    oplan = oirr.make_plan(in1, in2, out, "uvu")
    rng = np.random.default_rng(seed)
    dev = torch.device("cuda")
    b = {k: torch.from_numpy(rng.standard_normal((B, n))).to(dev).to(torch.bfloat16)
         for k, n in (("x1", oplan.d1), ("x2", oplan.d2), ("W", oplan.w_numel), ("g", oplan.d_out))}
    h = {k: v.float().cpu().numpy().astype(np.float64) for k, v in b.items()}
    plan = cg.Plan(in1, in2, out, "uvu", torch.bfloat16)
    out = cg.cgtp_forward(plan, b["x1"], b["x2"], b["W"])
    close("out", out, oconv.tp_uvu_forward(oplan, h["x1"], h["x2"], h["W"]))
    got = cg.cgtp_backward(plan, b["g"], b["x1"], b["x2"], b["W"])
    ref = oconv.tp_uvu_backward(oplan, h["g"], h["x1"], h["x2"], h["W"])
    for nm, a, r in zip(("gx1", "gx2", "gW"), got, ref):
        close(nm, a, r)


def test_bf16_batched_high_l():
    # multiplicity 16, l up to 7 (the high-L recipe's irreps): an odd batch and a single sample
    spec = wl.SPECS["highl"]
    _batched_bf16(spec["in1"], spec["in2"], spec["out"], 37, 21)
    _batched_bf16(spec["in1"], spec["in2"], spec["out"], 1, 22)


def test_bf16_batched_mul32():
    _batched_bf16("32x0e+32x1o+32x2e+32x3o+32x4e+32x5o", "1x0e+1x1o+1x2e+1x3o+1x4e+1x5o",
                  "1x0e+1x1o+1x2e+1x3o+1x4e+1x5o+1x0o+1x1e+1x2o+1x3e+1x4o+1x5e", 23, 23)


def test_bf16_outside_the_served_plans_is_unsupported():
    # blocks of different multiplicity: neither the v3 conv nor the batched kernels
    with pytest.raises(cg.CgtpError) as e:
        cg.Plan("32x0e+16x1o+16x2e", "1x0e+1x1o+1x2e", "1x0e+1x1o+1x2e", "uvu", torch.bfloat16)
    assert e.value.status == cg.CGTP_EUNSUPPORTED
    # multiplicity 8 (tiny): conv yes, batched no
    spec = wl.SPECS["tiny"]
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", torch.bfloat16)
    z = lambda n: torch.zeros(4, n, device="cuda", dtype=torch.bfloat16)   # noqa: E731
    with pytest.raises(cg.CgtpError) as e:
        cg.cgtp_forward(plan, z(plan.d1), z(plan.d2), z(plan.w_numel),
                        out=torch.zeros(4, plan.d_out, device="cuda", dtype=torch.float32))
    assert e.value.status == cg.CGTP_EUNSUPPORTED
    # l up to 7 (high-L irreps): batched yes, graph convolution no
    spec = wl.SPECS["highl"]
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", torch.bfloat16)
    w = wl.make("tiny", 1, N=4)
    graph = cg.Graph(torch.from_numpy(w["rowptr"]).cuda(), torch.from_numpy(w["col"]).cuda(), 4)
    with pytest.raises(cg.CgtpError) as e:
        cg.cgtp_conv_forward(plan, graph, torch.zeros(4, plan.d1, device="cuda", dtype=torch.bfloat16),
                             torch.zeros(w["E"], plan.d2, device="cuda", dtype=torch.bfloat16),
                             torch.zeros(w["E"], plan.w_numel, device="cuda", dtype=torch.bfloat16))
    assert e.value.status == cg.CGTP_EUNSUPPORTED


def _graph(rng, N, E):
    src = rng.integers(0, N, E)
    dst = rng.integers(0, N - 2, E)          # the last two receivers have no in-edges
    order = np.argsort(dst, kind="stable")
    rowptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))]).astype(np.int32)
    return rowptr, src[order].astype(np.int32)


def _bf(rng, shape, scale=1.0):
    """A bfloat16 device tensor and the FP64 copy of its exact values."""
    t = torch.from_numpy(rng.standard_normal(shape) * scale).cuda().to(torch.bfloat16)
    return t, t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("in1,out", [("16x0e+16x1o+16x2e", "16x0e+16x1o+16x2e"),        # 16-byte weight rows
                                     ("12x0e+5x1o+3x2e", "7x0e+9x1o+4x2e")])            # scalar weight rows
def test_bf16_per_edge_uvw(in1, out):
    rng = np.random.default_rng(41)
    in2 = "0e+1o+2e+3o"
    oplan = oirr.make_plan(in1, in2, out, "uvw")
    plan = cg.Plan(in1, in2, out, "uvw", torch.bfloat16, radial_k=0)
    N, E = 40, 300
    rowptr, col = _graph(rng, N, E)
    graph = cg.Graph(torch.from_numpy(rowptr).cuda(), torch.from_numpy(col).cuda(), N)
    (x, hx), (Y, hY), (W, hW), (g, hg) = (_bf(rng, (N, oplan.d1)), _bf(rng, (E, oplan.d2)),
                                          _bf(rng, (E, oplan.w_numel), 0.25), _bf(rng, (N, oplan.d_out)))
    close("out", cg.cgtp_conv_forward(plan, graph, x, Y, W), oconv.conv_uvw_forward(oplan, hx, hY, hW, rowptr, col))
    gx, gY, gW, _ = cg.cgtp_conv_backward(plan, graph, g, x, Y, W)
    for nm, a, r in zip(("gx", "gY", "gW"), (gx, gY, gW), oconv.conv_uvw_backward(oplan, hg, hx, hY, hW, rowptr, col)):
        close(nm, a, r)


def test_bf16_mixed_list():
    """32x(0e,1o,2e): the 0e outputs uvw (weights per edge), the others uvu (v3 kernels)."""
    rng = np.random.default_rng(43)
    in1 = out = "32x0e+32x1o+32x2e"
    in2 = "0e+1o+2e"
    a, b, o = oirr.parse_irreps(in1), oirr.parse_irreps(in2), oirr.parse_irreps(out)
    ins, modes = [], []
    for i1, (_, l1, p1) in enumerate(a):
        for i2, (_, l2, p2) in enumerate(b):
            for io, (_, l3, p3) in enumerate(o):
                if abs(l1 - l2) <= l3 <= l1 + l2 and p3 == p1 * p2:
                    ins.append((i1, i2, io))
                    modes.append("uvw" if l3 == 0 else "uvu")
    lay = oconv.mixed_layout(in1, in2, out, ins, modes)
    d1, d2, d_out, wu, ww, _ = lay
    plan = cg.MixedPlan(in1, in2, out, ins, modes, torch.bfloat16)
    N, E = 50, 420
    rowptr, col = _graph(rng, N, E)
    graph = cg.Graph(torch.from_numpy(rowptr).cuda(), torch.from_numpy(col).cuda(), N)
    (x, hx), (Y, hY), (Wu, hWu), (Ww, hWw), (g, hg) = (
        _bf(rng, (N, d1)), _bf(rng, (E, d2)), _bf(rng, (E, wu), 0.5), _bf(rng, (E, ww), 0.125), _bf(rng, (N, d_out)))
    close("out", cg.cgtp_mixed_conv_forward(plan, graph, x, Y, Wu, Ww),
          oconv.conv_mixed_forward(lay, hx, hY, hWu, hWw, rowptr, col))
    got = cg.cgtp_mixed_conv_backward(plan, graph, g, x, Y, Wu, Ww)
    for nm, a_, r in zip(("gx", "gY", "gWu", "gWw"), got, oconv.conv_mixed_backward(lay, hg, hx, hY, hWu, hWw,
                                                                                      rowptr, col)):
        close(nm, a_, r)
