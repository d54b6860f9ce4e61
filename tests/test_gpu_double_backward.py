"""GPU parity of the second derivatives ("double backward") against the FP64 oracle.

cgtp_conv_double_backward / cgtp_double_backward return the derivatives of
S = sum_j <c_j, dL/da_j> with respect to the output gradient and every operand
(x, Y, W; uvw: x, Y, R, M).  Each output tensor is compared element by element
with the oracle (itself pinned by exact directional differences of its
backward): max|err| <= 1e-4 * max|ref| in FP32, <= 1e-10 * max|ref| in FP64.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from clebsch_gordan_tensor_racah_gb300 import workloads as wl  # noqa: E402
from oracle import conv as oconv, irreps as oirr  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = {np.float32: 1e-4, np.float64: 1e-10}


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def close(name, got, ref, dtype):
    got = got.detach().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    err, scale = np.abs(got - ref).max(), np.abs(ref).max()
    assert err <= TOL[dtype] * scale, f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


@pytest.mark.parametrize("name,dtype,over", [
    ("tiny", np.float32, {}),
    ("nequip", np.float32, dict(N=20)),
    ("mace", np.float64, dict(N=15)),
])
def test_conv_uvu_double_backward(name, dtype, over):
    spec = wl.SPECS[name]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    w = wl.make(name, oplan.w_numel, seed=3, dtype=dtype, **over)
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", tdt)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    rng = np.random.default_rng(4)
    g = rng.standard_normal((w["N"], oplan.d_out)).astype(dtype)
    cx, cY, cW = (rng.standard_normal(w[k].shape).astype(dtype) for k in ("x", "Y", "W"))
    got = cg.cgtp_conv_double_backward(plan, graph, T(g), T(w["x"]), T(w["Y"]), T(w["W"]),
                                       T(cx), T(cY), T(cW))
    ref = oconv.conv_uvu_double_backward(oplan, g, w["x"], w["Y"], w["W"], cx, cY, cW, w["rowptr"], w["col"])
    for nm, a, b in zip(("d_gout", "d_x", "d_Y", "d_W"), got[:4], ref):
        close(nm, a, b, dtype)
    assert got[4] is None


def test_conv_uvw_double_backward():
    spec = wl.SPECS["uvw"]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvw")
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvw", torch.float32, radial_k=8)
    w = wl.make("uvw", oplan.w_numel, seed=5, N=12)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    rng = np.random.default_rng(6)
    g = rng.standard_normal((w["N"], oplan.d_out)).astype(np.float32)
    c = [rng.standard_normal(w[k].shape).astype(np.float32) for k in ("x", "Y", "R", "M")]
    got = cg.cgtp_conv_double_backward(plan, graph, T(g), T(w["x"]), T(w["Y"]), T(w["R"]),
                                       T(c[0]), T(c[1]), T(c[2]), M=T(w["M"]), ggM=T(c[3]))
    ref = oconv.conv_uvw_radial_double_backward(oplan, g, w["x"], w["Y"], w["R"], w["M"], *c,
                                                w["rowptr"], w["col"])
    for nm, a, b in zip(("d_gout", "d_x", "d_Y", "d_R", "d_M"), got, ref):
        close(nm, a, b, np.float32)


@pytest.mark.parametrize("B", [5, 13])
def test_batched_high_l_double_backward(B):
    spec = wl.SPECS["highl"]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", torch.float32)
    w = wl.make("highl", oplan.w_numel, seed=7, B=B)
    rng = np.random.default_rng(8)
    g = rng.standard_normal((B, oplan.d_out)).astype(np.float32)
    c = [rng.standard_normal(w[k].shape).astype(np.float32) for k in ("x1", "x2", "W")]
    got = cg.cgtp_double_backward(plan, T(g), T(w["x1"]), T(w["x2"]), T(w["W"]), *(T(v) for v in c))
    ref = oconv.tp_uvu_double_backward(oplan, g, w["x1"], w["x2"], w["W"], *c)
    for nm, a, b in zip(("d_gout", "d_x1", "d_x2", "d_W"), got, ref):
        close(nm, a, b, np.float32)


def test_double_backward_rejects_small_workspace():
    import ctypes
    spec = wl.SPECS["tiny"]
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", torch.float32)
    L = cg.lib()
    nb = ctypes.c_int64()
    assert L.cgtp_double_backward_workspace(plan.handle, 4, ctypes.byref(nb)) == cg.CGTP_OK
    assert nb.value > 0
    z = torch.zeros(4 * 4096, device="cuda")
    p = ctypes.c_void_p(z.data_ptr())
    st = L.cgtp_double_backward(plan.handle, p, p, p, p, p, p, p, p, p, p, p, 4, p, nb.value - 256,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == cg.CGTP_EINVAL
    assert b"workspace" in L.cgtp_last_error()
