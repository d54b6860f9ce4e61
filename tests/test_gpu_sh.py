"""GPU parity of the convolution fed by raw edge vectors (harmonics evaluated in
the kernels) against the FP64 oracle (scipy harmonics and their exact Jacobian).

max|err| <= 1e-4 * max|ref| (FP32), <= 1e-10 * max|ref| (FP64) for out, gx, gY,
grvec and gW.  Edge vectors have random lengths, so the normalisation and the
radial projection of the gradient are exercised.
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
    got = got.cpu().numpy().astype(np.float64)
    err, scale = np.abs(got - ref).max(), np.abs(ref).max()
    assert err <= TOL[dtype] * scale, f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


@pytest.mark.parametrize("name,dtype,over", [
    ("tiny", np.float32, {}),
    ("nequip", np.float32, dict(N=200)),
    ("mace", np.float64, dict(N=60)),
])
def test_edge_vector_conv(name, dtype, over):
    spec = wl.SPECS[name]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    w = wl.make(name, oplan.w_numel, seed=5, dtype=dtype, **over)
    rng = np.random.default_rng(6)
    rvec = (rng.normal(size=(w["E"], 3)) * rng.uniform(0.5, 5.0, size=(w["E"], 1))).astype(dtype)
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", tdt)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    out = cg.cgtp_conv_forward_sh(plan, graph, T(w["x"]), T(rvec), T(w["W"]))
    close("out", out, oconv.conv_uvu_forward_sh(oplan, w["x"], rvec, w["W"], w["rowptr"], w["col"]), dtype)
    g = rng.standard_normal((w["N"], oplan.d_out)).astype(dtype)
    got = cg.cgtp_conv_backward_sh(plan, graph, T(g), T(w["x"]), T(rvec), T(w["W"]))
    ref = oconv.conv_uvu_backward_sh(oplan, g, w["x"], rvec, w["W"], w["rowptr"], w["col"])
    for nm, a, b in zip(("gx", "gY", "grvec", "gW"), got, ref):
        close(nm, a, b, dtype)


def test_edge_vector_conv_needs_harmonic_in2():
    spec = wl.SPECS["uvw"]
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvw", torch.float32, radial_k=8)
    z = torch.zeros(16, 4096, device="cuda")
    graph = cg.Graph(torch.zeros(2, dtype=torch.int32, device="cuda"), torch.zeros(0, dtype=torch.int32,
                                                                                      device="cuda"), 1)
    with pytest.raises(cg.CgtpError) as e:
        cg.cgtp_conv_forward_sh(plan, graph, z, z, z, out=z)
    assert e.value.status == cg.CGTP_EUNSUPPORTED


def test_radial_edge_vector_uvw_conv():
    spec = wl.SPECS["uvw"]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvw")
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvw", torch.float32, radial_k=8)
    w = wl.make("uvw", oplan.w_numel, seed=8, N=12)
    rng = np.random.default_rng(9)
    rvec = (rng.normal(size=(w["E"], 3)) * rng.uniform(0.6, 4.5, size=(w["E"], 1))).astype(np.float32)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    out = cg.cgtp_conv_forward_sh_radial(plan, graph, T(w["x"]), T(rvec), T(w["M"]), 0.5, 5.0)
    close("out", out, oconv.conv_uvw_radial_forward_sh(oplan, w["x"], rvec, w["M"], 8, 0.5, 5.0,
                                                        w["rowptr"], w["col"]), np.float32)
    g = rng.standard_normal((w["N"], oplan.d_out)).astype(np.float32)
    got = cg.cgtp_conv_backward_sh_radial(plan, graph, T(g), T(w["x"]), T(rvec), T(w["M"]), 0.5, 5.0)
    ref = oconv.conv_uvw_radial_backward_sh(oplan, g, w["x"], rvec, w["M"], 8, 0.5, 5.0, w["rowptr"], w["col"])
    for nm, a, b in zip(("gx", "gY", "gR", "grvec", "gM"), got, ref):
        close(nm, a, b, np.float32)
