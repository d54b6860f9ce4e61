"""GPU parity of the uvu fused CG tensor-product convolution and the batched product.

Every test calls the CUDA path through the C ABI (Python binding) and compares it
element by element with the FP64 oracle on the same seeded inputs:
max|err| <= 1e-4 * max|ref| (FP32) and <= 1e-10 * max|ref| (FP64), per output
tensor; the graph transpose is compared bit for bit.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from clebsch_gordan_tensor_racah_gb300 import workloads as wl  # noqa: E402
from oracle import conv as oconv, graph as ograph, irreps as oirr  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = {np.float32: 1e-4, np.float64: 1e-10}


def dev():
    return torch.device("cuda:0")


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def close(name, got, ref, dtype):
    got = got.detach().cpu().numpy().astype(np.float64) if hasattr(got, "detach") else got
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    scale = np.abs(ref).max() if ref.size else 0.0
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= TOL[dtype] * max(scale, 1e-30), f"{name}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


def run_conv(spec_name, dtype=np.float32, seed=0, check_grad=True, **over):
    spec = dict(wl.SPECS[spec_name])
    spec.update(over)
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    w = wl.make(spec_name, oplan.w_numel, seed=seed, dtype=dtype, **over)
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", tdt)
    assert (plan.d1, plan.d2, plan.d_out, plan.w_numel) == (oplan.d1, oplan.d2, oplan.d_out, oplan.w_numel)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    x, Y, W = T(w["x"]), T(w["Y"]), T(w["W"])
    out = cg.cgtp_conv_forward(plan, graph, x, Y, W)
    ref = oconv.conv_uvu_forward(oplan, w["x"], w["Y"], w["W"], w["rowptr"], w["col"])
    close("out", out, ref, dtype)
    if check_grad:
        g = np.random.default_rng(seed + 100).standard_normal(ref.shape).astype(dtype)
        gx, gY, gW, _ = cg.cgtp_conv_backward(plan, graph, T(g), x, Y, W)
        rgx, rgY, rgW = oconv.conv_uvu_backward(oplan, g, w["x"], w["Y"], w["W"], w["rowptr"], w["col"])
        close("gx", gx, rgx, dtype)
        close("gY", gY, rgY, dtype)
        close("gW", gW, rgW, dtype)
    return plan, graph, w


def test_tiny_config_fwd_bwd():
    run_conv("tiny")


def test_nequip_like_small():
    run_conv("nequip", N=300)


def test_mace_like_small_fp32():
    run_conv("mace", N=120)


def test_mace_like_small_fp64():
    run_conv("mace", dtype=np.float64, N=120)


def test_nequip_like_fp64():
    run_conv("nequip", dtype=np.float64, N=64)


def test_graph_transpose_bit_exact():
    w = wl.make("mace", 2304, N=500)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    tr, te, td = graph.transpose()
    rr, re_, rd = ograph.transpose(w["rowptr"], w["col"], w["N"])
    assert np.array_equal(tr.cpu().numpy(), rr)
    assert np.array_equal(te.cpu().numpy(), re_)
    assert np.array_equal(td.cpu().numpy(), rd)


def test_graph_transpose_long_segment():
    # one hub sender with 3000 out-edges (block sort path) plus a uniform rest
    rng = np.random.default_rng(3)
    N, E = 400, 6000
    src = np.where(rng.random(E) < 0.5, 7, rng.integers(0, N, E))
    dst = rng.integers(0, N, E)
    order = np.argsort(dst, kind="stable")
    rowptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))]).astype(np.int32)
    col = src[order].astype(np.int32)
    graph = cg.Graph(T(rowptr), T(col), N)
    tr, te, td = graph.transpose()
    rr, re_, rd = ograph.transpose(rowptr, col, N)
    assert np.array_equal(te.cpu().numpy(), re_) and np.array_equal(td.cpu().numpy(), rd)


def test_graph_validation_errors():
    rowptr = T(np.array([0, 2, 1, 3], np.int32))
    col = T(np.array([0, 1, 2], np.int32))
    with pytest.raises(cg.CgtpError) as e:
        cg.Graph(rowptr, col, 3)
    assert e.value.status == cg.CGTP_EGRAPH
    with pytest.raises(cg.CgtpError) as e:
        cg.Graph(T(np.array([0, 1, 2, 3], np.int32)), T(np.array([0, 5, 2], np.int32)), 3)
    assert e.value.status == cg.CGTP_EGRAPH
    with pytest.raises(cg.CgtpError) as e:
        cg.Graph(T(np.array([0, 1, 2, 4], np.int32)), T(np.array([0, 1, 2], np.int32)), 3)
    assert e.value.status == cg.CGTP_EGRAPH


def _custom_conv(in1, in2, out, rowptr, col, N, dtype=np.float32, seed=0):
    rng = np.random.default_rng(seed)
    oplan = oirr.make_plan(in1, in2, out, "uvu")
    E = int(rowptr[-1])
    x = rng.standard_normal((N, oplan.d1)).astype(dtype)
    Y = rng.standard_normal((E, oplan.d2)).astype(dtype)
    W = rng.standard_normal((E, oplan.w_numel)).astype(dtype)
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.Plan(in1, in2, out, "uvu", tdt)
    graph = cg.Graph(T(rowptr.astype(np.int32)), T(col.astype(np.int32)), N)
    out_t = cg.cgtp_conv_forward(plan, graph, T(x), T(Y), T(W))
    close("out", out_t, oconv.conv_uvu_forward(oplan, x, Y, W, rowptr, col), dtype)
    g = rng.standard_normal((N, oplan.d_out)).astype(dtype)
    gx, gY, gW, _ = cg.cgtp_conv_backward(plan, graph, T(g), T(x), T(Y), T(W))
    rgx, rgY, rgW = oconv.conv_uvu_backward(oplan, g, x, Y, W, rowptr, col)
    close("gx", gx, rgx, dtype)
    close("gY", gY, rgY, dtype)
    close("gW", gW, rgW, dtype)


def test_edge_cases_empty_rows_self_loops_multi_edges():
    # node 0: no in-edges; node 1: self loop twice; node 2: 3 in-edges from 0; node 3: no out-edges
    rowptr = np.array([0, 0, 2, 5, 6, 6])
    col = np.array([1, 1, 0, 0, 0, 4])
    _custom_conv("3x0e+2x1o+1x2e", "0e+1o+2e", wl._all_out(2), rowptr, col, 5)


def test_single_node_and_l0_only():
    _custom_conv("5x0e", "0e", "0e", np.array([0, 3]), np.array([0, 0, 0]), 1)


def test_ragged_channel_blocks_and_long_rows():
    # 40 channels -> a full and a ragged 32-lane block; 70 in-edges -> ragged chunk tail
    rng = np.random.default_rng(9)
    N = 6
    deg = np.array([70, 0, 1, 33, 16, 17])
    rowptr = np.concatenate([[0], np.cumsum(deg)])
    col = rng.integers(0, N, rowptr[-1])
    _custom_conv("40x0e+40x1o+8x2e", "0e+1o+2e", wl._all_out(2), rowptr, col, N)


def test_zero_edges():
    N = 4
    rowptr = np.zeros(N + 1, np.int64)
    col = np.zeros(0, np.int64)
    oplan = oirr.make_plan("4x0e+4x1o", "0e+1o", "0e+1o+1e", "uvu")
    plan = cg.Plan("4x0e+4x1o", "0e+1o", "0e+1o+1e", "uvu", torch.float32)
    graph = cg.Graph(T(rowptr.astype(np.int32)), torch.zeros(0, dtype=torch.int32, device=dev()), N)
    x = T(np.ones((N, oplan.d1), np.float32))
    out = torch.full((N, oplan.d_out), 7.0, device=dev())
    cg.cgtp_conv_forward(plan, graph, x, torch.zeros(0, 4, device=dev()), torch.zeros(0, 10, device=dev()), out=out)
    assert torch.count_nonzero(out).item() == 0


def test_batched_high_l_small():
    spec = wl.SPECS["highl"]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    w = wl.make("highl", oplan.w_numel, B=48)
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", torch.float32)
    x1, x2, W = T(w["x1"]), T(w["x2"]), T(w["W"])
    out = cg.cgtp_forward(plan, x1, x2, W)
    close("out", out, oconv.tp_uvu_forward(oplan, w["x1"], w["x2"], w["W"]), np.float32)
    g = np.random.default_rng(5).standard_normal((48, oplan.d_out)).astype(np.float32)
    gx1, gx2, gW = cg.cgtp_backward(plan, T(g), x1, x2, W)
    r1, r2, rW = oconv.tp_uvu_backward(oplan, g, w["x1"], w["x2"], w["W"])
    close("gx1", gx1, r1, np.float32)
    close("gx2", gx2, r2, np.float32)
    close("gW", gW, rW, np.float32)


def _batched_case(in1, in2, out, B, seed):
    oplan = oirr.make_plan(in1, in2, out, "uvu")
    rng = np.random.default_rng(seed)
    x1 = rng.standard_normal((B, oplan.d1)).astype(np.float32)
    x2 = rng.standard_normal((B, oplan.d2)).astype(np.float32)
    W = rng.standard_normal((B, oplan.w_numel)).astype(np.float32)
    plan = cg.Plan(in1, in2, out, "uvu", torch.float32)
    out_d = cg.cgtp_forward(plan, T(x1), T(x2), T(W))
    close("out", out_d, oconv.tp_uvu_forward(oplan, x1, x2, W), np.float32)
    g = rng.standard_normal((B, oplan.d_out)).astype(np.float32)
    gx1, gx2, gW = cg.cgtp_backward(plan, T(g), T(x1), T(x2), T(W))
    r1, r2, rW = oconv.tp_uvu_backward(oplan, g, x1, x2, W)
    close("gx1", gx1, r1, np.float32)
    close("gx2", gx2, r2, np.float32)
    close("gW", gW, rW, np.float32)


def test_batched_high_l_odd_batch():
    # 16 channels: two samples per warp, an odd tail; l up to 7 spans several path groups
    spec = wl.SPECS["highl"]
    _batched_case(spec["in1"], spec["in2"], spec["out"], 37, 11)
    _batched_case(spec["in1"], spec["in2"], spec["out"], 1, 12)


def test_batched_mul32_mixed_l():
    # 32 channels: one sample per warp; in1 blocks shared by several path groups
    in1 = "32x0e+32x1o+32x2e+32x3o+32x4e+32x5o"
    in2 = "1x0e+1x1o+1x2e+1x3o+1x4e+1x5o"
    out = "1x0e+1x1o+1x2e+1x3o+1x4e+1x5o+1x0o+1x1e+1x2o+1x3e+1x4o+1x5e"
    _batched_case(in1, in2, out, 23, 13)


def test_deterministic_bitwise():
    plan, graph, w = run_conv("nequip", N=200, check_grad=False)
    x, Y, W = T(w["x"]), T(w["Y"]), T(w["W"])
    a = cg.cgtp_conv_forward(plan, graph, x, Y, W)
    b = cg.cgtp_conv_forward(plan, graph, x, Y, W)
    assert torch.equal(a, b)
    g = torch.randn_like(a)
    r1 = cg.cgtp_conv_backward(plan, graph, g, x, Y, W)
    r2 = cg.cgtp_conv_backward(plan, graph, g, x, Y, W)
    for u, v in zip(r1[:3], r2[:3]):
        assert torch.equal(u, v)
