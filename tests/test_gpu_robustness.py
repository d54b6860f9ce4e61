"""Failure handling and memory safety of the CUDA path, on the GPU.

* Bounded waits: the uvw node GEMM waits on mbarriers for its tensor-core
  MMAs.  A plan whose wait limit is 0 gives up at the first wait; the kernel
  records the failure in the plan's error word, lets the MMAs in flight finish,
  frees its tensor memory and exits.  That call's results are invalid, the
  plan's next call returns CGTP_ECUDA, and the GPU stays usable (a fresh plan
  on the same graph matches the oracle).
* Host checks: a misaligned tensor pointer is rejected with CGTP_EINVAL before
  anything is launched.
* Canaries: every output tensor is surrounded by guard words; forward and
  backward leave the guards untouched (no write outside the outputs).
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402
from clebsch_gordan_tensor_racah_gb300 import workloads as wl  # noqa: E402
from oracle import conv as oconv, irreps as oirr  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _workload(name="nequip", N=300, dtype=np.float32):
    spec = wl.SPECS[name]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    w = wl.make(name, oplan.w_numel, seed=3, dtype=dtype, N=N)
    return spec, oplan, w


def _plan(spec, dtype=torch.float32):
    return cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvu", dtype)


def _uvw_workload(N=48):
    spec = dict(wl.SPECS["uvw"])
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvw")
    w = wl.make("uvw", oplan.w_numel, seed=4, N=N)
    return spec, oplan, w


def _uvw_plan(spec):
    return cg.Plan(spec["in1"], spec["in2"], spec["out"], "uvw", torch.float32, radial_k=8)


@pytest.mark.parametrize("direction", ["forward", "backward"])
def test_wait_give_up_is_reported_and_the_gpu_stays_usable(direction):
    spec, oplan, w = _uvw_workload()
    d = {k: T(v) for k, v in w.items() if isinstance(v, np.ndarray)}
    graph = cg.Graph(d["rowptr"], d["col"], w["N"])
    g = T(np.random.default_rng(5).standard_normal((w["N"], oplan.d_out)).astype(np.float32))
    bad = _uvw_plan(spec)
    bad.set_wait_limit(0)
    if direction == "forward":
        cg.cgtp_conv_forward(bad, graph, d["x"], d["Y"], d["R"], d["M"])      # results invalid
    else:
        cg.cgtp_conv_backward(bad, graph, g, d["x"], d["Y"], d["R"], d["M"])
    torch.cuda.synchronize()                                                 # the kernels left on their own
    with pytest.raises(cg.CgtpError) as e:
        cg.cgtp_conv_forward(bad, graph, d["x"], d["Y"], d["R"], d["M"])
    assert e.value.status == cg.CGTP_ECUDA
    assert "gave up" in str(e.value)
    with pytest.raises(cg.CgtpError):                                        # sticky
        cg.cgtp_conv_backward(bad, graph, g, d["x"], d["Y"], d["R"], d["M"])
    good = _uvw_plan(spec)
    out = cg.cgtp_conv_forward(good, graph, d["x"], d["Y"], d["R"], d["M"])
    torch.cuda.synchronize()
    ref = oconv.conv_uvw_radial_forward(oplan, w["x"], w["Y"], w["R"], w["M"], w["rowptr"], w["col"])
    got = out.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()


def test_wait_limit_and_node_chunk_reject_bad_values():
    spec, _, _ = _uvw_workload(N=8)
    plan = _uvw_plan(spec)
    for call in (lambda: plan.set_wait_limit(-1), lambda: plan.set_node_chunk(0),
                 lambda: plan.set_node_chunk((1 << 20) + 1),
                 lambda: plan.set_node_chunk(200_000),   # 200k x 17,920 state values per node > 2^31
                 lambda: _plan(wl.SPECS["nequip"]).set_node_chunk(64)):   # uvu plans have no node state
        with pytest.raises(cg.CgtpError) as e:
            call()
        assert e.value.status == cg.CGTP_EINVAL


def test_misaligned_pointer_is_rejected_before_launch():
    spec, oplan, w = _workload(N=40)
    plan = _plan(spec)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    x, Y, W = T(w["x"]), T(w["Y"]), T(w["W"])
    out = torch.zeros(w["N"] * oplan.d_out + 4, dtype=torch.float32, device=DEV)
    L = cg.lib()
    st = torch.cuda.current_stream().cuda_stream
    vp = ctypes.c_void_p
    shifted = vp(out.data_ptr() + 4)                   # 4-byte offset: not 16-byte aligned
    s = L.cgtp_conv_forward(plan.handle, graph.handle, vp(x.data_ptr()), vp(Y.data_ptr()), vp(W.data_ptr()),
                            None, shifted, vp(st))
    assert s == cg.CGTP_EINVAL
    assert b"aligned" in L.cgtp_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0               # nothing ran


def _guarded(shape, dtype, guard=64):
    """A tensor of `shape` inside a buffer with `guard` sentinel words on each side."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * guard,), 7.25e30, dtype=dtype, device=DEV)
    return buf, buf[guard:guard + n].view(*shape), guard


@pytest.mark.parametrize("name,dtype", [("nequip", np.float32), ("mace", np.float64), ("tiny", np.float32)])
def test_outputs_leave_guard_words_untouched(name, dtype):
    if name == "tiny":
        spec, oplan, w = _workload_tiny(dtype)
    else:
        spec, oplan, w = _workload(name, N=64, dtype=dtype)
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = _plan(spec, tdt)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    x, Y, W = T(w["x"]), T(w["Y"]), T(w["W"])
    bo, out, k = _guarded((w["N"], oplan.d_out), tdt)
    cg.cgtp_conv_forward(plan, graph, x, Y, W, out=out)
    g = T(np.random.default_rng(9).standard_normal((w["N"], oplan.d_out)).astype(dtype))
    bufs = [_guarded(t.shape, tdt) for t in (x, Y, W)]
    cg.cgtp_conv_backward(plan, graph, g, x, Y, W, outs=(bufs[0][1], bufs[1][1], bufs[2][1], None))
    torch.cuda.synchronize()
    for b, _, kk in [(bo, out, k)] + bufs:
        assert torch.all(b[:kk] == 7.25e30) and torch.all(b[-kk:] == 7.25e30)
    ref = oconv.conv_uvu_forward(oplan, w["x"], w["Y"], w["W"], w["rowptr"], w["col"])
    tol = 1e-10 if dtype == np.float64 else 1e-4
    assert np.abs(out.cpu().numpy() - ref).max() <= tol * np.abs(ref).max()


def _workload_tiny(dtype):
    spec = wl.SPECS["tiny"]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    return spec, oplan, wl.make("tiny", oplan.w_numel, seed=3, dtype=dtype)


def _run_twice(plan, graph, args, g_shape, dtype, **kw):
    a = cg.cgtp_conv_forward(plan, graph, *args, **kw)
    b = cg.cgtp_conv_forward(plan, graph, *args, **kw)
    g = torch.randn(g_shape, dtype=dtype, device=DEV, generator=torch.Generator(DEV).manual_seed(11))
    r1 = cg.cgtp_conv_backward(plan, graph, g, *args, **kw)
    r2 = cg.cgtp_conv_backward(plan, graph, g, *args, **kw)
    return [(a, b)] + [(u, v) for u, v in zip(r1, r2) if u is not None]


@pytest.mark.parametrize("name,mode,dtype", [("nequip", "uvu", np.float32), ("mace", "uvu", np.float32),
                                             ("mace", "uvu", np.float64), ("mixedmul", "uvu", np.float32),
                                             ("uvw", "uvw", np.float32), ("uvw_edge", "uvw", np.float64)])
def test_conv_results_are_bitwise_reproducible(name, mode, dtype):
    """Reductions that use atomic additions (gx and gY of the uvu backward, gR and gY of the
    radial uvw backward) add at most one value per element between two block barriers, so the
    order of additions is fixed: two runs give identical bits."""
    spec = wl.SPECS[name]
    radial = name == "uvw"
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], mode)
    w = wl.make(name, oplan.w_numel, seed=13, dtype=dtype, N=300)
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    plan = cg.Plan(spec["in1"], spec["in2"], spec["out"], mode, tdt, radial_k=8 if radial else 0)
    graph = cg.Graph(T(w["rowptr"]), T(w["col"]), w["N"])
    if radial:
        pairs = _run_twice(plan, graph, (T(w["x"]), T(w["Y"]), T(w["R"]), T(w["M"])), (w["N"], oplan.d_out), tdt)
    else:
        pairs = _run_twice(plan, graph, (T(w["x"]), T(w["Y"]), T(w["W"])), (w["N"], oplan.d_out), tdt)
    for u, v in pairs:
        assert torch.equal(u, v)


def test_batched_results_are_bitwise_reproducible():
    spec = wl.SPECS["highl"]
    oplan = oirr.make_plan(spec["in1"], spec["in2"], spec["out"], "uvu")
    w = wl.make("highl", oplan.w_numel, seed=13, B=600)
    plan = _plan(spec)
    x1, x2, W = T(w["x1"]), T(w["x2"]), T(w["W"])
    a, b = cg.cgtp_forward(plan, x1, x2, W), cg.cgtp_forward(plan, x1, x2, W)
    assert torch.equal(a, b)
    g = torch.randn_like(a)
    for u, v in zip(cg.cgtp_backward(plan, g, x1, x2, W), cg.cgtp_backward(plan, g, x1, x2, W)):
        assert torch.equal(u, v)
