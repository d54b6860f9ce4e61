"""GB300 fused Clebsch-Gordan tensor-product convolution: Python binding of libcgtp.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libcgtp.so`` (built in-tree by ``_build.build()``).  PyTorch is used
for device memory and streams.  There is no CPU fallback: if the library is
missing or no GPU is present the calls raise.

Names follow the C ABI in ``include/cgtp.h`` (and ``include/cgtp_measure.h`` for the
measurement kernels ``measure_fma`` / ``measure_read``):

* ``Plan(irreps_in1, irreps_in2, irreps_out, mode, dtype, radial_k)`` --
  ``cgtp_plan_create``; ``plan.d1, d2, d_out, w_numel, n_paths``;
  ``plan.path(p)`` -> (ints, CG block).
* ``cgtp_forward(plan, x1, x2, W)`` / ``cgtp_backward(plan, gout, x1, x2, W)``.
* ``Graph(rowptr, col, N)`` -- ``cgtp_graph_create``; ``graph.transpose()``.
* ``cgtp_conv_forward(plan, graph, x, Y, W_or_R, M=None)`` and
  ``cgtp_conv_backward(plan, graph, gout, x, Y, W_or_R, M=None)``.
* ``cgtp_real_cg_block(l1, l2, l3)`` -- host-only query of the planner's block.
"""

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcgtp.so")

CGTP_OK, CGTP_EINVAL, CGTP_EUNSUPPORTED, CGTP_ENOMEM, CGTP_ECUDA, CGTP_EGRAPH = range(6)
CGTP_UVU, CGTP_UVW = 0, 1
CGTP_F32, CGTP_F64, CGTP_BF16 = 0, 1, 2

EXPORTS = ["cgtp_plan_create", "cgtp_plan_destroy", "cgtp_plan_info", "cgtp_plan_path",
           "cgtp_forward", "cgtp_backward", "cgtp_graph_create", "cgtp_graph_destroy",
           "cgtp_graph_transpose", "cgtp_conv_forward", "cgtp_conv_backward",
           "cgtp_real_cg_block", "cgtp_last_error", "cgtp_graph_transpose_noalloc",
           "cgtp_conv_double_backward_workspace", "cgtp_conv_double_backward",
           "cgtp_double_backward_workspace", "cgtp_double_backward",
           "cgtp_conv_forward_sh", "cgtp_conv_backward_sh", "cgtp_real_sh",
           "cgtp_conv_forward_sh_radial", "cgtp_conv_backward_sh_radial",
           "cgtp_mixed_plan_create", "cgtp_mixed_plan_destroy", "cgtp_mixed_plan_info",
           "cgtp_mixed_conv_workspace", "cgtp_mixed_conv_forward", "cgtp_mixed_conv_backward",
           "cgtp_mixed_conv_double_backward", "cgtp_measure_fma", "cgtp_measure_read",
           "cgtp_plan_device_bytes", "cgtp_graph_device_bytes", "cgtp_plan_set_wait_limit",
           "cgtp_plan_set_node_chunk", "cgtp_plan_node_chunk"]


class CgtpError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"cgtp status {status}: {msg}")
        self.status = status


_lib = None


def lib():
    """Load libcgtp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run __graft_entry__.build() "
                              "(or python -m clebsch_gordan_tensor_racah_gb300._build)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.cgtp_last_error.restype = ctypes.c_char_p
        L.cgtp_plan_create.argtypes = [ctypes.POINTER(vp), ctypes.c_char_p, ctypes.c_char_p,
                                       ctypes.c_char_p, vp, i32, i32, i32, i32]
        L.cgtp_plan_destroy.argtypes = [vp]
        L.cgtp_plan_destroy.restype = None
        L.cgtp_plan_info.argtypes = [vp] + [ctypes.POINTER(i64)] * 4 + [ctypes.POINTER(i32)]
        L.cgtp_plan_path.argtypes = [vp, i32, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_double), i64]
        L.cgtp_forward.argtypes = [vp, vp, vp, vp, vp, i64, vp]
        L.cgtp_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, vp]
        L.cgtp_graph_create.argtypes = [ctypes.POINTER(vp), vp, vp, i64, i64, vp]
        L.cgtp_graph_destroy.argtypes = [vp]
        L.cgtp_graph_destroy.restype = None
        L.cgtp_graph_transpose.argtypes = [vp, vp, vp, vp, vp]
        L.cgtp_conv_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.cgtp_conv_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.cgtp_real_cg_block.argtypes = [i32, i32, i32, ctypes.POINTER(ctypes.c_double), i64]
        L.cgtp_graph_transpose_noalloc.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp]
        L.cgtp_conv_double_backward_workspace.argtypes = [vp, vp, ctypes.POINTER(i64)]
        L.cgtp_conv_double_backward.argtypes = [vp] * 17 + [i64, vp]
        L.cgtp_double_backward_workspace.argtypes = [vp, i64, ctypes.POINTER(i64)]
        L.cgtp_double_backward.argtypes = [vp] * 12 + [i64, vp, i64, vp]
        L.cgtp_conv_forward_sh.argtypes = [vp] * 7
        L.cgtp_conv_backward_sh.argtypes = [vp] * 11
        L.cgtp_real_sh.argtypes = [i32, vp, i64, vp, vp]
        dbl = ctypes.c_double
        L.cgtp_conv_forward_sh_radial.argtypes = [vp] * 5 + [dbl, dbl, vp, vp]
        L.cgtp_conv_backward_sh_radial.argtypes = [vp] * 6 + [dbl, dbl] + [vp] * 6
        L.cgtp_mixed_plan_create.argtypes = [ctypes.POINTER(vp), ctypes.c_char_p, ctypes.c_char_p,
                                             ctypes.c_char_p, vp, vp, i32, i32]
        L.cgtp_mixed_plan_destroy.argtypes = [vp]
        L.cgtp_mixed_plan_destroy.restype = None
        L.cgtp_mixed_plan_info.argtypes = [vp] + [ctypes.POINTER(i64)] * 5
        L.cgtp_mixed_conv_workspace.argtypes = [vp, vp, ctypes.POINTER(i64)]
        L.cgtp_mixed_conv_forward.argtypes = [vp] * 8 + [i64, vp]
        L.cgtp_mixed_conv_backward.argtypes = [vp] * 12 + [i64, vp]
        L.cgtp_mixed_conv_double_backward.argtypes = [vp] * 17 + [i64, vp]
        L.cgtp_plan_device_bytes.argtypes = [vp, ctypes.POINTER(i64)]
        L.cgtp_plan_set_wait_limit.argtypes = [vp, i64]
        L.cgtp_plan_set_node_chunk.argtypes = [vp, i64]
        L.cgtp_plan_node_chunk.argtypes = [vp, ctypes.POINTER(i64)]
        L.cgtp_graph_device_bytes.argtypes = [vp, ctypes.POINTER(i64)]
        L.cgtp_measure_fma.argtypes = [i32, i32, i32, vp, ctypes.POINTER(ctypes.c_double), vp]
        L.cgtp_measure_read.argtypes = [vp, i64, i32, i32, vp, ctypes.POINTER(ctypes.c_double), vp]
        for name in EXPORTS:
            if name not in ("cgtp_last_error", "cgtp_plan_destroy", "cgtp_graph_destroy",
                            "cgtp_mixed_plan_destroy"):
                getattr(L, name).restype = i32
        _lib = L
    return _lib


def _check(status):
    if status != CGTP_OK:
        raise CgtpError(status, lib().cgtp_last_error().decode())


def cgtp_real_sh(lmax, rvec, jacobian=False):
    """Host query of the library's real spherical harmonics of the (normalised)
    vectors rvec [n,3]: Y [n,(lmax+1)^2] and, optionally, dY/drvec [n,(lmax+1)^2,3]."""
    r = np.ascontiguousarray(rvec, dtype=np.float64).reshape(-1, 3)
    d2 = (lmax + 1) ** 2
    Y = np.zeros((r.shape[0], d2))
    dY = np.zeros((r.shape[0], d2, 3)) if jacobian else None
    _check(lib().cgtp_real_sh(lmax, r.ctypes.data, r.shape[0], Y.ctypes.data,
                              dY.ctypes.data if jacobian else None))
    return (Y, dY) if jacobian else Y


def cgtp_real_cg_block(l1, l2, l3):
    n = (2 * l1 + 1) * (2 * l2 + 1) * (2 * l3 + 1)
    buf = np.zeros(n, dtype=np.float64)
    _check(lib().cgtp_real_cg_block(l1, l2, l3, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n))
    return buf.reshape(2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1)


# ---------------------------------------------------------------------------
# torch-facing helpers (imported lazily so host-only use needs no torch CUDA)
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t, name, dtype=None):
    torch = _torch()
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Plan:
    """cgtp_plan_create: paths, CG tables and (uvw) bounded scratch on the current device."""

    def __init__(self, irreps_in1, irreps_in2, irreps_out, mode="uvu", dtype=None, radial_k=0,
                 instructions=None):
        torch = _torch()
        dtype = dtype or torch.float32
        self.mode = mode
        self.dtype = dtype
        self.radial_k = radial_k
        m = CGTP_UVU if mode == "uvu" else CGTP_UVW
        dt = {torch.float64: CGTP_F64, torch.bfloat16: CGTP_BF16}.get(dtype, CGTP_F32)
        # bfloat16 plans read bfloat16 inputs and write float32 outputs
        self.out_dtype = torch.float32 if dtype == torch.bfloat16 else dtype
        h = ctypes.c_void_p()
        arr, n = None, 0
        if instructions:
            n = len(instructions)
            arr = (ctypes.c_int * (3 * n))(*[v for ins in instructions for v in ins])
        _check(lib().cgtp_plan_create(ctypes.byref(h), irreps_in1.encode(), irreps_in2.encode(),
                                      irreps_out.encode(), ctypes.cast(arr, ctypes.c_void_p) if arr else None,
                                      n, m, dt, radial_k))
        self._h = h
        d = [ctypes.c_int64() for _ in range(4)]
        npaths = ctypes.c_int()
        _check(lib().cgtp_plan_info(h, *[ctypes.byref(v) for v in d], ctypes.byref(npaths)))
        self.d1, self.d2, self.d_out, self.w_numel = (v.value for v in d)
        self.n_paths = npaths.value

    @property
    def handle(self):
        return self._h

    def set_wait_limit(self, polls):
        """Polls before a staging wait of the plan's kernels gives up (cgtp_plan_set_wait_limit)."""
        _check(lib().cgtp_plan_set_wait_limit(self._h, int(polls)))

    def device_bytes(self):
        """Device memory the library holds for this plan (cgtp_plan_device_bytes)."""
        nb = ctypes.c_int64()
        _check(lib().cgtp_plan_device_bytes(self._h, ctypes.byref(nb)))
        return nb.value

    @property
    def node_chunk(self):
        """Nodes per streamed chunk of a radial uvw plan's node state (cgtp_plan_node_chunk)."""
        nb = ctypes.c_int64()
        _check(lib().cgtp_plan_node_chunk(self._h, ctypes.byref(nb)))
        return nb.value

    def set_node_chunk(self, nodes):
        """cgtp_plan_set_node_chunk: stream the node state `nodes` nodes at a time."""
        _check(lib().cgtp_plan_set_node_chunk(self._h, int(nodes)))

    def launches_per_step(self, n_nodes):
        """Kernel launches of one forward + backward of a radial uvw plan on n_nodes nodes:
        per streamed node chunk of the plan, the forward's edge stage and node GEMM and
        the backward's GEMM, edge stage, two GEMMs and split-K reduction."""
        return 7 * max(1, -(-int(n_nodes) // max(1, self.node_chunk)))

    def path(self, p):
        ints = (ctypes.c_int * 10)()
        _check(lib().cgtp_plan_path(self._h, p, ints, None, 0))
        l1, l2, l3 = ints[0], ints[1], ints[2]
        n = (2 * l1 + 1) * (2 * l2 + 1) * (2 * l3 + 1)
        buf = np.zeros(n)
        _check(lib().cgtp_plan_path(self._h, p, ints, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n))
        return list(ints), buf.reshape(2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.cgtp_plan_destroy(h)
            self._h = None


class Graph:
    """cgtp_graph_create: validated receiver-sorted CSR + device transpose."""

    def __init__(self, rowptr, col, N, stream=None):
        torch = _torch()
        self.rowptr, self.col, self.N = rowptr, col, int(N)
        self.E = int(col.numel())
        h = ctypes.c_void_p()
        _check(lib().cgtp_graph_create(ctypes.byref(h), _ptr(rowptr, "rowptr", torch.int32),
                                       _ptr(col, "col", torch.int32) if self.E else None,
                                       self.N, self.E, _stream(stream)))
        self._h = h

    @property
    def handle(self):
        return self._h

    def device_bytes(self):
        """Device memory the library holds for this graph (cgtp_graph_device_bytes)."""
        nb = ctypes.c_int64()
        _check(lib().cgtp_graph_device_bytes(self._h, ctypes.byref(nb)))
        return nb.value

    def transpose(self, stream=None):
        torch = _torch()
        dev = self.rowptr.device
        t_rowptr = torch.empty(self.N + 1, dtype=torch.int32, device=dev)
        t_eid = torch.empty(max(self.E, 1), dtype=torch.int32, device=dev)
        t_dst = torch.empty(max(self.E, 1), dtype=torch.int32, device=dev)
        _check(lib().cgtp_graph_transpose(self._h, _ptr(t_rowptr, "t_rowptr"), _ptr(t_eid, "t_eid"),
                                          _ptr(t_dst, "t_dst"), _stream(stream)))
        return t_rowptr, t_eid[:self.E], t_dst[:self.E]

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.cgtp_graph_destroy(h)
            self._h = None


def cgtp_forward(plan, x1, x2, W, out=None, stream=None):
    torch = _torch()
    B = x1.shape[0]
    if out is None:
        out = torch.empty(B, plan.d_out, dtype=plan.out_dtype, device=x1.device)
    _check(lib().cgtp_forward(plan.handle, _ptr(x1, "x1", plan.dtype), _ptr(x2, "x2", plan.dtype),
                              _ptr(W, "W", plan.dtype), _ptr(out, "out", plan.out_dtype), B, _stream(stream)))
    return out


def cgtp_backward(plan, gout, x1, x2, W, stream=None):
    torch = _torch()
    B = x1.shape[0]
    od = plan.out_dtype   # bfloat16 plans write FP32 gradients
    gx1, gx2, gW = (torch.empty(t.shape, dtype=od, device=t.device) for t in (x1, x2, W))
    _check(lib().cgtp_backward(plan.handle, _ptr(gout, "gout", plan.dtype), _ptr(x1, "x1", plan.dtype),
                               _ptr(x2, "x2", plan.dtype), _ptr(W, "W", plan.dtype),
                               _ptr(gx1, "gx1", od), _ptr(gx2, "gx2", od), _ptr(gW, "gW", od), B,
                               _stream(stream)))
    return gx1, gx2, gW


def cgtp_conv_forward(plan, graph, x, Y, W_or_R, M=None, out=None, stream=None):
    torch = _torch()
    if out is None:
        out = torch.empty(graph.N, plan.d_out, dtype=plan.out_dtype, device=x.device)
    _check(lib().cgtp_conv_forward(plan.handle, graph.handle, _ptr(x, "x", plan.dtype),
                                   _ptr(Y, "Y", plan.dtype), _ptr(W_or_R, "W_or_R", plan.dtype),
                                   _ptr(M, "M", plan.dtype), _ptr(out, "out", plan.out_dtype), _stream(stream)))
    return out


def cgtp_conv_backward(plan, graph, gout, x, Y, W_or_R, M=None, stream=None, outs=None):
    torch = _torch()
    if outs is None:
        od = plan.out_dtype
        gx, gY, gW = (torch.empty(t.shape, dtype=od, device=t.device) for t in (x, Y, W_or_R))
        gM = torch.empty(M.shape, dtype=od, device=M.device) if M is not None else None
    else:
        gx, gY, gW, gM = outs
    _check(lib().cgtp_conv_backward(plan.handle, graph.handle, _ptr(gout, "gout", plan.dtype),
                                    _ptr(x, "x", plan.dtype), _ptr(Y, "Y", plan.dtype),
                                    _ptr(W_or_R, "W_or_R", plan.dtype), _ptr(M, "M", plan.dtype),
                                    _ptr(gx, "gx", plan.out_dtype), _ptr(gY, "gY", plan.out_dtype),
                                    _ptr(gW, "gW", plan.out_dtype), _ptr(gM, "gM", plan.out_dtype),
                                    _stream(stream)))
    return gx, gY, gW, gM


def _workspace(nbytes, device):
    torch = _torch()
    # 256-byte aligned: torch's caching allocator hands out 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def cgtp_conv_double_backward(plan, graph, gout, x, Y, W_or_R, ggx, ggY, ggW_or_ggR, M=None, ggM=None,
                              stream=None):
    """Second derivatives: (d_gout, d_x, d_Y, d_W_or_dR, d_M) of
    S = <ggx, gx> + <ggY, gY> + <ggW, gW> (+ <ggM, gM> for uvw)."""
    torch = _torch()
    nb = ctypes.c_int64()
    _check(lib().cgtp_conv_double_backward_workspace(plan.handle, graph.handle, ctypes.byref(nb)))
    ws = _workspace(nb.value, x.device)
    d_g, d_x, d_Y, d_W = torch.empty_like(gout), torch.empty_like(x), torch.empty_like(Y), torch.empty_like(W_or_R)
    d_M = torch.empty_like(M) if M is not None else None
    dt = plan.dtype
    _check(lib().cgtp_conv_double_backward(
        plan.handle, graph.handle, _ptr(gout, "gout", dt), _ptr(x, "x", dt), _ptr(Y, "Y", dt),
        _ptr(W_or_R, "W_or_R", dt), _ptr(M, "M", dt), _ptr(ggx, "ggx", dt), _ptr(ggY, "ggY", dt),
        _ptr(ggW_or_ggR, "ggW_or_ggR", dt), _ptr(ggM, "ggM", dt), _ptr(d_g, "d_gout"), _ptr(d_x, "d_x"),
        _ptr(d_Y, "d_Y"), _ptr(d_W, "d_W"), _ptr(d_M, "d_M"), _ptr(ws, "workspace"), nb.value, _stream(stream)))
    return d_g, d_x, d_Y, d_W, d_M


def cgtp_double_backward(plan, gout, x1, x2, W, gg1, gg2, ggW, stream=None):
    """Second derivatives of the batched product: (d_gout, d_x1, d_x2, d_W)."""
    torch = _torch()
    B = x1.shape[0]
    nb = ctypes.c_int64()
    _check(lib().cgtp_double_backward_workspace(plan.handle, B, ctypes.byref(nb)))
    ws = _workspace(nb.value, x1.device)
    d_g, d_1, d_2, d_W = torch.empty_like(gout), torch.empty_like(x1), torch.empty_like(x2), torch.empty_like(W)
    dt = plan.dtype
    _check(lib().cgtp_double_backward(
        plan.handle, _ptr(gout, "gout", dt), _ptr(x1, "x1", dt), _ptr(x2, "x2", dt), _ptr(W, "W", dt),
        _ptr(gg1, "gg1", dt), _ptr(gg2, "gg2", dt), _ptr(ggW, "ggW", dt), _ptr(d_g, "d_gout"),
        _ptr(d_1, "d_x1"), _ptr(d_2, "d_x2"), _ptr(d_W, "d_W"), B, _ptr(ws, "workspace"), nb.value,
        _stream(stream)))
    return d_g, d_1, d_2, d_W


def cgtp_conv_forward_sh(plan, graph, x, rvec, W, out=None, stream=None):
    """Fused convolution whose edge harmonics are evaluated in the kernel from rvec [E,3]."""
    torch = _torch()
    if out is None:
        out = torch.empty(graph.N, plan.d_out, dtype=plan.out_dtype, device=x.device)
    dt = plan.dtype
    _check(lib().cgtp_conv_forward_sh(plan.handle, graph.handle, _ptr(x, "x", dt), _ptr(rvec, "rvec", dt),
                                      _ptr(W, "W", dt), _ptr(out, "out", plan.out_dtype), _stream(stream)))
    return out


def cgtp_conv_backward_sh(plan, graph, gout, x, rvec, W, stream=None):
    """Adjoint of cgtp_conv_forward_sh: (gx, gY, grvec, gW)."""
    torch = _torch()
    dt = plan.dtype
    gx = torch.empty(x.shape, dtype=plan.out_dtype, device=x.device)
    gY = torch.empty(graph.E, plan.d2, dtype=plan.out_dtype, device=x.device)
    grvec = torch.empty(rvec.shape, dtype=plan.out_dtype, device=x.device)
    gW = torch.empty(W.shape, dtype=plan.out_dtype, device=x.device)
    _check(lib().cgtp_conv_backward_sh(plan.handle, graph.handle, _ptr(gout, "gout", dt), _ptr(x, "x", dt),
                                       _ptr(rvec, "rvec", dt), _ptr(W, "W", dt), _ptr(gx, "gx"), _ptr(gY, "gY"),
                                       _ptr(grvec, "grvec"), _ptr(gW, "gW"), _stream(stream)))
    return gx, gY, grvec, gW


def cgtp_conv_forward_sh_radial(plan, graph, x, rvec, M, rbf_lo=0.5, rbf_hi=5.0, out=None, stream=None):
    """uvw radial convolution whose harmonics and radial basis are evaluated in the kernels."""
    torch = _torch()
    if out is None:
        out = torch.empty(graph.N, plan.d_out, dtype=plan.out_dtype, device=x.device)
    dt = plan.dtype
    _check(lib().cgtp_conv_forward_sh_radial(plan.handle, graph.handle, _ptr(x, "x", dt), _ptr(rvec, "rvec", dt),
                                             _ptr(M, "M", dt), float(rbf_lo), float(rbf_hi),
                                             _ptr(out, "out", plan.out_dtype), _stream(stream)))
    return out


def cgtp_conv_backward_sh_radial(plan, graph, gout, x, rvec, M, rbf_lo=0.5, rbf_hi=5.0, stream=None):
    """Adjoint of cgtp_conv_forward_sh_radial: (gx, gY, gR, grvec, gM)."""
    torch = _torch()
    dt, od, dev = plan.dtype, plan.out_dtype, x.device
    gx = torch.empty(x.shape, dtype=od, device=dev)
    gY = torch.empty(graph.E, plan.d2, dtype=od, device=dev)
    gR = torch.empty(graph.E, plan.radial_k, dtype=od, device=dev)
    grvec = torch.empty(rvec.shape, dtype=od, device=dev)
    gM = torch.empty(M.shape, dtype=od, device=dev)
    _check(lib().cgtp_conv_backward_sh_radial(
        plan.handle, graph.handle, _ptr(gout, "gout", dt), _ptr(x, "x", dt), _ptr(rvec, "rvec", dt),
        _ptr(M, "M", dt), float(rbf_lo), float(rbf_hi), _ptr(gx, "gx"), _ptr(gY, "gY"), _ptr(gR, "gR"),
        _ptr(grvec, "grvec"), _ptr(gM, "gM"), _stream(stream)))
    return gx, gY, gR, grvec, gM


CGTP_MEASURE_FFMA, CGTP_MEASURE_FFMA2, CGTP_MEASURE_DFMA = 0, 1, 2


def measure_fma(kind, ctas, iters, sink, stream=None):
    """Enqueue one arithmetic-throughput launch (cgtp_measure_fma); returns its FLOPs."""
    fl = ctypes.c_double()
    _check(lib().cgtp_measure_fma(int(kind), int(ctas), int(iters), _ptr(sink, "sink"), ctypes.byref(fl),
                                  _stream(stream)))
    return fl.value


def measure_read(buf, reps, ctas, sink, stream=None):
    """Enqueue one read-bandwidth launch over buf (cgtp_measure_read); returns the bytes read."""
    nb = ctypes.c_double()
    _check(lib().cgtp_measure_read(_ptr(buf, "buf"), buf.numel() * buf.element_size(), int(reps), int(ctas),
                                   _ptr(sink, "sink"), ctypes.byref(nb), _stream(stream)))
    return nb.value


class MixedPlan:
    """cgtp_mixed_plan_create: a connection mode ("uvu" or "uvw") per instruction, every
    instruction summing into its block of irreps_out; weights Wu [E, wu_numel] and
    Ww [E, ww_numel] in instruction order."""

    def __init__(self, irreps_in1, irreps_in2, irreps_out, instructions, modes, dtype=None):
        torch = _torch()
        dtype = dtype or torch.float32
        self.dtype = dtype
        dt = {torch.float64: CGTP_F64, torch.bfloat16: CGTP_BF16}.get(dtype, CGTP_F32)
        n = len(instructions)
        if len(modes) != n:
            raise ValueError("one mode per instruction")
        ins = (ctypes.c_int * (3 * n))(*[v for t in instructions for v in t])
        md = (ctypes.c_int * n)(*[{"uvu": CGTP_UVU, "uvw": CGTP_UVW}.get(m, -1) for m in modes])
        h = ctypes.c_void_p()
        _check(lib().cgtp_mixed_plan_create(ctypes.byref(h), irreps_in1.encode(), irreps_in2.encode(),
                                            irreps_out.encode(), ctypes.cast(ins, ctypes.c_void_p),
                                            ctypes.cast(md, ctypes.c_void_p), n, dt))
        self._h = h
        d = [ctypes.c_int64() for _ in range(5)]
        _check(lib().cgtp_mixed_plan_info(h, *[ctypes.byref(v) for v in d]))
        self.d1, self.d2, self.d_out, self.wu_numel, self.ww_numel = (v.value for v in d)
        self.mode = "mixed"
        self.out_dtype = torch.float32 if dtype == torch.bfloat16 else dtype   # bfloat16 plans: FP32 outputs
        self.irreps = (irreps_in1, irreps_in2, irreps_out)
        self.instructions, self.modes = [tuple(t) for t in instructions], list(modes)

    @property
    def handle(self):
        return self._h

    def workspace(self, graph, device):
        nb = ctypes.c_int64()
        _check(lib().cgtp_mixed_conv_workspace(self._h, graph.handle, ctypes.byref(nb)))
        return _workspace(nb.value, device), nb.value

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.cgtp_mixed_plan_destroy(h)
            self._h = None


def _mixed_ws(plan, graph, device, workspace):
    if workspace is None:
        return plan.workspace(graph, device)
    return workspace, workspace.numel()


def cgtp_mixed_conv_forward(plan, graph, x, Y, Wu, Ww, out=None, stream=None, workspace=None):
    """out [N, d_out] of the convolution with mixed instruction modes (workspace: an
    optional uint8 device buffer of at least plan.workspace(...) bytes)."""
    torch = _torch()
    if out is None:
        out = torch.empty(graph.N, plan.d_out, dtype=plan.out_dtype, device=x.device)
    ws, nb = _mixed_ws(plan, graph, x.device, workspace)
    dt = plan.dtype
    _check(lib().cgtp_mixed_conv_forward(plan.handle, graph.handle, _ptr(x, "x", dt), _ptr(Y, "Y", dt),
                                         _ptr(Wu, "Wu", dt), _ptr(Ww, "Ww", dt), _ptr(out, "out", plan.out_dtype),
                                         _ptr(ws, "workspace"), nb, _stream(stream)))
    return out


def cgtp_mixed_conv_backward(plan, graph, gout, x, Y, Wu, Ww, stream=None, workspace=None, outs=None):
    """(gx, gY, gWu, gWw) of cgtp_mixed_conv_forward (outs: optional preallocated results)."""
    torch = _torch()
    if outs is None:
        od = plan.out_dtype
        gx, gY = (torch.empty(t.shape, dtype=od, device=t.device) for t in (x, Y))
        gWu = torch.empty(Wu.shape, dtype=od, device=Wu.device) if Wu is not None else None
        gWw = torch.empty(Ww.shape, dtype=od, device=Ww.device) if Ww is not None else None
    else:
        gx, gY, gWu, gWw = outs
    ws, nb = _mixed_ws(plan, graph, x.device, workspace)
    dt = plan.dtype
    _check(lib().cgtp_mixed_conv_backward(
        plan.handle, graph.handle, _ptr(gout, "gout", dt), _ptr(x, "x", dt), _ptr(Y, "Y", dt), _ptr(Wu, "Wu", dt),
        _ptr(Ww, "Ww", dt), _ptr(gx, "gx"), _ptr(gY, "gY"), _ptr(gWu, "gWu"), _ptr(gWw, "gWw"),
        _ptr(ws, "workspace"), nb, _stream(stream)))
    return gx, gY, gWu, gWw


def cgtp_mixed_conv_double_backward(plan, graph, gout, x, Y, Wu, Ww, ggx, ggY, ggWu, ggWw, stream=None,
                                    workspace=None):
    """(d_gout, d_x, d_Y, d_Wu, d_Ww) of S = <ggx, gx> + <ggY, gY> + <ggWu, gWu> + <ggWw, gWw>."""
    torch = _torch()
    d_g, d_x, d_Y = torch.empty_like(gout), torch.empty_like(x), torch.empty_like(Y)
    d_Wu = torch.empty_like(Wu) if Wu is not None else None
    d_Ww = torch.empty_like(Ww) if Ww is not None else None
    ws, nb = _mixed_ws(plan, graph, x.device, workspace)
    dt = plan.dtype
    _check(lib().cgtp_mixed_conv_double_backward(
        plan.handle, graph.handle, _ptr(gout, "gout", dt), _ptr(x, "x", dt), _ptr(Y, "Y", dt), _ptr(Wu, "Wu", dt),
        _ptr(Ww, "Ww", dt), _ptr(ggx, "ggx", dt), _ptr(ggY, "ggY", dt), _ptr(ggWu, "ggWu", dt),
        _ptr(ggWw, "ggWw", dt), _ptr(d_g, "d_gout"), _ptr(d_x, "d_x"), _ptr(d_Y, "d_Y"), _ptr(d_Wu, "d_Wu"),
        _ptr(d_Ww, "d_Ww"), _ptr(ws, "workspace"), nb, _stream(stream)))
    return d_g, d_x, d_Y, d_Wu, d_Ww
