"""The allocation-free transpose entry point against the allocating one.

cgtp_graph_transpose_noalloc serves callers that may not allocate device memory
where they need the sender transpose; it must give exactly what
cgtp_graph_create + cgtp_graph_transpose give.  Two calls in a row on different
graphs also show that the shared working array is cleared between calls, and a
graph at the largest accepted node count fills that array to its last word.  This
file is collected last so that a run stopping at its first failure has already
run every other test.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import clebsch_gordan_tensor_racah_gb300 as cg  # noqa: E402

pytestmark = pytest.mark.gpu


def _csr(seed, N, E, hub=None):
    rng = np.random.default_rng(seed)
    src = rng.integers(0, N, E)
    if hub is not None:
        src = np.where(rng.random(E) < 0.3, hub, src)
    dst = rng.integers(0, N, E)
    order = np.argsort(dst, kind="stable")
    rowptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))]).astype(np.int32)
    return rowptr, src[order].astype(np.int32)


def _noalloc(rowptr_d, col_d, N, E):
    L = cg.lib()
    dev = rowptr_d.device
    t_rowptr = torch.full((N + 1,), -1, dtype=torch.int32, device=dev)
    t_eid = torch.full((max(E, 1),), -1, dtype=torch.int32, device=dev)
    t_dst = torch.full((max(E, 1),), -1, dtype=torch.int32, device=dev)
    st = L.cgtp_graph_transpose_noalloc(
        ctypes.c_void_p(rowptr_d.data_ptr()), ctypes.c_void_p(col_d.data_ptr()), N, E,
        ctypes.c_void_p(t_rowptr.data_ptr()), ctypes.c_void_p(t_eid.data_ptr()),
        ctypes.c_void_p(t_dst.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == cg.CGTP_OK, L.cgtp_last_error()
    return t_rowptr, t_eid[:E], t_dst[:E]


def test_noalloc_transpose_matches_allocating_transpose_twice():
    # second call: smaller graph with a hub sender; third: the largest accepted node
    # count, where flag, total, counts and tile sums fill the working array exactly
    cases = [(0, 20000, 640000, None), (1, 777, 9000, 5), (2, 1 << 20, 300000, None)]
    for seed, N, E, hub in cases:
        rowptr, col = _csr(seed, N, E, hub)
        rd = torch.from_numpy(rowptr).cuda()
        cd = torch.from_numpy(col).cuda()
        ref = cg.Graph(rd, cd, N).transpose()
        got = _noalloc(rd, cd, N, E)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_rejects_oversized_graph():
    L = cg.lib()
    st = L.cgtp_graph_transpose_noalloc(None, None, (1 << 20) + 1, 0, None, None, None, None)
    assert st == cg.CGTP_EINVAL
    assert b"1048576" in L.cgtp_last_error()
