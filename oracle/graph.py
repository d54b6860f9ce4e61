"""Receiver-sorted CSR checks and the sender transpose (oracle side).

Test infrastructure only (see the package docstring).

The fused convolution of "An Efficient Sparse Kernel Generator for
O(3)-Equivariant Deep Networks" (Figure 4B) sums edge messages into the
receiving node; the edges are given as a CSR list sorted by receiver:
``rowptr[N+1]`` (monotone, rowptr[0] = 0, rowptr[N] = E) and ``col[E]`` = sender.

The gradient with respect to the node features is owned by the sender, so the
backward pass walks the transpose: ``t_rowptr[N+1]`` (prefix sum of out-degrees)
and ``t_eid[E]`` = the CSR positions ordered by sender, ties kept in CSR order
(a stable sort), with ``t_dst[E]`` the receiver of each such edge.
"""

import numpy as np


def check_csr(rowptr, col, N):
    rowptr = np.asarray(rowptr)
    col = np.asarray(col)
    if rowptr.shape != (N + 1,) or rowptr[0] != 0:
        return False
    if np.any(np.diff(rowptr) < 0) or rowptr[-1] != col.shape[0]:
        return False
    if col.size and (col.min() < 0 or col.max() >= N):
        return False
    return True


def csr_dst(rowptr):
    """Receiver of every CSR position."""
    return np.repeat(np.arange(len(rowptr) - 1, dtype=np.int64), np.diff(rowptr))


def transpose(rowptr, col, N):
    """(t_rowptr, t_eid, t_dst) of the sender-ordered view, int64, stable."""
    col = np.asarray(col, dtype=np.int64)
    t_eid = np.argsort(col, kind="stable")
    counts = np.bincount(col, minlength=N)
    t_rowptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    t_dst = csr_dst(rowptr)[t_eid]
    return t_rowptr, t_eid.astype(np.int64), t_dst
