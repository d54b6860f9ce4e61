"""CG tensor product and fused CG-tensor-product convolution, forward and backward.

Test infrastructure only (see the package docstring).  FP64 throughout; inputs
of any float type are promoted exactly.

Definitions followed
--------------------
"An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks":

* Figure 1 / Figure 4A (batched product, no graph), for every sample b and path
  (l1, l2 -> l3) of the plan::

      z[b][path, u, m3] = W[b][path, u] * sum_{m1, m2} C[m1, m2, m3] x1[b][u, m1] x2[b][m2]

* Figure 4B (fused graph convolution): the same message per edge e = (src -> dst)
  with x1 = x[src], x2 = Y[e], W = W[e], summed into the receiver::

      out[n] = sum_{e in row n of the CSR, in CSR order} message(e)

* Abstract ("optimized kernels for the gradient"): the adjoints with respect to
  x (or x1), Y (or x2) and W, written out by the chain rule.

"Sobek: Streaming Equivariant Tensor Product Convolutions", Abstract (radial
projection with fully connected multiplicity mixing): the uvw message with
per-edge weights W_e[path, u, w] = sum_k R[e, k] M[k, path, u, w], which this
oracle forms explicitly for every edge (the plain definition), summed into
output block i_out::

      out[dst][i_out][w, m3] += sum_u W_e[path, u, w] sum_{m1,m2} C x[src][u,m1] Y[e][m2]

``C`` is ``cg.real_cg_block(l1, l2, l3)``.  No path normalisation factor.
"""

import numpy as np

from .cg import real_cg_block, sh_real_concat, sh_real_concat_jacobian
from .graph import csr_dst


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _blocks(p, x1, y2):
    D1, D2 = 2 * p.l1 + 1, 2 * p.l2 + 1
    xs = x1[:, p.off1:p.off1 + p.mul1 * D1].reshape(-1, p.mul1, D1)
    ys = y2[:, p.off2:p.off2 + D2]
    return xs, ys


def _edges_of(rowptr, nodes):
    if len(nodes) == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    eidx = np.concatenate([np.arange(rowptr[n], rowptr[n + 1]) for n in nodes]).astype(np.int64)
    owner = np.repeat(np.arange(len(nodes)), rowptr[nodes + 1] - rowptr[nodes])
    return eidx, owner


# ---------------------------------------------------------------------------
# uvu: batched product (Figure 4A) and per-edge message
# ---------------------------------------------------------------------------

def tp_uvu_forward(plan, x1, x2, W):
    """z[b] for every sample: x1 [B, d1], x2 [B, d2], W [B, w_numel] -> [B, d_out]."""
    x1, x2, W = _f64(x1), _f64(x2), _f64(W)
    out = np.zeros((x1.shape[0], plan.d_out))
    for p in plan.paths:
        C = real_cg_block(p.l1, p.l2, p.l3)
        xs, ys = _blocks(p, x1, x2)
        w = W[:, p.woff:p.woff + p.mul1]
        z = np.einsum("ijk,bui,bj->buk", C, xs, ys) * w[:, :, None]
        D3 = 2 * p.l3 + 1
        out[:, p.ooff:p.ooff + p.mul1 * D3] += z.reshape(z.shape[0], -1)
    return out


def tp_uvu_backward(plan, g, x1, x2, W):
    """Adjoints of tp_uvu_forward: (gx1 [B,d1], gx2 [B,d2], gW [B,w_numel])."""
    g, x1, x2, W = _f64(g), _f64(x1), _f64(x2), _f64(W)
    B = x1.shape[0]
    gx1, gx2, gW = np.zeros((B, plan.d1)), np.zeros((B, plan.d2)), np.zeros((B, plan.w_numel))
    for p in plan.paths:
        C = real_cg_block(p.l1, p.l2, p.l3)
        D1, D2, D3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
        xs, ys = _blocks(p, x1, x2)
        w = W[:, p.woff:p.woff + p.mul1]
        gz = g[:, p.ooff:p.ooff + p.mul1 * D3].reshape(B, p.mul1, D3)
        gW[:, p.woff:p.woff + p.mul1] += np.einsum("ijk,bui,bj,buk->bu", C, xs, ys, gz)
        gx2[:, p.off2:p.off2 + D2] += np.einsum("ijk,bui,bu,buk->bj", C, xs, w, gz)
        gx1[:, p.off1:p.off1 + p.mul1 * D1] += np.einsum(
            "ijk,bj,bu,buk->bui", C, ys, w, gz).reshape(B, -1)
    return gx1, gx2, gW


# ---------------------------------------------------------------------------
# uvu fused convolution (Figure 4B)
# ---------------------------------------------------------------------------

def conv_uvu_forward(plan, x, Y, W, rowptr, col, nodes=None):
    """out[N, d_out] (or the rows of `nodes`, in that order)."""
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    x, Y, W = _f64(x), _f64(Y), _f64(W)
    if nodes is None:
        nodes = np.arange(len(rowptr) - 1)
    nodes = np.asarray(nodes, dtype=np.int64)
    eidx, owner = _edges_of(rowptr, nodes)
    out = np.zeros((len(nodes), plan.d_out))
    if eidx.size == 0:
        return out
    msg = tp_uvu_forward(plan, x[col[eidx]], Y[eidx], W[eidx])
    np.add.at(out, owner, msg)          # CSR order within each receiver
    return out


def conv_uvu_backward(plan, g, x, Y, W, rowptr, col, edges=None):
    """(gx [N,d1], gY [Es,d2], gW [Es,w_numel]) over CSR positions `edges` (all by default).

    gx only collects the contributions of the selected edges, summed over each
    sender's edges in CSR order.
    """
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    g, x, Y, W = _f64(g), _f64(x), _f64(Y), _f64(W)
    N = len(rowptr) - 1
    if edges is None:
        edges = np.arange(col.shape[0])
    edges = np.asarray(edges, dtype=np.int64)
    dst = csr_dst(rowptr)[edges]
    src = col[edges]
    gxe, gY, gW = tp_uvu_backward(plan, g[dst], x[src], Y[edges], W[edges])
    gx = np.zeros((N, plan.d1))
    np.add.at(gx, src, gxe)
    return gx, gY, gW


# ---------------------------------------------------------------------------
# uvw with radial weights (Sobek): plain definition, W_e formed per edge
# ---------------------------------------------------------------------------

def conv_uvw_radial_forward(plan, x, Y, R, M, rowptr, col, nodes=None, block=256):
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    x, Y, R, M = _f64(x), _f64(Y), _f64(R), _f64(M)
    if nodes is None:
        nodes = np.arange(len(rowptr) - 1)
    nodes = np.asarray(nodes, dtype=np.int64)
    out = np.zeros((len(nodes), plan.d_out))
    eidx, owner = _edges_of(rowptr, nodes)
    for s in range(0, eidx.size, block):
        e = eidx[s:s + block]
        We = R[e] @ M                       # per-edge weights, formed explicitly
        x1, y2 = x[col[e]], Y[e]
        msg = np.zeros((e.size, plan.d_out))
        for p in plan.paths:
            C = real_cg_block(p.l1, p.l2, p.l3)
            D3 = 2 * p.l3 + 1
            xs, ys = _blocks(p, x1, y2)
            t = np.einsum("ijk,eui,ej->euk", C, xs, ys)
            w = We[:, p.woff:p.woff + p.mul1 * p.mul_out].reshape(-1, p.mul1, p.mul_out)
            msg[:, p.ooff:p.ooff + p.mul_out * D3] += np.einsum("euw,euk->ewk", w, t).reshape(e.size, -1)
        np.add.at(out, owner[s:s + block], msg)
    return out


def conv_uvw_radial_backward(plan, g, x, Y, R, M, rowptr, col, edges=None, block=256):
    """(gx [N,d1], gY [Es,d2], gR [Es,K], gM [K,w_numel]) over CSR positions `edges`."""
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    g, x, Y, R, M = _f64(g), _f64(x), _f64(Y), _f64(R), _f64(M)
    N = len(rowptr) - 1
    if edges is None:
        edges = np.arange(col.shape[0])
    edges = np.asarray(edges, dtype=np.int64)
    dst_all = csr_dst(rowptr)
    gx = np.zeros((N, plan.d1))
    gY = np.zeros((edges.size, plan.d2))
    gR = np.zeros((edges.size, R.shape[1]))
    gM = np.zeros_like(M)
    for s in range(0, edges.size, block):
        e = edges[s:s + block]
        We = R[e] @ M
        gWe = np.zeros_like(We)
        x1, y2, gd = x[col[e]], Y[e], g[dst_all[e]]
        gxe = np.zeros((e.size, plan.d1))
        for p in plan.paths:
            C = real_cg_block(p.l1, p.l2, p.l3)
            D1, D2, D3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
            xs, ys = _blocks(p, x1, y2)
            t = np.einsum("ijk,eui,ej->euk", C, xs, ys)
            sl = slice(p.woff, p.woff + p.mul1 * p.mul_out)
            w = We[:, sl].reshape(-1, p.mul1, p.mul_out)
            go = gd[:, p.ooff:p.ooff + p.mul_out * D3].reshape(-1, p.mul_out, D3)
            gWe[:, sl] = np.einsum("ewk,euk->euw", go, t).reshape(e.size, -1)
            gt = np.einsum("euw,ewk->euk", w, go)
            gxe[:, p.off1:p.off1 + p.mul1 * D1] += np.einsum("ijk,ej,euk->eui", C, ys, gt).reshape(e.size, -1)
            gY[s:s + e.size, p.off2:p.off2 + D2] += np.einsum("ijk,eui,euk->ej", C, xs, gt)
        gR[s:s + e.size] = gWe @ M.T
        gM += R[e].T @ gWe
        np.add.at(gx, col[e], gxe)
    return gx, gY, gR, gM


# ---------------------------------------------------------------------------
# brute force: one dense bilinear tensor per edge (tiny inputs only)
# ---------------------------------------------------------------------------

def dense_tensor(plan, w_edge):
    """T[d1, d2, d_out] with out = einsum('ijk,i,j->k', T, x1, x2) for one edge.

    w_edge is that edge's uvu weight row [w_numel] or uvw weight row
    [sum_path mul1*mul_out].  Built entry by entry with explicit index
    arithmetic, independently of the vectorised per-path code above.
    """
    T = np.zeros((plan.d1, plan.d2, plan.d_out))
    for p in plan.paths:
        C = real_cg_block(p.l1, p.l2, p.l3)
        D1, D2, D3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
        for u in range(p.mul1):
            for m1 in range(D1):
                i = p.off1 + u * D1 + m1
                for m2 in range(D2):
                    j = p.off2 + m2
                    for m3 in range(D3):
                        c = C[m1, m2, m3]
                        if c == 0.0:
                            continue
                        if plan.mode == "uvu":
                            k = p.ooff + u * D3 + m3
                            T[i, j, k] += w_edge[p.woff + u] * c
                        else:
                            for w in range(p.mul_out):
                                k = p.ooff + w * D3 + m3
                                T[i, j, k] += w_edge[p.woff + u * p.mul_out + w] * c
    return T


def conv_uvw_radial_gM_entries(plan, g, x, Y, R, rowptr, col, entries):
    """Selected entries of gM, each summed over every edge (plain definition).

    entries: iterable of (k, path index, u, w).  gM[k][woff + u*mul_out + w] =
    sum_e R[e,k] sum_m3 g[dst][ooff + w*D3 + m3] t_e[u, m3] with
    t_e[u, m3] = sum_{m1,m2} C x[src][u, m1] Y[e][m2].
    """
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    g, x = np.asarray(g), np.asarray(x)
    Y, R = _f64(Y), _f64(R)
    dst = csr_dst(rowptr)
    out = []
    for (k, pi, u, w) in entries:
        p = plan.paths[pi]
        C = real_cg_block(p.l1, p.l2, p.l3)
        D1, D2, D3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
        xs = x[:, p.off1 + u * D1:p.off1 + (u + 1) * D1][col]
        ys = Y[:, p.off2:p.off2 + D2]
        t = np.einsum("ijk,ei,ej->ek", C, _f64(xs), ys)
        gw = g[:, p.ooff + w * D3:p.ooff + (w + 1) * D3][dst]
        out.append(float((R[:, k] * (_f64(gw) * t).sum(1)).sum()))
    return np.array(out)


def conv_uvw_radial_gM_slice(plan, g, x, Y, R, rowptr, col, k, pi, chunk=1 << 16):
    """One (k, path) slice of gM, [mul1, mul_out], summed over every edge.

    Same definition as conv_uvw_radial_gM_entries, for all (u, w) of the slice
    at once: gM[k][path][u][w] = sum_e R[e,k] sum_m3 t_e[u, m3] g[dst][w, m3],
    the edge sum taken in chunks of edges, each a matrix product over (e, m3).
    """
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    dst = csr_dst(rowptr)
    p = plan.paths[pi]
    C = real_cg_block(p.l1, p.l2, p.l3)
    D1, D2, D3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
    acc = np.zeros((p.mul1, p.mul_out))
    for e0 in range(0, col.size, chunk):
        e1 = min(col.size, e0 + chunk)
        xs = _f64(x[col[e0:e1], p.off1:p.off1 + p.mul1 * D1]).reshape(-1, p.mul1, D1)
        ys = _f64(Y[e0:e1, p.off2:p.off2 + D2])
        t = np.einsum("ijk,eui,ej->euk", C, xs, ys, optimize=True) * _f64(R[e0:e1, k])[:, None, None]
        gw = _f64(g[dst[e0:e1], p.ooff:p.ooff + p.mul_out * D3]).reshape(-1, p.mul_out, D3)
        acc += np.einsum("euk,ewk->uw", t, gw, optimize=True)
    return acc


# ---------------------------------------------------------------------------
# second derivatives ("double backward")
# ---------------------------------------------------------------------------
# "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
# Abstract: higher partial derivatives for force prediction, obtained from the
# forward and gradient operations through an identity.  With the backward
# (dL/da_j)_j = B_j(g; a) of a message that is linear in each operand a_j, and
# cotangents c_j of those gradients, the scalar
#     S = sum_j <c_j, B_j(g; a)> = <g, sum_i F(a with a_i replaced by c_i)>
# has the derivatives
#     dS/dg   = sum_i F(a with a_i -> c_i)
#     dS/da_j = sum_{i != j} B_j(g; a with a_i -> c_i)
# since B_j does not depend on a_j.  The tests pin these against exact
# directional differences of S computed with the backward alone.

def _double_backward(fwd, bwd, g, a, c):
    n = len(a)
    d_g = None
    d = [None] * n
    for i in range(n):
        ai = list(a)
        ai[i] = c[i]
        f = fwd(*ai)
        d_g = f if d_g is None else d_g + f
        grads = bwd(g, *ai)
        for j in range(n):
            if j != i:
                d[j] = grads[j] if d[j] is None else d[j] + grads[j]
    return (d_g, *d)


def conv_uvu_double_backward(plan, g, x, Y, W, ggx, ggY, ggW, rowptr, col):
    """(d_g [N,d_out], d_x [N,d1], d_Y [E,d2], d_W [E,w_numel]) for the uvu convolution."""
    fwd = lambda x_, Y_, W_: conv_uvu_forward(plan, x_, Y_, W_, rowptr, col)
    bwd = lambda g_, x_, Y_, W_: conv_uvu_backward(plan, g_, x_, Y_, W_, rowptr, col)
    return _double_backward(fwd, bwd, _f64(g), [_f64(x), _f64(Y), _f64(W)],
                            [_f64(ggx), _f64(ggY), _f64(ggW)])


def conv_uvw_radial_double_backward(plan, g, x, Y, R, M, ggx, ggY, ggR, ggM, rowptr, col):
    """(d_g, d_x, d_Y, d_R, d_M) for the uvw convolution with radial weights W = R M."""
    fwd = lambda x_, Y_, R_, M_: conv_uvw_radial_forward(plan, x_, Y_, R_, M_, rowptr, col)
    bwd = lambda g_, x_, Y_, R_, M_: conv_uvw_radial_backward(plan, g_, x_, Y_, R_, M_, rowptr, col)
    return _double_backward(fwd, bwd, _f64(g), [_f64(x), _f64(Y), _f64(R), _f64(M)],
                            [_f64(ggx), _f64(ggY), _f64(ggR), _f64(ggM)])


def tp_uvu_double_backward(plan, g, x1, x2, W, gg1, gg2, ggW):
    """(d_g, d_x1, d_x2, d_W) for the batched product."""
    fwd = lambda a_, b_, w_: tp_uvu_forward(plan, a_, b_, w_)
    bwd = lambda g_, a_, b_, w_: tp_uvu_backward(plan, g_, a_, b_, w_)
    return _double_backward(fwd, bwd, _f64(g), [_f64(x1), _f64(x2), _f64(W)],
                            [_f64(gg1), _f64(gg2), _f64(ggW)])


# ---------------------------------------------------------------------------
# convolution fed by raw edge vectors
# ---------------------------------------------------------------------------
# Figure 4B: the edge features are the spherical harmonics of the edge
# directions, Y[e] = sh_real_concat(L, rvec[e] / |rvec[e]|) with in2 = 0e+1o+...;
# the gradient with respect to rvec is the chain rule through that map.

def conv_uvu_forward_sh(plan, x, rvec, W, rowptr, col):
    lmax = len(plan.in2) - 1
    r = _f64(rvec)
    Y = sh_real_concat(lmax, r / np.linalg.norm(r, axis=1, keepdims=True))
    return conv_uvu_forward(plan, x, Y, W, rowptr, col)


def conv_uvu_backward_sh(plan, g, x, rvec, W, rowptr, col):
    """(gx, gY, grvec, gW): gY is the gradient with respect to the harmonics."""
    lmax = len(plan.in2) - 1
    r = _f64(rvec)
    Y = sh_real_concat(lmax, r / np.linalg.norm(r, axis=1, keepdims=True))
    gx, gY, gW = conv_uvu_backward(plan, g, x, Y, W, rowptr, col)
    grvec = np.einsum("ec,eck->ek", gY, sh_real_concat_jacobian(lmax, r))
    return gx, gY, grvec, gW


def radial_basis(d, K, lo, hi):
    """Gaussian radial basis of edge lengths d [E] and its derivative, both [E, K]:
    R_k = exp(-gamma (d - mu_k)^2), mu_k = lo + k step, step = (hi - lo)/(K - 1)
    (K = 1: hi - lo), gamma = 1/step^2 (Sobek, Abstract: radial projection)."""
    step = (hi - lo) / (K - 1) if K > 1 else (hi - lo)
    t = np.asarray(d, float)[:, None] - (lo + step * np.arange(K))[None, :]
    R = np.exp(-t * t / step ** 2)
    return R, -2.0 * t / step ** 2 * R


def conv_uvw_radial_forward_sh(plan, x, rvec, M, K, lo, hi, rowptr, col):
    """uvw radial convolution with Y and R evaluated from the edge vectors."""
    lmax = len(plan.in2) - 1
    r = _f64(rvec)
    d = np.linalg.norm(r, axis=1)
    Y = sh_real_concat(lmax, r / d[:, None])
    R, _ = radial_basis(d, K, lo, hi)
    return conv_uvw_radial_forward(plan, x, Y, R, M, rowptr, col)


def conv_uvw_radial_backward_sh(plan, g, x, rvec, M, K, lo, hi, rowptr, col):
    """(gx, gY, gR, grvec, gM): chain rule through the harmonics of the direction and
    the radial basis of the length."""
    lmax = len(plan.in2) - 1
    r = _f64(rvec)
    d = np.linalg.norm(r, axis=1)
    Y = sh_real_concat(lmax, r / d[:, None])
    R, dR = radial_basis(d, K, lo, hi)
    gx, gY, gR, gM = conv_uvw_radial_backward(plan, g, x, Y, R, M, rowptr, col)
    grvec = np.einsum("ec,eck->ek", gY, sh_real_concat_jacobian(lmax, r))
    grvec += ((gR * dR).sum(1) / d)[:, None] * r
    return gx, gY, gR, grvec, gM


# ---------------------------------------------------------------------------
# uvw with a weight matrix per edge (Figure 3B/C weights, no radial factorisation)
# ---------------------------------------------------------------------------

def conv_uvw_forward(plan, x, Y, W, rowptr, col):
    """out[n][i_out][w, m3] = sum_{e in row n} sum_{path -> i_out} sum_u W[e][path][u][w] t_e[u, m3]."""
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    x, Y, W = _f64(x), _f64(Y), _f64(W)
    dst = csr_dst(rowptr)
    msg = np.zeros((col.size, plan.d_out))
    x1 = x[col]
    for p in plan.paths:
        C = real_cg_block(p.l1, p.l2, p.l3)
        D3 = 2 * p.l3 + 1
        xs, ys = _blocks(p, x1, Y)
        t = np.einsum("ijk,eui,ej->euk", C, xs, ys)
        w = W[:, p.woff:p.woff + p.mul1 * p.mul_out].reshape(-1, p.mul1, p.mul_out)
        msg[:, p.ooff:p.ooff + p.mul_out * D3] += np.einsum("euw,euk->ewk", w, t).reshape(col.size, -1)
    out = np.zeros((len(rowptr) - 1, plan.d_out))
    np.add.at(out, dst, msg)              # CSR order within each receiver
    return out


def conv_uvw_backward(plan, g, x, Y, W, rowptr, col):
    """(gx [N,d1], gY [E,d2], gW [E,w_numel]) of conv_uvw_forward."""
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    g, x, Y, W = _f64(g), _f64(x), _f64(Y), _f64(W)
    dst = csr_dst(rowptr)
    x1, gd = x[col], g[dst]
    gxe = np.zeros((col.size, plan.d1))
    gY = np.zeros((col.size, plan.d2))
    gW = np.zeros_like(W)
    for p in plan.paths:
        C = real_cg_block(p.l1, p.l2, p.l3)
        D1, D2, D3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
        xs, ys = _blocks(p, x1, Y)
        t = np.einsum("ijk,eui,ej->euk", C, xs, ys)
        sl = slice(p.woff, p.woff + p.mul1 * p.mul_out)
        w = W[:, sl].reshape(-1, p.mul1, p.mul_out)
        go = gd[:, p.ooff:p.ooff + p.mul_out * D3].reshape(-1, p.mul_out, D3)
        gW[:, sl] = np.einsum("ewk,euk->euw", go, t).reshape(col.size, -1)
        gt = np.einsum("euw,ewk->euk", w, go)
        gxe[:, p.off1:p.off1 + p.mul1 * D1] += np.einsum("ijk,ej,euk->eui", C, ys, gt).reshape(col.size, -1)
        gY[:, p.off2:p.off2 + D2] += np.einsum("ijk,eui,euk->ej", C, xs, gt)
    gx = np.zeros((len(rowptr) - 1, plan.d1))
    np.add.at(gx, col, gxe)
    return gx, gY, gW


def conv_uvw_double_backward(plan, g, x, Y, W, ggx, ggY, ggW, rowptr, col):
    """(d_g, d_x, d_Y, d_W) for the uvw convolution with per-edge weights."""
    fwd = lambda x_, Y_, W_: conv_uvw_forward(plan, x_, Y_, W_, rowptr, col)
    bwd = lambda g_, x_, Y_, W_: conv_uvw_backward(plan, g_, x_, Y_, W_, rowptr, col)
    return _double_backward(fwd, bwd, _f64(g), [_f64(x), _f64(Y), _f64(W)],
                            [_f64(ggx), _f64(ggY), _f64(ggW)])


# ---------------------------------------------------------------------------
# Mixed instruction lists: a connection mode per instruction (Figure 3B/C)
# ---------------------------------------------------------------------------

def mixed_layout(irreps_in1, irreps_in2, irreps_out, instructions, modes):
    """Per-instruction offsets of the mixed convolution.

    Every instruction (i1, i2, i_out) sums into block i_out of irreps_out.  A
    "uvu" instruction keeps the channel (u -> u, so that block must have the
    multiplicity of in1 block i1) with one weight per (edge, u); a "uvw"
    instruction mixes channels with one weight per (edge, u, w).  Weights are
    two per-edge arrays, each in instruction order: Wu [E, sum_uvu mul1] and
    Ww [E, sum_uvw mul1*mul_out], each path's block of Ww laid out [u][w].
    Returns (d1, d2, d_out, wu_numel, ww_numel, rows) with rows = dicts of l1,
    l2, l3, mul1, mul_out, off1, off2, ooff, woff, mode."""
    from .irreps import parse_irreps, irreps_offsets, irreps_dim
    in1, in2, outr = parse_irreps(irreps_in1), parse_irreps(irreps_in2), parse_irreps(irreps_out)
    o1, o2, oo = irreps_offsets(in1), irreps_offsets(in2), irreps_offsets(outr)
    rows, wu, ww = [], 0, 0
    for (i1, i2, io), mode in zip(instructions, modes):
        m1, l1, p1 = in1[i1]
        _, l2, p2 = in2[i2]
        mo, l3, p3 = outr[io]
        if not (abs(l1 - l2) <= l3 <= l1 + l2) or p3 != p1 * p2:
            raise ValueError(f"forbidden path {(i1, i2, io)}")
        if mode == "uvu":
            if mo != m1:
                raise ValueError("a uvu instruction needs an output block of multiplicity mul1")
            rows.append(dict(l1=l1, l2=l2, l3=l3, mul1=m1, mul_out=m1, off1=o1[i1], off2=o2[i2],
                             ooff=oo[io], woff=wu, mode="uvu"))
            wu += m1
        elif mode == "uvw":
            rows.append(dict(l1=l1, l2=l2, l3=l3, mul1=m1, mul_out=mo, off1=o1[i1], off2=o2[i2],
                             ooff=oo[io], woff=ww, mode="uvw"))
            ww += m1 * mo
        else:
            raise ValueError(mode)
    return irreps_dim(in1), irreps_dim(in2), irreps_dim(outr), wu, ww, rows


def _mixed_t(r, xs_e, Y):
    """t_e[u, m3] = sum_{m1,m2} C[m1,m2,m3] x[src][u,m1] Y[e][m2] of one instruction."""
    C = real_cg_block(r["l1"], r["l2"], r["l3"])
    D1, D2 = 2 * r["l1"] + 1, 2 * r["l2"] + 1
    xs = xs_e[:, r["off1"]:r["off1"] + r["mul1"] * D1].reshape(-1, r["mul1"], D1)
    ys = Y[:, r["off2"]:r["off2"] + D2]
    return C, xs, ys, np.einsum("ijk,eui,ej->euk", C, xs, ys)


def conv_mixed_forward(layout, x, Y, Wu, Ww, rowptr, col):
    """out[n][i_out] = sum_{e in row n} sum_{instructions -> i_out} message, with
    uvu: msg[u, m3] = Wu[e][u] t[u, m3];  uvw: msg[w, m3] = sum_u Ww[e][u][w] t[u, m3]."""
    d1, d2, d_out, _, _, rows = layout
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    x, Y, Wu, Ww = _f64(x), _f64(Y), _f64(Wu), _f64(Ww)
    E = col.size
    msg = np.zeros((E, d_out))
    xs_e = x[col]
    for r in rows:
        D3 = 2 * r["l3"] + 1
        _, _, _, t = _mixed_t(r, xs_e, Y)
        if r["mode"] == "uvu":
            m = Wu[:, r["woff"]:r["woff"] + r["mul1"]][:, :, None] * t
        else:
            w = Ww[:, r["woff"]:r["woff"] + r["mul1"] * r["mul_out"]].reshape(-1, r["mul1"], r["mul_out"])
            m = np.einsum("euw,euk->ewk", w, t)
        msg[:, r["ooff"]:r["ooff"] + r["mul_out"] * D3] += m.reshape(E, -1)
    out = np.zeros((len(rowptr) - 1, d_out))
    np.add.at(out, csr_dst(rowptr), msg)     # CSR order within each receiver
    return out


def conv_mixed_backward(layout, g, x, Y, Wu, Ww, rowptr, col):
    """(gx [N,d1], gY [E,d2], gWu, gWw) of conv_mixed_forward, by the chain rule."""
    d1, d2, d_out, _, _, rows = layout
    rowptr = np.asarray(rowptr, dtype=np.int64)
    col = np.asarray(col, dtype=np.int64)
    g, x, Y, Wu, Ww = _f64(g), _f64(x), _f64(Y), _f64(Wu), _f64(Ww)
    E = col.size
    xs_e, gd = x[col], g[csr_dst(rowptr)]
    gxe, gY = np.zeros((E, d1)), np.zeros((E, d2))
    gWu, gWw = np.zeros_like(Wu), np.zeros_like(Ww)
    for r in rows:
        D1, D2, D3 = 2 * r["l1"] + 1, 2 * r["l2"] + 1, 2 * r["l3"] + 1
        C, xs, ys, t = _mixed_t(r, xs_e, Y)
        go = gd[:, r["ooff"]:r["ooff"] + r["mul_out"] * D3].reshape(E, r["mul_out"], D3)
        if r["mode"] == "uvu":
            sl = slice(r["woff"], r["woff"] + r["mul1"])
            gWu[:, sl] = np.einsum("euk,euk->eu", go, t)
            gt = Wu[:, sl][:, :, None] * go
        else:
            sl = slice(r["woff"], r["woff"] + r["mul1"] * r["mul_out"])
            w = Ww[:, sl].reshape(E, r["mul1"], r["mul_out"])
            gWw[:, sl] = np.einsum("ewk,euk->euw", go, t).reshape(E, -1)
            gt = np.einsum("euw,ewk->euk", w, go)
        gxe[:, r["off1"]:r["off1"] + r["mul1"] * D1] += np.einsum("ijk,ej,euk->eui", C, ys, gt).reshape(E, -1)
        gY[:, r["off2"]:r["off2"] + D2] += np.einsum("ijk,eui,euk->ej", C, xs, gt)
    gx = np.zeros((len(rowptr) - 1, d1))
    np.add.at(gx, col, gxe)
    return gx, gY, gWu, gWw


def conv_mixed_double_backward(layout, g, x, Y, Wu, Ww, ggx, ggY, ggWu, ggWw, rowptr, col):
    """(d_g, d_x, d_Y, d_Wu, d_Ww).  The message is linear in x, in Y and in the
    weights W = (Wu, Ww) taken together (each term holds one of them), so the
    multilinearity identity runs over the three operands x, Y, W, the two weight
    arrays being substituted together."""
    g, x, Y, Wu, Ww = _f64(g), _f64(x), _f64(Y), _f64(Wu), _f64(Ww)
    ggx, ggY, ggWu, ggWw = _f64(ggx), _f64(ggY), _f64(ggWu), _f64(ggWw)
    F = lambda *a: conv_mixed_forward(layout, *a, rowptr, col)
    B = lambda *a: conv_mixed_backward(layout, g, *a, rowptr, col)
    d_g = F(ggx, Y, Wu, Ww) + F(x, ggY, Wu, Ww) + F(x, Y, ggWu, ggWw)
    bx, by, bw = B(ggx, Y, Wu, Ww), B(x, ggY, Wu, Ww), B(x, Y, ggWu, ggWw)
    d_x = by[0] + bw[0]
    d_Y = bx[1] + bw[1]
    d_Wu = bx[2] + by[2]
    d_Ww = bx[3] + by[3]
    return d_g, d_x, d_Y, d_Wu, d_Ww
