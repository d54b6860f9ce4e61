"""Pins of the oracle's tensor product and convolution (CPU only).

* brute force: one dense [d1, d2, d_out] tensor per edge built entry by entry;
* closed forms for l <= 1 (products, dot, cross);
* equivariance of out (and of the gradients) under rotations and inversion;
* finite differences of the gradients;
* homogeneity: out is linear in each of x, Y, W (R, M), so
  <g, out> = <gx, x> = <gY, Y> = <gW, W>;
* the sender transpose against a plain loop.
"""

import numpy as np
import pytest

from oracle import cg, conv, graph, irreps
from clebsch_gordan_tensor_racah_gb300 import workloads as wl


def small_graph(rng, N, E):
    src = rng.integers(0, N, size=E)
    dst = rng.integers(0, N, size=E)
    order = np.argsort(dst, kind="stable")
    rowptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))])
    return rowptr, src[order]


UVU_CASES = [
    ("2x0e+2x1o", "0e+1o", "0e+1o+1e"),
    ("1x0e+2x1o+1x2e", "0e+1o+2e", "0e+0o+1e+1o+2e+2o"),
    ("2x1e+1x3o", "0e+1o+2e+3o", "1o+2e+3o+0e+1e"),
]


@pytest.mark.parametrize("case", UVU_CASES)
def test_uvu_conv_brute_force(case):
    rng = np.random.default_rng(1)
    plan = irreps.make_plan(*case, mode="uvu")
    N, E = 5, 12
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    Y = rng.normal(size=(E, plan.d2))
    W = rng.normal(size=(E, plan.w_numel))
    g = rng.normal(size=(N, plan.d_out))
    dst = graph.csr_dst(rowptr)
    out_ref = np.zeros((N, plan.d_out))
    gx_ref = np.zeros((N, plan.d1))
    gY_ref = np.zeros((E, plan.d2))
    gW_ref = np.zeros((E, plan.w_numel))
    for e in range(E):
        T = conv.dense_tensor(plan, W[e])
        out_ref[dst[e]] += np.einsum("ijk,i,j->k", T, x[col[e]], Y[e])
        gx_ref[col[e]] += np.einsum("ijk,j,k->i", T, Y[e], g[dst[e]])
        gY_ref[e] = np.einsum("ijk,i,k->j", T, x[col[e]], g[dst[e]])
        # dT/dW is T built from unit weight vectors
        for j in range(plan.w_numel):
            unit = np.zeros(plan.w_numel)
            unit[j] = 1.0
            Tj = conv.dense_tensor(plan, unit)
            gW_ref[e, j] = np.einsum("ijk,i,j,k->", Tj, x[col[e]], Y[e], g[dst[e]])
    out = conv.conv_uvu_forward(plan, x, Y, W, rowptr, col)
    assert np.abs(out - out_ref).max() < 1e-12
    gx, gY, gW = conv.conv_uvu_backward(plan, g, x, Y, W, rowptr, col)
    assert np.abs(gx - gx_ref).max() < 1e-12
    assert np.abs(gY - gY_ref).max() < 1e-12
    assert np.abs(gW - gW_ref).max() < 1e-12


def test_uvw_conv_brute_force():
    rng = np.random.default_rng(2)
    plan = irreps.make_plan("2x0e+2x1o", "0e+1o", "3x0e+2x1o+1x1e", mode="uvw")
    N, E, K = 4, 10, 3
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    Y = rng.normal(size=(E, plan.d2))
    R = rng.normal(size=(E, K))
    M = rng.normal(size=(K, plan.w_numel))
    g = rng.normal(size=(N, plan.d_out))
    dst = graph.csr_dst(rowptr)
    out_ref = np.zeros((N, plan.d_out))
    gx_ref = np.zeros((N, plan.d1))
    gY_ref = np.zeros((E, plan.d2))
    gR_ref = np.zeros((E, K))
    gM_ref = np.zeros_like(M)
    Tk = [conv.dense_tensor(plan, M[k]) for k in range(K)]
    for e in range(E):
        T = sum(R[e, k] * Tk[k] for k in range(K))
        out_ref[dst[e]] += np.einsum("ijk,i,j->k", T, x[col[e]], Y[e])
        gx_ref[col[e]] += np.einsum("ijk,j,k->i", T, Y[e], g[dst[e]])
        gY_ref[e] = np.einsum("ijk,i,k->j", T, x[col[e]], g[dst[e]])
        for k in range(K):
            gR_ref[e, k] = np.einsum("ijk,i,j,k->", Tk[k], x[col[e]], Y[e], g[dst[e]])
    for k in range(K):
        for j in range(plan.w_numel):
            unit = np.zeros(plan.w_numel)
            unit[j] = 1.0
            Tj = conv.dense_tensor(plan, unit)
            gM_ref[k, j] = sum(R[e, k] * np.einsum("ijk,i,j,k->", Tj, x[col[e]], Y[e], g[dst[e]])
                               for e in range(E))
    out = conv.conv_uvw_radial_forward(plan, x, Y, R, M, rowptr, col)
    assert np.abs(out - out_ref).max() < 1e-12
    gx, gY, gR, gM = conv.conv_uvw_radial_backward(plan, g, x, Y, R, M, rowptr, col, block=3)
    for a, b in ((gx, gx_ref), (gY, gY_ref), (gR, gR_ref), (gM, gM_ref)):
        assert np.abs(a - b).max() < 1e-11


def test_uvu_closed_forms_l_le_1():
    """Config-1 path list with one channel: products, dot/sqrt3 and cross/sqrt2."""
    plan = irreps.make_plan("1x0e+1x1o", "0e+1o", "0e+1o+1e", mode="uvu")
    rng = np.random.default_rng(4)
    a, v = rng.normal(), rng.normal(size=3)       # in1: scalar a, vector v (cartesian)
    s, w = rng.normal(), rng.normal(size=3)       # in2: scalar s, vector w
    perm = [1, 2, 0]                              # l = 1 components are (y, z, x)
    x1 = np.concatenate([[a], v[perm]])[None]
    x2 = np.concatenate([[s], w[perm]])[None]
    z = conv.tp_uvu_forward(plan, x1, x2, np.ones((1, 5)))[0]
    expect = np.concatenate([[a * s], (a * w)[perm], (v * s)[perm], [v @ w / np.sqrt(3)],
                             (np.cross(v, w) / np.sqrt(2))[perm]])
    assert np.abs(z - expect).max() < 1e-14


def _rot_features(irr, x, D_of_l, parity_flip):
    out = np.empty_like(x)
    o = 0
    for mul, l, p in irr:
        D = D_of_l(l) * (p if parity_flip else 1)
        d = 2 * l + 1
        blk = x[:, o:o + mul * d].reshape(x.shape[0], mul, d)
        out[:, o:o + mul * d] = np.einsum("ab,nub->nua", D, blk).reshape(x.shape[0], -1)
        o += mul * d
    return out


@pytest.mark.parametrize("invert", [False, True])
@pytest.mark.parametrize("mode", ["uvu", "uvw"])
def test_conv_equivariance(mode, invert):
    rng = np.random.default_rng(7 + invert)
    if mode == "uvu":
        plan = irreps.make_plan("2x0e+2x1o+2x2e+1x3o", "0e+1o+2e+3o", wl._all_out(3), mode="uvu")
    else:
        plan = irreps.make_plan("2x0e+2x1o+2x2e", "0e+1o+2e", "2x0e+2x1o+2x2e", mode="uvw")
    N, E, K = 6, 20, 4
    rowptr, col = small_graph(rng, N, E)
    lmax = max(l for _, l, _ in plan.in2)
    vec = wl.unit_vectors(rng, E)
    x = rng.normal(size=(N, plan.d1))
    axis, ang = rng.normal(size=3), rng.uniform(0, 2 * np.pi)
    Rm = cg.rotation_matrix(axis, ang) * (-1 if invert else 1)
    D = lambda l: cg.wigner_d_real(l, axis, ang)
    Y = cg.sh_real_concat(lmax, vec)
    Yr = cg.sh_real_concat(lmax, vec @ Rm.T)      # SH of the rotated (inverted) directions
    xr = _rot_features(plan.in1, x, D, invert)
    if mode == "uvu":
        W = rng.normal(size=(E, plan.w_numel))
        out = conv.conv_uvu_forward(plan, x, Y, W, rowptr, col)
        out_r = conv.conv_uvu_forward(plan, xr, Yr, W, rowptr, col)
        g = rng.normal(size=out.shape)
        gx, gY, gW = conv.conv_uvu_backward(plan, g, x, Y, W, rowptr, col)
        gr = _rot_features(plan.out, g, D, invert)
        gx_r, gY_r, gW_r = conv.conv_uvu_backward(plan, gr, xr, Yr, W, rowptr, col)
        assert np.abs(gW_r - gW).max() < 1e-10               # invariant
    else:
        R = rng.uniform(size=(E, K))
        M = rng.normal(size=(K, plan.w_numel))
        out = conv.conv_uvw_radial_forward(plan, x, Y, R, M, rowptr, col)
        out_r = conv.conv_uvw_radial_forward(plan, xr, Yr, R, M, rowptr, col)
        g = rng.normal(size=out.shape)
        gx, gY, gR, gM = conv.conv_uvw_radial_backward(plan, g, x, Y, R, M, rowptr, col)
        gr = _rot_features(plan.out, g, D, invert)
        gx_r, gY_r, gR_r, gM_r = conv.conv_uvw_radial_backward(plan, gr, xr, Yr, R, M, rowptr, col)
        assert np.abs(gR_r - gR).max() < 1e-10
        assert np.abs(gM_r - gM).max() < 1e-10
    assert np.abs(out_r - _rot_features(plan.out, out, D, invert)).max() < 1e-10
    assert np.abs(gx_r - _rot_features(plan.in1, gx, D, invert)).max() < 1e-10
    assert np.abs(gY_r - _rot_features(plan.in2, gY, D, invert)).max() < 1e-10


@pytest.mark.parametrize("mode", ["uvu", "uvw"])
def test_finite_differences(mode):
    rng = np.random.default_rng(11)
    if mode == "uvu":
        plan = irreps.make_plan("2x0e+1x1o+1x2e", "0e+1o+2e", wl._all_out(2), mode="uvu")
    else:
        plan = irreps.make_plan("2x0e+1x1o+1x2e", "0e+1o+2e", "1x0e+2x1o+1x2e", mode="uvw")
    N, E, K = 4, 9, 3
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    Y = rng.normal(size=(E, plan.d2))
    g = rng.normal(size=(N, plan.d_out))
    h = 1e-6
    if mode == "uvu":
        W = rng.normal(size=(E, plan.w_numel))
        f = lambda x_, Y_, W_: (g * conv.conv_uvu_forward(plan, x_, Y_, W_, rowptr, col)).sum()
        grads = conv.conv_uvu_backward(plan, g, x, Y, W, rowptr, col)
        args = [x, Y, W]
    else:
        R = rng.normal(size=(E, K))
        M = rng.normal(size=(K, plan.w_numel))
        f = lambda x_, Y_, R_, M_: (g * conv.conv_uvw_radial_forward(plan, x_, Y_, R_, M_, rowptr, col)).sum()
        grads = conv.conv_uvw_radial_backward(plan, g, x, Y, R, M, rowptr, col)
        args = [x, Y, R, M]
    for ai, (a, ga) in enumerate(zip(args, grads)):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in a.shape)
            ap, am = [b.copy() for b in args], [b.copy() for b in args]
            ap[ai][idx] += h
            am[ai][idx] -= h
            fd = (f(*ap) - f(*am)) / (2 * h)
            assert abs(fd - ga[idx]) < 1e-7 * max(1.0, abs(fd)), (ai, idx, fd, ga[idx])


def test_homogeneity_invariants():
    rng = np.random.default_rng(13)
    plan = irreps.make_plan("3x0e+3x1o+3x2e", "0e+1o+2e+3o", wl._all_out(3), mode="uvu")
    N, E = 8, 40
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    Y = rng.normal(size=(E, plan.d2))
    W = rng.normal(size=(E, plan.w_numel))
    out = conv.conv_uvu_forward(plan, x, Y, W, rowptr, col)
    g = rng.normal(size=out.shape)
    gx, gY, gW = conv.conv_uvu_backward(plan, g, x, Y, W, rowptr, col)
    ref = (g * out).sum()
    for a, ga in ((x, gx), (Y, gY), (W, gW)):
        assert abs((a * ga).sum() - ref) < 1e-10 * max(1, abs(ref))


def test_batched_equals_identity_graph_conv():
    rng = np.random.default_rng(17)
    plan = irreps.make_plan("2x0e+2x1o+1x2e", "0e+1o+2e", wl._all_out(2), mode="uvu")
    B = 7
    x1, x2 = rng.normal(size=(B, plan.d1)), rng.normal(size=(B, plan.d2))
    W = rng.normal(size=(B, plan.w_numel))
    rowptr, col = np.arange(B + 1), np.arange(B)
    assert np.abs(conv.tp_uvu_forward(plan, x1, x2, W)
                  - conv.conv_uvu_forward(plan, x1, x2, W, rowptr, col)).max() == 0.0


def test_transpose_against_loop():
    rng = np.random.default_rng(19)
    N, E = 30, 200
    rowptr, col = small_graph(rng, N, E)
    t_rowptr, t_eid, t_dst = graph.transpose(rowptr, col, N)
    dst = graph.csr_dst(rowptr)
    lists = [[] for _ in range(N)]
    for p in range(E):
        lists[col[p]].append(p)
    flat = [p for lst in lists for p in lst]
    assert list(t_eid) == flat
    assert list(t_rowptr) == list(np.cumsum([0] + [len(lst) for lst in lists]))
    assert list(t_dst) == [dst[p] for p in flat]
    assert graph.check_csr(rowptr, col, N)
    bad = rowptr.copy()
    bad[3], bad[4] = bad[4] + 1, bad[3]
    assert not graph.check_csr(bad, col, N)
    assert not graph.check_csr(rowptr, np.where(col == 0, N, col), N)


def test_workload_recipes_shapes():
    tiny = wl.make("tiny", 40)
    assert tiny["E"] == 512 and tiny["x"].shape == (64, 32) and tiny["Y"].shape == (512, 4)
    assert np.all(np.diff(tiny["rowptr"]) >= 0) and tiny["rowptr"][-1] == 512
    m = wl.make("mace", 2304, N=50)
    assert m["rowptr"][-1] == m["E"] and m["W"].shape == (m["E"], 2304)
    u = wl.make("uvw", 45056, N=10)
    assert u["R"].shape == (320, 8) and u["M"].shape == (8, 45056)
    assert np.all(u["R"] > 0) and np.all(u["R"] <= 1)


def test_uvw_gM_entries_match_full_backward():
    rng = np.random.default_rng(23)
    plan = irreps.make_plan("2x0e+2x1o+1x2e", "0e+1o+2e", "2x0e+1x1o+2x2e", mode="uvw")
    N, E, K = 5, 14, 3
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    Y = rng.normal(size=(E, plan.d2))
    R = rng.normal(size=(E, K))
    M = rng.normal(size=(K, plan.w_numel))
    g = rng.normal(size=(N, plan.d_out))
    _, _, _, gM = conv.conv_uvw_radial_backward(plan, g, x, Y, R, M, rowptr, col)
    entries = [(k, pi, u, w) for k in range(K) for pi, p in enumerate(plan.paths)
               for u in range(p.mul1) for w in range(p.mul_out)]
    vals = conv.conv_uvw_radial_gM_entries(plan, g, x, Y, R, rowptr, col, entries)
    for (k, pi, u, w), v in zip(entries, vals):
        p = plan.paths[pi]
        assert abs(gM[k, p.woff + u * p.mul_out + w] - v) < 1e-11


def test_uvw_gM_slice_matches_entries():
    # the chunked slice (matrix products over edge chunks) against the per-entry definition,
    # with a chunk smaller than E so several chunks and a ragged last one are summed
    rng = np.random.default_rng(29)
    plan = irreps.make_plan("3x0e+2x1o+2x2e", "0e+1o+2e", "2x0e+3x1o+2x2e", mode="uvw")
    N, E, K = 6, 23, 3
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    Y = rng.normal(size=(E, plan.d2))
    R = rng.normal(size=(E, K))
    g = rng.normal(size=(N, plan.d_out))
    for k in range(K):
        for pi, p in enumerate(plan.paths):
            sl = conv.conv_uvw_radial_gM_slice(plan, g, x, Y, R, rowptr, col, k, pi, chunk=5)
            ent = [(k, pi, u, w) for u in range(p.mul1) for w in range(p.mul_out)]
            ref = conv.conv_uvw_radial_gM_entries(plan, g, x, Y, R, rowptr, col, ent)
            assert np.abs(sl.reshape(-1) - ref).max() < 1e-12


@pytest.mark.parametrize("mode", ["uvu", "uvw", "batched"])
def test_double_backward_exact_directional_differences(mode):
    # S = sum_j <c_j, dL/da_j> is linear in g and in each operand separately, so
    # S(v + d) - S(v) = <dS/dv, d> holds exactly (up to rounding) for any
    # direction d; S itself is evaluated with the backward alone.
    rng = np.random.default_rng(23)
    N, E, K = 5, 11, 3
    if mode == "uvw":
        plan = irreps.make_plan("2x0e+1x1o+1x2e", "0e+1o+2e", "1x0e+2x1o+1x2e", mode="uvw")
    else:
        plan = irreps.make_plan("2x0e+1x1o+2x2e", "0e+1o+2e", wl._all_out(2), mode="uvu")
    if mode == "batched":
        B = 6
        shapes = [(B, plan.d1), (B, plan.d2), (B, plan.w_numel)]
        g = rng.normal(size=(B, plan.d_out))

        def bwd(g_, *a):
            return conv.tp_uvu_backward(plan, g_, *a)

        def dbl(g_, a, c):
            return conv.tp_uvu_double_backward(plan, g_, *a, *c)
    else:
        rowptr, col = small_graph(rng, N, E)
        g = rng.normal(size=(N, plan.d_out))
        if mode == "uvu":
            shapes = [(N, plan.d1), (E, plan.d2), (E, plan.w_numel)]

            def bwd(g_, *a):
                return conv.conv_uvu_backward(plan, g_, *a, rowptr, col)

            def dbl(g_, a, c):
                return conv.conv_uvu_double_backward(plan, g_, *a, *c, rowptr, col)
        else:
            shapes = [(N, plan.d1), (E, plan.d2), (E, K), (K, plan.w_numel)]

            def bwd(g_, *a):
                return conv.conv_uvw_radial_backward(plan, g_, *a, rowptr, col)

            def dbl(g_, a, c):
                return conv.conv_uvw_radial_double_backward(plan, g_, *a, *c, rowptr, col)
    a = [rng.normal(size=s) for s in shapes]
    c = [rng.normal(size=s) for s in shapes]

    def S(g_, a_):
        return sum((cj * bj).sum() for cj, bj in zip(c, bwd(g_, *a_)))

    d = dbl(g, a, c)
    assert d[0].shape == g.shape and all(dj.shape == aj.shape for dj, aj in zip(d[1:], a))
    base = S(g, a)
    for trial in range(3):
        dg = rng.normal(size=g.shape)
        lhs = S(g + dg, a) - base
        assert abs(lhs - (d[0] * dg).sum()) <= 1e-10 * (abs(lhs) + abs(base) + 1.0)
        for j in range(len(a)):
            dj = rng.normal(size=a[j].shape)
            aj = list(a)
            aj[j] = a[j] + dj
            lhs = S(g, aj) - base
            assert abs(lhs - (d[1 + j] * dj).sum()) <= 1e-10 * (abs(lhs) + abs(base) + 1.0), (mode, j)


def test_edge_vector_conv_gradient_finite_differences():
    # grvec of the edge-vector convolution against central differences of <g, out>
    rng = np.random.default_rng(37)
    plan = irreps.make_plan("2x0e+1x1o+1x2e", "0e+1o+2e", wl._all_out(2), mode="uvu")
    N, E = 4, 9
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    r = rng.normal(size=(E, 3)) * rng.uniform(0.5, 2.0, size=(E, 1))
    W = rng.normal(size=(E, plan.w_numel))
    g = rng.normal(size=(N, plan.d_out))
    f = lambda rr: (g * conv.conv_uvu_forward_sh(plan, x, rr, W, rowptr, col)).sum()  # noqa: E731
    _, _, grvec, _ = conv.conv_uvu_backward_sh(plan, g, x, r, W, rowptr, col)
    h = 1e-6
    for e in range(E):
        for k in range(3):
            rp, rm = r.copy(), r.copy()
            rp[e, k] += h
            rm[e, k] -= h
            fd = (f(rp) - f(rm)) / (2 * h)
            assert abs(fd - grvec[e, k]) < 1e-7 * max(1.0, abs(fd)), (e, k, fd, grvec[e, k])


def test_radial_edge_vector_conv_gradient_finite_differences():
    # uvw: grvec through both the harmonics of the direction and the radial basis of the length
    rng = np.random.default_rng(43)
    plan = irreps.make_plan("2x0e+1x1o+1x2e", "0e+1o+2e", "1x0e+2x1o+1x2e", mode="uvw")
    N, E, K, lo, hi = 4, 8, 3, 0.5, 5.0
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    r = rng.normal(size=(E, 3)) * rng.uniform(0.7, 3.0, size=(E, 1))
    M = rng.normal(size=(K, plan.w_numel))
    g = rng.normal(size=(N, plan.d_out))
    f = lambda rr: (g * conv.conv_uvw_radial_forward_sh(plan, x, rr, M, K, lo, hi, rowptr, col)).sum()  # noqa: E731
    grvec = conv.conv_uvw_radial_backward_sh(plan, g, x, r, M, K, lo, hi, rowptr, col)[3]
    h = 1e-6
    for e in range(E):
        for k in range(3):
            rp, rm = r.copy(), r.copy()
            rp[e, k] += h
            rm[e, k] -= h
            fd = (f(rp) - f(rm)) / (2 * h)
            assert abs(fd - grvec[e, k]) < 1e-7 * max(1.0, abs(fd)), (e, k, fd, grvec[e, k])


def test_uvw_per_edge_weights_brute_force_fd_and_radial_identity():
    rng = np.random.default_rng(47)
    plan = irreps.make_plan("2x0e+1x1o+1x2e", "0e+1o+2e", "1x0e+2x1o+1x2e", mode="uvw")
    N, E, K = 4, 9, 3
    rowptr, col = small_graph(rng, N, E)
    x = rng.normal(size=(N, plan.d1))
    Y = rng.normal(size=(E, plan.d2))
    W = rng.normal(size=(E, plan.w_numel))
    out = conv.conv_uvw_forward(plan, x, Y, W, rowptr, col)
    # brute force: one dense bilinear tensor per edge, summed into the receiver
    ref = np.zeros_like(out)
    dst = graph.csr_dst(rowptr)
    for e in range(E):
        ref[dst[e]] += np.einsum("ijk,i,j->k", conv.dense_tensor(plan, W[e]), x[col[e]], Y[e])
    assert np.abs(out - ref).max() < 1e-12
    # the radial convolution is the per-edge one at W = R M
    R = rng.normal(size=(E, K))
    M = rng.normal(size=(K, plan.w_numel))
    a = conv.conv_uvw_forward(plan, x, Y, R @ M, rowptr, col)
    b = conv.conv_uvw_radial_forward(plan, x, Y, R, M, rowptr, col)
    assert np.abs(a - b).max() < 1e-12 * max(1.0, np.abs(b).max())
    # gradients against central differences
    g = rng.normal(size=(N, plan.d_out))
    grads = conv.conv_uvw_backward(plan, g, x, Y, W, rowptr, col)
    f = lambda x_, Y_, W_: (g * conv.conv_uvw_forward(plan, x_, Y_, W_, rowptr, col)).sum()  # noqa: E731
    args, h = [x, Y, W], 1e-6
    for ai, (arr, ga) in enumerate(zip(args, grads)):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            ap, am = [b_.copy() for b_ in args], [b_.copy() for b_ in args]
            ap[ai][idx] += h
            am[ai][idx] -= h
            fd = (f(*ap) - f(*am)) / (2 * h)
            assert abs(fd - ga[idx]) < 1e-7 * max(1.0, abs(fd)), (ai, idx, fd, ga[idx])


def test_uvu_double_backward_against_autograd_hessian_vector_product():
    # A second, independent route to the second derivatives: the convolution
    # written as plain PyTorch CPU ops (per-path einsum with the oracle's CG
    # blocks, index_add over receivers), L = <g, out>, its gradients with
    # create_graph, S = sum_j <c_j, dL/da_j>, and autograd's dS/d(g, x, Y, W)
    # (a Hessian-vector product), against the oracle's identity-based result.
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    plan = irreps.make_plan("2x0e+1x1o+2x2e", "0e+1o+2e", wl._all_out(2), mode="uvu")
    N, E = 5, 12
    rowptr, col = small_graph(rng, N, E)
    dst = np.repeat(np.arange(N), np.diff(rowptr))
    x, Y, W = rng.normal(size=(N, plan.d1)), rng.normal(size=(E, plan.d2)), rng.normal(size=(E, plan.w_numel))
    g = rng.normal(size=(N, plan.d_out))
    cx, cY, cW = rng.normal(size=x.shape), rng.normal(size=Y.shape), rng.normal(size=W.shape)
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    xt, Yt, Wt, gt = t(x), t(Y), t(W), t(g)
    src_i, dst_i = torch.tensor(col, dtype=torch.long), torch.tensor(dst, dtype=torch.long)
    out = torch.zeros(N, plan.d_out, dtype=torch.float64)
    for p in plan.paths:
        C = torch.tensor(cg.real_cg_block(p.l1, p.l2, p.l3))
        D1, D2, D3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
        xs = xt[src_i, p.off1:p.off1 + p.mul1 * D1].reshape(E, p.mul1, D1)
        ys = Yt[:, p.off2:p.off2 + D2]
        msg = torch.einsum("ijk,eui,ej->euk", C, xs, ys) * Wt[:, p.woff:p.woff + p.mul1, None]
        pad = torch.zeros(N, plan.d_out, dtype=torch.float64)
        pad = pad.index_add(0, dst_i, torch.nn.functional.pad(msg.reshape(E, -1),
                                                             (p.ooff, plan.d_out - p.ooff - p.mul1 * D3)))
        out = out + pad
    L = (gt * out).sum()
    gx, gY, gW = torch.autograd.grad(L, (xt, Yt, Wt), create_graph=True)
    S = (gx * torch.tensor(cx)).sum() + (gY * torch.tensor(cY)).sum() + (gW * torch.tensor(cW)).sum()
    d_g, d_x, d_Y, d_W = torch.autograd.grad(S, (gt, xt, Yt, Wt), allow_unused=True)
    ref = conv.conv_uvu_double_backward(plan, g, x, Y, W, cx, cY, cW, rowptr, col)
    for name, got, r in (("d_gout", d_g, ref[0]), ("d_x", d_x, ref[1]), ("d_Y", d_Y, ref[2]), ("d_W", d_W, ref[3])):
        got = np.zeros_like(r) if got is None else got.detach().numpy()
        assert np.abs(got - r).max() <= 1e-11 * max(1.0, np.abs(r).max()), name
