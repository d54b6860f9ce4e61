"""Pins of the oracle's convolution with mixed uvu/uvw instruction lists (CPU only).

* brute force: scalar loops over edges, instructions, channels and components;
* an all-uvw list is the per-edge uvw convolution, an all-uvu list whose
  instructions own distinct output blocks is the uvu convolution (each pinned on
  its own in test_oracle_conv.py);
* the message is linear in each of x, Y, Wu, Ww, so directional differences of
  <g, out> give the gradients exactly (up to rounding), and directional
  differences of S = sum_j <c_j, dL/da_j> give the second derivatives.
"""

import numpy as np
import pytest

from oracle import cg, conv, graph, irreps

IN1, IN2, OUT = "2x0e+2x1o", "0e+1o", "2x0e+2x1o+3x1e"
INSTR = [(0, 0, 0), (1, 1, 0), (0, 1, 1), (1, 0, 1), (1, 1, 2)]
MODES = ["uvu", "uvw", "uvu", "uvw", "uvw"]


def small_graph(rng, N, E):
    src = rng.integers(0, N, size=E)
    dst = rng.integers(0, N, size=E)
    order = np.argsort(dst, kind="stable")
    rowptr = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))])
    return rowptr, src[order]


def operands(rng, layout, N, E):
    d1, d2, d_out, wu, ww, _ = layout
    return [rng.normal(size=(N, d1)), rng.normal(size=(E, d2)), rng.normal(size=(E, wu)),
            rng.normal(size=(E, ww))]


def brute_force(x, Y, Wu, Ww, rowptr, col):
    in1, in2, outr = irreps.parse_irreps(IN1), irreps.parse_irreps(IN2), irreps.parse_irreps(OUT)
    o1, o2, oo = irreps.irreps_offsets(in1), irreps.irreps_offsets(in2), irreps.irreps_offsets(outr)
    N = len(rowptr) - 1
    out = np.zeros((N, irreps.irreps_dim(outr)))
    wu = ww = 0
    for (i1, i2, io), mode in zip(INSTR, MODES):
        m1, l1, _ = in1[i1]
        _, l2, _ = in2[i2]
        mo, l3, _ = outr[io]
        C = cg.real_cg_block(l1, l2, l3)
        for n in range(N):
            for e in range(rowptr[n], rowptr[n + 1]):
                s = col[e]
                for u in range(m1):
                    for w in range(mo):
                        if mode == "uvu":
                            if w != u:
                                continue
                            coef = Wu[e, wu + u]
                        else:
                            coef = Ww[e, ww + u * mo + w]
                        for a in range(2 * l1 + 1):
                            for b in range(2 * l2 + 1):
                                for c in range(2 * l3 + 1):
                                    out[n, oo[io] + w * (2 * l3 + 1) + c] += (
                                        coef * C[a, b, c] * x[s, o1[i1] + u * (2 * l1 + 1) + a]
                                        * Y[e, o2[i2] + b])
        if mode == "uvu":
            wu += m1
        else:
            ww += m1 * mo
    return out


def test_mixed_forward_brute_force():
    rng = np.random.default_rng(3)
    lay = conv.mixed_layout(IN1, IN2, OUT, INSTR, MODES)
    assert lay[3] == 2 + 2 and lay[4] == 2 * 2 + 2 * 2 + 2 * 3
    rowptr, col = small_graph(rng, 4, 9)
    x, Y, Wu, Ww = operands(rng, lay, 4, 9)
    got = conv.conv_mixed_forward(lay, x, Y, Wu, Ww, rowptr, col)
    ref = brute_force(x, Y, Wu, Ww, rowptr, col)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_mixed_reduces_to_single_modes():
    rng = np.random.default_rng(4)
    rowptr, col = small_graph(rng, 5, 12)
    # all uvw: the per-edge uvw convolution
    ins = [(0, 0, 0), (1, 1, 0), (0, 1, 1), (1, 0, 1), (1, 1, 2)]
    lay = conv.mixed_layout(IN1, IN2, OUT, ins, ["uvw"] * len(ins))
    plan = irreps.make_plan(IN1, IN2, OUT, "uvw", instructions=ins)
    x, Y, Wu, Ww = operands(rng, lay, 5, 12)
    np.testing.assert_allclose(conv.conv_mixed_forward(lay, x, Y, Wu, Ww, rowptr, col),
                               conv.conv_uvw_forward(plan, x, Y, Ww, rowptr, col), rtol=1e-12, atol=1e-12)
    g = rng.normal(size=(5, lay[2]))
    gm = conv.conv_mixed_backward(lay, g, x, Y, Wu, Ww, rowptr, col)
    gr = conv.conv_uvw_backward(plan, g, x, Y, Ww, rowptr, col)
    for a, b in zip((gm[0], gm[1], gm[3]), gr):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    # all uvu, each instruction owning its own output block in the uvu order
    out_u = "2x0e+2x1o+2x0e+2x1o"
    ins = [(0, 0, 0), (0, 1, 1), (1, 0, 3), (1, 1, 2)]
    lay = conv.mixed_layout(IN1, IN2, out_u, ins, ["uvu"] * len(ins))
    plan = irreps.make_plan(IN1, IN2, out_u, "uvu", instructions=ins)
    x, Y, Wu, Ww = operands(rng, lay, 5, 12)
    ref = conv.conv_uvu_forward(plan, x, Y, Wu, rowptr, col)
    got = conv.conv_mixed_forward(lay, x, Y, Wu, Ww, rowptr, col)
    # the uvu plan appends blocks in instruction order; map them onto irreps_out
    for p, r in zip(plan.paths, lay[5]):
        n = p.mul1 * (2 * p.l3 + 1)
        np.testing.assert_allclose(got[:, r["ooff"]:r["ooff"] + n], ref[:, p.ooff:p.ooff + n],
                                   rtol=1e-12, atol=1e-12)


def test_mixed_layout_rejects_uvu_multiplicity_change():
    with pytest.raises(ValueError):
        conv.mixed_layout(IN1, IN2, "3x0e", [(0, 0, 0)], ["uvu"])
    with pytest.raises(ValueError):
        conv.mixed_layout(IN1, IN2, OUT, [(1, 1, 1)], ["uvw"])       # 1o x 1o -> 1o: parity


def test_mixed_backward_exact_directional_differences():
    rng = np.random.default_rng(5)
    lay = conv.mixed_layout(IN1, IN2, OUT, INSTR, MODES)
    N, E = 5, 13
    rowptr, col = small_graph(rng, N, E)
    a = operands(rng, lay, N, E)
    g = rng.normal(size=(N, lay[2]))
    grads = conv.conv_mixed_backward(lay, g, *a, rowptr, col)

    def L(ops):
        return float(np.sum(g * conv.conv_mixed_forward(lay, *ops, rowptr, col)))

    for j in range(4):
        d = rng.normal(size=a[j].shape)
        b = list(a)
        b[j] = a[j] + d
        lhs = L(b) - L(a)
        rhs = float(np.sum(grads[j] * d))
        assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs)), (j, lhs, rhs)


def test_mixed_double_backward_exact_directional_differences():
    rng = np.random.default_rng(6)
    lay = conv.mixed_layout(IN1, IN2, OUT, INSTR, MODES)
    N, E = 4, 10
    rowptr, col = small_graph(rng, N, E)
    a = operands(rng, lay, N, E)
    c = operands(rng, lay, N, E)
    g = rng.normal(size=(N, lay[2]))
    d = conv.conv_mixed_double_backward(lay, g, *a, *c, rowptr, col)

    def S(g_, ops):
        gr = conv.conv_mixed_backward(lay, g_, *ops, rowptr, col)
        return float(sum(np.sum(ci * gi) for ci, gi in zip(c, gr)))

    dg = rng.normal(size=g.shape)
    assert abs((S(g + dg, a) - S(g, a)) - np.sum(d[0] * dg)) <= 1e-10 * max(1.0, abs(np.sum(d[0] * dg)))
    for j in range(4):
        dj = rng.normal(size=a[j].shape)
        b = list(a)
        b[j] = a[j] + dj
        lhs = S(g, b) - S(g, a)
        rhs = float(np.sum(d[j + 1] * dj))
        assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs)), (j, lhs, rhs)


def test_mixed_bench_workload_lists_every_allowed_instruction():
    from clebsch_gordan_tensor_racah_gb300 import workloads as wl
    spec = wl.SPECS["mixed"]
    full = irreps.make_plan(spec["in1"], spec["in2"], spec["out"], "uvw")
    assert sorted(spec["instructions"]) == sorted((p.i1, p.i2, p.i_out) for p in full.paths)
    lay = conv.mixed_layout(spec["in1"], spec["in2"], spec["out"], spec["instructions"], spec["modes"])
    # uvw exactly for the instructions into the scalar block
    assert all((m == "uvw") == (r["l3"] == 0) for m, r in zip(spec["modes"], lay[5]))
    assert lay[4] == 3 * 32 * 32 and lay[3] == 8 * 32
