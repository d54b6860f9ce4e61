"""Irreps strings, path enumeration and feature layouts (oracle side).

Test infrastructure only (see the package docstring).

An irreps string is a '+'-separated list of ``MULxLP`` terms (``MULx`` may be
omitted for multiplicity 1), P in {e, o} for parity +1 / -1.  A feature vector
is the concatenation of its blocks; inside block i the element (u, m) sits at
``offset_i + u*(2l+1) + (m + l)`` (multiplicity-major).

Paths ("instructions") couple in1 block i1 with in2 block i2 into an output
irrep (l3, p3) with |l1-l2| <= l3 <= l1+l2 and p3 = p1*p2 (the selection rule of
the CG tensor product, "An Efficient Sparse Kernel Generator for
O(3)-Equivariant Deep Networks", Figure 1).  Without an explicit list every
allowed (i1, i2, l3) is taken, i1 outer, i2 next, l3 ascending, keeping those
whose (l3, p3) occurs in irreps_out.

Modes
-----
uvu : one weight per (path, channel u); each path writes its own output block
      of multiplicity mul1, appended in path order (the output irreps string is
      therefore derived from the paths).  Weights per edge: [paths, mul1].
uvw : fully connected multiplicity mixing, weights [path, u, w]; every path
      sums into the output block irreps_out[i_out].  With a radial basis of K
      functions the per-edge weights are W_e = sum_k R[e,k] M[k] with
      M of shape [K, sum_path mul1*mul_out] (path-major, then u, then w).
"""

from dataclasses import dataclass, field


def parse_irreps(s):
    """'8x0e+8x1o' -> [(8, 0, 1), (8, 1, -1)] as (mul, l, parity)."""
    out = []
    for term in s.replace(" ", "").split("+"):
        if not term:
            continue
        if "x" in term:
            mul_s, ir = term.split("x")
            mul = int(mul_s)
        else:
            mul, ir = 1, term
        l, p = int(ir[:-1]), {"e": 1, "o": -1}[ir[-1]]
        if mul < 0 or l < 0:
            raise ValueError(term)
        out.append((mul, l, p))
    return out


def irreps_dim(irr):
    return sum(mul * (2 * l + 1) for mul, l, _ in irr)


def irreps_offsets(irr):
    offs, o = [], 0
    for mul, l, _ in irr:
        offs.append(o)
        o += mul * (2 * l + 1)
    return offs


def irreps_str(irr):
    return "+".join(f"{mul}x{l}{'e' if p == 1 else 'o'}" for mul, l, p in irr)


@dataclass
class Path:
    i1: int
    i2: int
    i_out: int
    l1: int
    l2: int
    l3: int
    mul1: int
    mul_out: int
    off1: int       # offset of the in1 block
    off2: int       # offset of the in2 block
    ooff: int       # offset of the output block this path writes / sums into
    woff: int       # offset of this path's weights inside one edge's (or one k's) weight row


@dataclass
class Plan:
    in1: list
    in2: list
    out: list           # output irreps (derived per path for uvu)
    mode: str
    paths: list = field(default_factory=list)
    d1: int = 0
    d2: int = 0
    d_out: int = 0
    w_numel: int = 0    # per-edge weights (uvu) or per-k row of M (uvw)


def make_plan(irreps_in1, irreps_in2, irreps_out, mode="uvu", instructions=None):
    in1, in2, outr = parse_irreps(irreps_in1), parse_irreps(irreps_in2), parse_irreps(irreps_out)
    if mode not in ("uvu", "uvw"):
        raise ValueError(mode)
    if any(m != 1 for m, _, _ in in2):
        raise ValueError("in2 blocks must have multiplicity 1")
    if instructions is None:
        instructions = []
        for i1, (_, l1, p1) in enumerate(in1):
            for i2, (_, l2, p2) in enumerate(in2):
                for l3 in range(abs(l1 - l2), l1 + l2 + 1):
                    p3 = p1 * p2
                    for io, (_, lo, po) in enumerate(outr):
                        if lo == l3 and po == p3:
                            instructions.append((i1, i2, io))
                            break
    off1, off2, offo = irreps_offsets(in1), irreps_offsets(in2), irreps_offsets(outr)
    plan = Plan(in1, in2, [], mode)
    ooff_uvu, woff = 0, 0
    out_derived = []
    for (i1, i2, io) in instructions:
        m1, l1, p1 = in1[i1]
        _, l2, p2 = in2[i2]
        mo, l3, p3 = outr[io]
        if not (abs(l1 - l2) <= l3 <= l1 + l2) or p3 != p1 * p2:
            raise ValueError(f"forbidden path {(i1, i2, io)}")
        if mode == "uvu":
            p = Path(i1, i2, io, l1, l2, l3, m1, m1, off1[i1], off2[i2], ooff_uvu, woff)
            ooff_uvu += m1 * (2 * l3 + 1)
            woff += m1
            out_derived.append((m1, l3, p3))
        else:
            p = Path(i1, i2, io, l1, l2, l3, m1, mo, off1[i1], off2[i2], offo[io], woff)
            woff += m1 * mo
        plan.paths.append(p)
    plan.out = out_derived if mode == "uvu" else outr
    plan.d1, plan.d2, plan.d_out = irreps_dim(in1), irreps_dim(in2), irreps_dim(plan.out)
    plan.w_numel = woff
    return plan
