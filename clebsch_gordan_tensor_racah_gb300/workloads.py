"""Seeded synthetic inputs for the fused CG tensor-product convolution.

This module only draws inputs; it holds none of the tensor product's
arithmetic, and both the CUDA path and the CPU oracle consume what it returns.
The edge features are evaluated here because they are inputs of the
convolution, not steps of it:

* ``sh_real``: real spherical harmonics with component normalisation
  (sum_m Y_lm^2 = 2l+1; l = 1 gives sqrt(3) * (y, z, x)), computed from the
  associated-Legendre recurrence in the real (cos m phi / sin m phi) form;
* ``rbf``: K Gaussian radial-basis values of the edge length, centres evenly
  spaced over [0.5, 5], width 1 / (centre spacing)^2.

Recipes (one ``numpy.random.default_rng(seed)`` per workload; draw order:
graph, edge directions, node features, then weights or edge lengths; all draws
in FP64 and cast to the working precision; edge quantities are drawn after the
CSR sort, so draw i belongs to CSR position i):

* ``tiny``   64 nodes, 512 edges, src and dst uniform; in1 8x0e+8x1o, SH l<=1,
  uvu, paths with l3 <= 1, W ~ N(0,1).
* ``nequip`` 10,000 nodes, 32 in-edges each, senders uniform; in1
  32x(0e,1o,2e,3o), SH l<=3, uvu, all parity-allowed l3 <= 3,
  W ~ N(0,1)/sqrt(32) (fan-in = receiver in-degree).
* ``mace``   5,000 nodes, in-degree ~ Poisson(40), senders uniform; in1
  128x(0e,1o,2e), SH l<=3, uvu, l3 <= 2, W ~ N(0,1)/sqrt(40).
* ``highl``  batch 50,000, no graph; in1 16x l for l = 0..7 with parity (-1)^l,
  in2 = SH l<=7, uvu, all l3 <= 7, W ~ N(0,1).
* ``uvw``    200,000 nodes, 32 in-edges each, senders uniform; in1 = out =
  64x(0e,1o,2e), SH l<=2, uvw, 8 radial functions of a length ~ U[0.5, 5],
  M ~ N(0,1)/sqrt(8*64) of shape [8, paths*64*64].
* ``uvw_edge`` the NequIP-like graph (10,000 nodes x 32 in-edges) with
  in1 = out = 16x(0e,1o,2e), SH l<=2, uvw with a weight matrix per edge,
  W ~ N(0,1)/sqrt(32) of shape [E, paths*16*16].
* ``mixedmul`` the NequIP-like graph with in1 = 32x0e+16x1o+16x2e (blocks of
  different multiplicity), SH l<=2, uvu with every l3 <= 2, W ~ N(0,1)/sqrt(32).

Every recipe takes overrides (``N``, ``deg``, ``E``, ``B``) so tests can draw a
smaller instance with the same structure.
"""

import math

import numpy as np

_CHUNK = 1 << 22


def _normal(rng, shape, dtype, scale=1.0):
    """N(0,1)*scale drawn in FP64 chunk by chunk (same stream as one draw), cast to dtype."""
    shape = tuple(int(s) for s in shape)
    total = int(np.prod(shape)) if shape else 1
    out = np.empty(total, dtype=dtype)
    for s in range(0, total, _CHUNK):
        n = min(_CHUNK, total - s)
        v = rng.standard_normal(n)
        if scale != 1.0:
            v *= scale
        out[s:s + n] = v
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# graphs (CSR sorted by receiver, stable)
# ---------------------------------------------------------------------------

def _csr_from_coo(src, dst, N):
    order = np.argsort(dst, kind="stable")
    col = src[order].astype(np.int32)
    counts = np.bincount(dst, minlength=N)
    rowptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return rowptr, col


def graph_uniform(rng, N, E):
    src = rng.integers(0, N, size=E)
    dst = rng.integers(0, N, size=E)
    return _csr_from_coo(src, dst, N)


def graph_fixed_indegree(rng, N, deg):
    dst = np.repeat(np.arange(N), deg)
    src = rng.integers(0, N, size=N * deg)
    return _csr_from_coo(src, dst, N)


def graph_poisson_indegree(rng, N, lam):
    deg = rng.poisson(lam, size=N)
    dst = np.repeat(np.arange(N), deg)
    src = rng.integers(0, N, size=int(deg.sum()))
    return _csr_from_coo(src, dst, N)


def unit_vectors(rng, n):
    v = rng.standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# edge features (inputs of the convolution)
# ---------------------------------------------------------------------------

def sh_real(lmax, vec):
    """Real SH 0..lmax, component normalisation, shape [n, (lmax+1)^2], FP64."""
    x, y, z = vec[:, 0], vec[:, 1], vec[:, 2]
    n = vec.shape[0]
    rho = np.sqrt(np.maximum(x * x + y * y, 0.0))
    phi = np.arctan2(y, x)
    # P[l][m]: associated Legendre without the Condon-Shortley sign
    P = {}
    for m in range(lmax + 1):
        pmm = np.ones(n)
        dfact = 1.0
        for k in range(1, m + 1):
            dfact *= 2 * k - 1
        pmm = dfact * rho ** m
        P[(m, m)] = pmm
        if m + 1 <= lmax:
            P[(m + 1, m)] = z * (2 * m + 1) * pmm
        for l in range(m + 2, lmax + 1):
            P[(l, m)] = ((2 * l - 1) * z * P[(l - 1, m)] - (l + m - 1) * P[(l - 2, m)]) / (l - m)
    cols = []
    for l in range(lmax + 1):
        block = np.zeros((n, 2 * l + 1))
        block[:, l] = math.sqrt(2 * l + 1) * P[(l, 0)]
        for m in range(1, l + 1):
            c = math.sqrt(2 * l + 1) * math.sqrt(2.0 * math.factorial(l - m) / math.factorial(l + m))
            block[:, l + m] = c * P[(l, m)] * np.cos(m * phi)
            block[:, l - m] = c * P[(l, m)] * np.sin(m * phi)
        cols.append(block)
    return np.concatenate(cols, axis=1)


def rbf(r, K=8, lo=0.5, hi=5.0):
    mu = np.linspace(lo, hi, K)
    gamma = 1.0 / (mu[1] - mu[0]) ** 2
    return np.exp(-gamma * (r[:, None] - mu[None, :]) ** 2)


def _parity_str(l):
    return "e" if l % 2 == 0 else "o"


def _all_out(lmax):
    return "+".join(f"{l}{q}" for l in range(lmax + 1) for q in "eo")


def _sh_irreps(lmax):
    return "+".join(f"{l}{_parity_str(l)}" for l in range(lmax + 1))


# ---------------------------------------------------------------------------
# workload recipes
# ---------------------------------------------------------------------------

SPECS = {
    "tiny": dict(in1="8x0e+8x1o", in2="0e+1o", out="0e+1o+1e", mode="uvu", lmax_sh=1,
                 N=64, E=512, graph="uniform", wscale=None, dtype="float32"),
    "nequip": dict(in1="32x0e+32x1o+32x2e+32x3o", in2=_sh_irreps(3), out=_all_out(3),
                   mode="uvu", lmax_sh=3, N=10_000, deg=32, graph="fixed", wscale="deg",
                   dtype="float32"),
    "mace": dict(in1="128x0e+128x1o+128x2e", in2=_sh_irreps(3), out=_all_out(2), mode="uvu",
                 lmax_sh=3, N=5_000, deg=40, graph="poisson", wscale="deg", dtype="float32"),
    "highl": dict(in1="+".join(f"16x{l}{_parity_str(l)}" for l in range(8)), in2=_sh_irreps(7),
                  out=_all_out(7), mode="uvu", lmax_sh=7, B=50_000, graph=None, wscale=None,
                  dtype="float32"),
    "uvw": dict(in1="64x0e+64x1o+64x2e", in2=_sh_irreps(2), out="64x0e+64x1o+64x2e", mode="uvw",
                lmax_sh=2, N=200_000, deg=32, graph="fixed", K=8, dtype="float32"),
    # mixed instruction list on the NequIP-like graph: 32x(0e,1o,2e) x SH l<=2 -> 32x(0e,1o,2e),
    # the scalar output block fed fully connected (uvw), the others channel-wise (uvu);
    # every parity-allowed (i_in1, i_in2, i_out), written out
    "mixed": dict(in1="32x0e+32x1o+32x2e", in2=_sh_irreps(2), out="32x0e+32x1o+32x2e", mode="mixed",
                  instructions=[(0, 0, 0), (0, 1, 1), (0, 2, 2), (1, 0, 1), (1, 1, 0), (1, 1, 2), (1, 2, 1),
                                (2, 0, 2), (2, 1, 1), (2, 2, 0), (2, 2, 2)],
                  modes=["uvw", "uvu", "uvu", "uvu", "uvw", "uvu", "uvu", "uvu", "uvu", "uvw", "uvu"],
                  lmax_sh=2, N=10_000, deg=32, graph="fixed", wscale="deg", dtype="float32"),
    # channel-wise uvu with blocks of different multiplicity on the NequIP-like graph (the
    # general kernels serve it: the warp-autonomous ones need one multiplicity for all blocks)
    "mixedmul": dict(in1="32x0e+16x1o+16x2e", in2=_sh_irreps(2), out=_all_out(2), mode="uvu", lmax_sh=2,
                     N=10_000, deg=32, graph="fixed", wscale="deg", dtype="float32"),
    # uvw with a weight matrix per edge (K = 0): 16x(0e,1o,2e) on the NequIP-like graph
    "uvw_edge": dict(in1="16x0e+16x1o+16x2e", in2=_sh_irreps(2), out="16x0e+16x1o+16x2e", mode="uvw",
                     lmax_sh=2, N=10_000, deg=32, graph="fixed", K=0, wscale="deg", dtype="float32"),
}


def irreps_terms(s):
    """[(mul, l), ...] of an irreps string."""
    out = []
    for term in s.split("+"):
        mul, ir = (term.split("x") if "x" in term else ("1", term))
        out.append((int(mul), int(ir[:-1])))
    return out


def irreps_dim(s):
    d = 0
    for term in s.split("+"):
        mul, ir = (term.split("x") if "x" in term else ("1", term))
        d += int(mul) * (2 * int(ir[:-1]) + 1)
    return d


def make(name, w_numel, seed=0, dtype=None, **over):
    """Draw one workload.  Returns a dict of numpy arrays plus the spec entries.

    ``w_numel`` is the weight count of one edge (uvu) or of one radial row of M
    (uvw), taken from the caller's own plan; for a mixed instruction list it is the
    pair (uvu weights, uvw weights) of one edge.

    Keys: rowptr, col (int32) for graph workloads; x (or x1), Y (or x2), W for
    uvu; R, M for uvw; Wu, Ww for mixed lists; plus 'spec', 'N', 'E' (or 'B').
    """
    spec = dict(SPECS[name])
    spec.update(over)
    dt = np.dtype(dtype or spec["dtype"])
    rng = np.random.default_rng(seed)
    d1, d2 = irreps_dim(spec["in1"]), irreps_dim(spec["in2"])
    res = {"spec": spec, "name": name, "dtype": dt}
    if spec["graph"] is None:
        B = int(spec["B"])
        vec = unit_vectors(rng, B)
        x1 = _normal(rng, (B, d1), dt)
        x2 = sh_real(spec["lmax_sh"], vec).astype(dt)
        W = _normal(rng, (B, int(w_numel)), dt)
        res.update(x1=x1, x2=x2, W=W, B=B)
        return res
    N = int(spec["N"])
    if spec["graph"] == "uniform":
        rowptr, col = graph_uniform(rng, N, int(spec["E"]))
    elif spec["graph"] == "fixed":
        rowptr, col = graph_fixed_indegree(rng, N, int(spec["deg"]))
    else:
        rowptr, col = graph_poisson_indegree(rng, N, float(spec["deg"]))
    E = int(rowptr[-1])
    vec = unit_vectors(rng, E)
    Y = sh_real(spec["lmax_sh"], vec).astype(dt)
    x = _normal(rng, (N, d1), dt)
    res.update(rowptr=rowptr, col=col, N=N, E=E, x=x, Y=Y)
    if spec["mode"] == "mixed":   # two per-edge weight arrays
        scale = 1.0 / math.sqrt(float(spec["deg"]))
        wu, ww = (int(v) for v in w_numel)
        res.update(Wu=_normal(rng, (E, wu), dt, scale), Ww=_normal(rng, (E, ww), dt, scale / math.sqrt(32.0)))
    elif spec["mode"] == "uvu" or int(spec.get("K", 1)) == 0:   # weights per edge
        scale = 1.0 if spec["wscale"] is None else 1.0 / math.sqrt(float(spec["deg"]))
        W = _normal(rng, (E, int(w_numel)), dt, scale)
        res.update(W=W)
    else:
        K = int(spec["K"])
        r = rng.uniform(0.5, 5.0, size=E)
        R = rbf(r, K).astype(dt)
        M = _normal(rng, (K, int(w_numel)), dt, 1.0 / math.sqrt(K * 64))
        res.update(R=R, M=M)
    return res
