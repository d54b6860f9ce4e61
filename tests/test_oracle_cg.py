"""Pins of the oracle's coefficients, basis, harmonics and rotations (CPU only).

Nothing here compares the oracle with itself: each test checks it against a
textbook value, an identity of the mathematics, a closed form, or an
independent construction.
"""

import os
from math import sqrt  # also used by eval of the golden file

import numpy as np
import pytest

from oracle import cg
from clebsch_gordan_tensor_racah_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "cg_textbook.txt")


def _golden_rows():
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        *ints, expr = line.split(maxsplit=6)
        yield tuple(map(int, ints)), eval(expr)


@pytest.mark.parametrize("args,value", list(_golden_rows()))
def test_textbook_values(args, value):
    assert abs(cg.cg_complex(*args) - value) < 1e-15


def test_against_sympy_tables():
    sym = pytest.importorskip("sympy.physics.quantum.cg")
    for j1 in range(4):
        for j2 in range(3):
            for J in range(abs(j1 - j2), j1 + j2 + 1):
                for m1 in range(-j1, j1 + 1):
                    for m2 in range(-j2, j2 + 1):
                        M = m1 + m2
                        if abs(M) > J:
                            continue
                        ref = float(sym.CG(j1, m1, j2, m2, J, M).doit())
                        assert abs(cg.cg_complex(j1, m1, j2, m2, J, M) - ref) < 1e-14


def _cg_matrix(j1, j2):
    """Unitary map |j1 m1>|j2 m2> -> |J M>, rows (J, M), cols (m1, m2)."""
    rows = []
    for J in range(abs(j1 - j2), j1 + j2 + 1):
        for M in range(-J, J + 1):
            rows.append([cg.cg_complex(j1, m1, j2, m2, J, M)
                         for m1 in range(-j1, j1 + 1) for m2 in range(-j2, j2 + 1)])
    return np.array(rows)


@pytest.mark.parametrize("j1,j2", [(1, 1), (2, 1), (3, 2), (4, 4), (7, 7), (7, 3)])
def test_orthogonality_and_completeness(j1, j2):
    U = _cg_matrix(j1, j2)
    n = (2 * j1 + 1) * (2 * j2 + 1)
    assert U.shape == (n, n)
    assert np.abs(U @ U.T - np.eye(n)).max() < 1e-13      # sum over m1,m2
    assert np.abs(U.T @ U - np.eye(n)).max() < 1e-13      # sum over J,M


@pytest.mark.parametrize("l", range(8))
def test_real_basis_unitary(l):
    Q = cg.real_basis(l)
    assert np.abs(Q @ Q.conj().T - np.eye(2 * l + 1)).max() < 1e-15


def test_sh_closed_forms():
    rng = np.random.default_rng(3)
    v = rng.normal(size=(50, 3))
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    x, y, z = v.T
    assert np.abs(cg.sh_real(0, v)[:, 0] - 1).max() < 1e-14
    Y1 = cg.sh_real(1, v)
    assert np.abs(Y1 - np.sqrt(3) * np.stack([y, z, x], 1)).max() < 1e-14
    Y2 = cg.sh_real(2, v)
    ref2 = np.stack([np.sqrt(15) * x * y, np.sqrt(15) * y * z, np.sqrt(5) / 2 * (3 * z * z - 1),
                     np.sqrt(15) * x * z, np.sqrt(15) / 2 * (x * x - y * y)], 1)
    assert np.abs(Y2 - ref2).max() < 1e-13
    for l in range(8):
        Yl = cg.sh_real(l, v)
        assert np.abs((Yl ** 2).sum(1) - (2 * l + 1)).max() < 1e-11


def test_workload_sh_matches_oracle_sh():
    v = wl.unit_vectors(np.random.default_rng(5), 300)
    assert np.abs(wl.sh_real(7, v) - cg.sh_real_concat(7, v)).max() < 1e-12


@pytest.mark.parametrize("l", range(6))
def test_wigner_d_constructions_agree(l):
    rng = np.random.default_rng(10 + l)
    axis, ang = rng.normal(size=3), rng.uniform(0, 2 * np.pi)
    R = cg.rotation_matrix(axis, ang)
    D1 = cg.wigner_d_real(l, axis, ang)
    D2 = cg.wigner_d_lstsq(l, R, rng)
    assert np.abs(D1 - D2).max() < 1e-10
    assert np.abs(D1 @ D1.T - np.eye(2 * l + 1)).max() < 1e-12
    v = rng.normal(size=(20, 3))
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    assert np.abs(cg.sh_real(l, v @ R.T) - cg.sh_real(l, v) @ D1.T).max() < 1e-11


def test_real_block_closed_forms_l_le_1():
    C000 = cg.real_cg_block(0, 0, 0)
    assert C000.shape == (1, 1, 1) and abs(C000[0, 0, 0] - 1) < 1e-15
    # 0 x 1 -> 1 : z = x0 * y
    assert np.abs(cg.real_cg_block(0, 1, 1)[0] - np.eye(3)).max() < 1e-15
    assert np.abs(cg.real_cg_block(1, 0, 1)[:, 0, :] - np.eye(3)).max() < 1e-15
    # 1 x 1 -> 0 : z = (x . y) / sqrt3
    assert np.abs(cg.real_cg_block(1, 1, 0)[:, :, 0] - np.eye(3) / np.sqrt(3)).max() < 1e-15
    # 1 x 1 -> 1 : z = (x cross y) / sqrt2 with components ordered (y, z, x)
    rng = np.random.default_rng(0)
    a, b = rng.normal(size=3), rng.normal(size=3)           # cartesian (x, y, z)
    perm = [1, 2, 0]
    z = np.einsum("ijk,i,j->k", cg.real_cg_block(1, 1, 1), a[perm], b[perm])
    assert np.abs(z - np.cross(a, b)[perm] / np.sqrt(2)).max() < 1e-15


NNZ = {(1, 1, 0): 3, (1, 1, 1): 6, (1, 1, 2): 11, (2, 2, 2): 25, (3, 3, 3): 42, (7, 7, 7): 258}


@pytest.mark.parametrize("key", sorted(NNZ))
def test_real_block_nnz_and_norm(key):
    B = cg.real_cg_block(*key)
    assert np.count_nonzero(B) == NNZ[key]
    assert abs((B * B).sum() - (2 * key[2] + 1)) < 1e-12


def _all_triples(lmax):
    for l1 in range(lmax + 1):
        for l2 in range(lmax + 1):
            for l3 in range(abs(l1 - l2), min(l1 + l2, lmax) + 1):
                yield l1, l2, l3


@pytest.mark.parametrize("triple", list(_all_triples(4)) + [(7, 7, 7), (7, 6, 3), (5, 7, 2)])
def test_real_block_equivariance(triple):
    """C(D1 a, D2 b) = D3 C(a, b) for a random rotation (Wigner-D from generators)."""
    l1, l2, l3 = triple
    rng = np.random.default_rng(hash(triple) % (2 ** 31))
    axis, ang = rng.normal(size=3), rng.uniform(0, 2 * np.pi)
    D1, D2, D3 = (cg.wigner_d_real(l, axis, ang) for l in (l1, l2, l3))
    C = cg.real_cg_block(l1, l2, l3)
    lhs = np.einsum("ijk,ia,jb->abk", C, D1, D2)
    rhs = np.einsum("ijk,ck->ijc", C, D3)
    assert np.abs(lhs - rhs).max() < 1e-11


def test_real_block_orthogonality():
    """Distinct l3 blocks of the same (l1, l2) are orthogonal; each has norm^2 = 2l3+1."""
    for l1, l2 in [(1, 2), (3, 3), (2, 4)]:
        blocks = [cg.real_cg_block(l1, l2, l3) / np.sqrt(2 * l3 + 1)
                  for l3 in range(abs(l1 - l2), l1 + l2 + 1)]
        for i, a in enumerate(blocks):
            for j, b in enumerate(blocks):
                if a.shape != b.shape:
                    continue
                dot = (a * b).sum()
                assert abs(dot - (1.0 if i == j else 0.0)) < 1e-13


def test_sh_jacobian_against_finite_differences():
    # the generator-based Jacobian of Y(r/|r|) against central differences of
    # sh_real itself (any length of r, every l <= 7)
    rng = np.random.default_rng(31)
    r = rng.normal(size=(25, 3)) * rng.uniform(0.2, 4.0, size=(25, 1))
    h = 1e-6
    f = lambda rr: cg.sh_real_concat(7, rr / np.linalg.norm(rr, axis=1, keepdims=True))  # noqa: E731
    J = cg.sh_real_concat_jacobian(7, r)
    for k in range(3):
        rp, rm = r.copy(), r.copy()
        rp[:, k] += h
        rm[:, k] -= h
        fd = (f(rp) - f(rm)) / (2 * h)
        assert np.abs(J[:, :, k] - fd).max() < 1e-7 * max(1.0, np.abs(fd).max())
    # radial direction does not change the harmonics
    assert np.abs(np.einsum("eck,ek->ec", J, r)).max() < 1e-12


def test_real_block_sign_rule_every_triple_l_le_7():
    # The sign convention of the real blocks (the pages fix none): after the unit
    # Frobenius normalisation, the first entry above 1e-12 in row-major (m1, m2, m3)
    # order is positive, and the block carries the component factor sqrt(2 l3 + 1).
    # Equivariance, norms and nonzero counts are blind to a flipped sign, so the
    # rule is checked on its own for every triangle-valid triple with l <= 7.
    n = 0
    for l1 in range(8):
        for l2 in range(8):
            for l3 in range(abs(l1 - l2), min(l1 + l2, 7) + 1):
                C = cg.real_cg_block(l1, l2, l3)
                flat = C.reshape(-1)
                first = flat[np.flatnonzero(np.abs(flat) > 1e-12)[0]]
                assert first > 0, (l1, l2, l3, first)
                assert abs(np.linalg.norm(flat) - sqrt(2 * l3 + 1)) < 1e-12, (l1, l2, l3)
                n += 1
    assert n == sum(min(l1 + l2, 7) - abs(l1 - l2) + 1 for l1 in range(8) for l2 in range(8))
