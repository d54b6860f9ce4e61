"""Clebsch-Gordan coefficients, real basis, real spherical harmonics, Wigner-D.

Test infrastructure only (see the package docstring).

The pages ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep
Networks", Figures 1-2) describe the coefficient tensor only as block-sparse, one
block per (l1, l2, l3), each block itself sparse and repeated over the
multiplicities.  They print no formula, so this module writes out the standard
mathematics:

* ``cg_complex``: Racah's closed form for <j1 m1; j2 m2 | J M> with the
  Condon-Shortley phase, evaluated exactly (integers and Fractions; the single
  square root is taken last, in FP64).
* ``real_basis``: the unitary change of basis from complex to real spherical
  components (rows m = -l..l of the real basis).
* ``real_cg_block``: the complex block carried into the real basis, reduced to a
  real tensor, normalised to unit Frobenius norm (a 3j block), sign-fixed so the
  first entry above 1e-12 in row-major (m1, m2, m3) order is positive, and scaled
  by sqrt(2 l3 + 1) ("component" normalisation).
* ``sh_real``: real spherical harmonics with component normalisation
  (sum_m Y_lm^2 = 2l+1), built from scipy's complex harmonics and the same basis.
* ``wigner_d_real``: the real Wigner-D matrix of a rotation, two independent
  constructions (matrix exponential of the angular-momentum generators, and a
  least-squares fit of Y(R r) = D Y(r)).
"""

from fractions import Fraction
from functools import lru_cache
from math import factorial, sqrt, prod

import numpy as np
import scipy.linalg
import scipy.special


def cg_complex(j1, m1, j2, m2, J, M):
    """<j1 m1; j2 m2 | J M>, Condon-Shortley phase, exact Racah sum (FP64 result)."""
    if m1 + m2 != M:
        return 0.0
    if not (abs(j1 - j2) <= J <= j1 + j2):
        return 0.0
    if abs(m1) > j1 or abs(m2) > j2 or abs(M) > J:
        return 0.0
    f = factorial
    pref = Fraction((2 * J + 1) * f(J + j1 - j2) * f(J - j1 + j2) * f(j1 + j2 - J),
                    f(j1 + j2 + J + 1))
    pref *= f(J + M) * f(J - M) * f(j1 - m1) * f(j1 + m1) * f(j2 - m2) * f(j2 + m2)
    s = Fraction(0)
    for k in range(0, j1 + j2 - J + 1):
        d = (k, j1 + j2 - J - k, j1 - m1 - k, j2 + m2 - k, J - j2 + m1 + k, J - j1 - m2 + k)
        if min(d) < 0:
            continue
        s += Fraction((-1) ** k, prod(f(v) for v in d))
    if s == 0:
        return 0.0
    val = sqrt(float(s * s * pref))
    return val if s > 0 else -val


@lru_cache(maxsize=None)
def cg_complex_block(l1, l2, l3):
    """Dense complex-basis block C[m1+l1, m2+l2, m3+l3] (real numbers)."""
    out = np.zeros((2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1))
    for m1 in range(-l1, l1 + 1):
        for m2 in range(-l2, l2 + 1):
            m3 = m1 + m2
            if abs(m3) <= l3:
                out[m1 + l1, m2 + l2, m3 + l3] = cg_complex(l1, m1, l2, m2, l3, m3)
    return out


@lru_cache(maxsize=None)
def real_basis(l):
    """Q_l: row a (real m = a - l) expresses the real component in complex ones.

    m > 0 : (Y^{-m} + (-1)^m Y^{m}) / sqrt2
    m = 0 : Y^0
    m < 0 : i (Y^{m} - (-1)^m Y^{-m}) / sqrt2
    """
    Q = np.zeros((2 * l + 1, 2 * l + 1), dtype=complex)
    r = 1.0 / np.sqrt(2.0)
    for m in range(-l, l + 1):
        a = m + l
        if m > 0:
            Q[a, -m + l] = r
            Q[a, m + l] = (-1) ** m * r
        elif m == 0:
            Q[a, l] = 1.0
        else:
            Q[a, m + l] = 1j * r
            Q[a, -m + l] = -1j * (-1) ** (-m) * r
    return Q


@lru_cache(maxsize=None)
def real_cg_block(l1, l2, l3):
    """Real-basis, component-normalised coupling block C[m1, m2, m3] (FP64).

    Returns an array of shape (2l1+1, 2l2+1, 2l3+1).  Zero block if the
    triangle rule fails.
    """
    if not (abs(l1 - l2) <= l3 <= l1 + l2):
        return np.zeros((2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1))
    C = cg_complex_block(l1, l2, l3)
    Q1, Q2, Q3 = real_basis(l1), real_basis(l2), real_basis(l3)
    T = np.einsum("ai,bj,ck,ijk->abc", Q1, Q2, np.conj(Q3), C)
    re, im = np.abs(T.real).max(), np.abs(T.imag).max()
    R = T.real if re >= im else T.imag
    other = im if re >= im else re
    assert other < 1e-13, (l1, l2, l3, other)
    R = R / np.sqrt((R * R).sum())
    flat = R.ravel()
    first = np.flatnonzero(np.abs(flat) > 1e-12)[0]
    if flat[first] < 0:
        R = -R
    R = np.where(np.abs(R) > 1e-15, R, 0.0) * np.sqrt(2 * l3 + 1)
    return R


# ----------------------------------------------------------------------------
# spherical harmonics and rotations (used by the equivariance pins)
# ----------------------------------------------------------------------------

def sh_complex(l, vec):
    """Complex Y_l^m (Condon-Shortley) at unit vectors vec[..., 3]; shape [..., 2l+1]."""
    x, y, z = vec[..., 0], vec[..., 1], vec[..., 2]
    theta = np.arccos(np.clip(z, -1.0, 1.0))
    phi = np.arctan2(y, x)
    return np.stack([scipy.special.sph_harm_y(l, m, theta, phi) for m in range(-l, l + 1)], -1)


def sh_real(l, vec):
    """Real SH, component normalisation: sqrt(4 pi) * Q_l * Y_l^complex."""
    Yc = sh_complex(l, vec)
    Yr = np.sqrt(4 * np.pi) * np.einsum("am,...m->...a", real_basis(l), Yc)
    assert np.abs(Yr.imag).max() < 1e-12
    return Yr.real


def sh_real_concat(lmax, vec):
    """Concatenated real SH 0..lmax (component normalisation), shape [..., (lmax+1)^2]."""
    return np.concatenate([sh_real(l, vec) for l in range(lmax + 1)], -1)


def _angular_momentum(l):
    """J_x, J_y, J_z in the complex |l m> basis (m = -l..l), hbar = 1."""
    m = np.arange(-l, l + 1)
    Jz = np.diag(m).astype(complex)
    Jp = np.zeros((2 * l + 1, 2 * l + 1), dtype=complex)
    for i, mm in enumerate(m[:-1]):
        Jp[i + 1, i] = np.sqrt(l * (l + 1) - mm * (mm + 1))
    Jm = Jp.conj().T
    return (Jp + Jm) / 2, (Jp - Jm) / (2j), Jz


def rotation_matrix(axis, angle):
    """3x3 rotation by `angle` about unit `axis` (right-handed)."""
    axis = np.asarray(axis, float)
    axis = axis / np.linalg.norm(axis)
    K = np.array([[0, -axis[2], axis[1]], [axis[2], 0, -axis[0]], [-axis[1], axis[0], 0]])
    return scipy.linalg.expm(angle * K)


def wigner_d_real(l, axis, angle):
    """Real Wigner-D from the generators: D = Q conj(exp(-i angle n.J)) Q^dagger.

    Satisfies Y_l(R r) = D Y_l(r) for R = rotation_matrix(axis, angle).
    """
    axis = np.asarray(axis, float)
    axis = axis / np.linalg.norm(axis)
    Jx, Jy, Jz = _angular_momentum(l)
    U = scipy.linalg.expm(-1j * angle * (axis[0] * Jx + axis[1] * Jy + axis[2] * Jz))
    Q = real_basis(l)
    D = Q @ np.conj(U) @ Q.conj().T
    assert np.abs(D.imag).max() < 1e-12
    return D.real


def sh_real_jacobian(l, rvec):
    """d Y_l(r / |r|) / d r for vectors rvec [n, 3]: shape [n, 2l+1, 3].

    Exact, from the rotation generators: for the rotation R_a(t) about axis a,
    d/dt Y_l(R_a(t) u) at t = 0 equals G_a Y_l(u) with G_a = d/dt D_l(R_a(t)) =
    Q conj(-i J_a) Q^dagger (wigner_d_real at first order).  The same derivative
    is grad Y . (e_a x u) = e_a . (u x grad Y), so the tangential gradient t of
    Y on the sphere obeys u x t = w with w_a = G_a Y_l(u), hence t = -u x w;
    d/dr = t / |r| (the radial direction does not change Y(r/|r|)).
    """
    r = np.asarray(rvec, float)
    n = np.linalg.norm(r, axis=1)
    u = r / n[:, None]
    Y = sh_real(l, u)                                     # [n, 2l+1]
    Q = real_basis(l)
    w = np.zeros(Y.shape + (3,))
    for a, Ja in enumerate(_angular_momentum(l)):
        G = Q @ np.conj(-1j * Ja) @ Q.conj().T
        assert np.abs(G.imag).max() < 1e-12
        w[..., a] = Y @ G.real.T                           # (G_a Y)_m
    t = -np.cross(u[:, None, :], w)                        # [n, 2l+1, 3]
    return t / n[:, None, None]


def sh_real_concat_jacobian(lmax, rvec):
    """Jacobian of sh_real_concat(lmax, r / |r|) with respect to r: [n, (lmax+1)^2, 3]."""
    return np.concatenate([sh_real_jacobian(l, rvec) for l in range(lmax + 1)], axis=1)


def wigner_d_lstsq(l, R, rng):
    """Real Wigner-D by least squares: the D with Y_l(R r) = D Y_l(r) on random r."""
    pts = rng.normal(size=(4 * (2 * l + 1) + 8, 3))
    pts /= np.linalg.norm(pts, axis=1, keepdims=True)
    A = sh_real(l, pts)
    B = sh_real(l, pts @ R.T)
    Dt, *_ = np.linalg.lstsq(A, B, rcond=None)
    return Dt.T
