// sh.cuh -- real spherical harmonics of edge vectors, evaluated where they are
// consumed ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep
// Networks", Figure 4B: the edge features of the fused convolution are
// spherical harmonics of the edge directions).
//
// Convention (the one the library's CG tables are built for): component
// normalisation (sum_m Y_lm^2 = 2l+1 on the unit sphere), components ordered
// m = -l..l, real basis with
//   Y_l,+m = N_lm q_lm(z) Re((x + i y)^m),  Y_l,-m = N_lm q_lm(z) Im((x + i y)^m),
//   Y_l,0  = sqrt(2l+1) q_l0(z),
//   N_lm   = sqrt(2l+1) sqrt(2 (l-m)! / (l+m)!),
// where q_lm(z) is the associated Legendre function P_l^m (without the
// Condon-Shortley sign) divided by (1 - z^2)^(m/2), from the recurrence in l
//   q_mm = (2m-1)!!,  q_m+1,m = (2m+1) z q_mm,
//   q_lm = ((2l-1) z q_l-1,m - (l+m-1) q_l-2,m) / (l-m).
// For l = 1 this is sqrt(3) (y, z, x).  The formulas are polynomials in the
// unit vector (x, y, z), so instantiating them on a dual number gives the exact
// gradient of that polynomial; its projection on the tangent plane is the
// derivative on the sphere.
#pragma once
#include <cmath>

namespace cgtp {

// value and gradient with respect to (x, y, z)
template <typename T>
struct Dual3 {
  T v, dx, dy, dz;
};
template <typename T>
__host__ __device__ inline Dual3<T> operator+(Dual3<T> a, Dual3<T> b) {
  return {a.v + b.v, a.dx + b.dx, a.dy + b.dy, a.dz + b.dz};
}
template <typename T>
__host__ __device__ inline Dual3<T> operator-(Dual3<T> a, Dual3<T> b) {
  return {a.v - b.v, a.dx - b.dx, a.dy - b.dy, a.dz - b.dz};
}
template <typename T>
__host__ __device__ inline Dual3<T> operator*(Dual3<T> a, Dual3<T> b) {
  return {a.v * b.v, a.dx * b.v + a.v * b.dx, a.dy * b.v + a.v * b.dy, a.dz * b.v + a.v * b.dz};
}
template <typename T>
__host__ __device__ inline Dual3<T> operator*(T s, Dual3<T> a) {
  return {s * a.v, s * a.dx, s * a.dy, s * a.dz};
}
template <typename T>
__host__ __device__ inline T sh_scale(T s, T a) {
  return s * a;
}
template <typename T>
__host__ __device__ inline Dual3<T> sh_scale(T s, Dual3<T> a) {
  return s * a;
}
// the constant c as a value of the same kind as `like`
template <typename T>
__host__ __device__ inline T sh_const(T c, T) {
  return c;
}
template <typename T>
__host__ __device__ inline Dual3<T> sh_const(T c, Dual3<T>) {
  return {c, T(0), T(0), T(0)};
}

// Compile-time constants: N_lm^2 = (2l+1) [2 (l-m)! / (l+m)! for m > 0],
// (2m-1)!!, and a Newton square root (exact to double rounding for these sizes).
__host__ __device__ constexpr double sh_norm2(int l, int m) {
  double r = 2.0 * l + 1.0;
  if (m > 0) {
    double f = 2.0;
    for (int k = l - m + 1; k <= l + m; ++k) f /= k;
    r *= f;
  }
  return r;
}
__host__ __device__ constexpr double sh_dfact(int m) {
  double d = 1.0;
  for (int k = 1; k <= m; ++k) d *= 2 * k - 1;
  return d;
}
__host__ __device__ constexpr double sh_csqrt(double x) {
  double r = x > 1.0 ? x : 1.0;
  for (int i = 0; i < 64; ++i) r = 0.5 * (r + x / r);
  return r;
}

// the order-M terms of the degree-L block, then order M + 1
template <int L, int M, typename T, typename N>
__host__ __device__ inline void sh_order(N z, const N (&C)[L + 1], const N (&S)[L + 1], N (&out)[2 * L + 1]) {
  constexpr double nrm = sh_csqrt(sh_norm2(L, M));
  N q = sh_const(T(sh_dfact(M)), z);   // q_MM = (2M-1)!!
  if constexpr (L > M) {
    N q0 = q;
    N q1 = sh_scale(T(2 * M + 1), z * q0);
#pragma unroll
    for (int l = M + 2; l <= L; ++l) {
      const N q2 = sh_scale(T(1.0 / (l - M)), sh_scale(T(2 * l - 1), z * q1) - sh_scale(T(l + M - 1), q0));
      q0 = q1;
      q1 = q2;
    }
    q = q1;
  }
  out[L + M] = sh_scale(T(nrm), q * C[M]);
  if constexpr (M > 0) out[L - M] = sh_scale(T(nrm), q * S[M]);
  if constexpr (M < L) sh_order<L, M + 1, T, N>(z, C, S, out);
}

// Degree-L block at (x, y, z) (a unit vector for the harmonics; any point for
// the polynomial).  N is T or Dual3<T>; T is the arithmetic type.
template <int L, typename T, typename N>
__host__ __device__ inline void sh_block(N x, N y, N z, N (&out)[2 * L + 1]) {
  N C[L + 1], S[L + 1];   // C_m + i S_m = (x + i y)^m
  C[0] = sh_const(T(1), x);
  S[0] = sh_const(T(0), x);
#pragma unroll
  for (int m = 1; m <= L; ++m) {
    C[m] = x * C[m - 1] - y * S[m - 1];
    S[m] = x * S[m - 1] + y * C[m - 1];
  }
  sh_order<L, 0, T, N>(z, C, S, out);
}

}  // namespace cgtp
