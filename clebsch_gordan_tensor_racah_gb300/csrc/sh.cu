// sh.cu -- the fused convolution fed by raw edge vectors: the real spherical
// harmonics Y(r/|r|) are evaluated inside the kernels as each edge is loaded
// (sh.cuh), and the backward turns the harmonic gradient into the gradient
// with respect to the edge vectors ("An Efficient Sparse Kernel Generator for
// O(3)-Equivariant Deep Networks", Figure 4B: the edge features of the fused
// convolution are spherical harmonics of the edge directions).
//
// Chain rule: Y = P(u) with u = r/|r| and P the polynomials of sh.cuh, so
//   dL/dr = (g_u - (g_u . u) u) / |r|,   g_u = sum_lm (dL/dY_lm) grad P_lm(u),
// with grad P from the same polynomials evaluated on dual numbers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "internal.h"
#include "sh.cuh"

namespace cgtp {
namespace {

// g_u accumulated over the degree-L block of one edge
template <int L, typename T>
__host__ __device__ inline void sh_grad_block(T ux, T uy, T uz, const T* gy, T& gx_, T& gy_, T& gz_) {
  Dual3<T> x{ux, T(1), T(0), T(0)}, y{uy, T(0), T(1), T(0)}, z{uz, T(0), T(0), T(1)};
  Dual3<T> Yd[2 * L + 1];
  sh_block<L, T, Dual3<T>>(x, y, z, Yd);
#pragma unroll
  for (int m = 0; m < 2 * L + 1; ++m) {
    gx_ += gy[m] * Yd[m].dx;
    gy_ += gy[m] * Yd[m].dy;
    gz_ += gy[m] * Yd[m].dz;
  }
}

template <typename T>
__host__ __device__ inline void sh_grad_edge(const T* r, const T* gY, int lmax, T* out) {
  const T rx = r[0], ry = r[1], rz = r[2];
  const T n2 = rx * rx + ry * ry + rz * rz;
  if (!(n2 > T(0))) {
    out[0] = out[1] = out[2] = T(0);
    return;
  }
  const T n = sqrt(n2), ux = rx / n, uy = ry / n, uz = rz / n;
  T gx_ = 0, gy_ = 0, gz_ = 0;
  switch (lmax) {  // blocks l = 0..lmax sit at offsets l^2
    case 7: sh_grad_block<7, T>(ux, uy, uz, gY + 49, gx_, gy_, gz_); [[fallthrough]];
    case 6: sh_grad_block<6, T>(ux, uy, uz, gY + 36, gx_, gy_, gz_); [[fallthrough]];
    case 5: sh_grad_block<5, T>(ux, uy, uz, gY + 25, gx_, gy_, gz_); [[fallthrough]];
    case 4: sh_grad_block<4, T>(ux, uy, uz, gY + 16, gx_, gy_, gz_); [[fallthrough]];
    case 3: sh_grad_block<3, T>(ux, uy, uz, gY + 9, gx_, gy_, gz_); [[fallthrough]];
    case 2: sh_grad_block<2, T>(ux, uy, uz, gY + 4, gx_, gy_, gz_); [[fallthrough]];
    case 1: sh_grad_block<1, T>(ux, uy, uz, gY + 1, gx_, gy_, gz_); [[fallthrough]];
    default: break;  // Y_0 is constant
  }
  const T radial = gx_ * ux + gy_ * uy + gz_ * uz;
  out[0] = (gx_ - radial * ux) / n;
  out[1] = (gy_ - radial * uy) / n;
  out[2] = (gz_ - radial * uz) / n;
}

template <typename T>
__global__ void sh_grad_kernel(const T* __restrict__ rvec, const T* __restrict__ gY, int d2, int lmax,
                               int64_t E, T* __restrict__ grvec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride)
    sh_grad_edge<T>(rvec + 3 * e, gY + e * d2, lmax, grvec + 3 * e);
}

// uvw: the harmonic part plus the radial part sum_k gR_k dR_k/dd u, with
// R_k(d) = exp(-gamma (d - lo - k step)^2)
__global__ void sh_radial_grad_kernel(const float* __restrict__ rvec, const float* __restrict__ gY,
                                      const float* __restrict__ gR, int d2, int lmax, int K, float lo,
                                      float step, float gamma, int64_t E, float* __restrict__ grvec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride) {
    float* o = grvec + 3 * e;
    const float* r = rvec + 3 * e;
    sh_grad_edge<float>(r, gY + e * d2, lmax, o);
    const float d = sqrtf(r[0] * r[0] + r[1] * r[1] + r[2] * r[2]);
    if (!(d > 0.f)) continue;
    float s = 0.f;
    for (int k = 0; k < K; ++k) {
      const float t = d - (lo + k * step);
      s += gR[e * K + k] * (-2.f * gamma * t) * expf(-gamma * t * t);
    }
    const float inv = 1.f / d;
    o[0] += s * r[0] * inv;
    o[1] += s * r[1] * inv;
    o[2] += s * r[2] * inv;
  }
}

// in2 must be the harmonics 0..L in order (mul 1, parity (-1)^l): returns L or -1
int sh_lmax(const cgtp_plan_s* plan) {
  for (size_t i = 0; i < plan->in2.size(); ++i) {
    const Irrep& r = plan->in2[i];
    if (r.mul != 1 || r.l != static_cast<int>(i) || r.p != ((i & 1) ? -1 : 1)) return -1;
  }
  return static_cast<int>(plan->in2.size()) - 1;
}

cgtp_status sh_radial_check(const cgtp_plan_s* plan, double lo, double hi) {
  if (plan->mode != CGTP_UVW) return fail(CGTP_EUNSUPPORTED, "radial edge-vector input needs a uvw plan");
  if (sh_lmax(plan) < 0)
    return fail(CGTP_EUNSUPPORTED, "edge-vector input needs irreps_in2 = 0e+1o+2e+... (harmonics 0..L in order)");
  if (!(hi > lo)) return fail(CGTP_EINVAL, "radial basis needs rbf_hi > rbf_lo");
  return CGTP_OK;
}

cgtp_status sh_check(const cgtp_plan_s* plan) {
  if (plan->mode != CGTP_UVU) return fail(CGTP_EUNSUPPORTED, "edge-vector input needs a uvu plan");
  if (plan->dtype == CGTP_BF16) return fail(CGTP_EUNSUPPORTED, "edge-vector input has no CGTP_BF16 path");
  if (sh_lmax(plan) < 0)
    return fail(CGTP_EUNSUPPORTED, "edge-vector input needs irreps_in2 = 0e+1o+2e+... (harmonics 0..L in order)");
  if (!plan->v3.lpe)
    return fail(CGTP_EUNSUPPORTED, "edge-vector input needs a plan the fused l <= 3 kernels serve");
  return CGTP_OK;
}

}  // namespace
}  // namespace cgtp

using namespace cgtp;

extern "C" {

cgtp_status cgtp_real_sh(int lmax, const double* rvec, int64_t n, double* Y, double* dY) {
  clear_error();
  if (lmax < 0 || lmax > kMaxL) return fail(CGTP_EINVAL, "lmax must be in [0, 7]");
  if (n < 0 || (n > 0 && (!rvec || !Y))) return fail(CGTP_EINVAL, "null rvec or Y");
  const int d2 = (lmax + 1) * (lmax + 1);
  for (int64_t e = 0; e < n; ++e) {
    const double* r = rvec + 3 * e;
    const double n2 = r[0] * r[0] + r[1] * r[1] + r[2] * r[2];
    const double inv = n2 > 0 ? 1.0 / std::sqrt(n2) : 0.0;
    const double ux = r[0] * inv, uy = r[1] * inv, uz = r[2] * inv;
    double* y = Y + e * d2;
    switch (lmax) {
      case 7: { double b[15]; sh_block<7, double, double>(ux, uy, uz, b); std::memcpy(y + 49, b, sizeof b); } [[fallthrough]];
      case 6: { double b[13]; sh_block<6, double, double>(ux, uy, uz, b); std::memcpy(y + 36, b, sizeof b); } [[fallthrough]];
      case 5: { double b[11]; sh_block<5, double, double>(ux, uy, uz, b); std::memcpy(y + 25, b, sizeof b); } [[fallthrough]];
      case 4: { double b[9]; sh_block<4, double, double>(ux, uy, uz, b); std::memcpy(y + 16, b, sizeof b); } [[fallthrough]];
      case 3: { double b[7]; sh_block<3, double, double>(ux, uy, uz, b); std::memcpy(y + 9, b, sizeof b); } [[fallthrough]];
      case 2: { double b[5]; sh_block<2, double, double>(ux, uy, uz, b); std::memcpy(y + 4, b, sizeof b); } [[fallthrough]];
      case 1: { double b[3]; sh_block<1, double, double>(ux, uy, uz, b); std::memcpy(y + 1, b, sizeof b); } [[fallthrough]];
      default: { double b[1]; sh_block<0, double, double>(ux, uy, uz, b); y[0] = b[0]; }
    }
    if (dY) {  // dY[e][lm][k] = d Y_lm / d r_k, one unit cotangent at a time
      double gy[64];
      for (int c = 0; c < d2; ++c) {
        std::memset(gy, 0, sizeof gy);
        gy[c] = 1.0;
        sh_grad_edge<double>(r, gy, lmax, dY + (e * d2 + c) * 3);
      }
    }
  }
  return CGTP_OK;
}

cgtp_status cgtp_conv_forward_sh(cgtp_plan plan, cgtp_graph g, const void* x, const void* rvec, const void* W,
                                 void* out, void* stream) {
  clear_error();
  if (!plan || !g) return fail(CGTP_EINVAL, "null plan or graph");
  cgtp_status s;
  if ((s = sh_check(plan))) return s;
  if (!x || !out || (g->E > 0 && (!rvec || !W))) return fail(CGTP_EINVAL, "null x, rvec, W or out");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(W)) & 15u)
    return fail(CGTP_EINVAL, "x, W and out must be 16-byte aligned");
  if (g->N == 0) return CGTP_OK;
  cgtp_status st3 = CGTP_OK;
  if (!launch_v3_forward(plan, x, nullptr, W, out, g->rowptr, g->col, g->N, stream, &st3,
                         g->E > 0 ? rvec : nullptr))
    return fail(CGTP_EUNSUPPORTED, "edge-vector input: graph too large for the fused kernels");
  return st3;
}

cgtp_status cgtp_conv_backward_sh(cgtp_plan plan, cgtp_graph g, const void* gout, const void* x, const void* rvec,
                                  const void* W, void* gx, void* gY, void* grvec, void* gW, void* stream) {
  clear_error();
  if (!plan || !g) return fail(CGTP_EINVAL, "null plan or graph");
  cgtp_status s;
  if ((s = sh_check(plan))) return s;
  if (!gout || !x || !gx || (g->E > 0 && (!rvec || !W || !gY || !grvec || !gW)))
    return fail(CGTP_EINVAL, "null operand");
  if ((reinterpret_cast<uintptr_t>(gout) | reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(gx) |
       reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(gY) | reinterpret_cast<uintptr_t>(gW)) & 15u)
    return fail(CGTP_EINVAL, "tensors must be 16-byte aligned");
  if (g->N == 0) return CGTP_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cgtp_status st3 = CGTP_OK;
  if (!launch_v3_backward(plan, gout, x, nullptr, W, gx, gY, gW, g->t_rowptr, g->t_eid, g->t_dst, g->N, stream,
                          &st3, g->E > 0 ? rvec : nullptr))
    return fail(CGTP_EUNSUPPORTED, "edge-vector input: graph too large for the fused kernels");
  if (st3 != CGTP_OK || g->E == 0) return st3;
  const int lmax = sh_lmax(plan);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((g->E + 255) / 256, (int64_t)plan->num_sms * 8)));
  if (plan->dtype == CGTP_F64)
    sh_grad_kernel<double><<<grid, 256, 0, st>>>(static_cast<const double*>(rvec), static_cast<const double*>(gY),
                                                  static_cast<int>(plan->d2), lmax, g->E, static_cast<double*>(grvec));
  else
    sh_grad_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(rvec), static_cast<const float*>(gY),
                                                 static_cast<int>(plan->d2), lmax, g->E, static_cast<float*>(grvec));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CGTP_OK : fail(CGTP_ECUDA, std::string("edge-vector gradient launch: ") + cudaGetErrorString(e));
}

cgtp_status cgtp_conv_forward_sh_radial(cgtp_plan plan, cgtp_graph g, const void* x, const void* rvec,
                                        const void* M, double rbf_lo, double rbf_hi, void* out, void* stream) {
  clear_error();
  if (!plan || !g) return fail(CGTP_EINVAL, "null plan or graph");
  cgtp_status s;
  if ((s = sh_radial_check(plan, rbf_lo, rbf_hi))) return s;
  if (!x || !M || !out || (g->E > 0 && !rvec)) return fail(CGTP_EINVAL, "null x, rvec, M or out");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(M) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return fail(CGTP_EINVAL, "x, M and out must be 16-byte aligned");
  return uvw_forward(plan, g, x, nullptr, nullptr, M, out, stream, g->E > 0 ? rvec : nullptr, rbf_lo, rbf_hi);
}

cgtp_status cgtp_conv_backward_sh_radial(cgtp_plan plan, cgtp_graph g, const void* gout, const void* x,
                                         const void* rvec, const void* M, double rbf_lo, double rbf_hi,
                                         void* gx, void* gY, void* gR, void* grvec, void* gM, void* stream) {
  clear_error();
  if (!plan || !g) return fail(CGTP_EINVAL, "null plan or graph");
  cgtp_status s;
  if ((s = sh_radial_check(plan, rbf_lo, rbf_hi))) return s;
  if (!gout || !x || !M || !gx || !gM || (g->E > 0 && (!rvec || !gY || !gR || !grvec)))
    return fail(CGTP_EINVAL, "null operand");
  if ((reinterpret_cast<uintptr_t>(gout) | reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(M) |
       reinterpret_cast<uintptr_t>(gx) | reinterpret_cast<uintptr_t>(gY) | reinterpret_cast<uintptr_t>(gR) |
       reinterpret_cast<uintptr_t>(gM)) & 15u)
    return fail(CGTP_EINVAL, "tensors must be 16-byte aligned");
  if ((s = uvw_backward(plan, g, gout, x, nullptr, nullptr, M, gx, gY, gR, gM, stream, g->E > 0 ? rvec : nullptr,
                        rbf_lo, rbf_hi)))
    return s;
  if (g->E == 0) return CGTP_OK;
  const int K = plan->radial_k;
  const double step = K > 1 ? (rbf_hi - rbf_lo) / (K - 1) : (rbf_hi - rbf_lo);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((g->E + 255) / 256, (int64_t)plan->num_sms * 8)));
  sh_radial_grad_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const float*>(rvec), static_cast<const float*>(gY), static_cast<const float*>(gR),
      static_cast<int>(plan->d2), sh_lmax(plan), K, static_cast<float>(rbf_lo), static_cast<float>(step),
      static_cast<float>(1.0 / (step * step)), g->E, static_cast<float*>(grvec));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CGTP_OK : fail(CGTP_ECUDA, std::string("edge-vector gradient launch: ") + cudaGetErrorString(e));
}

}  // extern "C"
