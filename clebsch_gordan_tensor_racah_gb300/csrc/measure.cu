// measure.cu -- arithmetic and read-bandwidth kernels that give the roofline its
// measured denominators (declared in include/cgtp_measure.h).
//
// Each thread keeps 16 independent accumulator chains, so a warp always has an
// FMA ready to issue and the kernel measures the pipe's throughput, not its
// latency.  The constants keep every chain bounded (a*b + c with |a| < 1).
#include <cuda_runtime.h>

#include <string>

#include "cgtp_measure.h"
#include "internal.h"

namespace cgtp {
namespace {

constexpr int kMeasureThreads = 256;
constexpr int kChains = 16;

__global__ void __launch_bounds__(kMeasureThreads) ffma_kernel(int iters, float* sink) {
  float acc[kChains];
  const float a = 0.999f, b = 1e-3f * (threadIdx.x & 7);
#pragma unroll
  for (int i = 0; i < kChains; ++i) acc[i] = 1.0f + i;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int i = 0; i < kChains; ++i) acc[i] = fmaf(acc[i], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kChains; ++i) s += acc[i];
  sink[blockIdx.x * kMeasureThreads + threadIdx.x] = s;
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long x, unsigned long long m,
                                                    unsigned long long c) {
  unsigned long long d;
  asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(m), "l"(c));
  return d;
}

__global__ void __launch_bounds__(kMeasureThreads) ffma2_kernel(int iters, float* sink) {
  unsigned long long acc[kChains];
  const float2 a2 = make_float2(0.999f, 0.998f), b2 = make_float2(1e-3f, 2e-3f * (threadIdx.x & 7));
  const unsigned long long a = *reinterpret_cast<const unsigned long long*>(&a2);
  const unsigned long long b = *reinterpret_cast<const unsigned long long*>(&b2);
#pragma unroll
  for (int i = 0; i < kChains; ++i) {
    const float2 v = make_float2(1.0f + i, 2.0f + i);
    acc[i] = *reinterpret_cast<const unsigned long long*>(&v);
  }
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int i = 0; i < kChains; ++i) acc[i] = ffma2(acc[i], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kChains; ++i) {
    const float2 v = *reinterpret_cast<const float2*>(&acc[i]);
    s += v.x + v.y;
  }
  sink[blockIdx.x * kMeasureThreads + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kMeasureThreads) dfma_kernel(int iters, double* sink) {
  double acc[kChains];
  const double a = 0.999, b = 1e-3 * (threadIdx.x & 7);
#pragma unroll
  for (int i = 0; i < kChains; ++i) acc[i] = 1.0 + i;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int i = 0; i < kChains; ++i) acc[i] = fma(acc[i], a, b);
  }
  double s = 0.0;
#pragma unroll
  for (int i = 0; i < kChains; ++i) s += acc[i];
  sink[blockIdx.x * kMeasureThreads + threadIdx.x] = s;
}

// every CTA reads its own contiguous slice `reps` times (16-byte loads, 4 in flight per thread)
__global__ void __launch_bounds__(kMeasureThreads) read_kernel(const uint4* __restrict__ buf, int64_t per_cta,
                                                               int reps, unsigned* sink) {
  const uint4* p = buf + blockIdx.x * per_cta;
  unsigned acc = 0;
  for (int r = 0; r < reps; ++r) {
    for (int64_t i = threadIdx.x; i < per_cta; i += 4 * kMeasureThreads) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t k = i + j * kMeasureThreads;
        v[j] = k < per_cta ? __ldcg(p + k) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
    }
  }
  sink[blockIdx.x * kMeasureThreads + threadIdx.x] = acc;
}

}  // namespace
}  // namespace cgtp

extern "C" cgtp_status cgtp_measure_fma(int kind, int ctas, int iters, void* sink, double* flops, void* stream) {
  using namespace cgtp;
  clear_error();
  if (ctas < 1 || iters < 1) return fail(CGTP_EINVAL, "cgtp_measure_fma: ctas and iters must be >= 1");
  if (!sink) return fail(CGTP_EINVAL, "cgtp_measure_fma: null sink");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const double fma_per_thread = double(iters) * 8 * kChains;
  const double threads = double(ctas) * kMeasureThreads;
  switch (kind) {
    case CGTP_MEASURE_FFMA:
      ffma_kernel<<<ctas, kMeasureThreads, 0, st>>>(iters, static_cast<float*>(sink));
      if (flops) *flops = 2.0 * fma_per_thread * threads;
      break;
    case CGTP_MEASURE_FFMA2:
      ffma2_kernel<<<ctas, kMeasureThreads, 0, st>>>(iters, static_cast<float*>(sink));
      if (flops) *flops = 4.0 * fma_per_thread * threads;
      break;
    case CGTP_MEASURE_DFMA:
      dfma_kernel<<<ctas, kMeasureThreads, 0, st>>>(iters, static_cast<double*>(sink));
      if (flops) *flops = 2.0 * fma_per_thread * threads;
      break;
    default:
      return fail(CGTP_EINVAL, "cgtp_measure_fma: unknown kind");
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CGTP_ECUDA, std::string("cgtp_measure_fma launch: ") + cudaGetErrorString(e));
  return CGTP_OK;
}

extern "C" cgtp_status cgtp_measure_read(const void* buf, int64_t bytes, int reps, int ctas, void* sink,
                                         double* bytes_read, void* stream) {
  using namespace cgtp;
  clear_error();
  if (!buf || !sink) return fail(CGTP_EINVAL, "cgtp_measure_read: null buffer");
  if ((reinterpret_cast<uintptr_t>(buf) & 15u) != 0) return fail(CGTP_EINVAL, "cgtp_measure_read: buf not 16-byte aligned");
  if (ctas < 1 || reps < 1) return fail(CGTP_EINVAL, "cgtp_measure_read: ctas and reps must be >= 1");
  const int64_t quantum = int64_t(16) * kMeasureThreads * ctas;
  if (bytes <= 0 || bytes % quantum != 0)
    return fail(CGTP_EINVAL, "cgtp_measure_read: bytes must be a positive multiple of 4096*ctas");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  read_kernel<<<ctas, kMeasureThreads, 0, st>>>(static_cast<const uint4*>(buf), bytes / 16 / ctas, reps,
                                                static_cast<unsigned*>(sink));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CGTP_ECUDA, std::string("cgtp_measure_read launch: ") + cudaGetErrorString(e));
  if (bytes_read) *bytes_read = double(bytes) * reps;
  return CGTP_OK;
}
