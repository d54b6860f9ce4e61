// uvu3_launch.cuh -- host launch glue of the warp-autonomous uvu kernels
// (uvu3_impl.cuh), written once for every instance.
//
// An instance is (T, S, SH, LPE): arithmetic/output type, storage type of the
// inputs (T or bfloat16), edge vectors instead of harmonics, lanes per edge.
// Each uvu3_<variant>_<lanes>.cu translation unit only instantiates one of
// them (CGTP_V3_INSTANCE), so the kernels compile in parallel.
#pragma once
#include <algorithm>
#include <string>

#include "uvu3_impl.cuh"

namespace cgtp {
namespace uvu3_detail {

template <typename T, typename S>
Uvu3Args<T, S> v3_args(const cgtp_plan_s* plan) {
  Uvu3Args<T, S> a{};
  const V3Dev& v = plan->v3;
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.paths = v.paths;
  a.items = v.items;
  a.n_items = v.n_items;
  return a;
}

// shared memory for a CTA's edge indices: 16,384 ints (64 KB) in the backward
// (edge ids + receivers), half of it in the forward (sources)
constexpr int kV3IdxInts = 16384;

// persistent grid: every SM holds as many CTAs as fit, never more CTAs than nodes
inline int v3_grid(const void* kernel, int64_t N, int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kV3Threads, kV3IdxInts * sizeof(int)) !=
      cudaSuccess) {
    cudaGetLastError();
    per_sm = 1;
  }
  per_sm = std::max(per_sm, 1);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)num_sms * per_sm)));
}

inline const char* v3_variant_name(bool bf16, bool sh) {
  return sh ? " (edge vectors)" : bf16 ? " (bf16)" : "";
}

// forward: E_in is Y [E, d2] (SH = false) or the edge vectors [E, 3] (SH = true)
template <typename T, typename S, bool SH, int LPE>
cgtp_status v3_forward(const cgtp_plan_s* plan, const void* x, const void* E_in, const void* W, void* out,
                       const int32_t* rowptr, const int32_t* col, int64_t N, cudaStream_t st) {
  Uvu3Args<T, S> a = v3_args<T, S>(plan);
  a.x = static_cast<const S*>(x);
  if constexpr (SH) a.rvec = static_cast<const T*>(E_in);
  else a.Y = static_cast<const S*>(E_in);
  a.W = static_cast<const S*>(W);
  a.out = static_cast<T*>(out);
  a.rowptr = rowptr;
  a.col = col;
  a.N = static_cast<int>(N);
  auto k = uvu_forward3_kernel<T, LPE, S, SH>;
  a.idx_cap = kV3IdxInts / 2;  // the forward stages col only
  k<<<v3_grid(reinterpret_cast<const void*>(k), N, plan->num_sms), kV3Threads, a.idx_cap * sizeof(int), st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess)
    return fail(CGTP_ECUDA, std::string("uvu forward (v3") + v3_variant_name(sizeof(S) == 2, SH) +
                                ") launch: " + cudaGetErrorString(err));
  return CGTP_OK;
}

template <typename T, typename S, bool SH, int LPE>
cgtp_status v3_backward(const cgtp_plan_s* plan, const void* gout, const void* x, const void* E_in,
                        const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                        const int32_t* t_eid, const int32_t* t_dst, int64_t N, cudaStream_t st) {
  Uvu3Args<T, S> a = v3_args<T, S>(plan);
  a.x = static_cast<const S*>(x);
  if constexpr (SH) a.rvec = static_cast<const T*>(E_in);
  else a.Y = static_cast<const S*>(E_in);
  a.W = static_cast<const S*>(W);
  a.gout = static_cast<const S*>(gout);
  a.gx = static_cast<T*>(gx);
  a.gY = static_cast<T*>(gY);
  a.gW = static_cast<T*>(gW);
  a.rowptr = t_rowptr;
  a.col = t_eid;
  a.t_dst = t_dst;
  a.items = plan->v3.items_bwd;
  a.phase_begin = plan->v3.phase_begin;
  a.n_phases = plan->v3.n_phases;
  a.N = static_cast<int>(N);
  auto k = uvu_backward3_kernel<T, LPE, S, SH>;
  a.idx_cap = smem_cap_cached(reinterpret_cast<const void*>(k)) >= int(kV3IdxInts * sizeof(int)) ? kV3IdxInts : 0;
  k<<<v3_grid(reinterpret_cast<const void*>(k), N, plan->num_sms), kV3Threads, a.idx_cap * sizeof(int), st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess)
    return fail(CGTP_ECUDA, std::string("uvu backward (v3") + v3_variant_name(sizeof(S) == 2, SH) +
                                ") launch: " + cudaGetErrorString(err));
  return CGTP_OK;
}

}  // namespace uvu3_detail
}  // namespace cgtp

// One instance per translation unit.
#define CGTP_V3_INSTANCE(T, S, SH, LPE)                                                                   \
  namespace cgtp {                                                                                        \
  namespace uvu3_detail {                                                                                 \
  template cgtp_status v3_forward<T, S, SH, LPE>(const cgtp_plan_s*, const void*, const void*,            \
                                                 const void*, void*, const int32_t*, const int32_t*,      \
                                                 int64_t, cudaStream_t);                                  \
  template cgtp_status v3_backward<T, S, SH, LPE>(const cgtp_plan_s*, const void*, const void*,           \
                                                  const void*, const void*, void*, void*, void*,          \
                                                  const int32_t*, const int32_t*, const int32_t*, int64_t, \
                                                  cudaStream_t);                                          \
  }                                                                                                       \
  }
