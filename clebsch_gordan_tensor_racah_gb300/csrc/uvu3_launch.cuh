// uvu3_launch.cuh -- host launch glue of the warp-autonomous uvu kernels
// (uvu3_impl.cuh, and their staged form uvu4_impl.cuh when the plan's copies
// are 16-byte aligned), written once for every instance.
//
// An instance is (T, S, SH, LPE): arithmetic/output type, storage type of the
// inputs (T or bfloat16), edge vectors instead of harmonics, lanes per edge.
// Each uvu3_<variant>_<lanes>.cu translation unit only instantiates one of
// them (CGTP_V3_INSTANCE), so the kernels compile in parallel.
#pragma once
#include <algorithm>
#include <cstdio>
#include <string>

#include "uvu3_impl.cuh"
#include "uvu4_impl.cuh"

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

// persistent grid: every SM holds as many CTAs as fit, never more CTAs than nodes
inline int v3_grid(const void* kernel, int64_t N, int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kV3Threads, 0) != cudaSuccess) {
    cudaGetLastError();
    per_sm = 1;
  }
  per_sm = std::max(per_sm, 1);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)num_sms * per_sm)));
}

inline const char* v3_variant_name(bool bf16, bool sh) {
  return sh ? " (edge vectors)" : bf16 ? " (bf16)" : "";
}

// Staged (v4) launch: dynamic shared memory = 8 rings; the kernel's limit is
// raised to the device cap once per device.
template <typename T, typename S>
uvu4_detail::Uvu4Args<T, S> v4_args(const cgtp_plan_s* plan, const Uvu3Args<T, S>& b, const V4Ring& r) {
  uvu4_detail::Uvu4Args<T, S> a{};
  a.b = b;
  a.r = r;
  a.ublock = 4 * plan->v3.lpe;
  a.err = plan->v3.err_dev;
  a.wait_limit = plan->v3.wait_limit;
  return a;
}

template <typename K>
bool v4_ready(K kernel, size_t smem) {
  return smem_cap_cached(reinterpret_cast<const void*>(kernel)) >= static_cast<int>(smem);
}

inline cgtp_status v4_sticky(const cgtp_plan_s* plan) {
  const volatile int* e = plan->v3.err_host;
  if (e && e[0]) {
    char buf[256];
    snprintf(buf, sizeof buf,
             "a staging wait of an earlier call on this plan gave up (results of that call are invalid): "
             "block %d warp %d stage %d of %d fetched, slot %d parity %d, barrier %08x%08x, stage (%d,%d,%d,%d)",
             e[1] - 1, e[2], e[3], e[4], e[5], e[6], (unsigned)e[8], (unsigned)e[7], e[9], e[10], e[11], e[12]);
    return fail(CGTP_ECUDA, buf);
  }
  return CGTP_OK;
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
  const V4Ring& r4 = plan->v3.v4_fwd[SH ? 1 : 0];
  if (r4.S > 0) {
    if (cgtp_status e = v4_sticky(plan)) return e;
    auto k4 = uvu4_detail::uvu_forward4_kernel<T, LPE, S, SH>;
    const size_t smem = size_t(uvu4_detail::kV4Warps) * r4.warp_bytes;
    if (v4_ready(k4, smem)) {
      const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, plan->num_sms)));
      k4<<<grid, uvu4_detail::kV4Threads, smem, st>>>(v4_args(plan, a, r4));
      const cudaError_t err = cudaGetLastError();
      if (err != cudaSuccess)
        return fail(CGTP_ECUDA, std::string("uvu forward (v4") + v3_variant_name(sizeof(S) == 2, SH) +
                                    ") launch: " + cudaGetErrorString(err));
      return CGTP_OK;
    }
  }
  auto k = uvu_forward3_kernel<T, LPE, S, SH>;
  k<<<v3_grid(reinterpret_cast<const void*>(k), N, plan->num_sms), kV3Threads, 0, st>>>(a);
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
  const V4Ring& r4 = plan->v3.v4_bwd[SH ? 1 : 0];
  if (r4.S > 0) {
    if (cgtp_status e = v4_sticky(plan)) return e;
    auto k4 = uvu4_detail::uvu_backward4_kernel<T, LPE, S, SH>;
    const size_t smem = size_t(uvu4_detail::kV4Warps) * r4.warp_bytes;
    if (v4_ready(k4, smem)) {
      const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, plan->num_sms)));
      k4<<<grid, uvu4_detail::kV4Threads, smem, st>>>(v4_args(plan, a, r4));
      const cudaError_t err = cudaGetLastError();
      if (err != cudaSuccess)
        return fail(CGTP_ECUDA, std::string("uvu backward (v4") + v3_variant_name(sizeof(S) == 2, SH) +
                                    ") launch: " + cudaGetErrorString(err));
      return CGTP_OK;
    }
  }
  auto k = uvu_backward3_kernel<T, LPE, S, SH>;
  k<<<v3_grid(reinterpret_cast<const void*>(k), N, plan->num_sms), kV3Threads, 0, st>>>(a);
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
