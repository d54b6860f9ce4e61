// uvu.cu -- host launchers of the uvu kernels (templates in uvu_impl.cuh,
// instantiated in uvu_f32.cu, uvu_f32_l7.cu, uvu_f64.cu, uvu_f64_l7.cu).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>

#include "internal.h"

namespace cgtp {
namespace uvu_detail {
template <typename T, bool IDENT, int LMAX>
cgtp_status fwd_impl(const cgtp_plan_s* plan, const LayoutDev& lay, const void* x, const void* Y,
                     const void* W, void* out, const int32_t* rowptr, const int32_t* col, int64_t N,
                     cudaStream_t st);
template <typename T, bool IDENT, int LMAX>
cgtp_status bwd_impl(const cgtp_plan_s* plan, const LayoutDev& lay, const void* gout,
                     const void* x, const void* Y, const void* W, void* gx, void* gY, void* gW,
                     const int32_t* t_rowptr, const int32_t* t_eid, const int32_t* t_dst,
                     int64_t N, cudaStream_t st);
}  // namespace uvu_detail
namespace uvu2_detail {
template <typename T>
cgtp_status fwd2_impl(const cgtp_plan_s* plan, const LayoutDev& lay, const void* x, const void* Y,
                      const void* W, void* out, const int32_t* rowptr, const int32_t* col, int64_t N,
                      cudaStream_t st);
}  // namespace uvu2_detail
using uvu_detail::fwd_impl;
using uvu_detail::bwd_impl;

static int plan_lmax(const cgtp_plan_s* plan) {
  int l = 0;
  for (const auto& p : plan->paths) l = std::max(l, std::max(p.l1, p.l3));
  return l;
}

cgtp_status launch_uvu_forward(const cgtp_plan_s* plan, const LayoutDev& lay, const void* x,
                               const void* Y, const void* W, void* out, const int32_t* rowptr,
                               const int32_t* col, int64_t N, bool identity, void* stream) {
  if (N == 0) return CGTP_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool small = plan_lmax(plan) <= 3;
  if (!identity) {
    cgtp_status st3 = CGTP_OK;
    if (launch_v3_forward(plan, x, Y, W, out, rowptr, col, N, stream, &st3)) return st3;
  }
  if (plan->dtype == CGTP_BF16)  // only the v3 kernels take bfloat16 inputs
    return fail(CGTP_EUNSUPPORTED, "CGTP_BF16 graph convolutions need l <= 3 and one in1 multiplicity m "
                                   "with m/4 in {2, 8, 32} or m a multiple of 128");
  // graph convolutions with l <= 3 take the pipelined kernel
  if (!identity && small && lay.chunk2 > 0) {
    if (plan->dtype == CGTP_F64) return uvu2_detail::fwd2_impl<double>(plan, lay, x, Y, W, out, rowptr, col, N, st);
    return uvu2_detail::fwd2_impl<float>(plan, lay, x, Y, W, out, rowptr, col, N, st);
  }
#define CGTP_FWD_DISPATCH(T)                                                                         \
  if (identity)                                                                                      \
    return small ? fwd_impl<T, true, 3>(plan, lay, x, Y, W, out, rowptr, col, N, st)                 \
                 : fwd_impl<T, true, 7>(plan, lay, x, Y, W, out, rowptr, col, N, st);                \
  return small ? fwd_impl<T, false, 3>(plan, lay, x, Y, W, out, rowptr, col, N, st)                  \
               : fwd_impl<T, false, 7>(plan, lay, x, Y, W, out, rowptr, col, N, st);
  if (plan->dtype == CGTP_F64) {
    CGTP_FWD_DISPATCH(double)
  }
  CGTP_FWD_DISPATCH(float)
#undef CGTP_FWD_DISPATCH
}

cgtp_status launch_uvu_backward(const cgtp_plan_s* plan, const LayoutDev& lay, const void* gout,
                                const void* x, const void* Y, const void* W, void* gx, void* gY,
                                void* gW, const int32_t* t_rowptr, const int32_t* t_eid,
                                const int32_t* t_dst, int64_t N, bool identity, void* stream) {
  if (N == 0) return CGTP_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool small = plan_lmax(plan) <= 3;
  if (!identity) {
    cgtp_status st3 = CGTP_OK;
    if (launch_v3_backward(plan, gout, x, Y, W, gx, gY, gW, t_rowptr, t_eid, t_dst, N, stream, &st3))
      return st3;
  }
  if (plan->dtype == CGTP_BF16)  // only the v3 kernels take bfloat16 inputs
    return fail(CGTP_EUNSUPPORTED, "CGTP_BF16 graph convolutions need l <= 3 and one in1 multiplicity m "
                                   "with m/4 in {2, 8, 32} or m a multiple of 128");
#define CGTP_BWD_DISPATCH(T)                                                                            \
  if (identity)                                                                                         \
    return small ? bwd_impl<T, true, 3>(plan, lay, gout, x, Y, W, gx, gY, gW, t_rowptr, t_eid, t_dst, N, st) \
                 : bwd_impl<T, true, 7>(plan, lay, gout, x, Y, W, gx, gY, gW, t_rowptr, t_eid, t_dst, N, st); \
  return small ? bwd_impl<T, false, 3>(plan, lay, gout, x, Y, W, gx, gY, gW, t_rowptr, t_eid, t_dst, N, st)  \
               : bwd_impl<T, false, 7>(plan, lay, gout, x, Y, W, gx, gY, gW, t_rowptr, t_eid, t_dst, N, st);
  if (plan->dtype == CGTP_F64) {
    CGTP_BWD_DISPATCH(double)
  }
  CGTP_BWD_DISPATCH(float)
#undef CGTP_BWD_DISPATCH
}

}  // namespace cgtp
