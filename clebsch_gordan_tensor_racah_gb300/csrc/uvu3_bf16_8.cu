// uvu3_bf16_8.cu -- instantiation of the warp-autonomous uvu kernels with bfloat16 inputs
// (x, Y, W, output gradient), FP32 arithmetic and FP32 outputs, 8 lanes per edge.
#include <algorithm>

#include "uvu3_impl.cuh"

namespace cgtp {
namespace uvu3_detail {

namespace {
Uvu3Args<float, __nv_bfloat16> v3_args_bf16(const cgtp_plan_s* plan) {
  Uvu3Args<float, __nv_bfloat16> a{};
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
}  // namespace

template <int LPE>
cgtp_status fwd3_launch_bf16(const cgtp_plan_s* plan, const void* x, const void* Y, const void* W, void* out,
                             const int32_t* rowptr, const int32_t* col, int64_t N, cudaStream_t st);
template <int LPE>
cgtp_status bwd3_launch_bf16(const cgtp_plan_s* plan, const void* gout, const void* x, const void* Y,
                             const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                             const int32_t* t_eid, const int32_t* t_dst, int64_t N, cudaStream_t st);

template <>
cgtp_status fwd3_launch_bf16<8>(const cgtp_plan_s* plan, const void* x, const void* Y, const void* W, void* out,
                                const int32_t* rowptr, const int32_t* col, int64_t N, cudaStream_t st) {
  auto a = v3_args_bf16(plan);
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.Y = static_cast<const __nv_bfloat16*>(Y);
  a.W = static_cast<const __nv_bfloat16*>(W);
  a.out = static_cast<float*>(out);
  a.rowptr = rowptr;
  a.col = col;
  a.N = static_cast<int>(N);
  auto k = uvu_forward3_kernel<float, 8, __nv_bfloat16>;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kV3Threads, 0);
  per_sm = std::max(per_sm, 1);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)plan->num_sms * per_sm)));
  k<<<grid, kV3Threads, 0, st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu forward (v3, bf16) launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

template <>
cgtp_status bwd3_launch_bf16<8>(const cgtp_plan_s* plan, const void* gout, const void* x, const void* Y,
                                const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                                const int32_t* t_eid, const int32_t* t_dst, int64_t N, cudaStream_t st) {
  auto a = v3_args_bf16(plan);
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.Y = static_cast<const __nv_bfloat16*>(Y);
  a.W = static_cast<const __nv_bfloat16*>(W);
  a.gout = static_cast<const __nv_bfloat16*>(gout);
  a.gx = static_cast<float*>(gx);
  a.gY = static_cast<float*>(gY);
  a.gW = static_cast<float*>(gW);
  a.rowptr = t_rowptr;
  a.col = t_eid;
  a.t_dst = t_dst;
  a.items = plan->v3.items_bwd;
  a.phase_begin = plan->v3.phase_begin;
  a.n_phases = plan->v3.n_phases;
  a.N = static_cast<int>(N);
  auto k = uvu_backward3_kernel<float, 8, __nv_bfloat16>;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kV3Threads, 0);
  per_sm = std::max(per_sm, 1);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)plan->num_sms * per_sm)));
  k<<<grid, kV3Threads, 0, st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu backward (v3, bf16) launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

}  // namespace uvu3_detail
}  // namespace cgtp
