// uvu3_sh_f64_8.cu -- the warp-autonomous uvu kernels fed by edge vectors (harmonics
// evaluated in the kernel), double, 8 lanes per edge.
#include <algorithm>

#include "uvu3_impl.cuh"

namespace cgtp {
namespace uvu3_detail {

namespace {
Uvu3Args<double> v3_args_sh(const cgtp_plan_s* plan, const void* rvec) {
  Uvu3Args<double> a{};
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.paths = plan->v3.paths;
  a.items = plan->v3.items;
  a.n_items = plan->v3.n_items;
  a.rvec = static_cast<const double*>(rvec);
  return a;
}
int grid_for(const void* k, int64_t N, int num_sms) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kV3Threads, 0);
  per_sm = std::max(per_sm, 1);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)num_sms * per_sm)));
}
}  // namespace

template <typename T, int LPE>
cgtp_status fwd3_launch_sh(const cgtp_plan_s* plan, const void* x, const void* rvec, const void* W, void* out,
                           const int32_t* rowptr, const int32_t* col, int64_t N, cudaStream_t st);
template <typename T, int LPE>
cgtp_status bwd3_launch_sh(const cgtp_plan_s* plan, const void* gout, const void* x, const void* rvec,
                           const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                           const int32_t* t_eid, const int32_t* t_dst, int64_t N, cudaStream_t st);

template <>
cgtp_status fwd3_launch_sh<double, 8>(const cgtp_plan_s* plan, const void* x, const void* rvec, const void* W,
                                   void* out, const int32_t* rowptr, const int32_t* col, int64_t N,
                                   cudaStream_t st) {
  auto a = v3_args_sh(plan, rvec);
  a.x = static_cast<const double*>(x);
  a.W = static_cast<const double*>(W);
  a.out = static_cast<double*>(out);
  a.rowptr = rowptr;
  a.col = col;
  a.N = static_cast<int>(N);
  auto k = uvu_forward3_kernel<double, 8, double, true>;
  k<<<grid_for(reinterpret_cast<const void*>(k), N, plan->num_sms), kV3Threads, 0, st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu forward (edge vectors) launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

template <>
cgtp_status bwd3_launch_sh<double, 8>(const cgtp_plan_s* plan, const void* gout, const void* x, const void* rvec,
                                   const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                                   const int32_t* t_eid, const int32_t* t_dst, int64_t N, cudaStream_t st) {
  auto a = v3_args_sh(plan, rvec);
  a.x = static_cast<const double*>(x);
  a.W = static_cast<const double*>(W);
  a.gout = static_cast<const double*>(gout);
  a.gx = static_cast<double*>(gx);
  a.gY = static_cast<double*>(gY);
  a.gW = static_cast<double*>(gW);
  a.rowptr = t_rowptr;
  a.col = t_eid;
  a.t_dst = t_dst;
  a.items = plan->v3.items_bwd;
  a.phase_begin = plan->v3.phase_begin;
  a.n_phases = plan->v3.n_phases;
  a.N = static_cast<int>(N);
  auto k = uvu_backward3_kernel<double, 8, double, true>;
  k<<<grid_for(reinterpret_cast<const void*>(k), N, plan->num_sms), kV3Threads, 0, st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu backward (edge vectors) launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

}  // namespace uvu3_detail
}  // namespace cgtp
