// uvu3_f32_8.cu -- instantiation of the warp-autonomous uvu kernels for float, 8 lanes per edge.
#include <algorithm>

#include "uvu3_impl.cuh"

namespace cgtp {
namespace uvu3_detail {

template <typename T>
Uvu3Args<T> v3_args(const cgtp_plan_s* plan) {
  Uvu3Args<T> a{};
  const V3Dev& v = plan->v3;
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.paths = v.paths;
  a.items = v.items;
  a.n_items = v.n_items;
  a.gxp_off = v.gxp_off;
  a.gxp_size = v.gxp_size;
  a.in1_off = v.in1_off;
  a.n_in1 = v.n_in1;
  a.gx_begin = v.gx_begin;
  a.gx_paths = v.gx_paths;
  a.chunk_b = v.chunk_b;
  return a;
}

template <typename T, int LPE>
cgtp_status fwd3_launch(const cgtp_plan_s* plan, const void* x, const void* Y, const void* W, void* out,
                        const int32_t* rowptr, const int32_t* col, int64_t N, cudaStream_t st) {
  Uvu3Args<T> a = v3_args<T>(plan);
  a.x = static_cast<const T*>(x);
  a.Y = static_cast<const T*>(Y);
  a.W = static_cast<const T*>(W);
  a.out = static_cast<T*>(out);
  a.rowptr = rowptr;
  a.col = col;
  a.N = static_cast<int>(N);
  auto k = uvu_forward3_kernel<T, LPE>;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kV3Threads, 0);
  per_sm = std::max(per_sm, 1);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)plan->num_sms * per_sm)));
  k<<<grid, kV3Threads, 0, st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu forward (v3) launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

template <typename T, int LPE>
cgtp_status bwd3_launch(const cgtp_plan_s* plan, const void* gout, const void* x, const void* Y,
                        const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                        const int32_t* t_eid, const int32_t* t_dst, int64_t N, cudaStream_t st) {
  Uvu3Args<T> a = v3_args<T>(plan);
  a.x = static_cast<const T*>(x);
  a.Y = static_cast<const T*>(Y);
  a.W = static_cast<const T*>(W);
  a.gout = static_cast<const T*>(gout);
  a.gx = static_cast<T*>(gx);
  a.gY = static_cast<T*>(gY);
  a.gW = static_cast<T*>(gW);
  a.rowptr = t_rowptr;
  a.col = t_eid;
  a.items = plan->v3.items_bwd;
  a.phase_begin = plan->v3.phase_begin;
  a.n_phases = plan->v3.n_phases;
  a.t_dst = t_dst;
  a.N = static_cast<int>(N);
  auto k = uvu_backward3_kernel<T, LPE>;
  const size_t smem = 0;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kV3Threads, smem);
  per_sm = std::max(per_sm, 1);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)plan->num_sms * per_sm)));
  k<<<grid, kV3Threads, smem, st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu backward (v3) launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

template cgtp_status fwd3_launch<float, 8>(const cgtp_plan_s*, const void*, const void*, const void*, void*,
                                            const int32_t*, const int32_t*, int64_t, cudaStream_t);
template cgtp_status bwd3_launch<float, 8>(const cgtp_plan_s*, const void*, const void*, const void*,
                                            const void*, void*, void*, void*, const int32_t*,
                                            const int32_t*, const int32_t*, int64_t, cudaStream_t);

}  // namespace uvu3_detail
}  // namespace cgtp
