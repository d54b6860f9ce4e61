// uvu2.cu -- launchers of the pipelined uvu kernels (uvu2_impl.cuh), l <= 3.
#include <cuda_runtime.h>

#include <algorithm>

#include "uvu2_impl.cuh"

namespace cgtp {
namespace uvu2_detail {

template <typename T>
cgtp_status fwd2_impl(const cgtp_plan_s* plan, const LayoutDev& lay, const void* x, const void* Y,
                      const void* W, void* out, const int32_t* rowptr, const int32_t* col, int64_t N,
                      cudaStream_t st) {
  constexpr int VN = 16 / sizeof(T);
  Fwd2Args<T> a{};
  a.x = static_cast<const T*>(x);
  a.Y = static_cast<const T*>(Y);
  a.W = static_cast<const T*>(W);
  a.out = static_cast<T*>(out);
  a.rowptr = rowptr;
  a.col = col;
  a.N = static_cast<int>(N);
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.chunk = lay.chunk2;
  int wg = 0;
  bool wal = (a.w_numel * sizeof(T)) % 16 == 0;
  for (const auto& g : lay.groups_host) {
    wg = std::max(wg, g.w1 - g.w0);
    wal = wal && ((g.w0 * sizeof(T)) % 16 == 0) && (((g.w1 - g.w0) * sizeof(T)) % 16 == 0);
  }
  a.d1p = pad_up(a.d1, VN);
  a.d2p = pad_up(a.d2, VN);
  a.wgp = pad_up(wg, VN);
  a.vec_x = (a.d1 * sizeof(T)) % 16 == 0;
  a.vec_w = wal;
  a.vec_y = (a.d2 * sizeof(T)) % 16 == 0;
  a.n_groups = lay.n_groups;
  a.paths = lay.paths;
  a.groups = lay.groups;
  a.cy2_col = lay.cy2_col;
  a.cy2_coef = static_cast<const T*>(lay.cy2_coef);
  a.cy2_base = lay.cy2_base;
  a.item_begin = lay.item_begin;
  a.items = lay.items;
  auto k = uvu_forward2_kernel<T, 3>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.smem_fwd2) != cudaSuccess)
    return fail(CGTP_ECUDA, "uvu forward (pipelined): shared memory attribute rejected");
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, lay.smem_fwd2);
  per_sm = std::max(per_sm, 1);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(N, (int64_t)plan->num_sms * per_sm)));
  k<<<grid, kThreads, lay.smem_fwd2, st>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu forward (pipelined) launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

template cgtp_status fwd2_impl<float>(const cgtp_plan_s*, const LayoutDev&, const void*, const void*,
                                      const void*, void*, const int32_t*, const int32_t*, int64_t, cudaStream_t);
template cgtp_status fwd2_impl<double>(const cgtp_plan_s*, const LayoutDev&, const void*, const void*,
                                       const void*, void*, const int32_t*, const int32_t*, int64_t, cudaStream_t);

}  // namespace uvu2_detail
}  // namespace cgtp
