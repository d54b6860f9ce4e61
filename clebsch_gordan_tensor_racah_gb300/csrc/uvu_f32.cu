// uvu_f32.cu -- instantiation of the uvu kernels for float, l <= 3.
#include "uvu_impl.cuh"

namespace cgtp {
namespace uvu_detail {
template cgtp_status fwd_impl<float, false, 3>(const cgtp_plan_s*, const LayoutDev&, const void*,
                                             const void*, const void*, void*, const int32_t*,
                                             const int32_t*, int64_t, cudaStream_t);
template cgtp_status fwd_impl<float, true, 3>(const cgtp_plan_s*, const LayoutDev&, const void*,
                                            const void*, const void*, void*, const int32_t*,
                                            const int32_t*, int64_t, cudaStream_t);
template cgtp_status bwd_impl<float, false, 3>(const cgtp_plan_s*, const LayoutDev&, const void*,
                                             const void*, const void*, const void*, void*, void*,
                                             void*, const int32_t*, const int32_t*,
                                             const int32_t*, int64_t, cudaStream_t);
template cgtp_status bwd_impl<float, true, 3>(const cgtp_plan_s*, const LayoutDev&, const void*,
                                            const void*, const void*, const void*, void*, void*,
                                            void*, const int32_t*, const int32_t*, const int32_t*,
                                            int64_t, cudaStream_t);
}  // namespace uvu_detail
}  // namespace cgtp
