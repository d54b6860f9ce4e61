// uvu3_bf16_32.cu -- warp-autonomous uvu kernels, bfloat16 inputs (x, Y, W, output gradient), FP32 arithmetic and outputs, 32 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(float, __nv_bfloat16, false, 32)
