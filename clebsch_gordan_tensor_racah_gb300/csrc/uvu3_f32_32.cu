// uvu3_f32_32.cu -- warp-autonomous uvu kernels, float, 32 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(float, float, false, 32)
