// uvu3_f32_8.cu -- warp-autonomous uvu kernels, float, 8 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(float, float, false, 8)
