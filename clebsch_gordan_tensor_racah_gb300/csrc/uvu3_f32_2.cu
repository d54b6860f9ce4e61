// uvu3_f32_2.cu -- warp-autonomous uvu kernels, float, 2 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(float, float, false, 2)
