// uvu3_sh_f32_8.cu -- warp-autonomous uvu kernels, float, fed by edge vectors (harmonics evaluated in the kernel), 8 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(float, float, true, 8)
