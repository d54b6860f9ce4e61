// uvu3_sh_f32_32.cu -- warp-autonomous uvu kernels, float, fed by edge vectors (harmonics evaluated in the kernel), 32 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(float, float, true, 32)
