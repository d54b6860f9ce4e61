// uvu3_sh_f64_32.cu -- warp-autonomous uvu kernels, double, fed by edge vectors (harmonics evaluated in the kernel), 32 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(double, double, true, 32)
