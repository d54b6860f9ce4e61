// uvu3_sh_f64_2.cu -- warp-autonomous uvu kernels, double, fed by edge vectors (harmonics evaluated in the kernel), 2 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(double, double, true, 2)
