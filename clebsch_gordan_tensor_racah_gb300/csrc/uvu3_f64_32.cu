// uvu3_f64_32.cu -- warp-autonomous uvu kernels, double, 32 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(double, double, false, 32)
