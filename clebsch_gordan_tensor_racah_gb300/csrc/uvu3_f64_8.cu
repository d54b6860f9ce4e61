// uvu3_f64_8.cu -- warp-autonomous uvu kernels, double, 8 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(double, double, false, 8)
