// uvu3_f64_2.cu -- warp-autonomous uvu kernels, double, 2 lanes per edge.
#include "uvu3_launch.cuh"

CGTP_V3_INSTANCE(double, double, false, 2)
