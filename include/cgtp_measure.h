/*
 * cgtp_measure.h -- measurement kernels of libcgtp (not part of the operation).
 *
 * The roofline of the convolution kernels needs the chip's arithmetic and
 * cache peaks as measured on the part at hand, not a unit-count formula
 * ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep
 * Networks", Abstract, reports its kernels against the GPU's own throughput).
 * These entry points only ENQUEUE one launch on `stream`; the caller times it
 * with events on the same stream.  Pointers are DEVICE pointers on the
 * current device; errors come back as a status plus cgtp_last_error().
 */
#ifndef CGTP_MEASURE_H
#define CGTP_MEASURE_H

#include <stdint.h>

#include "cgtp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Kinds of arithmetic throughput kernels. */
enum {
  CGTP_MEASURE_FFMA = 0,    /* FP32 fused multiply-add, one value per instruction */
  CGTP_MEASURE_FFMA2 = 1,   /* FP32 paired fused multiply-add (fma.rn.f32x2) */
  CGTP_MEASURE_DFMA = 2     /* FP64 fused multiply-add */
};

/*
 * cgtp_measure_fma -- launches a grid of `ctas` CTAs x 256 threads; every
 *  thread runs `iters` rounds of 16 independent FMA chains (FFMA2: 16 paired
 *  chains).  *flops receives the floating-point operations of the launch (an
 *  FMA counts 2).  sink: device buffer of at least ctas*256*8 bytes (each
 *  thread stores its chain sum so nothing is optimised away); its contents
 *  are meaningless.  CGTP_EINVAL for an unknown kind, ctas < 1 or iters < 1.
 */
cgtp_status cgtp_measure_fma(int kind, int ctas, int iters, void* sink, double* flops, void* stream);

/*
 * cgtp_measure_read -- launches a grid of `ctas` CTAs x 256 threads that read
 *  the device buffer buf [bytes] `reps` times with 16-byte loads, each CTA
 *  walking its own contiguous slice (a buffer below the L2 size measures L2
 *  bandwidth after the first pass; one far above it measures HBM).  *bytes_read
 *  receives bytes*reps.  buf 16-byte aligned, bytes a positive multiple of
 *  16*256*ctas; sink as above (ctas*256*4 bytes).  CGTP_EINVAL otherwise.
 */
cgtp_status cgtp_measure_read(const void* buf, int64_t bytes, int reps, int ctas, void* sink,
                              double* bytes_read, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CGTP_MEASURE_H */
