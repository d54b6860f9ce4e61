/*
 * cgtp.h -- C ABI of the GB300 fused Clebsch-Gordan tensor-product convolution.
 *
 * The operation (from "An Efficient Sparse Kernel Generator for O(3)-Equivariant
 * Deep Networks", Figure 1 and Figure 4B; "Sobek: Streaming Equivariant Tensor
 * Product Convolutions", Abstract):
 *
 *   message(e)[path, u, m3] = W[e][path, u] * sum_{m1,m2} C[m1,m2,m3] x[src e][u,m1] Y[e][m2]
 *   out[n] = sum over the in-edges e of receiver n of message(e)            (uvu)
 *
 *   uvw with radial weights: W_e[path,u,w] = sum_k R[e,k] M[k,path,u,w] (never formed)
 *   out[n][i_out][w, m3] = sum_e sum_path sum_u W_e[path,u,w] sum C x[src][u,m1] Y[e][m2]
 *
 * C is the real-basis, component-normalised Clebsch-Gordan block of (l1,l2,l3),
 * computed by the planner from Racah's closed form.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Feature layout is multiplicity-major: inside irreps block i the element
 *    (u, m) of a row sits at offset_i + u*(2l+1) + (m+l).  Rows are contiguous,
 *    row-major, element type float (CGTP_F32) or double (CGTP_F64).
 *  - Tensor arguments are DEVICE pointers on the current CUDA device, aligned
 *    to 16 bytes; the caller owns them.  Outputs are overwritten, never
 *    accumulated; inputs are never modified.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Compute entry
 *    points are asynchronous: they enqueue kernels and return.
 *  - Arguments are validated on the host before anything is launched; a
 *    failed check returns a status and launches nothing.  cgtp_last_error()
 *    returns a message for the last failure of the calling thread.
 *  - Results are bitwise deterministic run to run: where a backward reduction
 *    uses floating-point atomic additions (gx, gY of the uvu kernels; gR, gY
 *    of the radial uvw edge stage), each element receives at most one
 *    addition between two block barriers, so the order of additions is fixed.
 *  - A plan holds device state used by its launches (work counters of the
 *    batched kernels, the uvw node-state scratch): calls that use the same
 *    plan must not overlap on the GPU (issue them on one stream).
 */
#ifndef CGTP_H
#define CGTP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cgtp_plan_s* cgtp_plan;
typedef struct cgtp_graph_s* cgtp_graph;

typedef enum {
  CGTP_OK = 0,
  CGTP_EINVAL = 1,        /* bad argument: null pointer, bad string, size mismatch, misalignment */
  CGTP_EUNSUPPORTED = 2,  /* valid request outside what this library implements */
  CGTP_ENOMEM = 3,        /* device allocation failed (plan or graph creation only) */
  CGTP_ECUDA = 4,         /* a CUDA call or kernel launch failed */
  CGTP_EGRAPH = 5         /* the CSR arrays are not a valid receiver-sorted edge list */
} cgtp_status;

typedef enum { CGTP_UVU = 0, CGTP_UVW = 1 } cgtp_mode;
/* CGTP_BF16: inputs x, Y, W and the output gradient stored as bfloat16; arithmetic
 * and every output (out, gx, gY, gW) in FP32. */
typedef enum { CGTP_F32 = 0, CGTP_F64 = 1, CGTP_BF16 = 2 } cgtp_dtype;

/* One path: in1 block i_in1 (x) in2 block i_in2 -> output irrep irreps_out[i_out]. */
typedef struct { int i_in1, i_in2, i_out; } cgtp_instr;

/*
 * cgtp_plan_create -- parse irreps, enumerate paths, compute the CG blocks and
 * upload the per-plan tables.  ("An Efficient Sparse Kernel Generator ...",
 * Abstract: static analysis at model compile time; Figures 1-2: the
 * block-sparse coefficient tensor.)
 *
 *  irreps_in1, irreps_in2, irreps_out : strings "MULxLP+..." (P = e|o, l <= 7).
 *      in2 blocks must have multiplicity 1 (spherical-harmonic edge features).
 *  instr, n_instr : explicit paths, or NULL/0 for every path allowed by the
 *      triangle and parity rules whose (l3, p3) occurs in irreps_out, ordered
 *      i_in1, then i_in2, then l3 ascending.
 *  mode : CGTP_UVU (weights [paths, mul1] per edge; each path writes its own
 *      output block of multiplicity mul1, appended in path order -- the muls of
 *      irreps_out are ignored) or CGTP_UVW (fully connected mixing into the
 *      blocks of irreps_out).
 *  dtype : CGTP_F32, CGTP_F64 or CGTP_BF16 (CGTP_UVW with radial_k > 0 supports
 *      CGTP_F32 only; with radial_k = 0, all three).
 *      CGTP_BF16 (bfloat16 inputs, FP32 arithmetic and outputs; the pages'
 *      lower-precision future work) serves graph convolutions whose plan has
 *      l <= 3 and one in1 multiplicity m with m/4 in {2, 8, 32} or m a multiple
 *      of 128, batched products (cgtp_forward / cgtp_backward) whose paths
 *      all have multiplicity 16 or 32 and l <= 7, and uvw with per-edge
 *      weights (radial_k = 0); a uvu plan that neither kernel family serves
 *      is CGTP_EUNSUPPORTED, and so is each entry point outside what its plan
 *      serves, and the double backward.
 *  radial_k : 0 for uvu.  For uvw, 0 selects one weight matrix per edge,
 *      W [E, sum_path mul1*mul_out] with each path's block laid out [u][w]
 *      (FP32 or FP64, l <= 3; "An Efficient Sparse Kernel Generator ...",
 *      Figure 3B/C), or the number K of radial functions (1..8), the weights
 *      then being W_e = R[e,:] @ M with M [K, sum_path mul1*mul_out].
 * Creates device tables (a few KB) and, for uvw, the bounded scratch used by
 * the streaming node stage: node state for a chunk of nodes (default 128 per
 * SM, 19,456 on a 152-SM GPU; cgtp_plan_set_node_chunk changes it),
 * 2 x chunk x K x sum_path mul*(2l+1) floats (2.8 GB for 64x(0e,1o,2e), K = 8
 * at the default chunk on 152 SMs).  uvw
 * limits: l <= 3, K <= 8.  Must be called with the target device current.
 */
cgtp_status cgtp_plan_create(cgtp_plan* plan, const char* irreps_in1, const char* irreps_in2,
                             const char* irreps_out, const cgtp_instr* instr, int n_instr,
                             int mode, int dtype, int radial_k);
void cgtp_plan_destroy(cgtp_plan plan);

/* Sizes of one row: d1 = dim(in1), d2 = dim(in2), d_out = dim(out), w_numel =
 * weights of one edge (uvu) or of one radial row of M (uvw). Any pointer may be NULL. */
cgtp_status cgtp_plan_info(cgtp_plan plan, int64_t* d1, int64_t* d2, int64_t* d_out,
                           int64_t* w_numel, int* n_paths);

/* Host copy of path `p`: ints[0..9] = l1, l2, l3, mul1, mul_out, off1, off2, ooff,
 * woff, i_out and the dense real CG block C[m1][m2][m3] (FP64) of
 * (2l1+1)(2l2+1)(2l3+1) entries into `block` (capacity in doubles). */
cgtp_status cgtp_plan_path(cgtp_plan plan, int p, int* ints10, double* block, int64_t capacity);

/*
 * cgtp_forward -- batched tensor product without a graph ("An Efficient Sparse
 * Kernel Generator ...", Figure 4A): out[b] = TP(x1[b], x2[b]; W[b]).
 *  x1 [B, d1], x2 [B, d2], W [B, w_numel] -> out [B, d_out].  uvu plans only.
 *  CGTP_BF16 plans: x1, x2, W (and gout below) bfloat16, outputs FP32.
 */
cgtp_status cgtp_forward(cgtp_plan plan, const void* x1, const void* x2, const void* W, void* out,
                         int64_t B, void* stream);

/* Adjoint of cgtp_forward: gout [B, d_out] -> gx1 [B,d1], gx2 [B,d2], gW [B,w_numel]. */
cgtp_status cgtp_backward(cgtp_plan plan, const void* gout, const void* x1, const void* x2,
                          const void* W, void* gx1, void* gx2, void* gW, int64_t B, void* stream);

/*
 * cgtp_graph_create -- validate a receiver-sorted CSR edge list and build the
 * sender transpose on the device ("An Efficient Sparse Kernel Generator ...",
 * Figure 4B: messages are summed into the receiving node).
 *  rowptr [N+1], col [E] : DEVICE int32 arrays; rowptr monotone, rowptr[0]=0,
 *      rowptr[N]=E, 0 <= col < N.  Self-loops and repeated edges are allowed.
 *  The graph keeps the two pointers (the caller must keep them alive and
 *  unchanged while the graph is used) and owns t_rowptr [N+1], t_eid [E]
 *  (CSR positions ordered by sender, ties in CSR order) and t_dst [E].
 *  Synchronises `stream` once to read the validation result.  Limits:
 *  N, E < 2^31; a sender may have at most 32768 out-edges (CGTP_EUNSUPPORTED).
 */
cgtp_status cgtp_graph_create(cgtp_graph* graph, const int32_t* rowptr, const int32_t* col,
                              int64_t N, int64_t E, void* stream);
void cgtp_graph_destroy(cgtp_graph graph);

/*
 * Device memory the library holds for a plan (constant tables, work counters,
 * the uvw node-state scratch and gM partials) or a graph (the transpose
 * arrays), in bytes.  Callers' tensors are not included.  Memory accounting
 * in the spirit of the allocated-memory checks of "The GPU memory
 * optimization with Larger angular momentum" and the peak-memory figures of
 * "Sobek ...", Abstract.  CGTP_EINVAL for a null argument.
 */
cgtp_status cgtp_plan_device_bytes(cgtp_plan plan, int64_t* bytes);
cgtp_status cgtp_graph_device_bytes(cgtp_graph graph, int64_t* bytes);

/*
 * cgtp_plan_set_wait_limit -- polls of an mbarrier before a wait of the
 *  plan's kernels gives up (default 4,194,304).  The uvw node GEMM runs on
 *  the tensor cores (tcgen05.mma, "An Efficient Sparse Kernel Generator ...",
 *  Figure 3B/C: the multiplicity-mixing matrix product) and waits on mbarriers
 *  for their completion; no wait is unbounded.  A wait that gives up records
 *  the failure in the plan's error word, lets the work in flight finish
 *  (bounded), frees its tensor memory and leaves the kernel; that call's
 *  results are invalid and every later call on the plan returns CGTP_ECUDA.
 *  0 makes the first wait give up at once (fault injection for tests: the GPU
 *  stays usable).  CGTP_EINVAL for a null plan or polls < 0.
 */
cgtp_status cgtp_plan_set_wait_limit(cgtp_plan plan, int64_t polls);

/*
 * Node chunk of a uvw plan with radial weights (radial_k > 0).  Its node state
 * ("Sobek ...", Abstract: bounded receiver-side state) is streamed through a
 * plan-owned scratch of 2 * nodes * K * sum_path(mul * (2l+1)) floats: the
 * forward and the backward walk the graph `nodes` receivers (senders) at a
 * time.  cgtp_plan_set_node_chunk replaces the scratch (it waits for work still
 * using the old one); nodes in [1, 1048576] with nodes * K * sum_path(mul *
 * (2l+1)) below 2^31 (one chunk's state is addressed with 32-bit offsets),
 * default 128 x the SM count (halved at plan creation until that bound
 * holds).  CGTP_EINVAL
 * for other plans or sizes, CGTP_ENOMEM when the scratch cannot be allocated.
 * cgtp_plan_node_chunk reports the chunk (0 for plans without node state).
 */
cgtp_status cgtp_plan_set_node_chunk(cgtp_plan plan, int64_t nodes);
cgtp_status cgtp_plan_node_chunk(cgtp_plan plan, int64_t* nodes);

/* Device-to-device copy of the transpose arrays (any pointer may be NULL). */
cgtp_status cgtp_graph_transpose(cgtp_graph graph, int32_t* t_rowptr, int32_t* t_eid,
                                 int32_t* t_dst, void* stream);

/*
 * cgtp_graph_transpose_noalloc -- the sender transpose of cgtp_graph_create,
 * built without allocating any device memory.  The paper has no counterpart.
 *
 *  For callers that may not call cudaMalloc where they need the transpose
 *  (their framework hands out all device memory from its own pool, they run
 *  under a device-memory budget fixed at start-up, or they cannot accept the
 *  device-wide synchronisation an allocation can cause).
 *  rowptr [N+1], col [E] : DEVICE int32 CSR, as for cgtp_graph_create.
 *  t_rowptr [N+1], t_eid [E], t_dst [E] : DEVICE int32 outputs owned by the
 *      caller, filled exactly as cgtp_graph_transpose would fill them.
 *  Working memory is a fixed ~4 MiB array inside the library that every GPU
 *  which loads the library keeps until the process exits; N above 1,048,576
 *  is rejected with CGTP_EINVAL.  The first call on a device looks up that
 *  array's device address (with the device current) and keeps it for the
 *  life of the process; make that first call before any stream capture, and
 *  do not call this function on a device after cudaDeviceReset.  All calls on
 *  a device share the one array and clear it before use: calls whose work
 *  overlaps on the GPU (different streams or threads, same device) race and
 *  must be serialised by the caller.  Every call synchronises `stream` twice
 *  and copies two status flags into host memory (validation, long segments).
 *  Errors as cgtp_graph_create; a refused launch is CGTP_ECUDA.
 */
cgtp_status cgtp_graph_transpose_noalloc(const int32_t* rowptr, const int32_t* col, int64_t N,
                                         int64_t E, int32_t* t_rowptr, int32_t* t_eid,
                                         int32_t* t_dst, void* stream);

/*
 * cgtp_conv_forward -- fused CG tensor product + receiver sum.
 *  uvu: x [N,d1], Y [E,d2], W_or_R = W [E,w_numel], M = NULL -> out [N,d_out].
 *  uvw, radial_k > 0: W_or_R = R [E,K], M [K,w_numel] -> out [N,d_out];
 *       per-edge weights are never formed; node state is streamed through
 *       bounded scratch owned by the plan ("Sobek ...", Abstract).
 *  uvw, radial_k == 0: W_or_R = W [E,w_numel], M = NULL (weights per edge).
 *  Receivers own their accumulation; no atomics; empty rows give zeros.
 */
cgtp_status cgtp_conv_forward(cgtp_plan plan, cgtp_graph graph, const void* x, const void* Y,
                              const void* W_or_R, const void* M, void* out, void* stream);

/*
 * cgtp_conv_backward -- adjoint of cgtp_conv_forward for an output gradient gout [N,d_out]:
 *  gx [N,d1] (sender-owned, summed over each sender's out-edges), gY [E,d2],
 *  uvu: gW_or_gR = gW [E,w_numel], gM = NULL;
 *  uvw: gW_or_gR = gR [E,K], gM [K,w_numel] (deterministic ordered reduction);
 *  uvw with per-edge weights: gW_or_gR = gW [E,w_numel], gM = NULL.
 */
cgtp_status cgtp_conv_backward(cgtp_plan plan, cgtp_graph graph, const void* gout, const void* x,
                               const void* Y, const void* W_or_R, const void* M, void* gx, void* gY,
                               void* gW_or_gR, void* gM, void* stream);

/*
 * cgtp_conv_double_backward -- second derivatives for force training
 * ("An Efficient Sparse Kernel Generator ...", Abstract: higher partial
 * derivatives from the gradient kernels through an identity; "Sobek ...",
 * Abstract: double backward).  Given cotangents of the backward's outputs,
 *   S = <ggx, gx> + <ggY, gY> + <ggW, gW>   (uvw: + <ggR, gR> + <ggM, gM>),
 * it returns dS/dgout, dS/dx, dS/dY, dS/dW (uvw: dS/dR, dS/dM).  The message is
 * multilinear in its operands, so dS/dgout is the sum of the forwards with one
 * operand replaced by its cotangent, and dS/da_j the sum of the backwards with
 * one other operand replaced (3 forwards + 3 backwards for uvu, 4 + 4 for uvw).
 *  gout [N,d_out], x, Y, W_or_R, M : as for cgtp_conv_backward (M = NULL for uvu).
 *  ggx [N,d1], ggY [E,d2], ggW_or_ggR [E,w_numel] or [E,K], ggM [K,w_numel] (uvw).
 *  d_gout [N,d_out], d_x [N,d1], d_Y [E,d2], d_W_or_dR, d_M : outputs (overwritten).
 *  workspace : caller-owned DEVICE buffer, 256-byte aligned, of at least the
 *      size cgtp_conv_double_backward_workspace reports (N*d_out plus one
 *      copy of every operand, in elements); nothing is allocated inside.
 *  Errors: CGTP_EINVAL for a missing or small workspace or a null operand;
 *  otherwise as cgtp_conv_forward / cgtp_conv_backward.
 */
cgtp_status cgtp_conv_double_backward_workspace(cgtp_plan plan, cgtp_graph graph, int64_t* bytes);
cgtp_status cgtp_conv_double_backward(cgtp_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                      const void* Y, const void* W_or_R, const void* M, const void* ggx,
                                      const void* ggY, const void* ggW_or_ggR, const void* ggM,
                                      void* d_gout, void* d_x, void* d_Y, void* d_W_or_dR, void* d_M,
                                      void* workspace, int64_t workspace_size, void* stream);

/* Double backward of the batched product (uvu plans): cotangents gg1 [B,d1],
 * gg2 [B,d2], ggW [B,w_numel] of cgtp_backward's outputs -> d_gout [B,d_out],
 * d_x1, d_x2, d_W.  Workspace as above, from cgtp_double_backward_workspace. */
cgtp_status cgtp_double_backward_workspace(cgtp_plan plan, int64_t B, int64_t* bytes);
cgtp_status cgtp_double_backward(cgtp_plan plan, const void* gout, const void* x1, const void* x2,
                                 const void* W, const void* gg1, const void* gg2, const void* ggW,
                                 void* d_gout, void* d_x1, void* d_x2, void* d_W, int64_t B,
                                 void* workspace, int64_t workspace_size, void* stream);

/*
 * cgtp_conv_forward_sh / cgtp_conv_backward_sh -- the uvu convolution fed by raw
 * edge vectors ("An Efficient Sparse Kernel Generator ...", Figure 4B: the edge
 * features are spherical harmonics of the edge directions).  The kernels
 * evaluate Y[e] = Y(rvec[e] / |rvec[e]|) (component normalisation, the
 * convention of cgtp_real_sh) as each edge is loaded, so no Y tensor is read.
 *  rvec [E,3] : DEVICE edge vectors (any length; a zero vector gives zero
 *      gradient), element type of the plan (CGTP_F32 or CGTP_F64).
 *  Other tensors as for cgtp_conv_forward / cgtp_conv_backward.  The backward
 *  also returns gY [E,d2] (the gradient with respect to the harmonics, which
 *  the caller provides as storage) and grvec [E,3] = dL/drvec.
 *  Needs irreps_in2 = 0e+1o+2e+... (harmonics 0..L in order, L <= 3) and a
 *  plan the fused l <= 3 kernels serve (one in1 multiplicity m with m/4 in
 *  {2, 8, 32} or m a multiple of 128); otherwise CGTP_EUNSUPPORTED.
 */
cgtp_status cgtp_conv_forward_sh(cgtp_plan plan, cgtp_graph graph, const void* x, const void* rvec,
                                 const void* W, void* out, void* stream);
cgtp_status cgtp_conv_backward_sh(cgtp_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                  const void* rvec, const void* W, void* gx, void* gY, void* grvec,
                                  void* gW, void* stream);

/*
 * cgtp_conv_forward_sh_radial / cgtp_conv_backward_sh_radial -- the uvw radial
 * convolution fed by raw edge vectors ("Sobek ...", Abstract: radial projection
 * and spherical-harmonic coupling streamed together).  The kernels evaluate the
 * harmonics Y(rvec/|rvec|) and the K Gaussian radial functions of d = |rvec|,
 *   R_k(d) = exp(-gamma (d - mu_k)^2),  mu_k = rbf_lo + k step,
 *   step = (rbf_hi - rbf_lo)/(K - 1) (K = 1: rbf_hi - rbf_lo),  gamma = 1/step^2,
 * so neither Y nor R is read.  rvec [E,3] DEVICE float; M, x, out, gout, gx, gM
 * as for cgtp_conv_forward / cgtp_conv_backward.  The backward also returns gY
 * [E,d2] and gR [E,K] (caller storage) and grvec [E,3] = dL/drvec.  Needs a uvw
 * plan with irreps_in2 = 0e+1o+2e+... and rbf_hi > rbf_lo.
 */
cgtp_status cgtp_conv_forward_sh_radial(cgtp_plan plan, cgtp_graph graph, const void* x, const void* rvec,
                                        const void* M, double rbf_lo, double rbf_hi, void* out, void* stream);
cgtp_status cgtp_conv_backward_sh_radial(cgtp_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                         const void* rvec, const void* M, double rbf_lo, double rbf_hi,
                                         void* gx, void* gY, void* gR, void* grvec, void* gM, void* stream);

/* Host only: the library's real spherical harmonics (component normalisation,
 * m = -l..l, l = 1 is sqrt(3) (y, z, x)) of n vectors rvec [n,3] after
 * normalisation: Y [n, (lmax+1)^2], and if dY is not NULL the Jacobian
 * dY [n, (lmax+1)^2, 3] = d Y / d rvec.  lmax <= 7. */
cgtp_status cgtp_real_sh(int lmax, const double* rvec, int64_t n, double* Y, double* dY);

/* Host only (no device needed): the planner's real-basis, component-normalised
 * CG block of (l1, l2, l3), l <= 7, as (2l1+1)(2l2+1)(2l3+1) doubles in
 * [m1][m2][m3] order; zeros if the triangle rule fails.  Same routine the plan
 * tables are built from ("An Efficient Sparse Kernel Generator ...", Figure 2:
 * the coefficient blocks). */
cgtp_status cgtp_real_cg_block(int l1, int l2, int l3, double* block, int64_t capacity);

/*
 * Mixed instruction lists: a connection mode per instruction ("An Efficient
 * Sparse Kernel Generator ...", Figure 3B/C: channel-wise (uvu) and fully
 * connected (uvw) weights; Figure 4B: fused with the receiver sum).
 *
 * cgtp_mixed_plan_create -- instr[i] = (i_in1, i_in2, i_out) with modes[i] in
 *  {CGTP_UVU, CGTP_UVW}; every instruction sums its message into block i_out of
 *  irreps_out (d_out = dim(irreps_out)).  A uvu instruction keeps the channel
 *  (block i_out must have the multiplicity of in1 block i_in1, else
 *  CGTP_EINVAL); a uvw instruction mixes channels.  Weights are two per-edge
 *  arrays in instruction order: Wu [E, wu_numel] (mul1 per uvu instruction) and
 *  Ww [E, ww_numel] (mul1*mul_out per uvw instruction, each block [u][w]).
 *  dtype CGTP_F32, CGTP_F64 or CGTP_BF16 (bfloat16 x, Y, Wu, Ww and output
 *  gradient, FP32 arithmetic and outputs; the uvu instructions must then be
 *  ones the v3 kernels serve, else CGTP_EUNSUPPORTED); the uvw instructions
 *  need l <= 3.  The plan owns two single-mode plans and a few KB of tables.
 * Must be called with the target device current.
 */
typedef struct cgtp_mixed_plan_s* cgtp_mixed_plan;
cgtp_status cgtp_mixed_plan_create(cgtp_mixed_plan* plan, const char* irreps_in1, const char* irreps_in2,
                                   const char* irreps_out, const cgtp_instr* instr, const int* modes, int n_instr,
                                   int dtype);
void cgtp_mixed_plan_destroy(cgtp_mixed_plan plan);
/* d1, d2, d_out and the row lengths of Wu and Ww (0 when the plan has no
 * instruction of that mode).  Any pointer may be NULL. */
cgtp_status cgtp_mixed_plan_info(cgtp_mixed_plan plan, int64_t* d1, int64_t* d2, int64_t* d_out,
                                 int64_t* wu_numel, int64_t* ww_numel);
/* Bytes of device workspace the three mixed entry points need on this graph
 * (one size for all three). */
cgtp_status cgtp_mixed_conv_workspace(cgtp_mixed_plan plan, cgtp_graph graph, int64_t* bytes);
/*
 * cgtp_mixed_conv_forward -- out [N,d_out] (overwritten) from x [N,d1], Y [E,d2],
 *  Wu, Ww (NULL allowed for a mode the plan does not use).
 * cgtp_mixed_conv_backward -- gx [N,d1], gY [E,d2], gWu, gWw (overwritten) for
 *  gout [N,d_out].
 * cgtp_mixed_conv_double_backward -- for cotangents ggx, ggY, ggWu, ggWw of
 *  (gx, gY, gWu, gWw): d_gout [N,d_out], d_x, d_Y, d_Wu, d_Ww (overwritten).  The
 *  message is linear in x, in Y and in the weights (Wu, Ww) taken together.
 * workspace: a 256-byte aligned device buffer of at least the size
 * cgtp_mixed_conv_workspace reports; errors as for the single-mode entry points.
 * Calls with the same plan must not overlap on the GPU.
 */
cgtp_status cgtp_mixed_conv_forward(cgtp_mixed_plan plan, cgtp_graph graph, const void* x, const void* Y,
                                    const void* Wu, const void* Ww, void* out, void* workspace,
                                    int64_t workspace_size, void* stream);
cgtp_status cgtp_mixed_conv_backward(cgtp_mixed_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                     const void* Y, const void* Wu, const void* Ww, void* gx, void* gY, void* gWu,
                                     void* gWw, void* workspace, int64_t workspace_size, void* stream);
cgtp_status cgtp_mixed_conv_double_backward(cgtp_mixed_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                            const void* Y, const void* Wu, const void* Ww, const void* ggx,
                                            const void* ggY, const void* ggWu, const void* ggWw, void* d_gout,
                                            void* d_x, void* d_Y, void* d_Wu, void* d_Ww, void* workspace,
                                            int64_t workspace_size, void* stream);

/* Message of the last failed call on this thread ("" if none). */
const char* cgtp_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* CGTP_H */
