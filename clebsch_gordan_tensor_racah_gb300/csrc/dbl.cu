// dbl.cu -- second derivatives of the fused CG tensor-product convolution and of
// the batched product ("double backward").
//
// "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
// Abstract: higher partial derivatives (needed for force prediction) obtained
// from the existing forward and gradient kernels through an identity; "Sobek:
// Streaming Equivariant Tensor Product Convolutions", Abstract: forward,
// backward and double backward.
//
// The message is multilinear in its operands a = (x, Y, W) for uvu, or
// (x, Y, R, M) for uvw with W = R M.  The backward maps an output gradient g to
// (dL/da_j)_j = B_j(g; a).  For cotangents c_j of those gradients, the scalar
//   S = sum_j < c_j, B_j(g; a) > = < g, sum_i F(a with a_i -> c_i) >
// so
//   dS/dg   = sum_i F(a with a_i -> c_i)                       (one forward each)
//   dS/da_j = sum_{i != j} B_j(g; a with a_i -> c_i)          (one backward each)
// because B_j does not depend on a_j.  The entry points here run the existing
// kernels with substituted operands and add the pieces with one elementwise
// kernel.  Temporaries live in a workspace the caller provides.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"

namespace cgtp {
namespace {

template <typename T>
__global__ void add_kernel(T* __restrict__ dst, const T* __restrict__ src, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] += src[i];
}

cgtp_status add_into(void* dst, const void* src, int64_t n, int dtype, int num_sms, cudaStream_t st) {
  if (n <= 0) return CGTP_OK;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)num_sms * 8)));
  if (dtype == CGTP_F64)
    add_kernel<double><<<grid, 256, 0, st>>>(static_cast<double*>(dst), static_cast<const double*>(src), n);
  else
    add_kernel<float><<<grid, 256, 0, st>>>(static_cast<float*>(dst), static_cast<const float*>(src), n);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CGTP_OK : fail(CGTP_ECUDA, std::string("double backward add: ") + cudaGetErrorString(e));
}

int64_t al256(int64_t v) { return (v + 255) / 256 * 256; }

// Operand sizes (elements) of a plan on a graph (uvu: x, Y, W; uvw: x, Y, R, M)
int operand_sizes(const cgtp_plan_s* plan, int64_t rows, int64_t E, int64_t* sz) {
  sz[0] = rows * plan->d1;
  sz[1] = E * plan->d2;
  if (plan->mode == CGTP_UVU || plan->radial_k == 0) {   // weights per edge
    sz[2] = E * plan->w_numel;
    return 3;
  }
  sz[2] = E * plan->radial_k;
  sz[3] = static_cast<int64_t>(plan->radial_k) * plan->w_numel;
  return 4;
}

int64_t workspace_bytes(const cgtp_plan_s* plan, int64_t rows, int64_t E) {
  const int64_t es = plan->dtype == CGTP_F64 ? 8 : 4;
  int64_t sz[4];
  const int n = operand_sizes(plan, rows, E, sz);
  int64_t b = al256(rows * plan->d_out * es);
  for (int j = 0; j < n; ++j) b += al256(sz[j] * es);
  return b;
}

struct Calls {  // forward / backward through the public entry points, graph or batched
  const cgtp_plan_s* plan;
  cgtp_graph_s* graph;  // null: batched product
  int64_t B;
  void* stream;
  cgtp_status fwd(const void* const* a, void* out) const {
    if (graph) return cgtp_conv_forward(const_cast<cgtp_plan_s*>(plan), graph, a[0], a[1], a[2],
                                        plan->radial_k > 0 ? a[3] : nullptr, out, stream);
    return cgtp_forward(const_cast<cgtp_plan_s*>(plan), a[0], a[1], a[2], out, B, stream);
  }
  cgtp_status bwd(const void* g, const void* const* a, void* const* o) const {
    if (graph)
      return cgtp_conv_backward(const_cast<cgtp_plan_s*>(plan), graph, g, a[0], a[1], a[2],
                                plan->radial_k > 0 ? a[3] : nullptr, o[0], o[1], o[2],
                                plan->radial_k > 0 ? o[3] : nullptr, stream);
    return cgtp_backward(const_cast<cgtp_plan_s*>(plan), g, a[0], a[1], a[2], o[0], o[1], o[2], B, stream);
  }
};

cgtp_status double_backward(const Calls& c, int64_t rows, int64_t E, const void* gout,
                            const void* const* a, const void* const* cot, void* d_gout, void* const* d,
                            void* workspace, int64_t ws_bytes) {
  const cgtp_plan_s* plan = c.plan;
  if (plan->dtype == CGTP_BF16) return fail(CGTP_EUNSUPPORTED, "double backward has no CGTP_BF16 path");
  const int64_t es = plan->dtype == CGTP_F64 ? 8 : 4;
  int64_t sz[4];
  const int n = operand_sizes(plan, rows, E, sz);
  if (ws_bytes < workspace_bytes(plan, rows, E))
    return fail(CGTP_EINVAL, "double backward: workspace too small (query the *_workspace entry point)");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(CGTP_EINVAL, "double backward: workspace must be a 256-byte aligned device pointer");
  for (int j = 0; j < n; ++j)
    if (sz[j] > 0 && (!a[j] || !cot[j] || !d[j])) return fail(CGTP_EINVAL, "double backward: null operand");
  if (!gout || !d_gout) return fail(CGTP_EINVAL, "double backward: null gout or d_gout");
  cudaStream_t st = static_cast<cudaStream_t>(c.stream);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  void* tg = w;
  void* tmp[4];
  int64_t off = al256(rows * plan->d_out * es);
  for (int j = 0; j < n; ++j) {
    tmp[j] = w + off;
    off += al256(sz[j] * es);
  }
  const int64_t n_out = rows * plan->d_out;
  cgtp_status s;
  // dS/dg: one forward per substituted operand
  for (int i = 0; i < n; ++i) {
    const void* ai[4] = {a[0], a[1], a[2], n > 3 ? a[3] : nullptr};
    ai[i] = cot[i];
    if ((s = c.fwd(ai, i == 0 ? d_gout : tg))) return s;
    if (i > 0 && (s = add_into(d_gout, tg, n_out, plan->dtype, plan->num_sms, st))) return s;
  }
  // dS/da_j: one backward per substituted operand; its own-operand gradient is discarded
  bool written[4] = {false, false, false, false};
  for (int i = 0; i < n; ++i) {
    const void* ai[4] = {a[0], a[1], a[2], n > 3 ? a[3] : nullptr};
    ai[i] = cot[i];
    void* o[4] = {nullptr, nullptr, nullptr, nullptr};
    bool add[4] = {false, false, false, false};
    for (int j = 0; j < n; ++j) {
      if (j == i || written[j]) {
        o[j] = tmp[j];
        add[j] = j != i;
      } else {
        o[j] = d[j];
        written[j] = true;
      }
    }
    if ((s = c.bwd(gout, ai, o))) return s;
    for (int j = 0; j < n; ++j)
      if (add[j] && (s = add_into(d[j], tmp[j], sz[j], plan->dtype, plan->num_sms, st))) return s;
  }
  return CGTP_OK;
}

}  // namespace
}  // namespace cgtp

using namespace cgtp;

extern "C" {

cgtp_status cgtp_conv_double_backward_workspace(cgtp_plan plan, cgtp_graph graph, int64_t* bytes) {
  clear_error();
  if (!plan || !graph || !bytes) return fail(CGTP_EINVAL, "null plan, graph or bytes");
  *bytes = workspace_bytes(plan, graph->N, graph->E);
  return CGTP_OK;
}

cgtp_status cgtp_conv_double_backward(cgtp_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                      const void* Y, const void* W_or_R, const void* M, const void* ggx,
                                      const void* ggY, const void* ggW_or_ggR, const void* ggM, void* d_gout,
                                      void* d_x, void* d_Y, void* d_W_or_dR, void* d_M, void* workspace,
                                      int64_t workspace_size, void* stream) {
  clear_error();
  if (!plan || !graph) return fail(CGTP_EINVAL, "null plan or graph");
  if (plan->radial_k == 0 && (M || ggM || d_M))
    return fail(CGTP_EINVAL, "M, ggM and d_M must be NULL for per-edge weights");
  const void* a[4] = {x, Y, W_or_R, M};
  const void* cot[4] = {ggx, ggY, ggW_or_ggR, ggM};
  void* d[4] = {d_x, d_Y, d_W_or_dR, d_M};
  Calls c{plan, graph, 0, stream};
  return double_backward(c, graph->N, graph->E, gout, a, cot, d_gout, d, workspace, workspace_size);
}

cgtp_status cgtp_double_backward_workspace(cgtp_plan plan, int64_t B, int64_t* bytes) {
  clear_error();
  if (!plan || !bytes || B < 0) return fail(CGTP_EINVAL, "null plan or bytes, or negative batch");
  if (plan->mode != CGTP_UVU) return fail(CGTP_EUNSUPPORTED, "the batched product needs a uvu plan");
  *bytes = workspace_bytes(plan, B, B);
  return CGTP_OK;
}

cgtp_status cgtp_double_backward(cgtp_plan plan, const void* gout, const void* x1, const void* x2,
                                 const void* W, const void* gg1, const void* gg2, const void* ggW,
                                 void* d_gout, void* d_x1, void* d_x2, void* d_W, int64_t B, void* workspace,
                                 int64_t workspace_size, void* stream) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (plan->mode != CGTP_UVU) return fail(CGTP_EUNSUPPORTED, "the batched product needs a uvu plan");
  if (B < 0 || B >= (int64_t(1) << 31)) return fail(CGTP_EINVAL, "batch size out of range");
  if (B == 0) return CGTP_OK;
  const void* a[4] = {x1, x2, W, nullptr};
  const void* cot[4] = {gg1, gg2, ggW, nullptr};
  void* d[4] = {d_x1, d_x2, d_W, nullptr};
  Calls c{plan, nullptr, B, stream};
  return double_backward(c, B, B, gout, a, cot, d_gout, d, workspace, workspace_size);
}

}  // extern "C"
