// mixed.cu -- fused CG tensor-product convolution with a connection mode per
// instruction ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep
// Networks", Figure 3B/C: channel-wise (uvu) and fully connected (uvw)
// weights; Figure 4B: fused with the receiver sum).
//
// Every instruction (i_in1, i_in2, i_out) sums its message into block i_out of
// irreps_out.  A uvu instruction keeps the channel (that block must have the
// multiplicity of in1 block i_in1) with weights Wu [E, sum_uvu mul1]; a uvw
// instruction mixes channels with weights Ww [E, sum_uvw mul1*mul_out], each
// path's block [u][w]; both weight arrays are in instruction order.
//
// The message is a sum of the uvu terms and the uvw terms, so the plan runs the
// two single-mode plans over the same graph: the uvw plan writes irreps_out
// directly, and the uvu plan (whose outputs are appended in instruction order)
// is folded into it by a gather that owns each output element (deterministic,
// no atomics).  The backward gathers the output gradient into the uvu layout
// and adds the two plans' gx and gY.  The double backward adds the two plans'
// double backwards: the second-order scalar is the sum of the two plans' own.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

struct cgtp_mixed_plan_s {
  cgtp_plan uvu = nullptr;   // uvu instructions; outputs appended in instruction order
  cgtp_plan uvw = nullptr;   // uvw instructions; weights per edge, outputs in irreps_out blocks
  int dtype = 0, num_sms = 0;
  int64_t d1 = 0, d2 = 0, d_out = 0, d_u = 0, wu = 0, ww = 0;
  int* tables = nullptr;     // device: dst [d_u], inv_ptr [d_out + 1], inv_idx [d_u]
  const int *dst = nullptr, *inv_ptr = nullptr, *inv_idx = nullptr;
};

namespace cgtp {
namespace {

// out[n][f] (+)= sum over the uvu columns c folded into f of u[n][c]
template <typename T>
__global__ void fold_kernel(T* __restrict__ out, const T* __restrict__ u, const int* __restrict__ inv_ptr,
                            const int* __restrict__ inv_idx, int64_t N, int d_out, int d_u, bool accumulate) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N * d_out; i += stride) {
    const int64_t n = i / d_out;
    const int f = static_cast<int>(i - n * d_out);
    const int k0 = __ldg(inv_ptr + f), k1 = __ldg(inv_ptr + f + 1);
    if (accumulate && k0 == k1) continue;
    T v = accumulate ? out[i] : T(0);
    for (int k = k0; k < k1; ++k) v += u[n * d_u + __ldg(inv_idx + k)];
    out[i] = v;
  }
}

// u[n][c] = g[n][dst[c]]: the output gradient in the uvu plan's layout
template <typename T>
__global__ void unfold_kernel(T* __restrict__ u, const T* __restrict__ g, const int* __restrict__ dst, int64_t N,
                              int d_out, int d_u) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N * d_u; i += stride) {
    const int64_t n = i / d_u;
    const int c = static_cast<int>(i - n * d_u);
    u[i] = g[n * d_out + __ldg(dst + c)];
  }
}

template <typename T>
__global__ void acc_kernel(T* __restrict__ dst, const T* __restrict__ src, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] += src[i];
}

int grid_for(int64_t n, int num_sms) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)num_sms * 8)));
}

cgtp_status launched(const char* what) {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CGTP_OK : fail(CGTP_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

cgtp_status fold(const cgtp_mixed_plan_s* p, void* out, const void* u, int64_t N, bool accumulate, cudaStream_t st) {
  if (N == 0) return CGTP_OK;
  const int grid = grid_for(N * p->d_out, p->num_sms);
  if (p->dtype == CGTP_F64)
    fold_kernel<double><<<grid, 256, 0, st>>>(static_cast<double*>(out), static_cast<const double*>(u), p->inv_ptr,
                                              p->inv_idx, N, (int)p->d_out, (int)p->d_u, accumulate);
  else
    fold_kernel<float><<<grid, 256, 0, st>>>(static_cast<float*>(out), static_cast<const float*>(u), p->inv_ptr,
                                             p->inv_idx, N, (int)p->d_out, (int)p->d_u, accumulate);
  return launched("mixed plan: fold");
}

cgtp_status unfold(const cgtp_mixed_plan_s* p, void* u, const void* g, int64_t N, cudaStream_t st) {
  if (N == 0) return CGTP_OK;
  const int grid = grid_for(N * p->d_u, p->num_sms);
  if (p->dtype == CGTP_F64)
    unfold_kernel<double><<<grid, 256, 0, st>>>(static_cast<double*>(u), static_cast<const double*>(g), p->dst, N,
                                                (int)p->d_out, (int)p->d_u);
  else if (p->dtype == CGTP_BF16)  // the stored bfloat16 gradient, moved bit for bit
    unfold_kernel<unsigned short><<<grid, 256, 0, st>>>(static_cast<unsigned short*>(u),
                                                        static_cast<const unsigned short*>(g), p->dst, N,
                                                        (int)p->d_out, (int)p->d_u);
  else
    unfold_kernel<float><<<grid, 256, 0, st>>>(static_cast<float*>(u), static_cast<const float*>(g), p->dst, N,
                                               (int)p->d_out, (int)p->d_u);
  return launched("mixed plan: unfold");
}

cgtp_status accumulate(const cgtp_mixed_plan_s* p, void* dst, const void* src, int64_t n, cudaStream_t st) {
  if (n <= 0) return CGTP_OK;
  const int grid = grid_for(n, p->num_sms);
  if (p->dtype == CGTP_F64)
    acc_kernel<double><<<grid, 256, 0, st>>>(static_cast<double*>(dst), static_cast<const double*>(src), n);
  else
    acc_kernel<float><<<grid, 256, 0, st>>>(static_cast<float*>(dst), static_cast<const float*>(src), n);
  return launched("mixed plan: add");
}

int64_t al256(int64_t v) { return (v + 255) / 256 * 256; }

// Workspace carve-up shared by the three entry points (offsets in bytes):
// [sub-plan double-backward workspace][u: N*d_u][du: N*d_u][x2: N*d1][y2: E*d2]
struct Carve {
  int64_t sub = 0, u = 0, du = 0, x2 = 0, y2 = 0, total = 0;
};

cgtp_status carve(const cgtp_mixed_plan_s* p, const cgtp_graph_s* g, Carve* c) {
  const int64_t es = p->dtype == CGTP_F64 ? 8 : 4;
  int64_t sub = 0, b = 0;
  cgtp_status s;
  if (p->uvu) {
    if ((s = cgtp_conv_double_backward_workspace(p->uvu, const_cast<cgtp_graph_s*>(g), &b))) return s;
    sub = std::max(sub, b);
  }
  if (p->uvw) {
    if ((s = cgtp_conv_double_backward_workspace(p->uvw, const_cast<cgtp_graph_s*>(g), &b))) return s;
    sub = std::max(sub, b);
  }
  c->sub = 0;
  c->u = al256(sub);
  c->du = c->u + al256(g->N * p->d_u * es);
  c->x2 = c->du + al256(g->N * p->d_u * es);
  c->y2 = c->x2 + al256(g->N * p->d1 * es);
  c->total = c->y2 + al256(g->E * p->d2 * es);
  c->sub = sub;
  return CGTP_OK;
}

cgtp_status check_ws(const cgtp_mixed_plan_s* p, const cgtp_graph_s* g, const void* ws, int64_t ws_size, Carve* c) {
  cgtp_status s;
  if ((s = carve(p, g, c))) return s;
  if (ws_size < c->total) return fail(CGTP_EINVAL, "mixed plan: workspace too small (query cgtp_mixed_conv_workspace)");
  if (c->total > 0 && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)))
    return fail(CGTP_EINVAL, "mixed plan: workspace must be a 256-byte aligned device pointer");
  return CGTP_OK;
}

unsigned char* at(void* ws, int64_t off) { return static_cast<unsigned char*>(ws) + off; }

}  // namespace
}  // namespace cgtp

using namespace cgtp;

extern "C" {

cgtp_status cgtp_mixed_plan_create(cgtp_mixed_plan* out, const char* irreps_in1, const char* irreps_in2,
                                   const char* irreps_out, const cgtp_instr* instr, const int* modes, int n_instr,
                                   int dtype) {
  clear_error();
  if (!out) return fail(CGTP_EINVAL, "null plan pointer");
  *out = nullptr;
  if (!irreps_in1 || !irreps_in2 || !irreps_out) return fail(CGTP_EINVAL, "null irreps string");
  if (!instr || !modes || n_instr <= 0) return fail(CGTP_EINVAL, "a mixed plan needs an explicit instruction list");
  if (dtype != CGTP_F32 && dtype != CGTP_F64 && dtype != CGTP_BF16)
    return fail(CGTP_EINVAL, "dtype must be CGTP_F32, CGTP_F64 or CGTP_BF16");
  std::vector<Irrep> in1, outr;
  std::string err;
  if (!parse_irreps(irreps_in1, &in1, &err)) return fail(CGTP_EINVAL, "irreps_in1: " + err);
  if (!parse_irreps(irreps_out, &outr, &err)) return fail(CGTP_EINVAL, "irreps_out: " + err);
  std::vector<cgtp_instr> iu, iw;
  for (int i = 0; i < n_instr; ++i) {
    const cgtp_instr& t = instr[i];
    if (t.i_in1 < 0 || t.i_in1 >= (int)in1.size() || t.i_out < 0 || t.i_out >= (int)outr.size())
      return fail(CGTP_EINVAL, "instruction " + std::to_string(i) + ": block index out of range");
    if (modes[i] == CGTP_UVU) {
      if (outr[t.i_out].mul != in1[t.i_in1].mul)
        return fail(CGTP_EINVAL, "instruction " + std::to_string(i) +
                                     ": a uvu instruction needs an output block of the in1 block's multiplicity");
      iu.push_back(t);
    } else if (modes[i] == CGTP_UVW) {
      iw.push_back(t);
    } else {
      return fail(CGTP_EINVAL, "instruction " + std::to_string(i) + ": mode must be CGTP_UVU or CGTP_UVW");
    }
  }
  cgtp_mixed_plan_s* p = new (std::nothrow) cgtp_mixed_plan_s();
  if (!p) return fail(CGTP_ENOMEM, "host allocation failed");
  p->dtype = dtype;
  cgtp_status s;
  if (!iu.empty() &&
      (s = cgtp_plan_create(&p->uvu, irreps_in1, irreps_in2, irreps_out, iu.data(), (int)iu.size(), CGTP_UVU, dtype, 0))) {
    cgtp_mixed_plan_destroy(p);
    return s;
  }
  if (!iw.empty() &&
      (s = cgtp_plan_create(&p->uvw, irreps_in1, irreps_in2, irreps_out, iw.data(), (int)iw.size(), CGTP_UVW, dtype, 0))) {
    cgtp_mixed_plan_destroy(p);
    return s;
  }
  const cgtp_plan_s* any = p->uvw ? p->uvw : p->uvu;
  p->d1 = any->d1;
  p->d2 = any->d2;
  p->num_sms = any->num_sms;
  int64_t d_out = 0;
  std::vector<int> ooff(outr.size());
  for (size_t k = 0; k < outr.size(); ++k) {
    ooff[k] = static_cast<int>(d_out);
    d_out += int64_t(outr[k].mul) * (2 * outr[k].l + 1);
  }
  p->d_out = d_out;
  p->ww = p->uvw ? p->uvw->w_numel : 0;
  // fold map: column c of the uvu layout -> column dst[c] of irreps_out
  std::vector<int> dst;
  if (p->uvu) {
    p->d_u = p->uvu->d_out;
    p->wu = p->uvu->w_numel;
    dst.resize(p->d_u);
    for (const auto& ph : p->uvu->paths) {
      const int n = ph.mul1 * (2 * ph.l3 + 1);
      for (int c = 0; c < n; ++c) dst[ph.ooff + c] = ooff[ph.io] + c;
    }
  }
  std::vector<int> inv_ptr(d_out + 1, 0), inv_idx(dst.size());
  for (int c : dst) ++inv_ptr[c + 1];
  for (int64_t f = 0; f < d_out; ++f) inv_ptr[f + 1] += inv_ptr[f];
  {
    std::vector<int> fill(inv_ptr.begin(), inv_ptr.end() - 1);
    for (size_t c = 0; c < dst.size(); ++c) inv_idx[fill[dst[c]]++] = static_cast<int>(c);  // ascending c
  }
  std::vector<int> tab;
  tab.insert(tab.end(), dst.begin(), dst.end());
  tab.insert(tab.end(), inv_ptr.begin(), inv_ptr.end());
  tab.insert(tab.end(), inv_idx.begin(), inv_idx.end());
  if (cudaMalloc(&p->tables, tab.size() * sizeof(int)) != cudaSuccess) {
    p->tables = nullptr;
    cgtp_mixed_plan_destroy(p);
    return fail(CGTP_ENOMEM, "mixed plan: table allocation failed");
  }
  if (cudaMemcpy(p->tables, tab.data(), tab.size() * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    cgtp_mixed_plan_destroy(p);
    return fail(CGTP_ECUDA, "mixed plan: table upload failed");
  }
  p->dst = p->tables;
  p->inv_ptr = p->tables + dst.size();
  p->inv_idx = p->inv_ptr + (d_out + 1);
  *out = p;
  return CGTP_OK;
}

void cgtp_mixed_plan_destroy(cgtp_mixed_plan plan) {
  if (!plan) return;
  if (plan->uvu) cgtp_plan_destroy(plan->uvu);
  if (plan->uvw) cgtp_plan_destroy(plan->uvw);
  if (plan->tables) cudaFree(plan->tables);
  delete plan;
}

cgtp_status cgtp_mixed_plan_info(cgtp_mixed_plan plan, int64_t* d1, int64_t* d2, int64_t* d_out, int64_t* wu_numel,
                                 int64_t* ww_numel) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (d1) *d1 = plan->d1;
  if (d2) *d2 = plan->d2;
  if (d_out) *d_out = plan->d_out;
  if (wu_numel) *wu_numel = plan->wu;
  if (ww_numel) *ww_numel = plan->ww;
  return CGTP_OK;
}

cgtp_status cgtp_mixed_conv_workspace(cgtp_mixed_plan plan, cgtp_graph graph, int64_t* bytes) {
  clear_error();
  if (!plan || !graph || !bytes) return fail(CGTP_EINVAL, "null plan, graph or bytes");
  Carve c;
  cgtp_status s = carve(plan, graph, &c);
  if (!s) *bytes = c.total;
  return s;
}

cgtp_status cgtp_mixed_conv_forward(cgtp_mixed_plan plan, cgtp_graph graph, const void* x, const void* Y,
                                    const void* Wu, const void* Ww, void* out, void* workspace,
                                    int64_t workspace_size, void* stream) {
  clear_error();
  if (!plan || !graph) return fail(CGTP_EINVAL, "null plan or graph");
  if (graph->N == 0) return CGTP_OK;
  Carve c;
  cgtp_status s;
  if ((s = check_ws(plan, graph, workspace, workspace_size, &c))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (plan->uvw && (s = cgtp_conv_forward(plan->uvw, graph, x, Y, Ww, nullptr, out, stream))) return s;
  if (plan->uvu) {
    void* u = at(workspace, c.u);
    if ((s = cgtp_conv_forward(plan->uvu, graph, x, Y, Wu, nullptr, u, stream))) return s;
    if ((s = fold(plan, out, u, graph->N, plan->uvw != nullptr, st))) return s;
  }
  return CGTP_OK;
}

cgtp_status cgtp_mixed_conv_backward(cgtp_mixed_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                     const void* Y, const void* Wu, const void* Ww, void* gx, void* gY, void* gWu,
                                     void* gWw, void* workspace, int64_t workspace_size, void* stream) {
  clear_error();
  if (!plan || !graph) return fail(CGTP_EINVAL, "null plan or graph");
  Carve c;
  cgtp_status s;
  if ((s = check_ws(plan, graph, workspace, workspace_size, &c))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool both = plan->uvu && plan->uvw;
  if (plan->uvu) {
    void* u = at(workspace, c.u);
    if ((s = unfold(plan, u, gout, graph->N, st))) return s;
    if ((s = cgtp_conv_backward(plan->uvu, graph, u, x, Y, Wu, nullptr, gx, gY, gWu, nullptr, stream))) return s;
  }
  if (plan->uvw) {
    void* gx2 = both ? at(workspace, c.x2) : gx;
    void* gY2 = both ? at(workspace, c.y2) : gY;
    if ((s = cgtp_conv_backward(plan->uvw, graph, gout, x, Y, Ww, nullptr, gx2, gY2, gWw, nullptr, stream)))
      return s;
    if (both) {
      if ((s = accumulate(plan, gx, gx2, graph->N * plan->d1, st))) return s;
      if ((s = accumulate(plan, gY, gY2, graph->E * plan->d2, st))) return s;
    }
  }
  return CGTP_OK;
}

cgtp_status cgtp_mixed_conv_double_backward(cgtp_mixed_plan plan, cgtp_graph graph, const void* gout, const void* x,
                                            const void* Y, const void* Wu, const void* Ww, const void* ggx,
                                            const void* ggY, const void* ggWu, const void* ggWw, void* d_gout,
                                            void* d_x, void* d_Y, void* d_Wu, void* d_Ww, void* workspace,
                                            int64_t workspace_size, void* stream) {
  clear_error();
  if (!plan || !graph) return fail(CGTP_EINVAL, "null plan or graph");
  Carve c;
  cgtp_status s;
  if ((s = check_ws(plan, graph, workspace, workspace_size, &c))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool both = plan->uvu && plan->uvw;
  void* sub = at(workspace, 0);
  if (plan->uvw &&
      (s = cgtp_conv_double_backward(plan->uvw, graph, gout, x, Y, Ww, nullptr, ggx, ggY, ggWw, nullptr, d_gout, d_x,
                                     d_Y, d_Ww, nullptr, sub, c.sub, stream)))
    return s;
  if (plan->uvu) {
    void* u = at(workspace, c.u);
    void* du = at(workspace, c.du);
    void* dx = both ? at(workspace, c.x2) : d_x;
    void* dY = both ? at(workspace, c.y2) : d_Y;
    if ((s = unfold(plan, u, gout, graph->N, st))) return s;
    if ((s = cgtp_conv_double_backward(plan->uvu, graph, u, x, Y, Wu, nullptr, ggx, ggY, ggWu, nullptr, du, dx, dY,
                                       d_Wu, nullptr, sub, c.sub, stream)))
      return s;
    if ((s = fold(plan, d_gout, du, graph->N, both, st))) return s;
    if (both) {
      if ((s = accumulate(plan, d_x, dx, graph->N * plan->d1, st))) return s;
      if ((s = accumulate(plan, d_Y, dY, graph->E * plan->d2, st))) return s;
    }
  }
  return CGTP_OK;
}

}  // extern "C"
