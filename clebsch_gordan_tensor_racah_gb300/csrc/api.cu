// api.cu -- the extern "C" boundary of libcgtp (declared in include/cgtp.h).
//
// Every entry point validates its arguments on the host and returns a status
// before anything is launched; compute entry points only enqueue kernels on
// the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>

#include "internal.h"

namespace cgtp {
const char* last_error_cstr();

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cgtp_status need(const void* p, const char* name) {
  if (!p) return fail(CGTP_EINVAL, std::string("null pointer: ") + name);
  if (!aligned16(p)) return fail(CGTP_EINVAL, std::string("pointer not 16-byte aligned: ") + name);
  return CGTP_OK;
}

template <typename T>
void append(std::vector<unsigned char>& buf, const std::vector<T>& v, size_t* off) {
  size_t o = (buf.size() + 15) / 16 * 16;
  buf.resize(o + v.size() * sizeof(T));
  if (!v.empty()) std::memcpy(buf.data() + o, v.data(), v.size() * sizeof(T));
  *off = o;
}

}  // namespace

int smem_cap_cached(const void* kernel) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> caps;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> lock(mu);
  auto it = caps.find({kernel, dev});
  if (it != caps.end()) return it->second;
  const int cap = raise_smem_limit(kernel);
  if (cap >= 0) caps[{kernel, dev}] = cap;
  return cap;
}

int raise_smem_limit(const void* kernel) {
  int dev = 0, optin = 0;
  cudaFuncAttributes fa{};
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  const int cap = optin - static_cast<int>(fa.sharedSizeBytes);
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return cap;
}

cgtp_status upload_layout(const cgtp_plan_s* plan, const LayoutHost& h, LayoutDev* d) {
  std::vector<unsigned char> buf;
  size_t o_paths, o_in1, o_groups, o_cyb, o_cyc, o_cyf, o_gyb, o_gys, o_gyn, o_gyf, o_ib, o_it, o_gxb,
      o_gxp;
  append(buf, h.paths, &o_paths);
  append(buf, h.in1_off, &o_in1);
  append(buf, h.groups, &o_groups);
  append(buf, h.cy_begin, &o_cyb);
  append(buf, h.cy_col, &o_cyc);
  if (plan->dtype == CGTP_F64) {
    append(buf, h.cy_coef, &o_cyf);
  } else {
    std::vector<float> f(h.cy_coef.begin(), h.cy_coef.end());
    append(buf, f, &o_cyf);
  }
  append(buf, h.gy_begin, &o_gyb);
  append(buf, h.gy_slot, &o_gys);
  append(buf, h.gy_nub, &o_gyn);
  if (plan->dtype == CGTP_F64) {
    append(buf, h.gy_coef, &o_gyf);
  } else {
    std::vector<float> f(h.gy_coef.begin(), h.gy_coef.end());
    append(buf, f, &o_gyf);
  }
  append(buf, h.item_begin, &o_ib);
  append(buf, h.items, &o_it);
  append(buf, h.gx_begin, &o_gxb);
  append(buf, h.gx_paths, &o_gxp);
  size_t o_c2c, o_c2f, o_c2b;
  append(buf, h.cy2_col, &o_c2c);
  if (plan->dtype == CGTP_F64) {
    append(buf, h.cy2_coef, &o_c2f);
  } else {
    std::vector<float> f(h.cy2_coef.begin(), h.cy2_coef.end());
    append(buf, f, &o_c2f);
  }
  append(buf, h.cy2_base, &o_c2b);
  void* base = nullptr;
  if (cudaMalloc(&base, std::max<size_t>(buf.size(), 16)) != cudaSuccess)
    return fail(CGTP_ENOMEM, "plan table allocation failed");
  const_cast<cgtp_plan_s*>(plan)->device_bytes += std::max<size_t>(buf.size(), 16);
  if (cudaMemcpy(base, buf.data(), buf.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(base);
    return fail(CGTP_ECUDA, "plan table upload failed");
  }
  auto at = [&](size_t o) { return static_cast<unsigned char*>(base) + o; };
  d->base = base;
  d->chunk = h.chunk;
  d->n_groups = static_cast<int>(h.groups.size());
  d->n_in1 = static_cast<int>(h.in1_off.size()) - 1;
  d->paths = reinterpret_cast<const PathDev*>(at(o_paths));
  d->in1_off = reinterpret_cast<const int*>(at(o_in1));
  d->groups = reinterpret_cast<const GroupDev*>(at(o_groups));
  d->cy_begin = reinterpret_cast<const int*>(at(o_cyb));
  d->cy_col = reinterpret_cast<const int*>(at(o_cyc));
  d->cy_coef = at(o_cyf);
  d->gy_begin = reinterpret_cast<const int*>(at(o_gyb));
  d->gy_slot = reinterpret_cast<const int*>(at(o_gys));
  d->gy_nub = reinterpret_cast<const int*>(at(o_gyn));
  d->gy_coef = at(o_gyf);
  d->item_begin = reinterpret_cast<const int*>(at(o_ib));
  d->items = reinterpret_cast<const Item*>(at(o_it));
  d->gx_begin = reinterpret_cast<const int*>(at(o_gxb));
  d->gx_paths = reinterpret_cast<const int*>(at(o_gxp));
  d->smem_fwd = h.smem_fwd;
  d->smem_bwd = h.smem_bwd;
  d->cy2_col = reinterpret_cast<const int*>(at(o_c2c));
  d->cy2_coef = at(o_c2f);
  d->cy2_base = reinterpret_cast<const int*>(at(o_c2b));
  d->chunk2 = h.chunk2;
  d->smem_fwd2 = h.smem_fwd2;
  d->smem_bwd2 = h.smem_bwd2;
  d->groups_host = h.groups;
  return CGTP_OK;
}

void free_layout(LayoutDev* d) {
  if (d->base) cudaFree(d->base);
  d->base = nullptr;
}

}  // namespace cgtp

using namespace cgtp;

extern "C" {

const char* cgtp_last_error(void) { return last_error_cstr(); }

cgtp_status cgtp_real_cg_block(int l1, int l2, int l3, double* block, int64_t capacity) {
  clear_error();
  if (l1 < 0 || l2 < 0 || l3 < 0 || l1 > kMaxL || l2 > kMaxL || l3 > kMaxL)
    return fail(CGTP_EINVAL, "l must be in [0, 7]");
  if (!block) return fail(CGTP_EINVAL, "null block");
  const int64_t n = int64_t(2 * l1 + 1) * (2 * l2 + 1) * (2 * l3 + 1);
  if (capacity < n) return fail(CGTP_EINVAL, "block capacity too small");
  const std::vector<double> C = real_cg_block(l1, l2, l3);
  std::memcpy(block, C.data(), n * sizeof(double));
  return CGTP_OK;
}

cgtp_status cgtp_plan_create(cgtp_plan* out, const char* irreps_in1, const char* irreps_in2,
                             const char* irreps_out, const cgtp_instr* instr, int n_instr, int mode,
                             int dtype, int radial_k) {
  clear_error();
  if (!out) return fail(CGTP_EINVAL, "null plan output pointer");
  *out = nullptr;
  if (mode != CGTP_UVU && mode != CGTP_UVW) return fail(CGTP_EINVAL, "mode must be CGTP_UVU or CGTP_UVW");
  if (dtype != CGTP_F32 && dtype != CGTP_F64 && dtype != CGTP_BF16)
    return fail(CGTP_EINVAL, "dtype must be CGTP_F32, CGTP_F64 or CGTP_BF16");
  if (mode == CGTP_UVU && radial_k != 0) return fail(CGTP_EINVAL, "radial_k must be 0 in uvu mode");
  if (mode == CGTP_UVW && (radial_k < 0 || radial_k > 8))
    return fail(CGTP_EUNSUPPORTED, "uvw mode needs 0 <= radial_k <= 8 (0: one weight matrix per edge)");
  if (mode == CGTP_UVW && radial_k > 0 && dtype != CGTP_F32)
    return fail(CGTP_EUNSUPPORTED, "uvw mode with radial weights supports CGTP_F32 only");
  if (mode == CGTP_UVW && dtype == CGTP_BF16 && radial_k > 0)
    return fail(CGTP_EUNSUPPORTED, "uvw with radial weights has no CGTP_BF16 kernels");
  if (n_instr < 0 || (n_instr > 0 && !instr)) return fail(CGTP_EINVAL, "bad instruction list");
  cgtp_plan_s* p = new (std::nothrow) cgtp_plan_s();
  if (!p) return fail(CGTP_ENOMEM, "host allocation failed");
  p->mode = mode;
  p->dtype = dtype;
  p->radial_k = radial_k;
  std::string err;
  if (!parse_irreps(irreps_in1, &p->in1, &err) || !parse_irreps(irreps_in2, &p->in2, &err) ||
      !parse_irreps(irreps_out, &p->out, &err)) {
    delete p;
    return fail(CGTP_EINVAL, err);
  }
  for (const auto& i : p->in2)
    if (i.mul != 1) {
      delete p;
      return fail(CGTP_EUNSUPPORTED, "irreps_in2 blocks must have multiplicity 1");
    }
  cgtp_status s = build_paths(p, instr, n_instr);
  if (s != CGTP_OK) {
    delete p;
    return s;
  }
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return fail(CGTP_ECUDA, "no CUDA device");
  }
  if (mode == CGTP_UVU) {
    LayoutHost conv, batch;
    const size_t budget = 96 * 1024;
    s = build_layout(p, 16, budget, &conv);
    if (s == CGTP_OK) s = build_layout(p, 1, budget, &batch);
    if (s == CGTP_OK) s = upload_layout(p, conv, &p->conv_layout);
    if (s == CGTP_OK) s = upload_layout(p, batch, &p->batch_layout);
    if (s == CGTP_OK) s = build_v3(p);
    if (s == CGTP_OK) s = bt_create(p);
    if (s == CGTP_OK && dtype == CGTP_BF16 && !p->v3.lpe && !p->bt)
      s = fail(CGTP_EUNSUPPORTED, "CGTP_BF16 needs l <= 3 and one in1 multiplicity m with m/4 in {2, 8, 32} "
                                  "or m a multiple of 128 (graph convolutions), or multiplicity 16 or 32 in "
                                  "every path and l <= 7 (batched products)");
  } else if (radial_k == 0) {
    s = uvwe_create(p);
  } else {
    s = uvw_create(p);
  }
  if (s != CGTP_OK) {
    cgtp_plan_destroy(p);
    return s;
  }
  *out = p;
  return CGTP_OK;
}

void cgtp_plan_destroy(cgtp_plan plan) {
  if (!plan) return;
  free_layout(&plan->conv_layout);
  free_layout(&plan->batch_layout);
  free_v3(plan);
  bt_destroy(plan);
  uvwe_destroy(plan);
  if (plan->uvw) uvw_destroy(plan);
  delete plan;
}

cgtp_status cgtp_plan_info(cgtp_plan plan, int64_t* d1, int64_t* d2, int64_t* d_out,
                           int64_t* w_numel, int* n_paths) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (d1) *d1 = plan->d1;
  if (d2) *d2 = plan->d2;
  if (d_out) *d_out = plan->d_out;
  if (w_numel) *w_numel = plan->w_numel;
  if (n_paths) *n_paths = static_cast<int>(plan->paths.size());
  return CGTP_OK;
}

cgtp_status cgtp_plan_set_wait_limit(cgtp_plan plan, int64_t polls) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (polls < 0) return fail(CGTP_EINVAL, "polls must be >= 0");
  plan->wait_limit = polls;
  return CGTP_OK;
}

cgtp_status cgtp_plan_set_node_chunk(cgtp_plan plan, int64_t nodes) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (!plan->uvw) return fail(CGTP_EINVAL, "node chunks belong to uvw plans with radial weights");
  if (nodes < 1 || nodes > (int64_t(1) << 20)) return fail(CGTP_EINVAL, "nodes must be in [1, 1048576]");
  return uvw_set_chunk(plan, static_cast<int>(nodes));
}

cgtp_status cgtp_plan_node_chunk(cgtp_plan plan, int64_t* nodes) {
  clear_error();
  if (!plan || !nodes) return fail(CGTP_EINVAL, "null plan or nodes");
  *nodes = plan->uvw ? uvw_chunk(plan) : 0;
  return CGTP_OK;
}

cgtp_status cgtp_plan_device_bytes(cgtp_plan plan, int64_t* bytes) {
  clear_error();
  if (!plan || !bytes) return fail(CGTP_EINVAL, "null plan or bytes");
  *bytes = static_cast<int64_t>(plan->device_bytes);
  return CGTP_OK;
}

cgtp_status cgtp_graph_device_bytes(cgtp_graph graph, int64_t* bytes) {
  clear_error();
  if (!graph || !bytes) return fail(CGTP_EINVAL, "null graph or bytes");
  *bytes = static_cast<int64_t>(sizeof(int32_t)) * (graph->N + 1 + 2 * std::max<int64_t>(graph->E, 1));
  return CGTP_OK;
}

cgtp_status cgtp_plan_path(cgtp_plan plan, int p, int* ints10, double* block, int64_t capacity) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (p < 0 || p >= static_cast<int>(plan->paths.size())) return fail(CGTP_EINVAL, "path index out of range");
  const auto& q = plan->paths[p];
  if (ints10) {
    const int v[10] = {q.l1, q.l2, q.l3, q.mul1, q.mul_out, q.off1, q.off2, q.ooff, q.woff, q.io};
    std::memcpy(ints10, v, sizeof(v));
  }
  if (block) {
    if (capacity < static_cast<int64_t>(q.C.size())) return fail(CGTP_EINVAL, "block capacity too small");
    std::memcpy(block, q.C.data(), q.C.size() * sizeof(double));
  }
  return CGTP_OK;
}

cgtp_status cgtp_forward(cgtp_plan plan, const void* x1, const void* x2, const void* W, void* out,
                         int64_t B, void* stream) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (plan->mode != CGTP_UVU) return fail(CGTP_EUNSUPPORTED, "cgtp_forward needs a uvu plan");
  if (plan->dtype == CGTP_BF16 && !plan->bt)
    return fail(CGTP_EUNSUPPORTED, "CGTP_BF16 batched products need multiplicity 16 or 32 in every path and l <= 7");
  if (B < 0 || B >= (int64_t(1) << 31)) return fail(CGTP_EINVAL, "batch size out of range");
  if (B == 0) return CGTP_OK;
  cgtp_status s;
  if ((s = need(x1, "x1")) || (s = need(x2, "x2")) || (s = need(W, "W")) || (s = need(out, "out"))) return s;
  if (bt_forward(plan, x1, x2, W, out, B, stream, &s)) return s;
  if (plan->dtype == CGTP_BF16) return fail(CGTP_EUNSUPPORTED, "batch too large for the CGTP_BF16 batched kernels");
  return launch_uvu_forward(plan, plan->batch_layout, x1, x2, W, out, nullptr, nullptr, B, true, stream);
}

cgtp_status cgtp_backward(cgtp_plan plan, const void* gout, const void* x1, const void* x2,
                          const void* W, void* gx1, void* gx2, void* gW, int64_t B, void* stream) {
  clear_error();
  if (!plan) return fail(CGTP_EINVAL, "null plan");
  if (plan->mode != CGTP_UVU) return fail(CGTP_EUNSUPPORTED, "cgtp_backward needs a uvu plan");
  if (plan->dtype == CGTP_BF16 && !plan->bt)
    return fail(CGTP_EUNSUPPORTED, "CGTP_BF16 batched products need multiplicity 16 or 32 in every path and l <= 7");
  if (B < 0 || B >= (int64_t(1) << 31)) return fail(CGTP_EINVAL, "batch size out of range");
  if (B == 0) return CGTP_OK;
  cgtp_status s;
  if ((s = need(gout, "gout")) || (s = need(x1, "x1")) || (s = need(x2, "x2")) || (s = need(W, "W")) ||
      (s = need(gx1, "gx1")) || (s = need(gx2, "gx2")) || (s = need(gW, "gW")))
    return s;
  if (bt_backward(plan, gout, x1, x2, W, gx1, gx2, gW, B, stream, &s)) return s;
  if (plan->dtype == CGTP_BF16) return fail(CGTP_EUNSUPPORTED, "batch too large for the CGTP_BF16 batched kernels");
  return launch_uvu_backward(plan, plan->batch_layout, gout, x1, x2, W, gx1, gx2, gW, nullptr, nullptr,
                             nullptr, B, true, stream);
}

cgtp_status cgtp_graph_create(cgtp_graph* out, const int32_t* rowptr, const int32_t* col, int64_t N,
                              int64_t E, void* stream) {
  clear_error();
  if (!out) return fail(CGTP_EINVAL, "null graph output pointer");
  *out = nullptr;
  if (N < 1 || N >= (int64_t(1) << 31) - 1 || E < 0 || E >= (int64_t(1) << 31))
    return fail(CGTP_EINVAL, "N must be in [1, 2^31-1) and E in [0, 2^31)");
  if (!rowptr) return fail(CGTP_EINVAL, "null rowptr");
  if (E > 0 && !col) return fail(CGTP_EINVAL, "null col");
  cgtp_graph_s* g = new (std::nothrow) cgtp_graph_s();
  if (!g) return fail(CGTP_ENOMEM, "host allocation failed");
  g->rowptr = rowptr;
  g->col = col;
  g->N = N;
  g->E = E;
  cudaGetDevice(&g->device);
  const size_t eb = std::max<int64_t>(E, 1) * sizeof(int32_t);
  if (cudaMalloc(&g->t_rowptr, (N + 1) * sizeof(int32_t)) != cudaSuccess ||
      cudaMalloc(&g->t_eid, eb) != cudaSuccess || cudaMalloc(&g->t_dst, eb) != cudaSuccess) {
    cgtp_graph_destroy(g);
    return fail(CGTP_ENOMEM, "graph allocation failed");
  }
  cgtp_status s = graph_build(g, stream);
  if (s != CGTP_OK) {
    cgtp_graph_destroy(g);
    return s;
  }
  *out = g;
  return CGTP_OK;
}

void cgtp_graph_destroy(cgtp_graph g) {
  if (!g) return;
  if (g->t_rowptr) cudaFree(g->t_rowptr);
  if (g->t_eid) cudaFree(g->t_eid);
  if (g->t_dst) cudaFree(g->t_dst);
  delete g;
}

cgtp_status cgtp_graph_transpose(cgtp_graph g, int32_t* t_rowptr, int32_t* t_eid, int32_t* t_dst,
                                 void* stream) {
  clear_error();
  if (!g) return fail(CGTP_EINVAL, "null graph");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (t_rowptr) e = cudaMemcpyAsync(t_rowptr, g->t_rowptr, (g->N + 1) * sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && t_eid && g->E)
    e = cudaMemcpyAsync(t_eid, g->t_eid, g->E * sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && t_dst && g->E)
    e = cudaMemcpyAsync(t_dst, g->t_dst, g->E * sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return fail(CGTP_ECUDA, cudaGetErrorString(e));
  return CGTP_OK;
}

cgtp_status cgtp_conv_forward(cgtp_plan plan, cgtp_graph g, const void* x, const void* Y,
                              const void* W_or_R, const void* M, void* out, void* stream) {
  clear_error();
  if (!plan || !g) return fail(CGTP_EINVAL, "null plan or graph");
  cgtp_status s;
  if ((s = need(x, "x")) || (s = need(out, "out"))) return s;
  if (g->E > 0 && ((s = need(Y, "Y")) || (s = need(W_or_R, plan->mode == CGTP_UVU ? "W" : "R")))) return s;
  if (plan->mode == CGTP_UVU) {
    if (M) return fail(CGTP_EINVAL, "M must be NULL for a uvu plan");
    return launch_uvu_forward(plan, plan->conv_layout, x, Y, W_or_R, out, g->rowptr, g->col, g->N,
                              false, stream);
  }
  if (plan->radial_k == 0) {
    if (M) return fail(CGTP_EINVAL, "M must be NULL for per-edge uvw weights");
    return uvwe_forward(plan, g, x, Y, W_or_R, out, stream);
  }
  if ((s = need(M, "M"))) return s;
  return uvw_forward(plan, g, x, Y, W_or_R, M, out, stream);
}

cgtp_status cgtp_conv_backward(cgtp_plan plan, cgtp_graph g, const void* gout, const void* x,
                               const void* Y, const void* W_or_R, const void* M, void* gx, void* gY,
                               void* gW_or_gR, void* gM, void* stream) {
  clear_error();
  if (!plan || !g) return fail(CGTP_EINVAL, "null plan or graph");
  cgtp_status s;
  if ((s = need(gout, "gout")) || (s = need(x, "x")) || (s = need(gx, "gx"))) return s;
  if (g->E > 0 && ((s = need(Y, "Y")) || (s = need(W_or_R, "W_or_R")) || (s = need(gY, "gY")) ||
                   (s = need(gW_or_gR, "gW_or_gR"))))
    return s;
  if (plan->mode == CGTP_UVU) {
    if (M || gM) return fail(CGTP_EINVAL, "M and gM must be NULL for a uvu plan");
    return launch_uvu_backward(plan, plan->conv_layout, gout, x, Y, W_or_R, gx, gY, gW_or_gR,
                               g->t_rowptr, g->t_eid, g->t_dst, g->N, false, stream);
  }
  if (plan->radial_k == 0) {
    if (M || gM) return fail(CGTP_EINVAL, "M and gM must be NULL for per-edge uvw weights");
    return uvwe_backward(plan, g, gout, x, Y, W_or_R, gx, gY, gW_or_gR, stream);
  }
  if ((s = need(M, "M")) || (s = need(gM, "gM"))) return s;
  return uvw_backward(plan, g, gout, x, Y, W_or_R, M, gx, gY, gW_or_gR, gM, stream);
}

}  // extern "C"
