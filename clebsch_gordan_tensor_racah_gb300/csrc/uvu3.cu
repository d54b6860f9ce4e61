// uvu3.cu -- host side of the warp-autonomous uvu kernels (uvu3_impl.cuh):
// qualification, work items, launches.  Kernels are instantiated in
// uvu3_<variant>_<lanes>.cu.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "internal.h"

namespace cgtp {
namespace uvu3_detail {
// instantiated in uvu3_<variant>_<lanes>.cu (uvu3_launch.cuh)
template <typename T, typename S, bool SH, int LPE>
cgtp_status v3_forward(const cgtp_plan_s* plan, const void* x, const void* E_in, const void* W, void* out,
                       const int32_t* rowptr, const int32_t* col, int64_t N, cudaStream_t st);
template <typename T, typename S, bool SH, int LPE>
cgtp_status v3_backward(const cgtp_plan_s* plan, const void* gout, const void* x, const void* E_in,
                        const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                        const int32_t* t_eid, const int32_t* t_dst, int64_t N, cudaStream_t st);

// calls f with the plan's lanes per edge as a compile-time constant
template <typename F>
bool v3_pick(int lpe, F&& f) {
  switch (lpe) {
    case 2: f(std::integral_constant<int, 2>{}); return true;
    case 8: f(std::integral_constant<int, 8>{}); return true;
    case 32: f(std::integral_constant<int, 32>{}); return true;
    default: return false;
  }
}
}  // namespace uvu3_detail

cgtp_status build_v3(cgtp_plan_s* plan) {
  plan->v3 = V3Dev{};
  if (plan->mode != CGTP_UVU || plan->paths.empty()) return CGTP_OK;
  const int m = plan->in1.front().mul;
  for (const auto& b : plan->in1)
    if (b.mul != m || b.l > 3) return CGTP_OK;
  for (const auto& p : plan->paths)
    if (p.l2 > 3 || p.l3 > 3) return CGTP_OK;
  int lpe = 0;
  if (m % 4 == 0 && (m / 4 == 2 || m / 4 == 8 || m / 4 == 32)) lpe = m / 4;
  else if (m % 128 == 0) lpe = 32;
  if (!lpe) return CGTP_OK;
  const int ublock = 4 * lpe;
  // work items: (path, channel block) in path order -- the kernels walk them
  // path-major, all warps of a CTA on the same path at a time
  std::vector<Item> items;
  for (size_t p = 0; p < plan->paths.size(); ++p)
    for (int u0 = 0; u0 < plan->paths[p].mul1; u0 += ublock) items.push_back({int(p), u0});
  std::vector<int> item_begin = {0, int(items.size())};
  // backward phases: at most kPhaseItems items that share no in1 block and no
  // in2 block (their gx / gY slices are disjoint), taken greedily from the
  // remaining items in path order
  constexpr int kPhaseItems = 4;
  std::vector<Item> items_bwd;
  std::vector<int> phase_begin = {0};
  {
    std::vector<char> used(items.size(), 0);
    size_t left = items.size();
    while (left) {
      std::vector<int> i1s, i2s;
      int taken = 0;
      for (size_t k = 0; k < items.size() && taken < kPhaseItems; ++k) {
        if (used[k]) continue;
        const PathHost& ph = plan->paths[items[k].path];
        if (std::find(i1s.begin(), i1s.end(), ph.i1) != i1s.end() ||
            std::find(i2s.begin(), i2s.end(), ph.i2) != i2s.end())
          continue;
        i1s.push_back(ph.i1);
        i2s.push_back(ph.i2);
        items_bwd.push_back(items[k]);
        used[k] = 1;
        --left;
        ++taken;
      }
      phase_begin.push_back(int(items_bwd.size()));
    }
  }
  // gx partial buffer: one [mul][D1] block per path
  std::vector<int> gxp_off;
  int gxp = 0;
  for (const auto& q : plan->paths) {
    gxp_off.push_back(gxp);
    gxp += q.mul1 * (2 * q.l1 + 1);
  }
  std::vector<int> in1_off;
  int o = 0;
  for (const auto& b : plan->in1) {
    in1_off.push_back(o);
    o += b.mul * (2 * b.l + 1);
  }
  in1_off.push_back(o);
  std::vector<int> gx_begin, gx_paths;
  for (size_t b = 0; b < plan->in1.size(); ++b) {
    gx_begin.push_back(int(gx_paths.size()));
    for (size_t p = 0; p < plan->paths.size(); ++p)
      if (plan->paths[p].i1 == int(b)) gx_paths.push_back(int(p));
  }
  gx_begin.push_back(int(gx_paths.size()));
  // upload
  std::vector<unsigned char> buf;
  auto put = [&](const void* src, size_t bytes) {
    const size_t off = (buf.size() + 15) / 16 * 16;
    buf.resize(off + bytes);
    if (bytes) std::memcpy(buf.data() + off, src, bytes);
    return off;
  };
  const size_t o_ib = put(item_begin.data(), item_begin.size() * sizeof(int));
  const size_t o_it = put(items.data(), items.size() * sizeof(Item));
  const size_t o_ib2 = put(items_bwd.data(), items_bwd.size() * sizeof(Item));
  const size_t o_ph = put(phase_begin.data(), phase_begin.size() * sizeof(int));
  const size_t o_gxo = put(gxp_off.data(), gxp_off.size() * sizeof(int));
  const size_t o_in1 = put(in1_off.data(), in1_off.size() * sizeof(int));
  const size_t o_gxb = put(gx_begin.data(), gx_begin.size() * sizeof(int));
  const size_t o_gxq = put(gx_paths.data(), std::max<size_t>(gx_paths.size(), 1) * sizeof(int));
  void* base = nullptr;
  if (cudaMalloc(&base, buf.size()) != cudaSuccess) return fail(CGTP_ENOMEM, "plan table allocation failed");
  plan->device_bytes += buf.size();
  if (cudaMemcpy(base, buf.data(), buf.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(base);
    return fail(CGTP_ECUDA, "plan table upload failed");
  }
  auto at = [&](size_t off) { return static_cast<unsigned char*>(base) + off; };
  V3Dev& v = plan->v3;
  v.base = base;
  v.lpe = lpe;
  v.paths = plan->conv_layout.paths;  // global offsets off1, off2, ooff, woff
  v.item_begin = reinterpret_cast<const int*>(at(o_ib));
  v.items = reinterpret_cast<const Item*>(at(o_it));
  v.n_items = int(items.size());
  v.items_bwd = reinterpret_cast<const Item*>(at(o_ib2));
  v.phase_begin = reinterpret_cast<const int*>(at(o_ph));
  v.n_phases = int(phase_begin.size()) - 1;
  v.gxp_off = reinterpret_cast<const int*>(at(o_gxo));
  v.gxp_size = gxp;
  v.in1_off = reinterpret_cast<const int*>(at(o_in1));
  v.n_in1 = int(plan->in1.size());
  v.gx_begin = reinterpret_cast<const int*>(at(o_gxb));
  v.gx_paths = reinterpret_cast<const int*>(at(o_gxq));
  const size_t es = plan->dtype == CGTP_F64 ? 8 : 4;
  v.chunk_b = 64;
  auto smem = [&](int cb) { return es * (size_t(gxp + 3) / 4 * 4 + size_t(kWarps) * cb * plan->d2); };
  while (v.chunk_b > 8 && smem(v.chunk_b) > 200 * 1024) v.chunk_b /= 2;
  v.smem_bwd = smem(v.chunk_b);
  if (v.smem_bwd > 220 * 1024) v.lpe = 0;  // gx partials too large: the general kernels serve this plan
  return CGTP_OK;
}

void free_v3(cgtp_plan_s* plan) {
  if (plan->v3.base) cudaFree(plan->v3.base);
  plan->v3 = V3Dev{};
}

bool launch_v3_forward(const cgtp_plan_s* plan, const void* x, const void* Y, const void* W, void* out,
                       const int32_t* rowptr, const int32_t* col, int64_t N, void* stream, cgtp_status* st,
                       const void* rvec) {
  using namespace uvu3_detail;
  if (!plan->v3.lpe) return false;
  if ((int64_t)plan->v3.n_items * N >= (int64_t(1) << 31)) {  // the kernels' 32-bit work counters
    if (plan->dtype != CGTP_BF16) return false;
    *st = fail(CGTP_EUNSUPPORTED, "graph too large for the bfloat16 kernels (paths x nodes >= 2^31)");
    return true;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int lpe = plan->v3.lpe;
  auto go = [&](auto tag_t, auto tag_s, auto sh) {
    using T = decltype(tag_t);
    using S = decltype(tag_s);
    constexpr bool SH = decltype(sh)::value;
    return v3_pick(lpe, [&](auto L) {
      *st = v3_forward<T, S, SH, decltype(L)::value>(plan, x, SH ? rvec : Y, W, out, rowptr, col, N, s);
    });
  };
  if (plan->dtype == CGTP_BF16)  // only these kernels read bfloat16 inputs
    return go(float{}, __nv_bfloat16{}, std::false_type{});
  const bool f64 = plan->dtype == CGTP_F64;
  if (rvec)  // edge vectors: the harmonics are evaluated in the kernels
    return f64 ? go(double{}, double{}, std::true_type{}) : go(float{}, float{}, std::true_type{});
  return f64 ? go(double{}, double{}, std::false_type{}) : go(float{}, float{}, std::false_type{});
}

bool launch_v3_backward(const cgtp_plan_s* plan, const void* gout, const void* x, const void* Y,
                        const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                        const int32_t* t_eid, const int32_t* t_dst, int64_t N, void* stream,
                        cgtp_status* st, const void* rvec) {
  using namespace uvu3_detail;
  if (!plan->v3.lpe) return false;
  if ((int64_t)plan->v3.n_items * N >= (int64_t(1) << 31)) {  // the kernels' 32-bit work counters
    if (plan->dtype != CGTP_BF16) return false;
    *st = fail(CGTP_EUNSUPPORTED, "graph too large for the bfloat16 kernels (paths x nodes >= 2^31)");
    return true;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int lpe = plan->v3.lpe;
  auto go = [&](auto tag_t, auto tag_s, auto sh) {
    using T = decltype(tag_t);
    using S = decltype(tag_s);
    constexpr bool SH = decltype(sh)::value;
    return v3_pick(lpe, [&](auto L) {
      *st = v3_backward<T, S, SH, decltype(L)::value>(plan, gout, x, SH ? rvec : Y, W, gx, gY, gW, t_rowptr,
                                                      t_eid, t_dst, N, s);
    });
  };
  if (plan->dtype == CGTP_BF16) return go(float{}, __nv_bfloat16{}, std::false_type{});
  const bool f64 = plan->dtype == CGTP_F64;
  if (rvec) return f64 ? go(double{}, double{}, std::true_type{}) : go(float{}, float{}, std::true_type{});
  return f64 ? go(double{}, double{}, std::false_type{}) : go(float{}, float{}, std::false_type{});
}

}  // namespace cgtp
