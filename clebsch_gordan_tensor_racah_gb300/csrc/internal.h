// internal.h -- host/device shared definitions of the cgtp library (not public).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "cgtp.h"

namespace cgtp {

constexpr int kMaxL = 7;          // largest l of any irrep (block dims up to 15)
constexpr int kWarps = 8;         // warps per CTA of the uvu kernels
constexpr int kThreads = kWarps * 32;

struct Irrep {
  int mul, l, p;
};

// ---------------------------------------------------------------------------
// Device-side tables (plain old data, uploaded once per plan).
// ---------------------------------------------------------------------------
struct PathDev {
  int l1, l2, l3, D1, D2, D3, mul, mul_out;
  int off1, off2, ooff, woff;       // offsets in the full rows
  int ooff_g, woff_g, cyoff_g;      // offsets inside the group's out slice / W slice / cy layout
  int gxpoff_g;                     // backward: offset of the path's gx partial [mul][D1]
  int i1;                           // in1 block
  int pad_;
};

struct GroupDev {
  int p0, p1;        // path range
  int o0, o1;        // output column range
  int w0, w1;        // weight column range
  int cy_size;       // per-edge cy / gc layout size (elements, padded)
  int cy_base;       // first index of this group's slots in cy_begin
  int gy_base;       // first index of this group's Y columns in gy_begin (d2 + 1 entries)
  int gxp_size;      // elements of the gx partial buffer
  int nub;           // max number of 32-channel blocks of a path in the group
  int item_base;     // first index of this group's per-warp lists in item_begin (kWarps + 1 entries)
  int gx_base;       // first index of this group's in1 blocks in gx_begin (n_in1 + 1 entries)
  int pad_;
};

struct Item {
  int path;  // global path index
  int u0;    // first channel of the 32-channel block
};

// One partition of the plan's paths into groups that fit the shared-memory
// budget of the uvu kernels for a given edge-chunk size.
struct LayoutHost {
  int chunk = 1;
  std::vector<PathDev> paths;      // group-relative offsets filled in
  std::vector<int> in1_off;        // n_in1 + 1 offsets of the in1 blocks (last = d1)
  std::vector<GroupDev> groups;
  std::vector<int> cy_begin;       // per group: cy_size + 1 offsets into cy terms
  std::vector<int> cy_col;         // Y column of each term
  std::vector<double> cy_coef;
  std::vector<int> gy_begin;       // per group: d2 + 1 offsets into gy terms
  std::vector<int> gy_slot;        // slot in the group's gc layout
  std::vector<int> gy_nub;         // number of channel blocks to sum for that slot
  std::vector<double> gy_coef;
  std::vector<int> item_begin;     // per group: kWarps + 1
  std::vector<Item> items;
  std::vector<int> gx_begin;       // per group: n_in1 + 1 offsets into gx_paths
  std::vector<int> gx_paths;       // global path indices, in path order
  size_t smem_fwd = 0, smem_bwd = 0;
  // two-term coefficient tables (every cy slot has at most two CG terms):
  // per group and slot, cy[slot] = c0 * Y[col0] + c1 * Y[col1]
  std::vector<int> cy2_col;        // 2 per slot, concatenated over groups (offset cy_base2)
  std::vector<double> cy2_coef;    // 2 per slot
  std::vector<int> cy2_base;       // per group: first slot
  // edge-chunk size of the pipelined kernels (even) and their shared memory
  int chunk2 = 0;
  size_t smem_fwd2 = 0, smem_bwd2 = 0;
};

// Device copy of a layout: one allocation, pointers into it.
struct LayoutDev {
  int chunk = 1;
  int n_groups = 0;
  int n_in1 = 0;
  const PathDev* paths = nullptr;
  const int* in1_off = nullptr;
  const GroupDev* groups = nullptr;
  const int* cy_begin = nullptr;
  const int* cy_col = nullptr;
  const void* cy_coef = nullptr;   // float or double
  const int* gy_begin = nullptr;
  const int* gy_slot = nullptr;
  const int* gy_nub = nullptr;
  const void* gy_coef = nullptr;
  const int* item_begin = nullptr;
  const Item* items = nullptr;
  const int* gx_begin = nullptr;
  const int* gx_paths = nullptr;
  size_t smem_fwd = 0, smem_bwd = 0;
  const int* cy2_col = nullptr;
  const void* cy2_coef = nullptr;
  const int* cy2_base = nullptr;
  int chunk2 = 0;
  size_t smem_fwd2 = 0, smem_bwd2 = 0;
  void* base = nullptr;            // owning allocation
  std::vector<GroupDev> groups_host;
};

// Tables of the warp-autonomous uvu kernels (uvu3_impl.cuh); lpe == 0 when the
// plan does not qualify (it needs l <= 3 and one multiplicity m for all in1
// blocks with m / 4 in {2, 8, 32} or m a multiple of 128).
struct V3Dev {
  int lpe = 0;
  const PathDev* paths = nullptr;
  const int* item_begin = nullptr;
  const Item* items = nullptr;    // path order
  int n_items = 0;
  const Item* items_bwd = nullptr;  // the same items grouped into backward phases
  const int* phase_begin = nullptr; // n_phases + 1 offsets into items_bwd
  int n_phases = 0;
  const int* gxp_off = nullptr;
  int gxp_size = 0;
  const int* in1_off = nullptr;
  int n_in1 = 0;
  const int* gx_begin = nullptr;
  const int* gx_paths = nullptr;
  int chunk_b = 0;
  size_t smem_bwd = 0;
  void* base = nullptr;
};

struct PathHost {
  int i1, i2, io;
  int l1, l2, l3, mul1, mul_out;
  int off1, off2, ooff, woff;
  std::vector<double> C;  // dense real CG block [D1][D2][D3]
};

}  // namespace cgtp

struct cgtp_plan_s {
  int mode = 0, dtype = 0, radial_k = 0;
  std::vector<cgtp::Irrep> in1, in2, out;
  std::vector<cgtp::PathHost> paths;
  int64_t d1 = 0, d2 = 0, d_out = 0, w_numel = 0;
  int device = 0;
  int num_sms = 0;
  // uvu
  cgtp::LayoutDev conv_layout, batch_layout;
  cgtp::V3Dev v3;
  // uvw (radial) state is kept opaque here; see uvw.cu
  void* uvw = nullptr;
  // batched-product kernels for multiplicity 16 / 32 (bt.cu); null when the plan does not qualify
  void* bt = nullptr;
  // uvw with a weight matrix per edge (radial_k == 0, uvwe.cu)
  void* uvwe = nullptr;
  // device memory the plan owns (tables, work counters, scratch), for cgtp_plan_device_bytes
  size_t device_bytes = 0;
  // polls of an mbarrier before a bounded wait of the plan's kernels gives up
  long long wait_limit = 1ll << 22;
};

struct cgtp_graph_s {
  const int32_t* rowptr = nullptr;
  const int32_t* col = nullptr;
  int64_t N = 0, E = 0;
  int32_t* t_rowptr = nullptr;
  int32_t* t_eid = nullptr;
  int32_t* t_dst = nullptr;
  int device = 0;
};

namespace cgtp {

// errors.cpp / planner.cpp
cgtp_status fail(cgtp_status s, const std::string& msg);
void clear_error();
// Raise a kernel's dynamic shared-memory limit to the device's opt-in cap minus
// the kernel's static shared memory and return that cap (-1 on a CUDA error).
// The limit belongs to the kernel and is shared by every plan, so it is only
// ever raised to the cap, never set to one plan's need.
int raise_smem_limit(const void* kernel);
// The same, done once per (kernel, device) and remembered (thread-safe).
int smem_cap_cached(const void* kernel);

bool parse_irreps(const char* s, std::vector<Irrep>* out, std::string* err);
double cg_complex(int j1, int m1, int j2, int m2, int J, int M);
std::vector<double> real_cg_block(int l1, int l2, int l3);
cgtp_status build_paths(cgtp_plan_s* plan, const cgtp_instr* instr, int n_instr);
cgtp_status build_layout(const cgtp_plan_s* plan, int chunk, size_t smem_budget, LayoutHost* out);

// device-side helpers (api.cu)
cgtp_status upload_layout(const cgtp_plan_s* plan, const LayoutHost& h, LayoutDev* d);
void free_layout(LayoutDev* d);

// uvu.cu
cgtp_status launch_uvu_forward(const cgtp_plan_s* plan, const LayoutDev& lay, const void* x,
                               const void* Y, const void* W, void* out, const int32_t* rowptr,
                               const int32_t* col, int64_t N, bool identity, void* stream);
cgtp_status launch_uvu_backward(const cgtp_plan_s* plan, const LayoutDev& lay, const void* gout,
                                const void* x, const void* Y, const void* W, void* gx, void* gY,
                                void* gW, const int32_t* t_rowptr, const int32_t* t_eid,
                                const int32_t* t_dst, int64_t N, bool identity, void* stream);

// uvu3.cu
cgtp_status build_v3(cgtp_plan_s* plan);
void free_v3(cgtp_plan_s* plan);
// rvec: edge vectors [E,3] whose harmonics replace Y (null: read Y)
bool launch_v3_forward(const cgtp_plan_s* plan, const void* x, const void* Y, const void* W, void* out,
                       const int32_t* rowptr, const int32_t* col, int64_t N, void* stream, cgtp_status* st,
                       const void* rvec = nullptr);
bool launch_v3_backward(const cgtp_plan_s* plan, const void* gout, const void* x, const void* Y,
                        const void* W, void* gx, void* gY, void* gW, const int32_t* t_rowptr,
                        const int32_t* t_eid, const int32_t* t_dst, int64_t N, void* stream,
                        cgtp_status* st, const void* rvec = nullptr);

// uvwe.cu (uvw with per-edge weights W [E, w_numel])
cgtp_status uvwe_create(cgtp_plan_s* plan);
void uvwe_destroy(cgtp_plan_s* plan);
cgtp_status uvwe_forward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* x, const void* Y,
                         const void* W, void* out, void* stream);
cgtp_status uvwe_backward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* gout, const void* x,
                          const void* Y, const void* W, void* gx, void* gY, void* gW, void* stream);

// bt.cu (batched product without a graph; return false when the plan does not qualify)
cgtp_status bt_create(cgtp_plan_s* plan);
void bt_destroy(cgtp_plan_s* plan);
bool bt_forward(const cgtp_plan_s* plan, const void* x1, const void* x2, const void* W, void* out,
                int64_t B, void* stream, cgtp_status* status);
bool bt_backward(const cgtp_plan_s* plan, const void* gout, const void* x1, const void* x2, const void* W,
                 void* gx1, void* gx2, void* gW, int64_t B, void* stream, cgtp_status* status);

// graph.cu
cgtp_status graph_build(cgtp_graph_s* g, void* stream);

// uvw.cu
cgtp_status uvw_create(cgtp_plan_s* plan);
// nodes per streamed chunk of the radial plan's node state (reallocates the scratch)
cgtp_status uvw_set_chunk(cgtp_plan_s* plan, int nodes);
int uvw_chunk(const cgtp_plan_s* plan);
void uvw_destroy(cgtp_plan_s* plan);
// rvec non-null: Y and R are evaluated from the edge vectors (harmonics of the
// direction, Gaussian radial basis of the length with centres lo..hi)
cgtp_status uvw_forward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* x,
                        const void* Y, const void* R, const void* M, void* out, void* stream,
                        const void* rvec = nullptr, double rbf_lo = 0.0, double rbf_hi = 0.0);
cgtp_status uvw_backward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* gout,
                         const void* x, const void* Y, const void* R, const void* M, void* gx,
                         void* gY, void* gR, void* gM, void* stream, const void* rvec = nullptr,
                         double rbf_lo = 0.0, double rbf_hi = 0.0);

}  // namespace cgtp
