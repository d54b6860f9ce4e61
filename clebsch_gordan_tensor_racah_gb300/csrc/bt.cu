// bt.cu -- batched uvu tensor product without a graph (one independent product
// per sample), for plans whose paths all have multiplicity 16 or 32 and l <= 7.
//
// "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
// Figure 4A (the batched product) and Figure 5 (its benchmark at batch 50K);
// the OEQ discussion "The GPU memory optimization with Larger angular
// momentum" (interactions up to L = 7, and nonzeros baked into the instruction
// stream spilling the instruction cache).  Per sample b and path p = (l1,l2,l3):
//
//   cy[m3][m1]   = sum_m2 C[m1,m2,m3] y[b][m2]                 (coupling matrix)
//   out[b][p][u][m3] = W[b][p,u] sum_m1 cy[m3][m1] x[b][u][m1]
//   gW[b][p,u]   = sum_m3 g[b][p][u][m3] sum_m1 cy[m3][m1] x[b][u][m1]
//   gx[b][u][m1] = sum_{p on that in1 block} sum_m3 cy[m3][m1] W[b][p,u] g[b][p][u][m3]
//   G[m3][m1]    = sum_u x[b][u][m1] W[b][p,u] g[b][p][u][m3]
//   gy[b][m2]    = sum_p sum_{m1,m3} C[m1,m2,m3] G[m3][m1]
//
// GB300 organisation.  At L = 7 there are 260 paths and ~24k CG nonzeros, far
// too many to bake into code, so the coefficients are tables: every cy entry
// has at most two CG terms (real basis), and the gy contraction is a list of
// (G slot, coefficient) per m2.  The paths are cut into contiguous groups whose
// tables fit a CTA's shared memory; grid.y is the group and grid.x a slice of
// the samples, so each CTA loads its tables once and then streams samples.
// Lanes map to channels (lanes per sample = multiplicity, 16 -> two samples a
// warp), every warp works on its own samples with only warp barriers:
//   * cy is formed by the sample's lanes into a per-warp buffer, rows padded
//     to a multiple of four so the contraction reads it as broadcast float4;
//   * the channel contraction uses the paired FP32 FMA (fma.rn.f32x2);
//   * outputs go through a per-warp tile and leave as streaming float4 stores
//     (the forward writes 7.7 GB at L = 7: the kernel is write-bandwidth bound);
//   * backward: lane u forms W*g for its channel and the lane holding m1 forms
//     G[.][m1] from the transposed W*g rows (into the dead cy buffer); lanes m2
//     then apply the gy table.
// gx blocks shared by several groups and gy (every group touches it) leave as
// per-group partials in a bounded plan-owned scratch (chunks of samples) and a
// reduce kernel adds them in group order: deterministic, no atomics.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "internal.h"

namespace cgtp {
namespace bt_detail {

constexpr int kBtWarps = 8;
constexpr int kBtThreads = kBtWarps * 32;
constexpr int kMaxD = 15;                // largest block dimension (l <= 7)
constexpr int kCyW = kMaxD * 16;         // per-sample cy / G buffer: [m3 < 15][m1 < 16]
constexpr int kGStride = 16;             // row stride of the G buffer
constexpr size_t kTableBudget = 44 * 1024;
constexpr size_t kScratchBytes = size_t(64) << 20;

struct BtPath {   // 16 ints
  int D1, D2, D3, Q;        // Q = D1 rounded up to a multiple of 4, divided by 4
  int off1, off2, ooff, woff;
  int ctab;                 // first cy entry of the path (group-relative), D3 * 4Q entries
  int grow;                 // first gy row pointer (group-relative), D2 + 1 of them
  int gxo;                  // gx destination: offset in the gx row (gxp = 0) or in the scratch row
  int gxp;                  // 1: the path's in1 block is shared with other groups
  int flush;                // 1: last path of its in1 run inside the group
  int pad0, pad1, pad2;
};
static_assert(sizeof(BtPath) == 64, "BtPath is 64 bytes");

struct BtGroup {
  int p0, p1;               // path range
  int ctab0, ctab_n;        // cy entries
  int grow0, grow_n;        // gy row pointers
  int gent0, gent_n;        // gy entries
  int gy_part;              // offset of the group's gy partial in the scratch row
  int pad0, pad1, pad2;
};

struct BtArgs {
  const float* x;
  const float* y;
  const float* W;
  const float* gout;
  float* out;
  float* gx;
  float* gW;
  float* scratch;
  int b0, b1;               // samples [b0, b1) of this launch
  int d1, d2, d2p, d_out, w_numel;
  int scratch_row;
  int slices;
  int warp_floats;
  const BtPath* paths;
  const BtGroup* groups;
  const float2* ccoef;
  const uint16_t* ccol;
  const int* grow;
  const float2* gent;
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
        "l"(*reinterpret_cast<unsigned long long*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

// cy[m3][m1] of one sample: the sample's lanes split the D3 x 4Q entries
template <int LPS, int Q>
__device__ __forceinline__ void coupling(const BtPath& p, const float2* sc, const uint16_t* scol,
                                         const float* ysw, float* cyw, int q) {
  const int ne = p.D3 * 4 * Q;
  const float* yb = ysw + p.off2;
  for (int e = q; e < ne; e += LPS) {
    const float2 c = sc[p.ctab + e];
    const unsigned cc = scol[p.ctab + e];
    cyw[e] = fmaf(c.y, yb[cc >> 8], c.x * yb[cc & 255u]);
  }
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <int LPS, int Q>
__device__ __forceinline__ void fwd_path(const BtPath& p, const BtArgs& a, const float2* sc,
                                         const uint16_t* scol, const float* ysw, float* cyw, float* tw,
                                         int b, bool valid, int q) {
  constexpr int D1P = 4 * Q;
  float xv[D1P];
  const float* xr = a.x + (size_t)b * a.d1 + p.off1 + q * p.D1;
#pragma unroll
  for (int m = 0; m < D1P; ++m) xv[m] = (valid && m < p.D1) ? __ldg(xr + m) : 0.f;
  const float w = valid ? __ldg(a.W + (size_t)b * a.w_numel + p.woff + q) : 0.f;
  coupling<LPS, Q>(p, sc, scol, ysw, cyw, q);
  __syncwarp();
  // m3 unrolled to its bound (warp-uniform guards): independent accumulators
#pragma unroll
  for (int m3 = 0; m3 < kMaxD; ++m3) {
    if (m3 < p.D3) {
      const float4* row = reinterpret_cast<const float4*>(cyw + m3 * D1P);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < Q; ++j) {
        const float4 c = row[j];
        acc = fma2(make_float2(c.x, c.y), make_float2(xv[4 * j], xv[4 * j + 1]), acc);
        acc = fma2(make_float2(c.z, c.w), make_float2(xv[4 * j + 2], xv[4 * j + 3]), acc);
      }
      tw[q * p.D3 + m3] = w * (acc.x + acc.y);
    }
  }
  __syncwarp();
  if (valid) {
    const int nv = p.D3 * LPS / 4;
    float4* dst = reinterpret_cast<float4*>(a.out + (size_t)b * a.d_out + p.ooff);
    const float4* src = reinterpret_cast<const float4*>(tw);
    for (int i = q; i < nv; i += LPS) __stcs(dst + i, src[i]);
  }
}

template <int LPS>
__global__ void __launch_bounds__(kBtThreads, 2) bt_forward_kernel(const BtArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int SPW = 32 / LPS;
  const BtGroup grp = a.groups[blockIdx.y];
  const int np = grp.p1 - grp.p0;
  BtPath* sp = reinterpret_cast<BtPath*>(smem);
  float2* sc = reinterpret_cast<float2*>(smem + (size_t)np * sizeof(BtPath));
  uint16_t* scol = reinterpret_cast<uint16_t*>(sc + grp.ctab_n);
  float* wbuf = reinterpret_cast<float*>(smem + al16((size_t)np * sizeof(BtPath) + (size_t)grp.ctab_n * 10));
  const int tid = threadIdx.x;
  for (int i = tid; i < np * 16; i += kBtThreads)
    reinterpret_cast<int*>(sp)[i] = reinterpret_cast<const int*>(a.paths + grp.p0)[i];
  for (int i = tid; i < grp.ctab_n; i += kBtThreads) {
    sc[i] = a.ccoef[grp.ctab0 + i];
    scol[i] = a.ccol[grp.ctab0 + i];
  }
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5, q = lane % LPS, s = lane / LPS;
  float* ys = wbuf + (size_t)warp * a.warp_floats;
  float* ysw = ys + s * a.d2p;
  float* cyw = ys + SPW * a.d2p + s * kCyW;
  float* tw = ys + SPW * (a.d2p + kCyW) + s * (LPS * kMaxD);
  const int nS = a.b1 - a.b0;
  const int sb = a.b0 + (int)((long long)nS * blockIdx.x / a.slices);
  const int se = a.b0 + (int)((long long)nS * (blockIdx.x + 1) / a.slices);
  for (int base = sb + warp * SPW; base < se; base += kBtWarps * SPW) {
    const int bs = base + s;
    const bool valid = bs < se;
    const int b = valid ? bs : base;
    for (int i = q; i < a.d2; i += LPS) ysw[i] = valid ? __ldg(a.y + (size_t)b * a.d2 + i) : 0.f;
    __syncwarp();
    for (int pi = 0; pi < np; ++pi) {
      const BtPath p = sp[pi];
      switch (p.Q) {
        case 1: fwd_path<LPS, 1>(p, a, sc, scol, ysw, cyw, tw, b, valid, q); break;
        case 2: fwd_path<LPS, 2>(p, a, sc, scol, ysw, cyw, tw, b, valid, q); break;
        case 3: fwd_path<LPS, 3>(p, a, sc, scol, ysw, cyw, tw, b, valid, q); break;
        default: fwd_path<LPS, 4>(p, a, sc, scol, ysw, cyw, tw, b, valid, q); break;
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
template <int LPS, int Q>
__device__ __forceinline__ void bwd_path(const BtPath& p, const BtArgs& a, const float2* sc,
                                         const uint16_t* scol, const int* sgrow, const float2* sgent,
                                         const float* ysw, float* cyw, float* wgw, float* gyw,
                                         float2 (&gxa)[8], int b, bool valid, int q, float* srow) {
  constexpr int D1P = 4 * Q;
  const float* xr = a.x + (size_t)b * a.d1 + p.off1;
  float xv[D1P], xt[LPS];
#pragma unroll
  for (int m = 0; m < D1P; ++m) xv[m] = (valid && m < p.D1) ? __ldg(xr + q * p.D1 + m) : 0.f;
  const bool own_m1 = valid && q < p.D1;
#pragma unroll
  for (int u = 0; u < LPS; ++u) xt[u] = own_m1 ? __ldg(xr + u * p.D1 + q) : 0.f;
  const float w = valid ? __ldg(a.W + (size_t)b * a.w_numel + p.woff + q) : 0.f;
  // the path's output-gradient slice of this channel, all loads in flight at once
  const float* gr = a.gout + (size_t)b * a.d_out + p.ooff + q * p.D3;
  float gv[kMaxD];
#pragma unroll
  for (int m3 = 0; m3 < kMaxD; ++m3) gv[m3] = (valid && m3 < p.D3) ? __ldg(gr + m3) : 0.f;
  coupling<LPS, Q>(p, sc, scol, ysw, cyw, q);
  __syncwarp();
  // t = cy x (-> gW), gx += cy^T (W g); W g goes to the transposed buffer
  float gw = 0.f;
#pragma unroll
  for (int m3 = 0; m3 < kMaxD; ++m3) {
    if (m3 < p.D3) {
      const float wg = w * gv[m3];
      wgw[m3 * LPS + q] = wg;
      const float2 wg2 = make_float2(wg, wg);
      const float4* row = reinterpret_cast<const float4*>(cyw + m3 * D1P);
      float2 t = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < Q; ++j) {
        const float4 c = row[j];
        const float2 c01 = make_float2(c.x, c.y), c23 = make_float2(c.z, c.w);
        t = fma2(c01, make_float2(xv[4 * j], xv[4 * j + 1]), t);
        t = fma2(c23, make_float2(xv[4 * j + 2], xv[4 * j + 3]), t);
        gxa[2 * j] = fma2(c01, wg2, gxa[2 * j]);
        gxa[2 * j + 1] = fma2(c23, wg2, gxa[2 * j + 1]);
      }
      gw = fmaf(gv[m3], t.x + t.y, gw);
    }
  }
  if (valid) a.gW[(size_t)b * a.w_numel + p.woff + q] = gw;
  __syncwarp();
  // G[m3][m1] = sum_u x[u][m1] (W g)[u][m3]; lane q holds m1 = q.  G reuses the
  // cy buffer (cy is dead once the contraction above is done).
  float* Gw = cyw;
  if (q < p.D1) {
#pragma unroll
    for (int m3 = 0; m3 < kMaxD; ++m3) {
      if (m3 < p.D3) {
        const float4* r = reinterpret_cast<const float4*>(wgw + m3 * LPS);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < LPS / 4; ++j) {
          const float4 c = r[j];
          acc = fma2(make_float2(c.x, c.y), make_float2(xt[4 * j], xt[4 * j + 1]), acc);
          acc = fma2(make_float2(c.z, c.w), make_float2(xt[4 * j + 2], xt[4 * j + 3]), acc);
        }
        Gw[m3 * kGStride + q] = acc.x + acc.y;
      }
    }
  }
  __syncwarp();
  // gy[m2] += sum C[m1,m2,m3] G[m3][m1]; lane q holds m2 = q
  if (q < p.D2) {
    const int r0 = sgrow[p.grow + q], r1 = sgrow[p.grow + q + 1];
    float v = 0.f;
    for (int r = r0; r < r1; ++r) {
      const float2 t = sgent[r];
      v = fmaf(t.x, Gw[__float_as_int(t.y)], v);
    }
    gyw[p.off2 + q] += v;
  }
  __syncwarp();  // G (the cy buffer) is rewritten by the next path's coupling stage
  if (p.flush) {
    if (valid) {
      float* dst = (p.gxp ? srow + p.gxo : a.gx + (size_t)b * a.d1 + p.gxo) + q * p.D1;
#pragma unroll
      for (int m = 0; m < D1P; ++m)
        if (m < p.D1) dst[m] = (m & 1) ? gxa[m >> 1].y : gxa[m >> 1].x;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) gxa[j] = make_float2(0.f, 0.f);
  }
}

template <int LPS>
__global__ void __launch_bounds__(kBtThreads, 2) bt_backward_kernel(const BtArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int SPW = 32 / LPS;
  const BtGroup grp = a.groups[blockIdx.y];
  const int np = grp.p1 - grp.p0;
  BtPath* sp = reinterpret_cast<BtPath*>(smem);
  float2* sc = reinterpret_cast<float2*>(smem + (size_t)np * sizeof(BtPath));
  uint16_t* scol = reinterpret_cast<uint16_t*>(sc + grp.ctab_n);
  const size_t o_grow = al16((size_t)np * sizeof(BtPath) + (size_t)grp.ctab_n * 10);
  int* sgrow = reinterpret_cast<int*>(smem + o_grow);
  const size_t o_gent = al16(o_grow + (size_t)grp.grow_n * 4);
  float2* sgent = reinterpret_cast<float2*>(smem + o_gent);
  float* wbuf = reinterpret_cast<float*>(smem + al16(o_gent + (size_t)grp.gent_n * 8));
  const int tid = threadIdx.x;
  for (int i = tid; i < np * 16; i += kBtThreads)
    reinterpret_cast<int*>(sp)[i] = reinterpret_cast<const int*>(a.paths + grp.p0)[i];
  for (int i = tid; i < grp.ctab_n; i += kBtThreads) {
    sc[i] = a.ccoef[grp.ctab0 + i];
    scol[i] = a.ccol[grp.ctab0 + i];
  }
  for (int i = tid; i < grp.grow_n; i += kBtThreads) sgrow[i] = a.grow[grp.grow0 + i];
  for (int i = tid; i < grp.gent_n; i += kBtThreads) sgent[i] = a.gent[grp.gent0 + i];
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5, q = lane % LPS, s = lane / LPS;
  float* wb = wbuf + (size_t)warp * a.warp_floats;
  float* ysw = wb + s * a.d2p;
  float* gyw = wb + SPW * a.d2p + s * a.d2p;
  float* cyw = wb + 2 * SPW * a.d2p + s * kCyW;
  float* wgw = wb + 2 * SPW * a.d2p + SPW * kCyW + s * (kMaxD * LPS);
  const int nS = a.b1 - a.b0;
  const int sb = a.b0 + (int)((long long)nS * blockIdx.x / a.slices);
  const int se = a.b0 + (int)((long long)nS * (blockIdx.x + 1) / a.slices);
  for (int base = sb + warp * SPW; base < se; base += kBtWarps * SPW) {
    const int bs = base + s;
    const bool valid = bs < se;
    const int b = valid ? bs : base;
    float* srow = a.scratch + (size_t)(b - a.b0) * a.scratch_row;
    for (int i = q; i < a.d2; i += LPS) {
      ysw[i] = valid ? __ldg(a.y + (size_t)b * a.d2 + i) : 0.f;
      gyw[i] = 0.f;
    }
    __syncwarp();
    float2 gxa[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) gxa[j] = make_float2(0.f, 0.f);
    for (int pi = 0; pi < np; ++pi) {
      const BtPath p = sp[pi];
      switch (p.Q) {
        case 1: bwd_path<LPS, 1>(p, a, sc, scol, sgrow, sgent, ysw, cyw, wgw, gyw, gxa, b, valid, q, srow); break;
        case 2: bwd_path<LPS, 2>(p, a, sc, scol, sgrow, sgent, ysw, cyw, wgw, gyw, gxa, b, valid, q, srow); break;
        case 3: bwd_path<LPS, 3>(p, a, sc, scol, sgrow, sgent, ysw, cyw, wgw, gyw, gxa, b, valid, q, srow); break;
        default: bwd_path<LPS, 4>(p, a, sc, scol, sgrow, sgent, ysw, cyw, wgw, gyw, gxa, b, valid, q, srow); break;
      }
    }
    __syncwarp();
    if (valid)
      for (int i = q; i < a.d2; i += LPS) srow[grp.gy_part + i] = gyw[i];
    __syncwarp();
  }
}

// gy = sum of the groups' partials; gx blocks shared by several groups = sum of
// their partials (in group order); blocks no path touches are zero.
struct BtReduceArgs {
  const float* scratch;
  float* gx;
  float* gy;
  int scratch_row, d1, d2, G, n_in1;
  const int* blk;       // per in1 block: off1, size, parts, first part
  const int* part_off;  // scratch-row offsets of the parts
  int b0, n;
};

__global__ void __launch_bounds__(256) bt_reduce_kernel(const BtReduceArgs r) {
  for (int i = blockIdx.x; i < r.n; i += gridDim.x) {
    const float* row = r.scratch + (size_t)i * r.scratch_row;
    const size_t b = (size_t)(r.b0 + i);
    for (int m = threadIdx.x; m < r.d2; m += blockDim.x) {
      float v = 0.f;
      for (int g = 0; g < r.G; ++g) v += row[g * r.d2 + m];
      r.gy[b * r.d2 + m] = v;
    }
    for (int k = 0; k < r.n_in1; ++k) {
      const int off1 = __ldg(r.blk + 4 * k), size = __ldg(r.blk + 4 * k + 1);
      const int np = __ldg(r.blk + 4 * k + 2), p0 = __ldg(r.blk + 4 * k + 3);
      if (np == 1) continue;
      for (int j = threadIdx.x; j < size; j += blockDim.x) {
        float v = 0.f;
        for (int t = 0; t < np; ++t) v += row[__ldg(r.part_off + p0 + t) + j];
        r.gx[b * r.d1 + off1 + j] = v;
      }
    }
  }
}

struct BtState {
  int lps = 0;
  int G = 0;
  int d2p = 0;
  int scratch_row = 0;
  int chunk = 0;
  int wf_fwd = 0, wf_bwd = 0;
  size_t smem_fwd = 0, smem_bwd = 0;
  int slices_fwd = 1, slices_bwd = 1;
  int n_in1 = 0;
  void* tables = nullptr;
  float* scratch = nullptr;
  const BtPath* paths = nullptr;
  const BtGroup* groups = nullptr;
  const float2* ccoef = nullptr;
  const uint16_t* ccol = nullptr;
  const int* grow = nullptr;
  const float2* gent = nullptr;
  const int* blk = nullptr;
  const int* part_off = nullptr;
};

}  // namespace bt_detail

using namespace bt_detail;

cgtp_status bt_create(cgtp_plan_s* plan) {
  plan->bt = nullptr;
  if (plan->mode != CGTP_UVU || plan->dtype != CGTP_F32 || plan->paths.empty()) return CGTP_OK;
  const int m = plan->paths.front().mul1;
  if (m != 16 && m != 32) return CGTP_OK;
  for (const auto& p : plan->paths)
    if (p.mul1 != m || p.l1 > 7 || p.l2 > 7 || p.l3 > 7 || p.ooff % 4 || p.woff % 4) return CGTP_OK;
  if (plan->d_out % 4) return CGTP_OK;
  const int P = static_cast<int>(plan->paths.size());
  const int d2 = static_cast<int>(plan->d2);
  // per-path tables
  std::vector<BtPath> bp(P);
  std::vector<std::vector<float2>> pc(P);
  std::vector<std::vector<uint16_t>> pcol(P);
  std::vector<std::vector<int>> prow(P);
  std::vector<std::vector<float2>> pent(P);
  std::vector<size_t> bytes(P);
  for (int i = 0; i < P; ++i) {
    const PathHost& h = plan->paths[i];
    const int D1 = 2 * h.l1 + 1, D2 = 2 * h.l2 + 1, D3 = 2 * h.l3 + 1;
    const int Q = (D1 + 3) / 4, D1P = 4 * Q;
    auto C = [&](int m1, int m2, int m3) { return h.C[(size_t(m1) * D2 + m2) * D3 + m3]; };
    BtPath& b = bp[i];
    std::memset(&b, 0, sizeof(b));
    b.D1 = D1; b.D2 = D2; b.D3 = D3; b.Q = Q;
    b.off1 = h.off1; b.off2 = h.off2; b.ooff = h.ooff; b.woff = h.woff;
    pc[i].assign(size_t(D3) * D1P, make_float2(0.f, 0.f));
    pcol[i].assign(size_t(D3) * D1P, 0);
    for (int m3 = 0; m3 < D3; ++m3)
      for (int m1 = 0; m1 < D1; ++m1) {
        int k = 0;
        float co[2] = {0.f, 0.f};
        int cl[2] = {0, 0};
        for (int m2 = 0; m2 < D2; ++m2) {
          const double c = C(m1, m2, m3);
          if (std::fabs(c) < 1e-15) continue;
          if (k == 2) return CGTP_OK;   // not a two-term block: the general kernels serve this plan
          co[k] = static_cast<float>(c);
          cl[k] = m2;
          ++k;
        }
        pc[i][size_t(m3) * D1P + m1] = make_float2(co[0], co[1]);
        pcol[i][size_t(m3) * D1P + m1] = static_cast<uint16_t>(cl[0] | (cl[1] << 8));
      }
    prow[i].push_back(0);
    for (int m2 = 0; m2 < D2; ++m2) {
      for (int m3 = 0; m3 < D3; ++m3)
        for (int m1 = 0; m1 < D1; ++m1) {
          const double c = C(m1, m2, m3);
          if (std::fabs(c) < 1e-15) continue;
          int slot = m3 * kGStride + m1;
          float sf;
          std::memcpy(&sf, &slot, 4);
          pent[i].push_back(make_float2(static_cast<float>(c), sf));
        }
      prow[i].push_back(static_cast<int>(pent[i].size()));
    }
    bytes[i] = sizeof(BtPath) + pc[i].size() * 10 + prow[i].size() * 4 + pent[i].size() * 8;
  }
  // contiguous path groups within the table budget; an in1 block's paths must
  // be contiguous inside a group (one gx flush per block and group)
  std::vector<BtGroup> groups;
  {
    int p0 = 0;
    size_t acc = 0;
    for (int i = 0; i < P; ++i) {
      if (i > p0 && acc + bytes[i] > kTableBudget) {
        BtGroup g{};
        g.p0 = p0; g.p1 = i;
        groups.push_back(g);
        p0 = i;
        acc = 0;
      }
      acc += bytes[i];
    }
    BtGroup g{};
    g.p0 = p0; g.p1 = P;
    groups.push_back(g);
  }
  const int G = static_cast<int>(groups.size());
  const int n_in1 = static_cast<int>(plan->in1.size());
  std::vector<std::vector<int>> touch(n_in1);  // groups touching each in1 block, in order
  for (int g = 0; g < G; ++g) {
    std::vector<int> seen;
    int last = -1;
    for (int i = groups[g].p0; i < groups[g].p1; ++i) {
      const int i1 = plan->paths[i].i1;
      if (i1 != last) {
        if (std::find(seen.begin(), seen.end(), i1) != seen.end()) return CGTP_OK;  // non-contiguous
        seen.push_back(i1);
        touch[i1].push_back(g);
        last = i1;
      }
    }
  }
  // scratch row: G gy partials, then the partial gx blocks
  std::vector<int> in1_off(n_in1 + 1, 0);
  for (int k = 0; k < n_in1; ++k) in1_off[k + 1] = in1_off[k] + plan->in1[k].mul * (2 * plan->in1[k].l + 1);
  int row = G * d2;
  std::vector<int> blk(4 * n_in1), part_off;
  std::vector<std::vector<int>> part_of(n_in1);  // per block, per touching group: scratch offset
  for (int k = 0; k < n_in1; ++k) {
    const int size = in1_off[k + 1] - in1_off[k];
    blk[4 * k] = in1_off[k];
    blk[4 * k + 1] = size;
    blk[4 * k + 2] = static_cast<int>(touch[k].size());
    blk[4 * k + 3] = static_cast<int>(part_off.size());
    if (touch[k].size() >= 2)
      for (size_t t = 0; t < touch[k].size(); ++t) {
        part_of[k].push_back(row);
        part_off.push_back(row);
        row += size;
      }
  }
  row = (row + 3) / 4 * 4;
  // finish the path records and the group tables
  std::vector<float2> ccoef, gent;
  std::vector<uint16_t> ccol;
  std::vector<int> growv;
  for (int g = 0; g < G; ++g) {
    BtGroup& gr = groups[g];
    gr.ctab0 = static_cast<int>(ccoef.size());
    gr.grow0 = static_cast<int>(growv.size());
    gr.gent0 = static_cast<int>(gent.size());
    gr.gy_part = g * d2;
    for (int i = gr.p0; i < gr.p1; ++i) {
      BtPath& b = bp[i];
      const int i1 = plan->paths[i].i1;
      b.ctab = static_cast<int>(ccoef.size()) - gr.ctab0;
      b.grow = static_cast<int>(growv.size()) - gr.grow0;
      const int ent_base = static_cast<int>(gent.size()) - gr.gent0;
      ccoef.insert(ccoef.end(), pc[i].begin(), pc[i].end());
      ccol.insert(ccol.end(), pcol[i].begin(), pcol[i].end());
      for (int r : prow[i]) growv.push_back(ent_base + r);
      gent.insert(gent.end(), pent[i].begin(), pent[i].end());
      b.flush = (i + 1 == gr.p1 || plan->paths[i + 1].i1 != i1) ? 1 : 0;
      if (touch[i1].size() >= 2) {
        const size_t t = std::find(touch[i1].begin(), touch[i1].end(), g) - touch[i1].begin();
        b.gxp = 1;
        b.gxo = part_of[i1][t];
      } else {
        b.gxp = 0;
        b.gxo = in1_off[i1];
      }
    }
    gr.ctab_n = static_cast<int>(ccoef.size()) - gr.ctab0;
    gr.grow_n = static_cast<int>(growv.size()) - gr.grow0;
    gr.gent_n = static_cast<int>(gent.size()) - gr.gent0;
  }
  BtState* st = new BtState();
  st->lps = m;
  st->G = G;
  st->n_in1 = n_in1;
  st->d2p = (d2 + 3) / 4 * 4;
  st->scratch_row = row;
  const int spw = 32 / m;
  st->wf_fwd = (spw * (st->d2p + kCyW + m * kMaxD) + 3) / 4 * 4;
  st->wf_bwd = (spw * (2 * st->d2p + kCyW + m * kMaxD) + 3) / 4 * 4;
  for (const BtGroup& g : groups) {
    const size_t np = g.p1 - g.p0;
    const size_t t_fwd = al16(np * sizeof(BtPath) + size_t(g.ctab_n) * 10);
    const size_t t_grow = al16(t_fwd + size_t(g.grow_n) * 4);
    const size_t t_bwd = al16(t_grow + size_t(g.gent_n) * 8);
    st->smem_fwd = std::max(st->smem_fwd, t_fwd + size_t(kBtWarps) * st->wf_fwd * 4);
    st->smem_bwd = std::max(st->smem_bwd, t_bwd + size_t(kBtWarps) * st->wf_bwd * 4);
  }
  if (st->smem_fwd > 200 * 1024 || st->smem_bwd > 200 * 1024) {
    delete st;
    return CGTP_OK;
  }
  // upload
  std::vector<unsigned char> buf;
  auto put = [&](const void* src, size_t nbytes) {
    const size_t off = (buf.size() + 15) / 16 * 16;
    buf.resize(off + std::max<size_t>(nbytes, 16));
    if (nbytes) std::memcpy(buf.data() + off, src, nbytes);
    return off;
  };
  const size_t o_p = put(bp.data(), bp.size() * sizeof(BtPath));
  const size_t o_g = put(groups.data(), groups.size() * sizeof(BtGroup));
  const size_t o_cc = put(ccoef.data(), ccoef.size() * sizeof(float2));
  const size_t o_cl = put(ccol.data(), ccol.size() * sizeof(uint16_t));
  const size_t o_gr = put(growv.data(), growv.size() * sizeof(int));
  const size_t o_ge = put(gent.data(), gent.size() * sizeof(float2));
  const size_t o_bk = put(blk.data(), blk.size() * sizeof(int));
  const size_t o_po = put(part_off.data(), part_off.size() * sizeof(int));
  if (cudaMalloc(&st->tables, buf.size()) != cudaSuccess) {
    delete st;
    return fail(CGTP_ENOMEM, "batched-product table allocation failed");
  }
  if (cudaMemcpy(st->tables, buf.data(), buf.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(st->tables);
    delete st;
    return fail(CGTP_ECUDA, "batched-product table upload failed");
  }
  auto at = [&](size_t off) { return static_cast<unsigned char*>(st->tables) + off; };
  st->paths = reinterpret_cast<const BtPath*>(at(o_p));
  st->groups = reinterpret_cast<const BtGroup*>(at(o_g));
  st->ccoef = reinterpret_cast<const float2*>(at(o_cc));
  st->ccol = reinterpret_cast<const uint16_t*>(at(o_cl));
  st->grow = reinterpret_cast<const int*>(at(o_gr));
  st->gent = reinterpret_cast<const float2*>(at(o_ge));
  st->blk = reinterpret_cast<const int*>(at(o_bk));
  st->part_off = reinterpret_cast<const int*>(at(o_po));
  // backward partials: a bounded chunk of samples at a time
  st->chunk = static_cast<int>(std::min<size_t>(16384, std::max<size_t>(256, kScratchBytes / (size_t(row) * 4))));
  if (cudaMalloc(&st->scratch, size_t(st->chunk) * row * 4) != cudaSuccess) {
    cudaFree(st->tables);
    delete st;
    return fail(CGTP_ENOMEM, "batched-product scratch allocation failed");
  }
  // kernel attributes and occupancy -> slices per group
  auto setup = [&](const void* k, size_t smem, int* slices) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kBtThreads, smem);
    per_sm = std::max(per_sm, 1);
    *slices = std::max(1, (plan->num_sms * per_sm + G - 1) / G);
  };
  if (m == 16) {
    setup(reinterpret_cast<const void*>(bt_forward_kernel<16>), st->smem_fwd, &st->slices_fwd);
    setup(reinterpret_cast<const void*>(bt_backward_kernel<16>), st->smem_bwd, &st->slices_bwd);
  } else {
    setup(reinterpret_cast<const void*>(bt_forward_kernel<32>), st->smem_fwd, &st->slices_fwd);
    setup(reinterpret_cast<const void*>(bt_backward_kernel<32>), st->smem_bwd, &st->slices_bwd);
  }
  cudaGetLastError();
  plan->bt = st;
  return CGTP_OK;
}

void bt_destroy(cgtp_plan_s* plan) {
  BtState* st = static_cast<BtState*>(plan->bt);
  if (!st) return;
  if (st->tables) cudaFree(st->tables);
  if (st->scratch) cudaFree(st->scratch);
  delete st;
  plan->bt = nullptr;
}

static BtArgs bt_args(const cgtp_plan_s* plan, const BtState* st) {
  BtArgs a{};
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d2p = st->d2p;
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.scratch_row = st->scratch_row;
  a.paths = st->paths;
  a.groups = st->groups;
  a.ccoef = st->ccoef;
  a.ccol = st->ccol;
  a.grow = st->grow;
  a.gent = st->gent;
  a.scratch = st->scratch;
  return a;
}

bool bt_forward(const cgtp_plan_s* plan, const void* x1, const void* x2, const void* W, void* out,
                int64_t B, void* stream, cgtp_status* status) {
  const BtState* st = static_cast<const BtState*>(plan->bt);
  if (!st) return false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  BtArgs a = bt_args(plan, st);
  a.x = static_cast<const float*>(x1);
  a.y = static_cast<const float*>(x2);
  a.W = static_cast<const float*>(W);
  a.out = static_cast<float*>(out);
  a.b0 = 0;
  a.b1 = static_cast<int>(B);
  a.slices = st->slices_fwd;
  a.warp_floats = st->wf_fwd;
  const dim3 grid(st->slices_fwd, st->G);
  if (st->lps == 16)
    bt_forward_kernel<16><<<grid, kBtThreads, st->smem_fwd, s>>>(a);
  else
    bt_forward_kernel<32><<<grid, kBtThreads, st->smem_fwd, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  *status = e == cudaSuccess ? CGTP_OK
                             : fail(CGTP_ECUDA, std::string("batched forward launch: ") + cudaGetErrorString(e));
  return true;
}

bool bt_backward(const cgtp_plan_s* plan, const void* gout, const void* x1, const void* x2, const void* W,
                 void* gx1, void* gx2, void* gW, int64_t B, void* stream, cgtp_status* status) {
  const BtState* st = static_cast<const BtState*>(plan->bt);
  if (!st) return false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  BtArgs a = bt_args(plan, st);
  a.x = static_cast<const float*>(x1);
  a.y = static_cast<const float*>(x2);
  a.W = static_cast<const float*>(W);
  a.gout = static_cast<const float*>(gout);
  a.gx = static_cast<float*>(gx1);
  a.gW = static_cast<float*>(gW);
  a.slices = st->slices_bwd;
  a.warp_floats = st->wf_bwd;
  BtReduceArgs r{};
  r.scratch = st->scratch;
  r.gx = static_cast<float*>(gx1);
  r.gy = static_cast<float*>(gx2);
  r.scratch_row = st->scratch_row;
  r.d1 = a.d1;
  r.d2 = a.d2;
  r.G = st->G;
  r.n_in1 = st->n_in1;
  r.blk = st->blk;
  r.part_off = st->part_off;
  const dim3 grid(st->slices_bwd, st->G);
  for (int64_t c0 = 0; c0 < B; c0 += st->chunk) {
    const int n = static_cast<int>(std::min<int64_t>(st->chunk, B - c0));
    a.b0 = static_cast<int>(c0);
    a.b1 = static_cast<int>(c0 + n);
    if (st->lps == 16)
      bt_backward_kernel<16><<<grid, kBtThreads, st->smem_bwd, s>>>(a);
    else
      bt_backward_kernel<32><<<grid, kBtThreads, st->smem_bwd, s>>>(a);
    r.b0 = a.b0;
    r.n = n;
    bt_reduce_kernel<<<std::min(n, plan->num_sms * 8), 256, 0, s>>>(r);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      *status = fail(CGTP_ECUDA, std::string("batched backward launch: ") + cudaGetErrorString(e));
      return true;
    }
  }
  *status = CGTP_OK;
  return true;
}

}  // namespace cgtp
