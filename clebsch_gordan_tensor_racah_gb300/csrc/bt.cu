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
// too many to bake into code, so the coefficients are tables in shared memory:
// every cy entry has at most two CG terms (real basis), and the gy contraction
// is a list of (G slot, coefficient) per m2.  The paths are cut into contiguous
// groups whose tables fit a CTA's shared memory.
//
// A lane owns one channel u of a PAIR of samples: every paired FP32 FMA
// (fma.rn.f32x2) advances both samples, so the table reads, the index
// arithmetic and the loop overhead are shared by two samples and no
// horizontal adds are needed.  Multiplicity 16 gives two pairs per warp.
//   * cy of the pair is formed by the pair's lanes into a per-warp buffer as
//     interleaved (sample 0, sample 1) values, rows padded to a multiple of
//     four, read back as broadcast float4 (two m1 of both samples);
//   * x of the pair stays in registers for a run of paths on one in1 block;
//   * forward outputs go through per-sample tiles and leave as streaming
//     float4 stores (7.7 GB at L = 7: the forward is write-bandwidth bound);
//   * backward: lane u forms W*g of its channel; the lane of m1 contracts the
//     transposed W*g rows with x[.][m1] into G; lanes m2 apply the gy table.
// Both kernels are persistent (SMs x resident CTAs) and take work units from a
// device counter zeroed before the launch.  Forward unit: (path group, chunk of
// 32 samples), group-major, so a CTA reloads tables only when its group
// changes.  Backward unit: a 32-sample batch that the CTA walks through all
// groups (reloading the tables), so gx and gy of a sample are owned by one
// warp: deterministic, no floating-point atomics, no scratch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

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
constexpr int kMaxD = 15;                 // largest block dimension (l <= 7)
constexpr int kCyPair = kMaxD * 16 + 8;   // float2 per pair: cy / G [m3][m1 < 16] (+8: bank offset)
constexpr int kGStride = 16;              // row stride (float2) of the G buffer
constexpr size_t kTableBudget = 24 * 1024;

struct BtPath {   // 16 ints
  int D1, D2, D3, Q;        // Q = D1 rounded up to a multiple of 4, divided by 4
  int off1, off2, ooff, woff;
  int ctab;                 // first cy entry of the path (group-relative), D3 * 4Q entries
  int grow;                 // first gy row pointer (group-relative), D2 + 1 of them
  int run;                  // first path of a run on one in1 block: paths in the run; else 0
  int gxfirst;              // backward: the run is the first to touch its in1 block (store, not add)
  int pad0, pad1, pad2, pad3;
};
static_assert(sizeof(BtPath) == 64, "BtPath is 64 bytes");

struct BtGroup {
  int p0, p1;               // path range
  int ctab0, ctab_n;        // cy entries
  int grow0, grow_n;        // gy row pointers
  int gent0, gent_n;        // gy entries
};

struct BtArgs {
  const void* x;     // inputs and output gradient: float, or bfloat16 for CGTP_BF16 plans
  const void* y;
  const void* W;
  const void* gout;
  float* out;
  float* gx;
  float* gy;
  float* gW;
  int B;
  int d1, d2, d_out, w_numel;
  int G;
  int unit;                 // samples per work unit (8 warps x 2 pairs x 2 samples for multiplicity 16)
  int chunks;               // forward: sample chunks per group (units = G * chunks)
  int n_units;
  int* counter;             // work-unit counter, zeroed before each launch
  int y2s;                  // float2 stride of a pair's y / gy buffer
  int tile;                 // float stride of a sample's output tile (forward)
  int wgs;                  // float2 stride of a pair's W*g buffer (backward)
  int warp_floats;
  int table_bytes;          // backward: shared-memory bytes reserved for one group's tables
  int n_zero;               // in1 blocks no path touches (gx = 0 there)
  const int* zero_blk;      // (offset, size) pairs
  const BtPath* paths;
  const BtGroup* groups;
  const float4* ctab;       // (c_a, c_b, byte offset of y[m2_a], byte offset of y[m2_b]) in the pair's y row
  const int* grow;
  const float2* gent;       // (coefficient, byte offset of the G slot)
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
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
// element i of a float or bfloat16 array as float (bfloat16 widens exactly)
template <typename S>
__device__ __forceinline__ float ld_s(const void* base, size_t i) {
  if constexpr (std::is_same<S, float>::value) {
    return __ldg(static_cast<const float*>(base) + i);
  } else {
    return __uint_as_float(static_cast<unsigned>(__ldg(static_cast<const unsigned short*>(base) + i)) << 16);
  }
}
// elements ia and ib of `base` for the two samples of a pair (zero where invalid)
template <typename S>
__device__ __forceinline__ float2 ld_pair(const void* base, size_t ia, size_t ib, bool va, bool vb) {
  return make_float2(va ? ld_s<S>(base, ia) : 0.f, vb ? ld_s<S>(base, ib) : 0.f);
}

// Group tables into shared memory: paths, cy entries [, gy row pointers, gy entries].
__device__ __forceinline__ void load_tables(const BtArgs& a, const BtGroup& g, unsigned char* smem,
                                            bool with_gy) {
  const int np = g.p1 - g.p0;
  int4* sp = reinterpret_cast<int4*>(smem);
  const int4* gp = reinterpret_cast<const int4*>(a.paths + g.p0);
  for (int i = threadIdx.x; i < np * 4; i += blockDim.x) sp[i] = gp[i];
  float4* sc = reinterpret_cast<float4*>(smem + (size_t)np * sizeof(BtPath));
  for (int i = threadIdx.x; i < g.ctab_n; i += blockDim.x) sc[i] = a.ctab[g.ctab0 + i];
  if (with_gy) {
    const size_t o_grow = (size_t)np * sizeof(BtPath) + (size_t)g.ctab_n * 16;
    int* sg = reinterpret_cast<int*>(smem + o_grow);
    for (int i = threadIdx.x; i < g.grow_n; i += blockDim.x) sg[i] = a.grow[g.grow0 + i];
    float2* se = reinterpret_cast<float2*>(smem + al16(o_grow + (size_t)g.grow_n * 4));
    for (int i = threadIdx.x; i < g.gent_n; i += blockDim.x) se[i] = a.gent[g.gent0 + i];
  }
}

// cy of a sample pair: the pair's lanes split the D3 x 4Q entries
template <int LPP, int Q>
__device__ __forceinline__ void coupling(const BtPath& p, const float4* sc, const float2* y2, float2* cy2,
                                         int u) {
  const int ne = p.D3 * 4 * Q;
  const char* yb = reinterpret_cast<const char*>(y2);
  for (int e = u; e < ne; e += LPP) {
    const float4 c = sc[p.ctab + e];
    const float2 ya = *reinterpret_cast<const float2*>(yb + __float_as_int(c.z));
    const float2 yv = *reinterpret_cast<const float2*>(yb + __float_as_int(c.w));
    cy2[e] = fma2(make_float2(c.y, c.y), yv, mul2(make_float2(c.x, c.x), ya));
  }
}

// x of the lane's channel for both samples of the pair (zero past D1)
template <int Q, typename S>
__device__ __forceinline__ void load_x2(const BtArgs& a, const BtPath& p, int b0, int b1, bool v0, bool v1,
                                        int u, float2 (&x2)[4 * Q]) {
  const size_t xa = (size_t)b0 * a.d1 + p.off1 + u * p.D1;
  const size_t xb = (size_t)b1 * a.d1 + p.off1 + u * p.D1;
#pragma unroll
  for (int m = 0; m < 4 * Q; ++m) x2[m] = ld_pair<S>(a.x, xa + m, xb + m, v0 && m < p.D1, v1 && m < p.D1);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <int LPP, int Q, typename S>
__device__ __forceinline__ void fwd_run(const BtArgs& a, const BtPath* sp, int n, const float4* sc,
                                        const float2* y2, float2* cy2, float* t0, float* t1, int b0, int b1,
                                        bool v0, bool v1, int u) {
  constexpr int D1P = 4 * Q;
  float2 x2[D1P];
  load_x2<Q, S>(a, sp[0], b0, b1, v0, v1, u, x2);
  for (int k = 0; k < n; ++k) {
    const BtPath p = sp[k];
    const float2 w2 = ld_pair<S>(a.W, (size_t)b0 * a.w_numel + p.woff + u, (size_t)b1 * a.w_numel + p.woff + u,
                                 v0, v1);
    coupling<LPP, Q>(p, sc, y2, cy2, u);
    __syncwarp();
    // D3 = 2 l3 + 1 is odd: (D3 - 1) / 2 guarded row pairs and the last row,
    // each row as two independent FMA chains
    auto row_out = [&](int m3) {
      const float4* row = reinterpret_cast<const float4*>(cy2 + m3 * D1P);
      float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 2 * Q; ++j) {
        const float4 c = row[j];
        a0 = fma2(make_float2(c.x, c.y), x2[2 * j], a0);
        a1 = fma2(make_float2(c.z, c.w), x2[2 * j + 1], a1);
      }
      const float2 o = mul2(make_float2(a0.x + a1.x, a0.y + a1.y), w2);
      t0[u * p.D3 + m3] = o.x;
      t1[u * p.D3 + m3] = o.y;
    };
#pragma unroll
    for (int m3 = 0; m3 + 1 < kMaxD; m3 += 2) {
      if (m3 + 1 < p.D3) {
        row_out(m3);
        row_out(m3 + 1);
      }
    }
    row_out(p.D3 - 1);
    __syncwarp();
    const int nv = p.D3 * LPP / 4;
    if (v0) {
      float4* dst = reinterpret_cast<float4*>(a.out + (size_t)b0 * a.d_out + p.ooff);
      for (int i = u; i < nv; i += LPP) __stcs(dst + i, reinterpret_cast<const float4*>(t0)[i]);
    }
    if (v1) {
      float4* dst = reinterpret_cast<float4*>(a.out + (size_t)b1 * a.d_out + p.ooff);
      for (int i = u; i < nv; i += LPP) __stcs(dst + i, reinterpret_cast<const float4*>(t1)[i]);
    }
  }
}

template <int LPP, typename S>
__global__ void __launch_bounds__(kBtThreads, 2) bt_forward_kernel(const BtArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int PPW = 32 / LPP;
  __shared__ int s_unit;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, pr = lane / LPP, u = lane % LPP;
  // persistent CTAs take (group, sample chunk) units in group-major order from a
  // counter, so a CTA reloads its tables only when its group changes
  int cur = -1, np = 0;
  const BtPath* sp = reinterpret_cast<const BtPath*>(smem);
  const float4* sc = nullptr;
  float* wb = nullptr;
  for (;;) {
    __syncthreads();  // the previous unit is done with the tables and buffers
    if (threadIdx.x == 0) s_unit = atomicAdd(a.counter, 1);
    __syncthreads();
    const int unit = s_unit;
    if (unit >= a.n_units) break;
    const int gi = unit / a.chunks, chunk = unit - gi * a.chunks;
    if (gi != cur) {
      const BtGroup grp = a.groups[gi];
      load_tables(a, grp, smem, false);
      __syncthreads();
      cur = gi;
      np = grp.p1 - grp.p0;
      sc = reinterpret_cast<const float4*>(smem + (size_t)np * sizeof(BtPath));
      wb = reinterpret_cast<float*>(smem + al16((size_t)np * sizeof(BtPath) + (size_t)grp.ctab_n * 16)) +
           (size_t)warp * a.warp_floats;
    }
    float2* y2 = reinterpret_cast<float2*>(wb) + pr * a.y2s;
    float2* cy2 = reinterpret_cast<float2*>(wb) + PPW * a.y2s + pr * kCyPair;
    float* t0 = wb + 2 * (PPW * a.y2s + PPW * kCyPair) + (2 * pr) * a.tile;
    float* t1 = t0 + a.tile;
    const int base = chunk * a.unit + warp * 2 * PPW;
    if (base >= a.B) continue;
    const int s0 = base + 2 * pr, s1 = s0 + 1;
    const bool v0 = s0 < a.B, v1 = s1 < a.B;
    const int b0 = v0 ? s0 : base, b1 = v1 ? s1 : base;
    for (int i = u; i < a.d2; i += LPP)
      y2[i] = ld_pair<S>(a.y, (size_t)b0 * a.d2 + i, (size_t)b1 * a.d2 + i, v0, v1);
    __syncwarp();
    for (int pi = 0; pi < np;) {
      const int n = sp[pi].run;
      switch (sp[pi].Q) {
        case 1: fwd_run<LPP, 1, S>(a, sp + pi, n, sc, y2, cy2, t0, t1, b0, b1, v0, v1, u); break;
        case 2: fwd_run<LPP, 2, S>(a, sp + pi, n, sc, y2, cy2, t0, t1, b0, b1, v0, v1, u); break;
        case 3: fwd_run<LPP, 3, S>(a, sp + pi, n, sc, y2, cy2, t0, t1, b0, b1, v0, v1, u); break;
        default: fwd_run<LPP, 4, S>(a, sp + pi, n, sc, y2, cy2, t0, t1, b0, b1, v0, v1, u); break;
      }
      pi += n;
    }
  }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
template <int LPP, int Q, typename S>
__device__ __forceinline__ void bwd_run(const BtArgs& a, const BtPath* sp, int n, const float4* sc,
                                        const int* sgrow, const float2* sgent, const float2* y2, float2* gy2,
                                        float2* cy2, float2* wg2, int b0, int b1, bool v0, bool v1, int u) {
  constexpr int D1P = 4 * Q;
  const BtPath p0 = sp[0];
  float2 x2[D1P], gxa[D1P];
  load_x2<Q, S>(a, p0, b0, b1, v0, v1, u, x2);
#pragma unroll
  for (int m = 0; m < D1P; ++m) gxa[m] = make_float2(0.f, 0.f);
  const size_t xa = (size_t)b0 * a.d1 + p0.off1;
  const size_t xb = (size_t)b1 * a.d1 + p0.off1;
  // G stage lanes: m1 = u % 16, channel half h = u / 16 (multiplicity 32 only)
  const int gm1 = u & 15, gh = u >> 4;
  const unsigned gmask = LPP == 32 ? (((1u << p0.D1) - 1u) | (((1u << p0.D1) - 1u) << 16)) : 0u;
  for (int k = 0; k < n; ++k) {
    const BtPath p = sp[k];
    const float2 w2 = ld_pair<S>(a.W, (size_t)b0 * a.w_numel + p.woff + u, (size_t)b1 * a.w_numel + p.woff + u,
                                 v0, v1);
    const size_t ga = (size_t)b0 * a.d_out + p.ooff + u * p.D3;
    const size_t gb = (size_t)b1 * a.d_out + p.ooff + u * p.D3;
    float2 g2[kMaxD];
#pragma unroll
    for (int m3 = 0; m3 < kMaxD; ++m3)
      g2[m3] = ld_pair<S>(a.gout, ga + m3, gb + m3, v0 && m3 < p.D3, v1 && m3 < p.D3);
    coupling<LPP, Q>(p, sc, y2, cy2, u);
    __syncwarp();
    // t = cy x (-> gW), gx += cy^T (W g); W g goes to the transposed buffer.
    // One row per guarded block (registers are full); the gx updates of a row
    // are independent and t is split into two chains.
    float2 gw = make_float2(0.f, 0.f);
    auto row_bwd = [&](int m3, float2 gv) {
      const float2 wg = mul2(w2, gv);
      wg2[m3 * LPP + u] = wg;
      const float4* row = reinterpret_cast<const float4*>(cy2 + m3 * D1P);
      float2 ta = make_float2(0.f, 0.f), tb = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 2 * Q; ++j) {
        const float4 c = row[j];
        const float2 c0 = make_float2(c.x, c.y), c1 = make_float2(c.z, c.w);
        ta = fma2(c0, x2[2 * j], ta);
        tb = fma2(c1, x2[2 * j + 1], tb);
        gxa[2 * j] = fma2(c0, wg, gxa[2 * j]);
        gxa[2 * j + 1] = fma2(c1, wg, gxa[2 * j + 1]);
      }
      gw = fma2(gv, make_float2(ta.x + tb.x, ta.y + tb.y), gw);
    };
#pragma unroll
    for (int m3 = 0; m3 < kMaxD; ++m3)
      if (m3 < p.D3) row_bwd(m3, g2[m3]);
    if (v0) a.gW[(size_t)b0 * a.w_numel + p.woff + u] = gw.x;
    if (v1) a.gW[(size_t)b1 * a.w_numel + p.woff + u] = gw.y;
    __syncwarp();
    // G[m3][m1] = sum_u x[u][m1] (W g)[u][m3] into the dead cy buffer
    float2* G2 = cy2;
    if (gm1 < p.D1) {
      float2 xt[16];
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        const int uu = gh * 16 + v;
        xt[v] = ld_pair<S>(a.x, xa + uu * p.D1 + gm1, xb + uu * p.D1 + gm1, v0, v1);
      }
      auto row_g = [&](int m3) {
        const float4* r = reinterpret_cast<const float4*>(wg2 + m3 * LPP + gh * 16);
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 c = r[j];
          a0 = fma2(make_float2(c.x, c.y), xt[2 * j], a0);
          a1 = fma2(make_float2(c.z, c.w), xt[2 * j + 1], a1);
        }
        float2 acc = make_float2(a0.x + a1.x, a0.y + a1.y);
        if (LPP == 32) {
          acc.x += __shfl_xor_sync(gmask, acc.x, 16);
          acc.y += __shfl_xor_sync(gmask, acc.y, 16);
        }
        if (gh == 0) G2[m3 * kGStride + gm1] = acc;
      };
#pragma unroll
      for (int m3 = 0; m3 + 1 < kMaxD; m3 += 2) {
        if (m3 + 1 < p.D3) {
          row_g(m3);
          row_g(m3 + 1);
        }
      }
      row_g(p.D3 - 1);
    }
    __syncwarp();
    // gy[m2] += sum C[m1,m2,m3] G[m3][m1]; lane u holds m2 = u
    if (u < p.D2) {
      const int r0 = sgrow[p.grow + u], r1 = sgrow[p.grow + u + 1];
      const char* gbase = reinterpret_cast<const char*>(G2);
      float2 v = make_float2(0.f, 0.f);
      for (int r = r0; r < r1; ++r) {
        const float2 t = sgent[r];
        v = fma2(make_float2(t.x, t.x), *reinterpret_cast<const float2*>(gbase + __float_as_int(t.y)), v);
      }
      float2& acc = gy2[p.off2 + u];
      acc = make_float2(acc.x + v.x, acc.y + v.y);
    }
    __syncwarp();  // G (the cy buffer) and W*g are rewritten by the next path
  }
  // gx of the run's in1 block: the first run on the block stores, later runs add (group order)
  float* da = a.gx + (size_t)b0 * a.d1 + p0.off1 + u * p0.D1;
  float* db = a.gx + (size_t)b1 * a.d1 + p0.off1 + u * p0.D1;
#pragma unroll
  for (int m = 0; m < D1P; ++m) {
    if (m < p0.D1) {
      if (v0) da[m] = p0.gxfirst ? gxa[m].x : da[m] + gxa[m].x;
      if (v1) db[m] = p0.gxfirst ? gxa[m].y : db[m] + gxa[m].y;
    }
  }
}

template <int LPP, typename S>
__global__ void __launch_bounds__(kBtThreads, 2) bt_backward_kernel(const BtArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int PPW = 32 / LPP;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, pr = lane / LPP, u = lane % LPP;
  float* wb = reinterpret_cast<float*>(smem + a.table_bytes) + (size_t)warp * a.warp_floats;
  float2* y2 = reinterpret_cast<float2*>(wb) + pr * a.y2s;
  float2* gy2 = reinterpret_cast<float2*>(wb) + PPW * a.y2s + pr * a.y2s;
  float2* cy2 = reinterpret_cast<float2*>(wb) + 2 * PPW * a.y2s + pr * kCyPair;
  float2* wg2 = reinterpret_cast<float2*>(wb) + 2 * PPW * a.y2s + PPW * kCyPair + pr * a.wgs;
  __shared__ int s_unit;
  // persistent CTAs take batches of a.unit samples from a counter
  for (;;) {
    __syncthreads();
    if (threadIdx.x == 0) s_unit = atomicAdd(a.counter, 1);
    __syncthreads();
    const int unit = s_unit;
    if (unit >= a.n_units) break;
    const int base = unit * a.unit;
    const int s0 = base + warp * 2 * PPW + 2 * pr, s1 = s0 + 1;
    const bool v0 = s0 < a.B, v1 = s1 < a.B;
    const int b0 = v0 ? s0 : base, b1 = v1 ? s1 : base;
    for (int i = u; i < a.d2; i += LPP) {
      y2[i] = ld_pair<S>(a.y, (size_t)b0 * a.d2 + i, (size_t)b1 * a.d2 + i, v0, v1);
      gy2[i] = make_float2(0.f, 0.f);
    }
    for (int z = 0; z < a.n_zero; ++z) {
      const int off = a.zero_blk[2 * z], size = a.zero_blk[2 * z + 1];
      for (int i = u; i < size; i += LPP) {
        if (v0) a.gx[(size_t)b0 * a.d1 + off + i] = 0.f;
        if (v1) a.gx[(size_t)b1 * a.d1 + off + i] = 0.f;
      }
    }
    __syncwarp();
    for (int gi = 0; gi < a.G; ++gi) {
      const BtGroup grp = a.groups[gi];
      __syncthreads();  // every warp is done with the previous group's tables
      load_tables(a, grp, smem, true);
      __syncthreads();
      const int np = grp.p1 - grp.p0;
      const BtPath* sp = reinterpret_cast<const BtPath*>(smem);
      const float4* sc = reinterpret_cast<const float4*>(smem + (size_t)np * sizeof(BtPath));
      const size_t o_grow = (size_t)np * sizeof(BtPath) + (size_t)grp.ctab_n * 16;
      const int* sgrow = reinterpret_cast<const int*>(smem + o_grow);
      const float2* sgent = reinterpret_cast<const float2*>(smem + al16(o_grow + (size_t)grp.grow_n * 4));
      for (int pi = 0; pi < np;) {
        const int n = sp[pi].run;
        switch (sp[pi].Q) {
          case 1: bwd_run<LPP, 1, S>(a, sp + pi, n, sc, sgrow, sgent, y2, gy2, cy2, wg2, b0, b1, v0, v1, u); break;
          case 2: bwd_run<LPP, 2, S>(a, sp + pi, n, sc, sgrow, sgent, y2, gy2, cy2, wg2, b0, b1, v0, v1, u); break;
          case 3: bwd_run<LPP, 3, S>(a, sp + pi, n, sc, sgrow, sgent, y2, gy2, cy2, wg2, b0, b1, v0, v1, u); break;
          default: bwd_run<LPP, 4, S>(a, sp + pi, n, sc, sgrow, sgent, y2, gy2, cy2, wg2, b0, b1, v0, v1, u); break;
        }
        pi += n;
      }
    }
    __syncwarp();
    for (int i = u; i < a.d2; i += LPP) {
      if (v0) a.gy[(size_t)b0 * a.d2 + i] = gy2[i].x;
      if (v1) a.gy[(size_t)b1 * a.d2 + i] = gy2[i].y;
    }
    __syncwarp();
  }
}

struct BtState {
  int lpp = 0;
  bool bf16 = false;        // inputs and output gradient stored as bfloat16 (FP32 arithmetic and outputs)
  int G = 0;
  int y2s = 0, tile = 0, wgs = 0;
  int wf_fwd = 0, wf_bwd = 0;
  int table_bytes = 0;      // largest group's full tables (backward)
  size_t smem_fwd = 0, smem_bwd = 0;
  int grid_fwd = 1, grid_bwd = 1;
  int n_zero = 0;
  void* tables = nullptr;
  int* counter = nullptr;   // [0] forward, [1] backward work-unit counters
  const BtPath* paths = nullptr;
  const BtGroup* groups = nullptr;
  const float4* ctab = nullptr;
  const int* grow = nullptr;
  const float2* gent = nullptr;
  const int* zero_blk = nullptr;
};

}  // namespace bt_detail

using namespace bt_detail;

cgtp_status bt_create(cgtp_plan_s* plan) {
  plan->bt = nullptr;
  if (plan->mode != CGTP_UVU || (plan->dtype != CGTP_F32 && plan->dtype != CGTP_BF16) || plan->paths.empty())
    return CGTP_OK;
  const int m = plan->paths.front().mul1;
  if (m != 16 && m != 32) return CGTP_OK;
  for (const auto& p : plan->paths)
    if (p.mul1 != m || p.l1 > 7 || p.l2 > 7 || p.l3 > 7 || p.ooff % 4) return CGTP_OK;
  if (plan->d_out % 4) return CGTP_OK;
  const int P = static_cast<int>(plan->paths.size());
  const int d2 = static_cast<int>(plan->d2);
  if (d2 > 4096) return CGTP_OK;
  // per-path tables
  std::vector<BtPath> bp(P);
  std::vector<std::vector<float4>> pc(P);
  std::vector<std::vector<int>> prow(P);
  std::vector<std::vector<float2>> pent(P);
  std::vector<size_t> bytes(P);
  auto as_float = [](int v) {
    float f;
    std::memcpy(&f, &v, 4);
    return f;
  };
  for (int i = 0; i < P; ++i) {
    const PathHost& h = plan->paths[i];
    const int D1 = 2 * h.l1 + 1, D2 = 2 * h.l2 + 1, D3 = 2 * h.l3 + 1;
    const int Q = (D1 + 3) / 4, D1P = 4 * Q;
    auto C = [&](int m1, int m2, int m3) { return h.C[(size_t(m1) * D2 + m2) * D3 + m3]; };
    BtPath& b = bp[i];
    std::memset(&b, 0, sizeof(b));
    b.D1 = D1; b.D2 = D2; b.D3 = D3; b.Q = Q;
    b.off1 = h.off1; b.off2 = h.off2; b.ooff = h.ooff; b.woff = h.woff;
    const float zoff = as_float(h.off2 * 8);
    pc[i].assign(size_t(D3) * D1P, make_float4(0.f, 0.f, zoff, zoff));
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
        pc[i][size_t(m3) * D1P + m1] =
            make_float4(co[0], co[1], as_float((h.off2 + cl[0]) * 8), as_float((h.off2 + cl[1]) * 8));
      }
    prow[i].push_back(0);
    for (int m2 = 0; m2 < D2; ++m2) {
      for (int m3 = 0; m3 < D3; ++m3)
        for (int m1 = 0; m1 < D1; ++m1) {
          const double c = C(m1, m2, m3);
          if (std::fabs(c) < 1e-15) continue;
          pent[i].push_back(make_float2(static_cast<float>(c), as_float((m3 * kGStride + m1) * 8)));
        }
      prow[i].push_back(static_cast<int>(pent[i].size()));
    }
    bytes[i] = sizeof(BtPath) + pc[i].size() * 16 + prow[i].size() * 4 + pent[i].size() * 8 + 16;
  }
  // contiguous path groups within the table budget
  std::vector<BtGroup> groups;
  {
    int p0 = 0;
    size_t acc = 0;
    for (int i = 0; i < P; ++i) {
      if (i > p0 && acc + bytes[i] > kTableBudget) {
        BtGroup g{};
        g.p0 = p0;
        g.p1 = i;
        groups.push_back(g);
        p0 = i;
        acc = 0;
      }
      acc += bytes[i];
    }
    BtGroup g{};
    g.p0 = p0;
    g.p1 = P;
    groups.push_back(g);
  }
  const int G = static_cast<int>(groups.size());
  const int n_in1 = static_cast<int>(plan->in1.size());
  std::vector<int> in1_off(n_in1 + 1, 0);
  for (int k = 0; k < n_in1; ++k) in1_off[k + 1] = in1_off[k] + plan->in1[k].mul * (2 * plan->in1[k].l + 1);
  std::vector<char> touched(n_in1, 0);
  std::vector<float4> ctab;
  std::vector<float2> gent;
  std::vector<int> growv;
  for (int g = 0; g < G; ++g) {
    BtGroup& gr = groups[g];
    gr.ctab0 = static_cast<int>(ctab.size());
    gr.grow0 = static_cast<int>(growv.size());
    gr.gent0 = static_cast<int>(gent.size());
    int run_start = gr.p0;
    for (int i = gr.p0; i < gr.p1; ++i) {
      BtPath& b = bp[i];
      const int i1 = plan->paths[i].i1;
      b.ctab = static_cast<int>(ctab.size()) - gr.ctab0;
      b.grow = static_cast<int>(growv.size()) - gr.grow0;
      const int ent_base = static_cast<int>(gent.size()) - gr.gent0;
      ctab.insert(ctab.end(), pc[i].begin(), pc[i].end());
      for (int r : prow[i]) growv.push_back(ent_base + r);
      gent.insert(gent.end(), pent[i].begin(), pent[i].end());
      if (i == gr.p0 || plan->paths[i - 1].i1 != i1) {
        run_start = i;
        b.gxfirst = touched[i1] ? 0 : 1;
        touched[i1] = 1;
      }
      bp[run_start].run = i - run_start + 1;
    }
    gr.ctab_n = static_cast<int>(ctab.size()) - gr.ctab0;
    gr.grow_n = static_cast<int>(growv.size()) - gr.grow0;
    gr.gent_n = static_cast<int>(gent.size()) - gr.gent0;
  }
  std::vector<int> zero_blk;
  for (int k = 0; k < n_in1; ++k)
    if (!touched[k] && in1_off[k + 1] > in1_off[k]) {
      zero_blk.push_back(in1_off[k]);
      zero_blk.push_back(in1_off[k + 1] - in1_off[k]);
    }
  BtState* st = new BtState();
  st->lpp = m;
  st->G = G;
  st->n_zero = static_cast<int>(zero_blk.size() / 2);
  const int ppw = 32 / m;
  auto eight_mod16 = [](int v) {  // smallest value >= v that is 8 (mod 16)
    int r = (v + 15) / 16 * 16 - 8;
    return r < v ? r + 16 : r;
  };
  st->y2s = eight_mod16(d2);                 // pairs' y rows 16 banks apart
  st->tile = eight_mod16(m * kMaxD);         // sample tiles of a pair 16 banks apart
  st->wgs = m * kMaxD + 8;
  st->wf_fwd = 2 * (ppw * st->y2s + ppw * kCyPair) + 2 * ppw * st->tile;
  st->wf_bwd = 2 * (2 * ppw * st->y2s + ppw * kCyPair + ppw * st->wgs);
  size_t tb_max = 0;
  for (const BtGroup& g : groups) {
    const size_t np = g.p1 - g.p0;
    const size_t t_fwd = al16(np * sizeof(BtPath) + size_t(g.ctab_n) * 16);
    const size_t t_grow = np * sizeof(BtPath) + size_t(g.ctab_n) * 16;
    const size_t t_bwd = al16(al16(t_grow + size_t(g.grow_n) * 4) + size_t(g.gent_n) * 8);
    st->smem_fwd = std::max(st->smem_fwd, t_fwd + size_t(kBtWarps) * st->wf_fwd * 4);
    tb_max = std::max(tb_max, t_bwd);
  }
  st->table_bytes = static_cast<int>(tb_max);
  st->smem_bwd = tb_max + size_t(kBtWarps) * st->wf_bwd * 4;
  if (st->smem_fwd > 220 * 1024 || st->smem_bwd > 220 * 1024) {
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
  const size_t o_c = put(ctab.data(), ctab.size() * sizeof(float4));
  const size_t o_r = put(growv.data(), growv.size() * sizeof(int));
  const size_t o_e = put(gent.data(), gent.size() * sizeof(float2));
  const size_t o_z = put(zero_blk.data(), zero_blk.size() * sizeof(int));
  if (cudaMalloc(&st->tables, buf.size()) != cudaSuccess) {
    delete st;
    return fail(CGTP_ENOMEM, "batched-product table allocation failed");
  }
  if (cudaMemcpy(st->tables, buf.data(), buf.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(st->tables);
    delete st;
    return fail(CGTP_ECUDA, "batched-product table upload failed");
  }
  if (cudaMalloc(&st->counter, 2 * sizeof(int)) != cudaSuccess) {
    cudaFree(st->tables);
    delete st;
    return fail(CGTP_ENOMEM, "batched-product counter allocation failed");
  }
  plan->device_bytes += buf.size() + 2 * sizeof(int);
  auto at = [&](size_t off) { return static_cast<unsigned char*>(st->tables) + off; };
  st->paths = reinterpret_cast<const BtPath*>(at(o_p));
  st->groups = reinterpret_cast<const BtGroup*>(at(o_g));
  st->ctab = reinterpret_cast<const float4*>(at(o_c));
  st->grow = reinterpret_cast<const int*>(at(o_r));
  st->gent = reinterpret_cast<const float2*>(at(o_e));
  st->zero_blk = reinterpret_cast<const int*>(at(o_z));
  // kernel attributes and occupancy -> grid sizes
  auto occupancy = [&](const void* k, size_t smem) {
    raise_smem_limit(k);
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kBtThreads, smem);
    return std::max(per_sm, 1);
  };
  st->bf16 = plan->dtype == CGTP_BF16;
  const void* kf = st->bf16 ? (m == 16 ? reinterpret_cast<const void*>(bt_forward_kernel<16, __nv_bfloat16>)
                                       : reinterpret_cast<const void*>(bt_forward_kernel<32, __nv_bfloat16>))
                            : (m == 16 ? reinterpret_cast<const void*>(bt_forward_kernel<16, float>)
                                       : reinterpret_cast<const void*>(bt_forward_kernel<32, float>));
  const void* kb = st->bf16 ? (m == 16 ? reinterpret_cast<const void*>(bt_backward_kernel<16, __nv_bfloat16>)
                                       : reinterpret_cast<const void*>(bt_backward_kernel<32, __nv_bfloat16>))
                            : (m == 16 ? reinterpret_cast<const void*>(bt_backward_kernel<16, float>)
                                       : reinterpret_cast<const void*>(bt_backward_kernel<32, float>));
  st->grid_fwd = plan->num_sms * occupancy(kf, st->smem_fwd);
  st->grid_bwd = plan->num_sms * occupancy(kb, st->smem_bwd);
  cudaGetLastError();
  plan->bt = st;
  return CGTP_OK;
}

void bt_destroy(cgtp_plan_s* plan) {
  BtState* st = static_cast<BtState*>(plan->bt);
  if (!st) return;
  if (st->tables) cudaFree(st->tables);
  if (st->counter) cudaFree(st->counter);
  delete st;
  plan->bt = nullptr;
}

static BtArgs bt_args(const cgtp_plan_s* plan, const BtState* st, int64_t B) {
  BtArgs a{};
  a.B = static_cast<int>(B);
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.G = st->G;
  a.unit = kBtWarps * 64 / st->lpp;
  a.y2s = st->y2s;
  a.tile = st->tile;
  a.wgs = st->wgs;
  a.table_bytes = st->table_bytes;
  a.n_zero = st->n_zero;
  a.zero_blk = st->zero_blk;
  a.paths = st->paths;
  a.groups = st->groups;
  a.ctab = st->ctab;
  a.grow = st->grow;
  a.gent = st->gent;
  return a;
}

bool bt_forward(const cgtp_plan_s* plan, const void* x1, const void* x2, const void* W, void* out,
                int64_t B, void* stream, cgtp_status* status) {
  const BtState* st = static_cast<const BtState*>(plan->bt);
  if (!st) return false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  BtArgs a = bt_args(plan, st, B);
  a.x = x1;
  a.y = x2;
  a.W = W;
  a.out = static_cast<float*>(out);
  a.warp_floats = st->wf_fwd;
  a.chunks = static_cast<int>((B + a.unit - 1) / a.unit);
  if ((int64_t)a.G * a.chunks + st->grid_fwd >= (int64_t(1) << 31)) return false;  // 32-bit unit counter
  a.n_units = a.G * a.chunks;
  a.counter = st->counter;
  if (cudaMemsetAsync(st->counter, 0, sizeof(int), s) != cudaSuccess) {
    *status = fail(CGTP_ECUDA, "batched forward: counter reset failed");
    return true;
  }
  const int grid = std::max(1, std::min(st->grid_fwd, a.n_units));
  if (st->bf16) {
    if (st->lpp == 16) bt_forward_kernel<16, __nv_bfloat16><<<grid, kBtThreads, st->smem_fwd, s>>>(a);
    else bt_forward_kernel<32, __nv_bfloat16><<<grid, kBtThreads, st->smem_fwd, s>>>(a);
  } else {
    if (st->lpp == 16) bt_forward_kernel<16, float><<<grid, kBtThreads, st->smem_fwd, s>>>(a);
    else bt_forward_kernel<32, float><<<grid, kBtThreads, st->smem_fwd, s>>>(a);
  }
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
  BtArgs a = bt_args(plan, st, B);
  a.x = x1;
  a.y = x2;
  a.W = W;
  a.gout = gout;
  a.gx = static_cast<float*>(gx1);
  a.gy = static_cast<float*>(gx2);
  a.gW = static_cast<float*>(gW);
  a.warp_floats = st->wf_bwd;
  a.n_units = static_cast<int>((B + a.unit - 1) / a.unit);
  a.counter = st->counter + 1;
  if (cudaMemsetAsync(st->counter + 1, 0, sizeof(int), s) != cudaSuccess) {
    *status = fail(CGTP_ECUDA, "batched backward: counter reset failed");
    return true;
  }
  const int grid = std::max(1, std::min(st->grid_bwd, a.n_units));
  if (st->bf16) {
    if (st->lpp == 16) bt_backward_kernel<16, __nv_bfloat16><<<grid, kBtThreads, st->smem_bwd, s>>>(a);
    else bt_backward_kernel<32, __nv_bfloat16><<<grid, kBtThreads, st->smem_bwd, s>>>(a);
  } else {
    if (st->lpp == 16) bt_backward_kernel<16, float><<<grid, kBtThreads, st->smem_bwd, s>>>(a);
    else bt_backward_kernel<32, float><<<grid, kBtThreads, st->smem_bwd, s>>>(a);
  }
  const cudaError_t e = cudaGetLastError();
  *status = e == cudaSuccess ? CGTP_OK
                             : fail(CGTP_ECUDA, std::string("batched backward launch: ") + cudaGetErrorString(e));
  return true;
}

}  // namespace cgtp
