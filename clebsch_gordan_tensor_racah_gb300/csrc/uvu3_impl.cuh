// uvu3_impl.cuh -- warp-autonomous uvu convolution kernels for plans with l <= 3.
//
// Same operation as uvu_impl.cuh ("An Efficient Sparse Kernel Generator for
// O(3)-Equivariant Deep Networks", Figure 4B: the CG tensor product fused with
// the receiver sum; gradients from its Abstract).  GB300 organisation:
//   * a lane owns four consecutive channels u of one edge; mul/4 lanes (LPE)
//     cover a path's channels, so one warp instruction advances 32/LPE edges;
//   * the CG nonzeros of each (l1, l2, l3) are compiled in as immediates
//     (cg_baked.cuh, generated from the planner's Racah tables), so every lane
//     forms its edge's coupling matrix cy[m1][m3] = sum_m2 C Y[m2] in registers
//     -- no shared tables, no block-wide barriers in the forward -- and the
//     contractions skip the (m1, m3) entries of cy that are structurally zero;
//   * node features, weights and output gradients arrive as 128-bit loads of
//     four channels; the channel pairs (u0,u1), (u2,u3) go through the paired
//     FP32 FMA (fma.rn.f32x2);
//   * sums over the edge slots of a warp use xor shuffles; the backward's gY
//     contraction applies the baked C per lane first, so only 2l2+1 values per
//     (edge, path) cross lanes;
//   * the forward writes every output once (its receiver's warp); the backward
//     writes gW once per edge and adds gx / gY partials with one atomic
//     addition per element per phase -- the items of a phase touch disjoint
//     in1 and in2 blocks and block barriers separate the phases, so the order
//     of additions is fixed (bitwise reproducible).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "sh.cuh"

namespace cgtp {
namespace uvu3_detail {

__host__ __device__ inline int pad_up(int v, int q) { return (v + q - 1) / q * q; }

// one 16-warp CTA per SM: the whole SM walks one path at a time
constexpr int kV3Warps = 16;
constexpr int kV3Threads = kV3Warps * 32;
constexpr int kV3OrderCap = 512;  // senders a backward CTA orders longest first

template <typename T>
struct PairT;
template <>
struct PairT<float> {
  using P = float2;
};
template <>
struct PairT<double> {
  using P = double2;
};

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
        "l"(*reinterpret_cast<unsigned long long*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ double2 fma2(double2 a, double2 b, double2 c) {
  return make_double2(fma(a.x, b.x, c.x), fma(a.y, b.y, c.y));
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ double2 mul2(double2 a, double2 b) { return make_double2(a.x * b.x, a.y * b.y); }

// Accumulation into gY / gx without reading back: each element receives at most
// one contribution per backward phase and phases are separated by block
// barriers, so the order of the additions is fixed (deterministic), and the
// warp does not wait for a read of the old value.
__device__ __forceinline__ void red_add3(float* p, float v) { atomicAdd(p, v); }
__device__ __forceinline__ void red_add3(double* p, double v) { atomicAdd(p, v); }

template <typename T>
__device__ __forceinline__ T shfl_x(T v, int o) {
  return __shfl_xor_sync(0xffffffffu, v, o);
}

// Sum V values over the L lanes of a lane group (L a power of two <= 32; the
// group's lanes differ in the low log2(L) bits of q).  Recursive halving: after
// the call lane q of the group holds slots [q*V/L, (q+1)*V/L) of the group
// total in v[0 .. V/L).  V must be a multiple of L.
template <typename T, int V, int O, int N>
__device__ __forceinline__ void gr_step(T (&v)[V], int q) {
  if constexpr (O >= 1) {
    constexpr int H = N / 2;
    const bool up = (q & O) != 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const T send = up ? v[i] : v[i + H];
      const T keep = up ? v[i + H] : v[i];
      v[i] = keep + shfl_x(send, O);
    }
    gr_step<T, V, O / 2, H>(v, q);
  }
}
template <typename T, int V, int L>
__device__ __forceinline__ void group_reduce(T (&v)[V], int q) {
  static_assert(V % L == 0, "pad V to a multiple of L");
  gr_step<T, V, L / 2, V>(v, q);
}

}  // namespace uvu3_detail
}  // namespace cgtp

#include "cg_baked.cuh"

namespace cgtp {
namespace uvu3_detail {

// T: arithmetic and output type; S: storage type of the inputs x, Y, W and the
// output gradient (T, or bfloat16 with FP32 arithmetic and outputs)
template <typename T, typename S = T>
struct Uvu3Args {
  const S* x;
  const S* Y;
  const S* W;
  const S* gout;
  const T* rvec;          // non-null: edge vectors [E,3]; Y is evaluated from them (in2 = SH 0..L)
  T* out;
  T* gx;
  T* gY;
  T* gW;
  const int* rowptr;  // forward: CSR rowptr; backward: transpose rowptr
  const int* col;     // forward: CSR col; backward: transpose edge ids
  const int* t_dst;
  int N, d1, d2, d_out, w_numel;
  const PathDev* paths;
  const Item* items;      // in path order (forward); grouped by phase (backward)
  int n_items;
  const int* phase_begin; // backward: n_phases + 1 offsets into items_bwd
  int n_phases;
  // backward
  const int* gxp_off;     // per path: offset of its [mul][D1] partial in the gx buffer
  int gxp_size;
  const int* in1_off;     // n_in1 + 1
  int n_in1;
  const int* gx_begin;    // n_in1 + 1 offsets into gx_paths
  const int* gx_paths;
  int chunk_b;            // edges of a sender processed per round (bounded by shared memory)
  int idx_cap;            // ints of dynamic shared memory for the CTA's edge indices
};

template <typename T, int N>
__device__ __forceinline__ void ldvec(const T* p, T (&v)[N]) {  // N consecutive, 16-byte aligned
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p) + i);
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const double2 q = __ldg(reinterpret_cast<const double2*>(p) + i);
      v[2 * i] = q.x;
      v[2 * i + 1] = q.y;
    }
  }
}

// N consecutive bfloat16 values (8-byte aligned), widened exactly to T
template <typename T, int N>
__device__ __forceinline__ void ldvec(const __nv_bfloat16* p, T (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N / 4; ++i) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p) + i);
    v[4 * i] = T(__uint_as_float(q.x << 16));
    v[4 * i + 1] = T(__uint_as_float(q.x & 0xffff0000u));
    v[4 * i + 2] = T(__uint_as_float(q.y << 16));
    v[4 * i + 3] = T(__uint_as_float(q.y & 0xffff0000u));
  }
}
__device__ __forceinline__ float ld1(const float* p) { return __ldg(p); }
__device__ __forceinline__ double ld1(const double* p) { return __ldg(p); }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<unsigned>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
}
// Edge features of edge e for one path: Y[e][off2 .. off2 + D2), or, in the
// edge-vector kernels (SH = true, Y then points at the vectors [E,3]), the
// degree-L2 harmonics of the normalised vector evaluated here.
template <int L2, typename T, bool SH, typename S>
__device__ __forceinline__ void edge_y(const S* __restrict__ Y, int e, int d2, int off2, T (&yv)[2 * L2 + 1]) {
  if constexpr (SH) {
    const T* r = reinterpret_cast<const T*>(Y) + 3 * (size_t)e;
    const T rx = __ldg(r), ry = __ldg(r + 1), rz = __ldg(r + 2);
    const T n2 = rx * rx + ry * ry + rz * rz;
    const T inv = n2 > T(0) ? T(1) / sqrt(n2) : T(0);
    sh_block<L2, T, T>(rx * inv, ry * inv, rz * inv, yv);
  } else {
#pragma unroll
    for (int m = 0; m < 2 * L2 + 1; ++m) yv[m] = ld1(Y + (size_t)e * d2 + off2 + m);
  }
}

// Rows [nb, ne) of a CTA split into contiguous warp ranges of about equal work
// (edges + rows): warp w gets [lo, hi).
__device__ __forceinline__ void warp_rows(const int* rowptr, int nb, int ne, int warp, int nwarps,
                                          int* lo, int* hi) {
  const long long w0 = (long long)rowptr[nb] + nb, w1 = (long long)rowptr[ne] + ne;
  auto lb = [&](long long target) {
    int a = nb, b = ne;
    while (a < b) {
      const int mid = (a + b) >> 1;
      if ((long long)rowptr[mid] + mid < target) a = mid + 1; else b = mid;
    }
    return a;
  };
  *lo = lb(w0 + (w1 - w0) * warp / nwarps);
  *hi = (warp + 1 == nwarps) ? ne : lb(w0 + (w1 - w0) * (warp + 1) / nwarps);
}

// ---------------------------------------------------------------------------
// forward: one (receiver, path, 4*LPE-channel block) per call, all 32 lanes
// ---------------------------------------------------------------------------
template <typename T, int D1, int D2, int D3>
struct FwdEdge {  // one edge's operands, loaded before any arithmetic
  T yv[D2];
  T xs[4 * D1];
  T wv[4];
};

template <typename T, int LPE, int L1, int L2, int L3, bool SH, typename S>
__device__ __forceinline__ void fwd3_load(FwdEdge<T, 2 * L1 + 1, 2 * L2 + 1, 2 * L3 + 1>& E,
                                          const S* __restrict__ x, const S* __restrict__ Y,
                                          const S* __restrict__ W, int e, int s, bool ok, int d1,
                                          int d2, int w_numel, int off1, int off2, int woff, int u) {
  constexpr int D1 = 2 * L1 + 1, D2 = 2 * L2 + 1;
  if (ok) {
    edge_y<L2, T, SH>(Y, e, d2, off2, E.yv);
    ldvec<T, 4 * D1>(x + (size_t)s * d1 + off1 + u * D1, E.xs);
    ldvec<T, 4>(W + (size_t)e * w_numel + woff + u, E.wv);
  } else {
#pragma unroll
    for (int m = 0; m < D2; ++m) E.yv[m] = T(0);
#pragma unroll
    for (int i = 0; i < 4 * D1; ++i) E.xs[i] = T(0);
#pragma unroll
    for (int i = 0; i < 4; ++i) E.wv[i] = T(0);
  }
}

template <typename T, int LPE, int L1, int L2, int L3>
__device__ __forceinline__ void fwd3_math(const FwdEdge<T, 2 * L1 + 1, 2 * L2 + 1, 2 * L3 + 1>& E,
                                          typename PairT<T>::P (&t01)[2 * L3 + 1],
                                          typename PairT<T>::P (&t23)[2 * L3 + 1]) {
  using P = typename PairT<T>::P;
  constexpr int D1 = 2 * L1 + 1, D3 = 2 * L3 + 1, NF = D1 * D3;
  T cy[NF];
#pragma unroll
  for (int f = 0; f < NF; ++f) cy[f] = T(0);
  CGB<L1, L2, L3>::each([&](int m1, int m2, int m3, double c) { cy[m1 * D3 + m3] += T(c) * E.yv[m2]; });
#pragma unroll
  for (int m1 = 0; m1 < D1; ++m1) {
    const P xw01{E.wv[0] * E.xs[m1], E.wv[1] * E.xs[D1 + m1]};
    const P xw23{E.wv[2] * E.xs[2 * D1 + m1], E.wv[3] * E.xs[3 * D1 + m1]};
#pragma unroll
    for (int m3 = 0; m3 < D3; ++m3) {
      if (!((CGB<L1, L2, L3>::mask >> (m1 * D3 + m3)) & 1ull)) continue;  // C.Y is zero there
      const P cp{cy[m1 * D3 + m3], cy[m1 * D3 + m3]};
      t01[m3] = fma2(cp, xw01, t01[m3]);
      t23[m3] = fma2(cp, xw23, t23[m3]);
    }
  }
}

// forward: one (receiver, path, 4*LPE-channel block) per call, all 32 lanes;
// each lane walks its edge slot two edges at a time, loads first
template <typename T, int LPE, int L1, int L2, int L3, bool SH, typename S>
__device__ __noinline__ void fwd3_item(const S* __restrict__ x, const S* __restrict__ Y,
                                       const S* __restrict__ W, T* __restrict__ out,
                                       const int* __restrict__ col, int e_begin, int deg, int n,
                                       int d1, int d2, int d_out, int w_numel, int off1, int off2,
                                       int ooff, int woff, int u, bool active, int g) {
  using P = typename PairT<T>::P;
  constexpr int D1 = 2 * L1 + 1, D2 = 2 * L2 + 1, D3 = 2 * L3 + 1;
  constexpr int EPW = 32 / LPE;
  P t01[D3], t23[D3];
#pragma unroll
  for (int k = 0; k < D3; ++k) t01[k] = t23[k] = P{T(0), T(0)};
  if (active) {
    for (int j = g; j < deg; j += 2 * EPW) {
      const int ja = j, jb = j + EPW;
      const bool okb = jb < deg;
      const int ea = e_begin + ja, eb = e_begin + (okb ? jb : ja);
      const int sa = col[ea], sb = col[eb];  // staged in shared memory (or global)
      FwdEdge<T, D1, D2, D3> A, B;
      fwd3_load<T, LPE, L1, L2, L3, SH>(A, x, Y, W, ea, sa, true, d1, d2, w_numel, off1, off2, woff, u);
      fwd3_load<T, LPE, L1, L2, L3, SH>(B, x, Y, W, eb, sb, okb, d1, d2, w_numel, off1, off2, woff, u);
      fwd3_math<T, LPE, L1, L2, L3>(A, t01, t23);
      fwd3_math<T, LPE, L1, L2, L3>(B, t01, t23);
    }
  }
  T v[4 * D3];
#pragma unroll
  for (int m = 0; m < D3; ++m) {
    v[m] = t01[m].x;
    v[D3 + m] = t01[m].y;
    v[2 * D3 + m] = t23[m].x;
    v[3 * D3 + m] = t23[m].y;
  }
#pragma unroll
  for (int o = 16; o >= LPE; o >>= 1)
#pragma unroll
    for (int i = 0; i < 4 * D3; ++i) v[i] += shfl_x(v[i], o);
  if (active && g == 0) {
    T* dst = out + (size_t)n * d_out + ooff + u * D3;
#pragma unroll
    for (int i = 0; i < 4 * D3; ++i) dst[i] = v[i];
  }
}

#define CGTP3_TRIPLES(M)                                                                          \
  M(0, 0, 0) M(0, 1, 1) M(0, 2, 2) M(0, 3, 3) M(1, 0, 1) M(1, 1, 0) M(1, 1, 1) M(1, 1, 2)         \
  M(1, 2, 1) M(1, 2, 2) M(1, 2, 3) M(1, 3, 2) M(1, 3, 3) M(2, 0, 2) M(2, 1, 1) M(2, 1, 2)         \
  M(2, 1, 3) M(2, 2, 0) M(2, 2, 1) M(2, 2, 2) M(2, 2, 3) M(2, 3, 1) M(2, 3, 2) M(2, 3, 3)         \
  M(3, 0, 3) M(3, 1, 2) M(3, 1, 3) M(3, 2, 1) M(3, 2, 2) M(3, 2, 3) M(3, 3, 0) M(3, 3, 1)         \
  M(3, 3, 2) M(3, 3, 3) M(1, 3, 4) M(0, 0, 1)

// only triangle-valid triples with l <= 3 are instantiated; the two trailing
// entries above are placeholders that never match a path (l3 = 4, or 0x0->1).
#define CGTP3_FWD_CASE(L1, L2, L3)                                                                  \
  case (L1)*16 + (L2)*4 + (L3):                                                                     \
    if constexpr ((L3) <= 3 && (L3) >= ((L1) > (L2) ? (L1) - (L2) : (L2) - (L1)) && (L3) <= (L1) + (L2)) \
      fwd3_item<T, LPE, L1, L2, L3, SH>(a.x, Yp, a.W, a.out, colp, e_begin, deg, n, a.d1, a.d2, a.d_out,  \
                                    a.w_numel, p.off1, p.off2, p.ooff, p.woff, u, active, g);      \
    break;

// Edge indices of the CTA's rows are read once into shared memory (when they
// fit `cap` ints), so the gathers of an edge never wait for an index load from
// global memory.  Returns the pointer to index with CSR positions.
__device__ __forceinline__ const int* stage_idx(const int* __restrict__ src, int p0, int p1, int* s_buf, int cap) {
  if (p1 - p0 > cap) return src;
  for (int i = threadIdx.x; i < p1 - p0; i += blockDim.x) s_buf[i] = __ldg(src + p0 + i);
  return s_buf - p0;
}

template <typename T, int LPE, typename S = T, bool SH = false>
__global__ void __launch_bounds__(kV3Threads, 1) uvu_forward3_kernel(const Uvu3Args<T, S> a) {
  extern __shared__ int v3_idx[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = lane % LPE, g = lane / LPE;
  const S* Yp = SH ? reinterpret_cast<const S*>(a.rvec) : a.Y;   // edge vectors or harmonics
  __shared__ int s_range[2];
  if (tid == 0) {
    const long long total = (long long)a.rowptr[a.N] + a.N;
    const long long t0 = total * blockIdx.x / gridDim.x, t1 = total * (blockIdx.x + 1) / gridDim.x;
    auto lb = [&](long long target) {
      int lo = 0, hi = a.N;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)a.rowptr[mid] + mid < target) lo = mid + 1; else hi = mid;
      }
      return lo;
    };
    s_range[0] = lb(t0);
    s_range[1] = (blockIdx.x + 1 == gridDim.x) ? a.N : lb(t1);
  }
  __syncthreads();
  const int nb = s_range[0], nr = s_range[1] - s_range[0];
  const int* colp = stage_idx(a.col, a.rowptr[nb], a.rowptr[s_range[1]], v3_idx, a.idx_cap);
  // One counter sweeps the (item, receiver) pairs item-major: the warps stay on
  // (nearly) the same path -- one hot instruction stream -- and never wait for
  // each other.  Each receiver's slice of a path is written by one warp.
  // (the host guarantees n_items * N < 2^31, so the counter stays 32-bit)
  __shared__ int s_ctr;
  if (tid == 0) s_ctr = 0;
  __syncthreads();
  const int total = a.n_items * nr;
  for (;;) {
    int k = 0;
    if (lane == 0) k = atomicAdd(&s_ctr, 1);
    k = __shfl_sync(0xffffffffu, k, 0);
    if (k >= total) break;
    const int it = k / nr, n = nb + (k - it * nr);
    const Item item = a.items[it];
    const PathDev p = a.paths[item.path];
    const int u = item.u0 + 4 * q;
    const bool active = u < p.mul;
    const int e_begin = a.rowptr[n], deg = a.rowptr[n + 1] - e_begin;
    switch (p.l1 * 16 + p.l2 * 4 + p.l3) {
      CGTP3_TRIPLES(CGTP3_FWD_CASE)
      default: break;
    }
  }
}

// ---------------------------------------------------------------------------
// backward: one (sender, path, channel block) per call over `cnt` out-edges
// ---------------------------------------------------------------------------
// backward, one (sender, path, channel block) per call over the sender's
// out-edges in one pass (each edge's Y, W and output-gradient slice gathered once):
//   cy, t = cy.x -> gW (stored), gx partial (registers);
//   h[m2] = sum C[m1,m2,m3] sum_lane x w g (baked C) -> reduced over the path's
//   lanes -> one atomic addition per gY element (the only one in this phase)
template <typename T, int LPE, int L1, int L2, int L3, bool SH, typename S>
__device__ __noinline__ void bwd3_item(const S* __restrict__ x, const S* __restrict__ Y,
                                       const S* __restrict__ W, const S* __restrict__ gout,
                                       T* __restrict__ gW, const int* __restrict__ t_eid,
                                       const int* __restrict__ t_dst, int te_begin, int cnt, int s,
                                       int d1, int d2, int d_out, int w_numel, int off1, int off2,
                                       int ooff, int woff, int u, bool active, int g, int q,
                                       T* __restrict__ gY, T* __restrict__ gx) {
  using P = typename PairT<T>::P;
  constexpr int D1 = 2 * L1 + 1, D2 = 2 * L2 + 1, D3 = 2 * L3 + 1, NF = D1 * D3;
  constexpr int EPW = 32 / LPE;
  constexpr int HV = (D2 + LPE - 1) / LPE * LPE;  // h values padded to a multiple of LPE
  T xs[4 * D1];
  if (active) {
    ldvec<T, 4 * D1>(x + (size_t)s * d1 + off1 + u * D1, xs);
  } else {
#pragma unroll
    for (int i = 0; i < 4 * D1; ++i) xs[i] = T(0);
  }
  P x01[D1], x23[D1];
#pragma unroll
  for (int m = 0; m < D1; ++m) {
    x01[m] = P{xs[m], xs[D1 + m]};
    x23[m] = P{xs[2 * D1 + m], xs[3 * D1 + m]};
  }
  // one pass over the out-edges (uniform trip count: the gY reduction shuffles
  // across the path's lanes); every edge's operands are gathered once
  P gxa01[D1], gxa23[D1];
#pragma unroll
  for (int m = 0; m < D1; ++m) gxa01[m] = gxa23[m] = P{T(0), T(0)};
  for (int j0 = 0; j0 < cnt; j0 += EPW) {
    const int j = j0 + g;
    const bool valid = active && j < cnt;
    int e = 0;
    T yv[D2], gs[4 * D3], wv[4];
    if (valid) {
      e = t_eid[te_begin + j];  // staged in shared memory (or global)
      const int d = t_dst[te_begin + j];
      edge_y<L2, T, SH>(Y, e, d2, off2, yv);
      ldvec<T, 4>(W + (size_t)e * w_numel + woff + u, wv);
      ldvec<T, 4 * D3>(gout + (size_t)d * d_out + ooff + u * D3, gs);
    } else {
#pragma unroll
      for (int m = 0; m < D2; ++m) yv[m] = T(0);
#pragma unroll
      for (int i = 0; i < 4; ++i) wv[i] = T(0);
#pragma unroll
      for (int i = 0; i < 4 * D3; ++i) gs[i] = T(0);
    }
    P wg01[D3], wg23[D3];
#pragma unroll
    for (int m3 = 0; m3 < D3; ++m3) {
      wg01[m3] = P{wv[0] * gs[m3], wv[1] * gs[D3 + m3]};
      wg23[m3] = P{wv[2] * gs[2 * D3 + m3], wv[3] * gs[3 * D3 + m3]};
    }
    // gW and the gx partial through cy = C.Y
    {
      T cy[NF];
#pragma unroll
      for (int f = 0; f < NF; ++f) cy[f] = T(0);
      CGB<L1, L2, L3>::each([&](int m1, int m2, int m3, double c) { cy[m1 * D3 + m3] += T(c) * yv[m2]; });
      T gw[4] = {T(0), T(0), T(0), T(0)};
#pragma unroll
      for (int m3 = 0; m3 < D3; ++m3) {
        P t01{T(0), T(0)}, t23{T(0), T(0)};
#pragma unroll
        for (int m1 = 0; m1 < D1; ++m1) {
          if (!((CGB<L1, L2, L3>::mask >> (m1 * D3 + m3)) & 1ull)) continue;  // C.Y is zero there
          const P cp{cy[m1 * D3 + m3], cy[m1 * D3 + m3]};
          t01 = fma2(cp, x01[m1], t01);
          t23 = fma2(cp, x23[m1], t23);
          gxa01[m1] = fma2(cp, wg01[m3], gxa01[m1]);
          gxa23[m1] = fma2(cp, wg23[m3], gxa23[m1]);
        }
        gw[0] += gs[m3] * t01.x;
        gw[1] += gs[D3 + m3] * t01.y;
        gw[2] += gs[2 * D3 + m3] * t23.x;
        gw[3] += gs[3 * D3 + m3] * t23.y;
      }
      if (valid) {
        T* gp = gW + (size_t)e * w_numel + woff + u;
        if constexpr (sizeof(T) == 4) {
          *reinterpret_cast<float4*>(gp) = make_float4(gw[0], gw[1], gw[2], gw[3]);
        } else {
          reinterpret_cast<double2*>(gp)[0] = make_double2(gw[0], gw[1]);
          reinterpret_cast<double2*>(gp)[1] = make_double2(gw[2], gw[3]);
        }
      }
    }
    // gY: h[m2] = sum C[m1,m2,m3] sum_lane x w g (baked C), reduced over the path's lanes
    T h[HV];
#pragma unroll
    for (int i = 0; i < HV; ++i) h[i] = T(0);
    CGB<L1, L2, L3>::each([&](int m1, int m2, int m3, double c) {
      const P pr = fma2(x23[m1], wg23[m3], mul2(x01[m1], wg01[m3]));
      h[m2] += T(c) * (pr.x + pr.y);
    });
    group_reduce<T, HV, LPE>(h, q);
    if (valid) {
#pragma unroll
      for (int k = 0; k < HV / LPE; ++k) {
        const int slot = q * (HV / LPE) + k;
        if (slot < D2) red_add3(gY + (size_t)e * d2 + off2 + slot, h[k]);
      }
    }
  }
  // gx partial of this path: sum over the edge slots; slot 0 adds it (one addition
  // per element in this phase)
  {
    T v[4 * D1];
#pragma unroll
    for (int m = 0; m < D1; ++m) {
      v[m] = gxa01[m].x;
      v[D1 + m] = gxa01[m].y;
      v[2 * D1 + m] = gxa23[m].x;
      v[3 * D1 + m] = gxa23[m].y;
    }
#pragma unroll
    for (int o = 16; o >= LPE; o >>= 1)
#pragma unroll
      for (int i = 0; i < 4 * D1; ++i) v[i] += shfl_x(v[i], o);
    if (active && g == 0) {
      T* dst = gx + (size_t)s * d1 + off1 + u * D1;
#pragma unroll
      for (int i = 0; i < 4 * D1; ++i) red_add3(dst + i, v[i]);
    }
  }
}

#define CGTP3_BWD_CASE(L1, L2, L3)                                                                   \
  case (L1)*16 + (L2)*4 + (L3):                                                                      \
    if constexpr ((L3) <= 3 && (L3) >= ((L1) > (L2) ? (L1) - (L2) : (L2) - (L1)) && (L3) <= (L1) + (L2)) \
      bwd3_item<T, LPE, L1, L2, L3, SH>(a.x, Yp, a.W, a.gout, a.gW, eidp, dstp, te0, cnt, s, a.d1,        \
                                    a.d2, a.d_out, a.w_numel, p.off1, p.off2, p.ooff, p.woff, u,     \
                                    active, g, q, a.gY, a.gx);                                       \
    break;

template <typename T, int LPE, typename S = T, bool SH = false>
__global__ void __launch_bounds__(kV3Threads, 1) uvu_backward3_kernel(const Uvu3Args<T, S> a) {
  extern __shared__ int v3_idx[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = lane % LPE, g = lane / LPE;
  const S* Yp = SH ? reinterpret_cast<const S*>(a.rvec) : a.Y;   // edge vectors or harmonics
  __shared__ int s_range[2];
  if (tid == 0) {
    const long long total = (long long)a.rowptr[a.N] + a.N;
    const long long t0 = total * blockIdx.x / gridDim.x, t1 = total * (blockIdx.x + 1) / gridDim.x;
    auto lb = [&](long long target) {
      int lo = 0, hi = a.N;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)a.rowptr[mid] + mid < target) lo = mid + 1; else hi = mid;
      }
      return lo;
    };
    s_range[0] = lb(t0);
    s_range[1] = (blockIdx.x + 1 == gridDim.x) ? a.N : lb(t1);
  }
  __syncthreads();
  const int sb = s_range[0], se = s_range[1], nr = se - sb;
  // the CTA's transpose slice (edge ids, receivers) in shared memory when it fits
  const int tp0 = a.rowptr[sb], tp1 = a.rowptr[se];
  const bool staged = tp1 - tp0 <= a.idx_cap / 2;
  const int* eidp = staged ? stage_idx(a.col, tp0, tp1, v3_idx, a.idx_cap / 2) : a.col;
  const int* dstp = staged ? stage_idx(a.t_dst, tp0, tp1, v3_idx + a.idx_cap / 2, a.idx_cap / 2) : a.t_dst;
  // clear gx and gY of the CTA's senders (and their out-edges) before the first path
  for (int s = sb + warp; s < se; s += kV3Warps) {
    for (int i = lane; i < a.d1; i += 32) a.gx[(size_t)s * a.d1 + i] = T(0);
    const int tb = a.rowptr[s], te = a.rowptr[s + 1];
    for (int i = lane; i < (te - tb) * a.d2; i += 32) {
      const int j = i / a.d2, c = i - j * a.d2;
      a.gY[(size_t)a.col[tb + j] * a.d2 + c] = T(0);
    }
  }
  // The CTA's senders longest first (out-degree, then index): a phase then ends
  // with its shortest units, so fewer warps wait at the phase barrier.  (A rank
  // sort in shared memory, for ranges of up to kV3OrderCap senders.)
  __shared__ int s_order[kV3OrderCap];
  const bool ordered = nr <= kV3OrderCap;
  if (ordered) {
    for (int i = tid; i < nr; i += kV3Threads) {
      const int di = a.rowptr[sb + i + 1] - a.rowptr[sb + i];
      int rank = 0;
      for (int j = 0; j < nr; ++j) {
        const int dj = a.rowptr[sb + j + 1] - a.rowptr[sb + j];
        rank += (dj > di) || (dj == di && j < i);
      }
      s_order[rank] = i;
    }
    __syncthreads();
  }
  // Items come in phases whose items share no in1 block and no in2 block, so
  // within a phase every gx / gY slice has one writer; a block barrier separates
  // the phases, and every gx / gY element receives its contributions in phase
  // order (deterministic, whatever order the units of a phase run in).  Inside a
  // phase a counter hands out (sender, item) pairs sender-major: the phase's few
  // paths share the instruction cache and a sender's operands stay in L1.
  __shared__ int s_next[2];
  for (int ph = 0; ph < a.n_phases; ++ph) {
    const int i0 = a.phase_begin[ph], ni = a.phase_begin[ph + 1] - i0;
    if (tid == 0) s_next[ph & 1] = 0;
    __syncthreads();
    const int total = ni * nr;
    for (;;) {
      int k = 0;
      if (lane == 0) k = atomicAdd(&s_next[ph & 1], 1);
      k = __shfl_sync(0xffffffffu, k, 0);
      if (k >= total) break;
      const int sl = k / ni, ii = k - sl * ni;
      const int s = sb + (ordered ? s_order[sl] : sl);
      const Item item = a.items[i0 + ii];
      const PathDev p = a.paths[item.path];
      const int u = item.u0 + 4 * q;
      const bool active = u < p.mul;
      const int te0 = a.rowptr[s], cnt = a.rowptr[s + 1] - te0;
      switch (p.l1 * 16 + p.l2 * 4 + p.l3) {
        CGTP3_TRIPLES(CGTP3_BWD_CASE)
        default: break;
      }
    }
  }
}

}  // namespace uvu3_detail
}  // namespace cgtp
