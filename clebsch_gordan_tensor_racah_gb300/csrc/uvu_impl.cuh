// uvu_impl.cuh -- fused CG tensor product + receiver sum (uvu, one weight per channel),
// forward and backward, for graph convolutions and for the batched product.
//
// "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks":
//   Figure 1: z = W * (P contracted with x and y), P block-sparse;
//   Figure 4A: batched product (here: the identity graph, one edge per row);
//   Figure 4B: the product fused with a graph convolution -- messages are
//              summed into the receiver without duplicating inputs;
//   Abstract: gradient kernels with respect to both inputs and the weights.
// "LunaTP ...", Abstract: node-centric execution and path-group parallelism --
// here one CTA owns a receiver (forward) or a sender (backward) and its warps
// split the paths.
//
// Forward, per receiver n (one CTA, edges in chunks of `chunk`):
//   cy[e][path][m1][m3] = sum_m2 C[m1,m2,m3] Y[e][m2]       (table-driven, shared memory)
//   acc[path][u][m3]   += W[e][path,u] * sum_m1 cy[m1][m3] x[src][u][m1]
//   out[n] = acc       (written once; no atomics, no edge-sized intermediates)
// Backward, per sender s over its out-edges (transpose order):
//   gW[e][path,u] = sum_m3 g[dst][path,u,m3] * sum_m1 cy[m1][m3] x[s][u][m1]
//   gx[s][u][m1] += sum_path W[e][path,u] sum_m3 cy[m1][m3] g[dst][path,u,m3]
//   gc[m1][m3]    = sum_u W x[s][u][m1] g[dst][path,u,m3]   (warp transpose-reduction)
//   gY[e][c]      = sum over table terms coef * gc[slot]
// uvu_impl.cuh holds the templates; uvu_*.cu instantiate them per element type and
// largest l so the translation units compile in parallel.
// The shape-dependent inner loops are instantiated for every (2l1+1, 2l3+1)
// with l <= 7, so per-lane operands stay in registers; the CG nonzeros come
// from per-plan tables.
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>

#include "internal.h"

namespace cgtp {
namespace uvu_detail {

template <typename T>
struct V16;
template <>
struct V16<float> {
  using type = float4;
  static constexpr int n = 4;
};
template <>
struct V16<double> {
  using type = double2;
  static constexpr int n = 2;
};

template <typename T>
struct UvuArgs {
  const T* x;
  const T* Y;
  const T* W;
  const T* gout;
  T* out;
  T* gx;
  T* gY;
  T* gW;
  const int* rowptr;  // forward: CSR rowptr; backward: transpose rowptr
  const int* col;     // forward: CSR col;    backward: transpose edge ids
  const int* t_dst;   // backward: receiver of each transposed edge
  int N;
  int d1, d2, d_out, w_numel;
  int chunk;
  int n_groups, n_in1;
  const PathDev* paths;
  const int* in1_off;
  const GroupDev* groups;
  const int* cy_begin;
  const int* cy_col;
  const T* cy_coef;
  const int* gy_begin;
  const int* gy_slot;
  const int* gy_nub;
  const T* gy_coef;
  const int* item_begin;
  const Item* items;
  const int* gx_begin;
  const int* gx_paths;
};

__host__ __device__ inline int pad_up(int v, int q) { return (v + q - 1) / q * q; }

// First row n in [0, N] whose work position (edges before it + n) reaches target.
template <bool IDENT>
__device__ int work_lower_bound(const int* rowptr, int N, long long target) {
  int lo = 0, hi = N;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const long long w = (IDENT ? (long long)mid : (long long)rowptr[mid]) + mid;
    if (w < target)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

template <bool IDENT>
__device__ void cta_row_range(const int* rowptr, int N, int* nb, int* ne) {
  __shared__ int s_range[2];
  if (threadIdx.x == 0) {
    const long long total = (IDENT ? (long long)N : (long long)rowptr[N]) + N;
    const long long G = gridDim.x;
    const long long t0 = total * blockIdx.x / G;
    const long long t1 = total * (blockIdx.x + 1) / G;
    s_range[0] = work_lower_bound<IDENT>(rowptr, N, t0);
    s_range[1] = (blockIdx.x + 1 == gridDim.x) ? N : work_lower_bound<IDENT>(rowptr, N, t1);
  }
  __syncthreads();
  *nb = s_range[0];
  *ne = s_range[1];
}

// ---------------------------------------------------------------------------
// forward item: one (path, 32-channel block) over the chunk's edges
// ---------------------------------------------------------------------------
template <typename T, int D1, int D3>
__device__ __noinline__ void fwd_item(const T* __restrict__ x, const T* __restrict__ W, int d1,
                                      int w_numel, int off1, int woff, int cyoff, int ooff, int u,
                                      int e0, int cnt, const int* src_s, const T* cys, int cy_size,
                                      T* acc) {
  using V = typename V16<T>::type;
  constexpr int VN = V16<T>::n;
  constexpr int NF = D1 * D3;
  constexpr int NV = (NF + VN - 1) / VN;
  T t[D3];
#pragma unroll
  for (int k = 0; k < D3; ++k) t[k] = T(0);
  const T* xcol = x + off1 + u * D1;
  const T* wcol = W + (size_t)e0 * w_numel + woff + u;
  const T* cyp = cys + cyoff;
#pragma unroll 2
  for (int j = 0; j < cnt; ++j) {
    const T* xr = xcol + (size_t)src_s[j] * d1;
    const T w = __ldg(wcol + (size_t)j * w_numel);
    T xw[D1];
#pragma unroll
    for (int m = 0; m < D1; ++m) xw[m] = w * __ldg(xr + m);
    const V* c = reinterpret_cast<const V*>(cyp + j * cy_size);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const V cv = c[v];
      const T* cs = reinterpret_cast<const T*>(&cv);
#pragma unroll
      for (int q = 0; q < VN; ++q) {
        const int f = v * VN + q;
        if (f < NF) t[f % D3] += cs[q] * xw[f / D3];
      }
    }
  }
  T* ap = acc + ooff + u * D3;
#pragma unroll
  for (int k = 0; k < D3; ++k) ap[k] += t[k];
}

#define CGTP_L_CASES(M, ...)                                                                      \
  M(0, 0, __VA_ARGS__) M(0, 1, __VA_ARGS__) M(0, 2, __VA_ARGS__) M(0, 3, __VA_ARGS__)             \
  M(0, 4, __VA_ARGS__) M(0, 5, __VA_ARGS__) M(0, 6, __VA_ARGS__) M(0, 7, __VA_ARGS__)             \
  M(1, 0, __VA_ARGS__) M(1, 1, __VA_ARGS__) M(1, 2, __VA_ARGS__) M(1, 3, __VA_ARGS__)             \
  M(1, 4, __VA_ARGS__) M(1, 5, __VA_ARGS__) M(1, 6, __VA_ARGS__) M(1, 7, __VA_ARGS__)             \
  M(2, 0, __VA_ARGS__) M(2, 1, __VA_ARGS__) M(2, 2, __VA_ARGS__) M(2, 3, __VA_ARGS__)             \
  M(2, 4, __VA_ARGS__) M(2, 5, __VA_ARGS__) M(2, 6, __VA_ARGS__) M(2, 7, __VA_ARGS__)             \
  M(3, 0, __VA_ARGS__) M(3, 1, __VA_ARGS__) M(3, 2, __VA_ARGS__) M(3, 3, __VA_ARGS__)             \
  M(3, 4, __VA_ARGS__) M(3, 5, __VA_ARGS__) M(3, 6, __VA_ARGS__) M(3, 7, __VA_ARGS__)             \
  M(4, 0, __VA_ARGS__) M(4, 1, __VA_ARGS__) M(4, 2, __VA_ARGS__) M(4, 3, __VA_ARGS__)             \
  M(4, 4, __VA_ARGS__) M(4, 5, __VA_ARGS__) M(4, 6, __VA_ARGS__) M(4, 7, __VA_ARGS__)             \
  M(5, 0, __VA_ARGS__) M(5, 1, __VA_ARGS__) M(5, 2, __VA_ARGS__) M(5, 3, __VA_ARGS__)             \
  M(5, 4, __VA_ARGS__) M(5, 5, __VA_ARGS__) M(5, 6, __VA_ARGS__) M(5, 7, __VA_ARGS__)             \
  M(6, 0, __VA_ARGS__) M(6, 1, __VA_ARGS__) M(6, 2, __VA_ARGS__) M(6, 3, __VA_ARGS__)             \
  M(6, 4, __VA_ARGS__) M(6, 5, __VA_ARGS__) M(6, 6, __VA_ARGS__) M(6, 7, __VA_ARGS__)             \
  M(7, 0, __VA_ARGS__) M(7, 1, __VA_ARGS__) M(7, 2, __VA_ARGS__) M(7, 3, __VA_ARGS__)             \
  M(7, 4, __VA_ARGS__) M(7, 5, __VA_ARGS__) M(7, 6, __VA_ARGS__) M(7, 7, __VA_ARGS__)

#define CGTP_FWD_CASE(L1, L3, ...)                                                      \
  case (L1)*8 + (L3):                                                                     \
    if constexpr ((L1) <= LMAX && (L3) <= LMAX)                                           \
      fwd_item<T, 2 * (L1) + 1, 2 * (L3) + 1>(a.x, a.W, a.d1, a.w_numel, p.off1, p.woff,   \
        p.cyoff_g, p.ooff_g, u, e0, cnt, src_s, cys, cy_size, acc);                        \
    break;

template <typename T, bool IDENT, int LMAX>
__global__ void __launch_bounds__(kThreads, 2) uvu_forward_kernel(const UvuArgs<T> a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int VN = V16<T>::n;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = a.chunk;
  const int d2p = pad_up(a.d2, VN);
  int nb, ne;
  cta_row_range<IDENT>(a.rowptr, a.N, &nb, &ne);
  for (int gi = 0; gi < a.n_groups; ++gi) {
    const GroupDev g = a.groups[gi];
    const int dog = g.o1 - g.o0;
    const int cy_size = g.cy_size;
    T* acc = reinterpret_cast<T*>(smem);
    T* Ys = acc + pad_up(dog, VN);
    T* cys = Ys + chunk * d2p;
    int* src_s = reinterpret_cast<int*>(cys + chunk * cy_size);
    const int ib = a.item_begin[g.item_base + warp];
    const int ie = a.item_begin[g.item_base + warp + 1];
    for (int n = nb; n < ne; ++n) {
      const int e_begin = IDENT ? n : a.rowptr[n];
      const int e_end = IDENT ? n + 1 : a.rowptr[n + 1];
      for (int i = tid; i < dog; i += kThreads) acc[i] = T(0);
      for (int e0 = e_begin; e0 < e_end; e0 += chunk) {
        const int cnt = min(chunk, e_end - e0);
        __syncthreads();  // previous chunk done with Ys / cys / src_s; acc zeroing visible
        for (int i = tid; i < cnt; i += kThreads) src_s[i] = IDENT ? e0 + i : a.col[e0 + i];
        for (int i = tid; i < cnt * a.d2; i += kThreads) {
          const int j = i / a.d2, c = i - j * a.d2;
          Ys[j * d2p + c] = a.Y[(size_t)(e0 + j) * a.d2 + c];
        }
        __syncthreads();
        for (int i = tid; i < cnt * cy_size; i += kThreads) {
          const int j = i / cy_size, s = i - j * cy_size;
          const int t0 = a.cy_begin[g.cy_base + s], t1 = a.cy_begin[g.cy_base + s + 1];
          T v = T(0);
          for (int t = t0; t < t1; ++t) v += a.cy_coef[t] * Ys[j * d2p + a.cy_col[t]];
          cys[i] = v;
        }
        __syncthreads();
        for (int it = ib; it < ie; ++it) {
          const Item item = a.items[it];
          const PathDev p = a.paths[item.path];
          const int u = item.u0 + lane;
          if (u >= p.mul) continue;
          switch (p.l1 * 8 + p.l3) { CGTP_L_CASES(CGTP_FWD_CASE, 0) default: break; }
        }
      }
      __syncthreads();
      T* orow = a.out + (size_t)n * a.d_out + g.o0;
      for (int i = tid; i < dog; i += kThreads) orow[i] = acc[i];
    }
  }
}

// ---------------------------------------------------------------------------
// backward item
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ T shfl_xor(T v, int o) {
  return __shfl_xor_sync(0xffffffffu, v, o);
}

// Sum the outer product gc[f] = xv[f / D3] * wg[f % D3] over the 32 lanes
// (recursive halving: after five exchange steps lane l holds slot l of each
// 32-slot block) and store slot f to dst[f].
template <typename T, int D1, int D3>
__device__ __forceinline__ void reduce_outer(const T (&xv)[D1], const T (&wg)[D3], T* dst,
                                             int lane) {
  constexpr int NF = D1 * D3;
  constexpr int NB = (NF + 31) / 32;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    T v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int f = b * 32 + i;
      v[i] = (f < NF) ? xv[(f < NF ? f : 0) / D3] * wg[(f < NF ? f : 0) % D3] : T(0);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const T send = up ? v[i] : v[i + o];
        const T keep = up ? v[i + o] : v[i];
        v[i] = keep + shfl_xor(send, o);
      }
    }
    const int f = b * 32 + lane;
    if (f < NF) dst[f] = v[0];
  }
}

template <typename T, int D1, int D3>
__device__ __noinline__ void bwd_item(const T* __restrict__ W, const T* __restrict__ gout,
                                      T* __restrict__ gW, int w_numel, int d_out, int mul,
                                      int off1, int woff, int ooff, int cyoff, int gxpoff, int u0,
                                      int lane, int cnt, const int* eid_s, const int* dst_s,
                                      const T* xs, const T* cys, T* gcp, int cy_size, int nub,
                                      T* gxp) {
  using V = typename V16<T>::type;
  constexpr int VN = V16<T>::n;
  constexpr int NF = D1 * D3;
  constexpr int NV = (NF + VN - 1) / VN;
  const int u = u0 + lane;
  const bool active = u < mul;
  const int ub = u0 >> 5;
  T xv[D1], gxa[D1];
#pragma unroll
  for (int m = 0; m < D1; ++m) {
    xv[m] = active ? xs[off1 + u * D1 + m] : T(0);
    gxa[m] = T(0);
  }
  for (int j = 0; j < cnt; ++j) {
    const int e = eid_s[j], d = dst_s[j];
    T w = T(0), gv[D3];
    if (active) w = __ldg(W + (size_t)e * w_numel + woff + u);
    const T* grow = gout + (size_t)d * d_out + ooff + u * D3;
#pragma unroll
    for (int k = 0; k < D3; ++k) gv[k] = active ? __ldg(grow + k) : T(0);
    T t[D3], wg[D3];
#pragma unroll
    for (int k = 0; k < D3; ++k) {
      t[k] = T(0);
      wg[k] = w * gv[k];
    }
    const V* c = reinterpret_cast<const V*>(cys + j * cy_size + cyoff);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const V cv = c[v];
      const T* cs = reinterpret_cast<const T*>(&cv);
#pragma unroll
      for (int q = 0; q < VN; ++q) {
        const int f = v * VN + q;
        if (f < NF) {
          t[f % D3] += cs[q] * xv[f / D3];
          gxa[f / D3] += cs[q] * wg[f % D3];
        }
      }
    }
    T gw = T(0);
#pragma unroll
    for (int k = 0; k < D3; ++k) gw += gv[k] * t[k];
    if (active) gW[(size_t)e * w_numel + woff + u] = gw;
    reduce_outer<T, D1, D3>(xv, wg, gcp + (j * nub + ub) * cy_size + cyoff, lane);
  }
  if (active) {
    T* gp = gxp + gxpoff + u * D1;
#pragma unroll
    for (int m = 0; m < D1; ++m) gp[m] += gxa[m];
  }
}

#define CGTP_BWD_CASE(L1, L3, ...)                                                           \
  case (L1)*8 + (L3):                                                                          \
    if constexpr ((L1) <= LMAX && (L3) <= LMAX)                                                \
      bwd_item<T, 2 * (L1) + 1, 2 * (L3) + 1>(a.W, a.gout, a.gW, a.w_numel, a.d_out, p.mul,   \
          p.off1, p.woff, p.ooff, p.cyoff_g, p.gxpoff_g, item.u0, lane, cnt, eid_s, dst_s, xs, \
          cys, gcp, cy_size, nub, gxp);                                                          \
    break;

template <typename T, bool IDENT, int LMAX>
__global__ void __launch_bounds__(kThreads, 2) uvu_backward_kernel(const UvuArgs<T> a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int VN = V16<T>::n;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = a.chunk;
  const int d2p = pad_up(a.d2, VN);
  const int d1p = pad_up(a.d1, VN);
  int sb, se;
  cta_row_range<IDENT>(a.rowptr, a.N, &sb, &se);
  for (int gi = 0; gi < a.n_groups; ++gi) {
    const GroupDev g = a.groups[gi];
    const int cy_size = g.cy_size, nub = g.nub;
    T* xs = reinterpret_cast<T*>(smem);
    T* Ys = xs + d1p;
    T* cys = Ys + chunk * d2p;
    T* gcp = cys + chunk * cy_size;
    T* gxp = gcp + chunk * nub * cy_size;
    int* eid_s = reinterpret_cast<int*>(gxp + pad_up(g.gxp_size, VN));
    int* dst_s = eid_s + chunk;
    const int ib = a.item_begin[g.item_base + warp];
    const int ie = a.item_begin[g.item_base + warp + 1];
    for (int s = sb; s < se; ++s) {
      const int e_begin = IDENT ? s : a.rowptr[s];
      const int e_end = IDENT ? s + 1 : a.rowptr[s + 1];
      __syncthreads();  // previous sender's gx reduction done with xs / gxp
      for (int i = tid; i < a.d1; i += kThreads) xs[i] = a.x[(size_t)s * a.d1 + i];
      for (int i = tid; i < g.gxp_size; i += kThreads) gxp[i] = T(0);
      for (int e0 = e_begin; e0 < e_end; e0 += chunk) {
        const int cnt = min(chunk, e_end - e0);
        __syncthreads();
        for (int i = tid; i < cnt; i += kThreads) {
          eid_s[i] = IDENT ? e0 + i : a.col[e0 + i];
          dst_s[i] = IDENT ? e0 + i : a.t_dst[e0 + i];
        }
        __syncthreads();
        for (int i = tid; i < cnt * a.d2; i += kThreads) {
          const int j = i / a.d2, c = i - j * a.d2;
          Ys[j * d2p + c] = a.Y[(size_t)eid_s[j] * a.d2 + c];
        }
        __syncthreads();
        for (int i = tid; i < cnt * cy_size; i += kThreads) {
          const int j = i / cy_size, sl = i - j * cy_size;
          const int t0 = a.cy_begin[g.cy_base + sl], t1 = a.cy_begin[g.cy_base + sl + 1];
          T v = T(0);
          for (int t = t0; t < t1; ++t) v += a.cy_coef[t] * Ys[j * d2p + a.cy_col[t]];
          cys[i] = v;
        }
        __syncthreads();
        for (int it = ib; it < ie; ++it) {
          const Item item = a.items[it];
          const PathDev p = a.paths[item.path];
          switch (p.l1 * 8 + p.l3) { CGTP_L_CASES(CGTP_BWD_CASE, 0) default: break; }
        }
        __syncthreads();
        for (int i = tid; i < cnt * a.d2; i += kThreads) {
          const int j = i / a.d2, c = i - j * a.d2;
          const int t0 = a.gy_begin[g.gy_base + c], t1 = a.gy_begin[g.gy_base + c + 1];
          T v = T(0);
          for (int t = t0; t < t1; ++t) {
            const int sl = a.gy_slot[t], nb = a.gy_nub[t];
            T gsum = T(0);
            for (int b = 0; b < nb; ++b) gsum += gcp[(j * nub + b) * cy_size + sl];
            v += a.gy_coef[t] * gsum;
          }
          T* dstp = a.gY + (size_t)eid_s[j] * a.d2 + c;
          if (gi == 0)
            *dstp = v;
          else
            *dstp += v;
        }
      }
      __syncthreads();
      // gx[s] = sum over the group's paths of the per-path partials, in path order
      for (int b = 0; b < a.n_in1; ++b) {
        const int o0 = a.in1_off[b], len = a.in1_off[b + 1] - o0;
        const int q0 = a.gx_begin[g.gx_base + b], q1 = a.gx_begin[g.gx_base + b + 1];
        for (int i = tid; i < len; i += kThreads) {
          T v = T(0);
          for (int q = q0; q < q1; ++q) v += gxp[a.paths[a.gx_paths[q]].gxpoff_g + i];
          T* dstp = a.gx + (size_t)s * a.d1 + o0 + i;
          if (gi == 0)
            *dstp = v;
          else
            *dstp += v;
        }
      }
    }
  }
}

template <typename T>
UvuArgs<T> make_args(const cgtp_plan_s* plan, const LayoutDev& lay) {
  UvuArgs<T> a{};
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.chunk = lay.chunk;
  a.n_groups = lay.n_groups;
  a.n_in1 = lay.n_in1;
  a.paths = lay.paths;
  a.in1_off = lay.in1_off;
  a.groups = lay.groups;
  a.cy_begin = lay.cy_begin;
  a.cy_col = lay.cy_col;
  a.cy_coef = static_cast<const T*>(lay.cy_coef);
  a.gy_begin = lay.gy_begin;
  a.gy_slot = lay.gy_slot;
  a.gy_nub = lay.gy_nub;
  a.gy_coef = static_cast<const T*>(lay.gy_coef);
  a.item_begin = lay.item_begin;
  a.items = lay.items;
  a.gx_begin = lay.gx_begin;
  a.gx_paths = lay.gx_paths;
  return a;
}

template <typename K>
int grid_for(K kernel, size_t smem, int num_sms, int64_t rows) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
  if (per_sm < 1) per_sm = 1;
  int64_t g = static_cast<int64_t>(num_sms) * per_sm;
  if (g > rows) g = rows;
  return static_cast<int>(g < 1 ? 1 : g);
}

template <typename T, bool IDENT, int LMAX>
cgtp_status fwd_impl(const cgtp_plan_s* plan, const LayoutDev& lay, const void* x, const void* Y,
                     const void* W, void* out, const int32_t* rowptr, const int32_t* col, int64_t N,
                     cudaStream_t st) {
  UvuArgs<T> a = make_args<T>(plan, lay);
  a.x = static_cast<const T*>(x);
  a.Y = static_cast<const T*>(Y);
  a.W = static_cast<const T*>(W);
  a.out = static_cast<T*>(out);
  a.rowptr = rowptr;
  a.col = col;
  a.N = static_cast<int>(N);
  auto k = uvu_forward_kernel<T, IDENT, LMAX>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.smem_fwd);
  const int grid = grid_for(k, lay.smem_fwd, plan->num_sms, N);
  k<<<grid, kThreads, lay.smem_fwd, st>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu forward launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

template <typename T, bool IDENT, int LMAX>
cgtp_status bwd_impl(const cgtp_plan_s* plan, const LayoutDev& lay, const void* gout,
                     const void* x, const void* Y, const void* W, void* gx, void* gY, void* gW,
                     const int32_t* t_rowptr, const int32_t* t_eid, const int32_t* t_dst,
                     int64_t N, cudaStream_t st) {
  UvuArgs<T> a = make_args<T>(plan, lay);
  a.x = static_cast<const T*>(x);
  a.Y = static_cast<const T*>(Y);
  a.W = static_cast<const T*>(W);
  a.gout = static_cast<const T*>(gout);
  a.gx = static_cast<T*>(gx);
  a.gY = static_cast<T*>(gY);
  a.gW = static_cast<T*>(gW);
  a.rowptr = t_rowptr;
  a.col = t_eid;
  a.t_dst = t_dst;
  a.N = static_cast<int>(N);
  auto k = uvu_backward_kernel<T, IDENT, LMAX>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.smem_bwd);
  const int grid = grid_for(k, lay.smem_bwd, plan->num_sms, N);
  k<<<grid, kThreads, lay.smem_bwd, st>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("uvu backward launch: ") + cudaGetErrorString(err));
  return CGTP_OK;
}

}  // namespace uvu_detail
}  // namespace cgtp
