// uvu2_impl.cuh -- pipelined uvu convolution kernels for plans with l <= 3.
//
// Same operation as uvu_impl.cuh ("An Efficient Sparse Kernel Generator for
// O(3)-Equivariant Deep Networks", Figure 4B: CG tensor product fused with the
// receiver sum), organised for GB300:
//   * the x rows of a chunk's senders, its W rows and its Y rows are staged into
//     shared memory with cp.async, one chunk ahead of the compute (double
//     buffer), so the HBM stream of W overlaps the arithmetic;
//   * cy[slot] = c0 * Y[col0] + c1 * Y[col1] (every slot of a real CG block has
//     at most two nonzero terms), computed once per edge and shared by all lanes;
//   * edges are processed in pairs with the paired FP32 FMA (fma.rn.f32x2):
//     one instruction updates the accumulators of both edges.
#pragma once
#include <cuda_runtime.h>

#include "internal.h"

namespace cgtp {
namespace uvu2_detail {

__host__ __device__ inline int pad_up(int v, int q) { return (v + q - 1) / q * q; }

template <typename T>
struct P2;  // a pair of values, one per edge of an edge pair
template <>
struct P2<float> {
  using type = float2;
  static constexpr int vn = 4;
};
template <>
struct P2<double> {
  using type = double2;
  static constexpr int vn = 2;
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

// ---- cp.async ---------------------------------------------------------------
__device__ __forceinline__ void cp16(void* s, const void* g) {
  const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(s));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(g));
}
template <int B>
__device__ __forceinline__ void cpN(void* s, const void* g) {
  const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(s));
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(sa), "l"(g), "n"(B));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Copy `rows` rows of n elements (row r from src(r)) into shared memory rows of
// stride dstride, 16-byte pieces when vec is true, element pieces otherwise.
template <typename T, typename Src>
__device__ __forceinline__ void stage_rows(T* dst, int dstride, int rows, int n, bool vec, Src src,
                                           int tid, int nthr) {
  if (vec) {
    constexpr int VN = 16 / sizeof(T);
    const int units = n / VN;
    for (int i = tid; i < rows * units; i += nthr) {
      const int r = i / units, q = i - r * units;
      cp16(dst + r * dstride + q * VN, src(r) + q * VN);
    }
  } else {
    for (int i = tid; i < rows * n; i += nthr) {
      const int r = i / n, q = i - r * n;
      cpN<sizeof(T)>(dst + r * dstride + q, src(r) + q);
    }
  }
}

template <typename T>
struct Fwd2Args {
  const T* x;
  const T* Y;
  const T* W;
  T* out;
  const int* rowptr;
  const int* col;
  int N;
  int d1, d2, d_out, w_numel;
  int chunk;                     // even
  int d1p, d2p, wgp;             // padded row strides in shared memory
  bool vec_x, vec_w, vec_y;      // 16-byte staging allowed
  int n_groups;
  const PathDev* paths;
  const GroupDev* groups;
  const int* cy2_col;
  const T* cy2_coef;
  const int* cy2_base;
  const int* item_begin;
  const Item* items;
};

// One (path, 32-channel block) item over the staged chunk, edges in pairs.
template <typename T, int D1, int D3>
__device__ __noinline__ void fwd2_item(const T* xs, int d1p, const T* ws, int wgp, const T* cyp,
                                       int cy_size, int cnt, int off1, int woff, int cyoff,
                                       int ooff, int u, T* acc) {
  using Q = typename P2<T>::type;
  constexpr int NF = D1 * D3;
  Q t[D3];
#pragma unroll
  for (int k = 0; k < D3; ++k) t[k] = Q{T(0), T(0)};
  const int npair = (cnt + 1) >> 1;
  for (int pr = 0; pr < npair; ++pr) {
    const int j0 = 2 * pr, j1 = j0 + 1;
    const bool has1 = j1 < cnt;
    Q w;
    w.x = ws[j0 * wgp + woff + u];
    w.y = has1 ? ws[j1 * wgp + woff + u] : T(0);
    Q xw[D1];
    const T* x0 = xs + j0 * d1p + off1 + u * D1;
    const T* x1 = xs + j1 * d1p + off1 + u * D1;
#pragma unroll
    for (int m = 0; m < D1; ++m) {
      Q xv;
      xv.x = x0[m];
      xv.y = has1 ? x1[m] : T(0);
      xw[m] = mul2(w, xv);
    }
    // cy pairs: [pair][slot] of Q, this path's slots at cyoff
    const Q* c = reinterpret_cast<const Q*>(cyp) + pr * cy_size + cyoff;
#pragma unroll
    for (int f = 0; f < NF; ++f) t[f % D3] = fma2(c[f], xw[f / D3], t[f % D3]);
  }
  T* ap = acc + ooff + u * D3;
#pragma unroll
  for (int k = 0; k < D3; ++k) ap[k] += t[k].x + t[k].y;
}

#define CGTP2_L3_CASES(M) \
  M(0, 0) M(0, 1) M(0, 2) M(0, 3) M(1, 0) M(1, 1) M(1, 2) M(1, 3) M(2, 0) M(2, 1) M(2, 2) M(2, 3) \
  M(3, 0) M(3, 1) M(3, 2) M(3, 3)

#define CGTP2_FWD_CASE(L1, L3)                                                                  \
  case (L1)*8 + (L3):                                                                           \
    fwd2_item<T, 2 * (L1) + 1, 2 * (L3) + 1>(xs, a.d1p, ws, a.wgp, cyb, cy_size, cnt, p.off1,   \
                                             p.woff_g, p.cyoff_g, p.ooff_g, u, acc);            \
    break;

// Chunk cursor: receiver n, first edge e0 (n == ne: none).
struct Cursor {
  int n, e0;
};

__device__ __forceinline__ Cursor first_chunk(const int* rowptr, int nb, int ne) {
  int n = nb;
  while (n < ne && rowptr[n] == rowptr[n + 1]) ++n;
  return Cursor{n, n < ne ? rowptr[n] : 0};
}
__device__ __forceinline__ Cursor next_chunk(const int* rowptr, Cursor c, int chunk, int ne) {
  if (c.e0 + chunk < rowptr[c.n + 1]) return Cursor{c.n, c.e0 + chunk};
  int n = c.n + 1;
  while (n < ne && rowptr[n] == rowptr[n + 1]) ++n;
  return Cursor{n, n < ne ? rowptr[n] : 0};
}

template <typename T, int LMAX>
__global__ void __launch_bounds__(kThreads) uvu_forward2_kernel(const Fwd2Args<T> a) {
  using Q = typename P2<T>::type;
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int VN = 16 / sizeof(T);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = a.chunk;
  // receiver range of this CTA, balanced by edges + rows
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
  const int nb = s_range[0], ne = s_range[1];
  // empty receivers: zero rows
  for (int n = nb; n < ne; ++n)
    if (a.rowptr[n] == a.rowptr[n + 1])
      for (int i = tid; i < a.d_out; i += kThreads) a.out[(size_t)n * a.d_out + i] = T(0);

  int dog_max = 0;
  for (int gi = 0; gi < a.n_groups; ++gi) dog_max = max(dog_max, a.groups[gi].o1 - a.groups[gi].o0);
  T* acc = reinterpret_cast<T*>(smem);
  T* stage0 = acc + pad_up(dog_max, VN);
  const int stage_elems = chunk * (a.d1p + a.wgp + a.d2p);
  int* src_base = reinterpret_cast<int*>(stage0 + 2 * stage_elems);
  T* cyb = reinterpret_cast<T*>(src_base + pad_up(2 * chunk, 4));  // [chunk/2][cy_size] of Q

  for (int gi = 0; gi < a.n_groups; ++gi) {
    const GroupDev g = a.groups[gi];
    const int dog = g.o1 - g.o0, cy_size = g.cy_size, wg = g.w1 - g.w0;
    const int c2b = a.cy2_base[gi];
    const int ib = a.item_begin[g.item_base + warp], ie = a.item_begin[g.item_base + warp + 1];
    auto issue = [&](Cursor c, int buf) {
      T* xs = stage0 + buf * stage_elems;
      T* ws = xs + chunk * a.d1p;
      T* ys = ws + chunk * a.wgp;
      int* src = src_base + buf * chunk;
      const int cnt = min(chunk, a.rowptr[c.n + 1] - c.e0);
      for (int i = tid; i < cnt; i += kThreads) src[i] = a.col[c.e0 + i];
      const int* colp = a.col + c.e0;
      stage_rows<T>(xs, a.d1p, cnt, a.d1, a.vec_x, [&](int r) { return a.x + (size_t)colp[r] * a.d1; }, tid,
                    kThreads);
      stage_rows<T>(ws, a.wgp, cnt, wg, a.vec_w,
                    [&](int r) { return a.W + (size_t)(c.e0 + r) * a.w_numel + g.w0; }, tid, kThreads);
      stage_rows<T>(ys, a.d2p, cnt, a.d2, a.vec_y, [&](int r) { return a.Y + (size_t)(c.e0 + r) * a.d2; }, tid,
                    kThreads);
      if (cnt & 1)  // the unused partner of the last pair: zero Y so its cy is zero
        for (int i = tid; i < a.d2; i += kThreads) ys[cnt * a.d2p + i] = T(0);
      cp_commit();
    };
    for (int i = tid; i < dog; i += kThreads) acc[i] = T(0);
    Cursor cur = first_chunk(a.rowptr, nb, ne);
    int buf = 0;
    if (cur.n < ne) issue(cur, 0);
    while (cur.n < ne) {
      const Cursor nxt = next_chunk(a.rowptr, cur, chunk, ne);
      if (nxt.n < ne) {
        issue(nxt, buf ^ 1);
        cp_wait<1>();
      } else {
        cp_wait<0>();
      }
      __syncthreads();  // chunk `cur` landed; acc zeroing visible
      const int cnt = min(chunk, a.rowptr[cur.n + 1] - cur.e0);
      const int npair = (cnt + 1) >> 1;
      T* xs = stage0 + buf * stage_elems;
      T* ws = xs + chunk * a.d1p;
      T* ys = ws + chunk * a.wgp;
      // cy for the pairs: cyb[pr][slot] = (cy of edge 2pr, cy of edge 2pr+1)
      for (int i = tid; i < npair * cy_size; i += kThreads) {
        const int pr = i / cy_size, sl = i - pr * cy_size;
        const int k = 2 * (c2b + sl);
        const int i0 = a.cy2_col[k], i1 = a.cy2_col[k + 1];
        const T c0 = a.cy2_coef[k], c1 = a.cy2_coef[k + 1];
        const T* y0 = ys + (2 * pr) * a.d2p;
        const T* y1 = y0 + a.d2p;
        Q v;
        v.x = c0 * y0[i0] + c1 * y0[i1];
        v.y = c0 * y1[i0] + c1 * y1[i1];
        reinterpret_cast<Q*>(cyb)[i] = v;
      }
      __syncthreads();
      for (int it = ib; it < ie; ++it) {
        const Item item = a.items[it];
        const PathDev p = a.paths[item.path];
        const int u = item.u0 + lane;
        if (u >= p.mul) continue;
        switch (p.l1 * 8 + p.l3) {
          CGTP2_L3_CASES(CGTP2_FWD_CASE)
          default: break;
        }
      }
      __syncthreads();  // items done with this stage and cyb; acc complete if last chunk
      if (nxt.n != cur.n) {
        T* orow = a.out + (size_t)cur.n * a.d_out + g.o0;
        for (int i = tid; i < dog; i += kThreads) {
          orow[i] = acc[i];
          acc[i] = T(0);
        }
      }
      cur = nxt;
      buf ^= 1;
    }
    __syncthreads();
  }
}

}  // namespace uvu2_detail
}  // namespace cgtp
