// uvwe.cu -- fully connected (uvw) CG tensor-product convolution with a weight
// matrix per edge (no radial factorisation): W [E, sum_path mul1 * mul_out],
// each path's block laid out [u][w].
//
// "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
// Figure 1 (the product followed by a structured weight multiplication),
// Figure 3B/C (multiplicity-mixing weights) and Figure 4B (fused with the
// receiver sum):
//   t_e[path][u][m3] = sum_{m1,m2} C[m1,m2,m3] x[src][u][m1] Y[e][m2]
//   out[n][i_out][w][m3] = sum_{e in row n} sum_{path -> i_out} sum_u W_e[path][u][w] t_e[path][u][m3]
// Backward, sender-owned over the transpose (every per-edge result written once,
// gx summed per sender, deterministic, no atomics):
//   gt[u][m3] = sum_w W_e[u][w] g[dst][w][m3],   gW_e[u][w] = sum_m3 t[u][m3] g[dst][w][m3]
//   gx[s][u][m1] += sum_m3 cy[m1][m3] gt[u][m3], cy = C.Y[e]
//   gY[e][m2] += sum_{m1,m3} C[m1,m2,m3] sum_u x[s][u][m1] gt[u][m3]
// One CTA owns a receiver (forward) or a sender (backward) and walks its edges
// in chunks of eight; every stage runs over all paths of the chunk at once,
// staged through shared memory.  The weight stream is read with consecutive
// threads on consecutive weights (forward: one thread per (path, w), all the
// chunk's edges in flight; backward: one thread per (edge, path, u) walking its
// row); the forward prefetches each chunk's contiguous rows into L2.  Every
// output, gx and gY element has one owning thread, so no atomics are needed.
// This serves plans of any multiplicities with l <= 3; the per-edge weights are
// the dominant stream.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <type_traits>
#include <vector>

#include "internal.h"

namespace cgtp {
namespace uvwe_detail {

constexpr int kThr = 256;
constexpr int kCh = 8;   // edges per chunk: every stage runs over all paths of a chunk at once
constexpr int kSmemCap = 200 * 1024;

struct EPath {
  int D1, D2, D3, mul1, mul_out;
  int off1, off2, ooff, woff, coff;  // coff: first entry of the dense C block [D1][D2][D3]
  int cyo, tso;                      // offsets of the path's cy [D1][D3] and t [mul1][D3] in a chunk row
  int aco;                           // offset of the path's out[w][m3] partials (prefix sum of mul_out * D3)
  int i1, i2, io;
};

// T: arithmetic and output type; S: storage type of x, Y, W and the output
// gradient (T, or bfloat16 with T = float)
template <typename T, typename S = T>
struct EArgs {
  const S* x;
  const S* Y;
  const S* W;
  const S* g;
  T* out;
  T* gx;
  T* gY;
  T* gW;
  const int* rowptr;   // forward: CSR; backward: transpose
  const int* col;      // forward: CSR col; backward: t_eid
  const int* t_dst;
  int N, d1, d2, d_out, w_numel, n_paths;
  int ncy, nts;        // per-edge sizes of the cy and t rows (all paths)
  int n_pw, nac, n_pu; // (path, w) pairs, per-path output partials, (path, u) pairs
  const EPath* paths;
  const T* C;
  // output blocks (forward), in1 blocks (backward gx) and in2 blocks (backward gY):
  // [begin, end) element ranges and the paths that feed each block
  int n_ob, n_ib, n_yb;
  const int* ob;       // per out block: elem0, elem1, path list begin, end (4 ints)
  const int* ib;       // per in1 block: same
  const int* yb;       // per in2 block: same
  const int* plist;
  // per-entry tables, packed path | sub-index << 16:
  const int* cy_path;  // entries of a cy row [ncy]: path | m1 << 16 | m3 << 24
  const int* pu_path;  // (path, u) pairs [n_pu], ordered by D3: path | u << 16
  const int* pw_path;  // (path, w) pairs [n_pw], ordered by D3: path | w << 16
};

// Ask L2 for the 128-byte lines of [p, p + bytes), spread over the block's threads.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
  const char* c = static_cast<const char*>(p);
  for (size_t o = (size_t)threadIdx.x * 128; o < bytes; o += (size_t)kThr * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
}

// one stored value as T (bfloat16 widens exactly)
template <typename T>
__device__ __forceinline__ T to_t(T v) { return v; }
template <typename T>
__device__ __forceinline__ T to_t(__nv_bfloat16 v) { return T(__bfloat162float(v)); }
template <typename T, typename S>
__device__ __forceinline__ T ld_t(const S* p) {
  if constexpr (std::is_same<S, __nv_bfloat16>::value) {
    return T(__uint_as_float(static_cast<unsigned>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16));
  } else {
    return __ldg(p);
  }
}

// V consecutive elements of a weight row (V = 1, or one 16-byte vector of T; for
// bfloat16 storage the same V values in one 8-byte load)
template <int V, typename T>
__device__ __forceinline__ void ldrow(const __nv_bfloat16* p, T (&r)[V]) {
  if constexpr (V == 1) {
    r[0] = ld_t<T>(p);
  } else {
    static_assert(V == 4, "bfloat16 rows come in vectors of four");
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
    r[0] = __uint_as_float(q.x << 16);
    r[1] = __uint_as_float(q.x & 0xffff0000u);
    r[2] = __uint_as_float(q.y << 16);
    r[3] = __uint_as_float(q.y & 0xffff0000u);
  }
}
template <int V, typename T>
__device__ __forceinline__ void ldrow(const T* p, T (&r)[V]) {
  if constexpr (V == 1) {
    r[0] = __ldg(p);
  } else if constexpr (sizeof(T) == 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
  } else {
    const double2 v = __ldg(reinterpret_cast<const double2*>(p));
    r[0] = v.x; r[1] = v.y;
  }
}
template <int V, typename T>
__device__ __forceinline__ void strow(T* p, const T (&r)[V]) {
  if constexpr (V == 1) {
    p[0] = r[0];
  } else if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(r[0], r[1], r[2], r[3]);
  } else {
    *reinterpret_cast<double2*>(p) = make_double2(r[0], r[1]);
  }
}

// Call f with the block size D3 as a compile-time constant (a std::integral_constant).
template <typename F>
__device__ __forceinline__ void with_d3(int D3, F&& f) {
  switch (D3) {
    case 1: f(std::integral_constant<int, 1>{}); break;
    case 3: f(std::integral_constant<int, 3>{}); break;
    case 5: f(std::integral_constant<int, 5>{}); break;
    default: f(std::integral_constant<int, 7>{}); break;
  }
}

// (j, r) = divmod(f, n) for f = threadIdx.x, threadIdx.x + kThr, ...: two
// divisions per stage instead of one per element
struct JR {
  int j, r, q, rem, n;
  __device__ __forceinline__ explicit JR(int n_) : n(n_) {
    j = threadIdx.x / n;
    r = threadIdx.x - j * n;
    q = kThr / n;
    rem = kThr - q * n;
  }
  __device__ __forceinline__ void next() {
    r += rem;
    j += q;
    if (r >= n) {
      r -= n;
      ++j;
    }
  }
};

// cy rows of a chunk: cy[j][path][m1][m3] = sum_m2 C Y[j][m2] (yrow(j): the
// chunk's j-th Y row, in shared or global memory)
template <typename T, typename S, typename YRow>
__device__ __forceinline__ void chunk_cy(const EArgs<T, S>& a, YRow yrow, T* cy, int cnt) {
  if (a.ncy == 0) return;
  for (JR it(a.ncy); it.j < cnt; it.next()) {
    const int e = __ldg(a.cy_path + it.r);
    const EPath p = a.paths[e & 0xffff];
    const int m1 = (e >> 16) & 0xff, m3 = e >> 24;
    const T* Cp = a.C + p.coff + m1 * p.D2 * p.D3 + m3;
    const auto* yr = yrow(it.j) + p.off2;   // T (shared memory) or S (global) values
    T v = T(0);
    for (int m2 = 0; m2 < p.D2; ++m2) v += __ldg(Cp + m2 * p.D3) * to_t<T>(yr[m2]);
    cy[it.j * a.ncy + it.r] = v;
  }
}

// t[m3] = sum_m1 cy[m1][m3] x[m1] of one (edge, path, u)
template <int D3, typename T>
__device__ __forceinline__ void t_row(const T* c, const T* xr, int D1, T (&t)[D3]) {
#pragma unroll
  for (int m3 = 0; m3 < D3; ++m3) t[m3] = T(0);
  for (int m1 = 0; m1 < D1; ++m1) {
    const T xv = xr[m1];
#pragma unroll
    for (int m3 = 0; m3 < D3; ++m3) t[m3] += c[m1 * D3 + m3] * xv;
  }
}

// Forward, software-pipelined over a receiver's chunks in steps of two phases:
//   phase 1 of step k: weight stage of chunk k - 1 beside the staging of chunk k
//                      (x gather, cy from the Y rows, weight prefetch)
//   phase 2 of step k: t stage of chunk k
// so a chunk costs two block barriers.  Every stage has one call site.
template <typename T, typename S>
__global__ void __launch_bounds__(kThr) uvwe_fwd_kernel(const EArgs<T, S> a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* accs = reinterpret_cast<T*>(smem_raw);   // [nac]: per path, out[w][m3] partials
  T* xs = accs + a.nac;             // [kCh][d1]
  T* cy = xs + kCh * a.d1;          // [kCh][ncy]
  T* ts = cy + kCh * a.ncy;         // [kCh][nts]
  const int tid = threadIdx.x;
  // per (path, w): acc[m3] += sum_{j, u} W_j[u][w] t_j[u][m3] over the chunk at e0;
  // a warp's weight loads cover consecutive w, and the chunk's edges are in flight together
  auto weights = [&](int e0, int cnt) {
    for (int pw = tid; pw < a.n_pw; pw += kThr) {
      const int e = __ldg(a.pw_path + pw);
      const EPath p = a.paths[e & 0xffff];
      const int w = e >> 16;
      const S* Wp = a.W + (size_t)e0 * a.w_numel + p.woff + w;
      with_d3(p.D3, [&](auto d3c) {
        constexpr int D3 = decltype(d3c)::value;
        T acc0[D3], acc1[D3];   // even and odd edges: two independent FMA chains
#pragma unroll
        for (int m3 = 0; m3 < D3; ++m3) acc0[m3] = acc1[m3] = T(0);
        for (int u = 0; u < p.mul1; ++u) {
          T wv[kCh];
#pragma unroll
          for (int j = 0; j < kCh; ++j) wv[j] = j < cnt ? ld_t<T>(Wp + (size_t)j * a.w_numel + u * p.mul_out) : T(0);
#pragma unroll
          for (int j = 0; j < kCh; ++j) {
            if (j < cnt) {
              const T* tj = ts + j * a.nts + p.tso + u * D3;
#pragma unroll
              for (int m3 = 0; m3 < D3; ++m3) {
                if (j & 1) acc1[m3] += wv[j] * tj[m3];
                else acc0[m3] += wv[j] * tj[m3];
              }
            }
          }
        }
        T* dst = accs + p.aco + w * D3;
#pragma unroll
        for (int m3 = 0; m3 < D3; ++m3) dst[m3] += acc0[m3] + acc1[m3];
      });
    }
  };
  for (int n = blockIdx.x; n < a.N; n += gridDim.x) {
    for (int i = tid; i < a.nac; i += kThr) accs[i] = T(0);
    const int e_begin = a.rowptr[n], e_end = a.rowptr[n + 1];
    auto count = [&](int k) { return k < 0 ? 0 : max(0, min(kCh, e_end - e_begin - k * kCh)); };
    for (int k = -1;; ++k) {
      const int e0 = e_begin + k * kCh, cnt = count(k);
      if (k >= 1) weights(e0 - kCh, count(k - 1));
      if (cnt > 0) {
        // the chunk's weight rows are contiguous: have L2 fetch them while the
        // product stages run
        prefetch_l2(a.W + (size_t)e0 * a.w_numel, sizeof(S) * (size_t)cnt * a.w_numel);
        for (JR it(a.d1); it.j < cnt; it.next())
          xs[it.j * a.d1 + it.r] = to_t<T>(a.x[(size_t)a.col[e0 + it.j] * a.d1 + it.r]);
        chunk_cy(a, [&](int j) { return a.Y + (size_t)(e0 + j) * a.d2; }, cy, cnt);
      }
      __syncthreads();  // x and cy of chunk k staged; the weight stage is done with ts
      if (k >= 0 && cnt == 0) break;
      // t[j][path][u][:] = cy x[u], one (edge, path, u) per item
      for (JR it(a.n_pu > 0 ? a.n_pu : 1); a.n_pu > 0 && it.j < cnt; it.next()) {
        const int j = it.j, e = __ldg(a.pu_path + it.r);
        const EPath p = a.paths[e & 0xffff];
        const int u = e >> 16;
        with_d3(p.D3, [&](auto d3c) {
          constexpr int D3 = decltype(d3c)::value;
          T t[D3];
          t_row<D3>(cy + j * a.ncy + p.cyo, xs + j * a.d1 + p.off1 + u * p.D1, p.D1, t);
          T* dst = ts + j * a.nts + p.tso + u * D3;
#pragma unroll
          for (int m3 = 0; m3 < D3; ++m3) dst[m3] = t[m3];
        });
      }
      __syncthreads();  // ts of chunk k ready; xs and cy free for the next chunk
    }
    // out[n] block by block: the sum of the partials of the paths feeding it
    for (int b = 0; b < a.n_ob; ++b) {
      const int o0 = a.ob[4 * b], o1 = a.ob[4 * b + 1], q0 = a.ob[4 * b + 2], q1 = a.ob[4 * b + 3];
      for (int f = o0 + tid; f < o1; f += kThr) {
        T v = T(0);
        for (int q = q0; q < q1; ++q) {
          const EPath p = a.paths[a.plist[q]];
          v += accs[p.aco + f - p.ooff];
        }
        a.out[(size_t)n * a.d_out + f] = v;
      }
    }
    __syncthreads();
  }
}

// V: weight-row vector width (1, or 16 bytes when every row segment is aligned)
//
// Backward over a sender's chunks: staging (edge ids, g rows, Y rows), cy, the
// fused t / gW / gt stage, G and gx, gY -- five block
// barriers a chunk.  (Overlapping gY and G with the next chunk's staging
// measured slower: the gathers' latency then sits inside the compute phases.)
template <typename T, int V, typename S>
__global__ void __launch_bounds__(kThr) uvwe_bwd_kernel(const EArgs<T, S> a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* xs = reinterpret_cast<T*>(smem_raw);   // [d1]
  T* gxs = xs + a.d1;                       // [d1]
  T* gs = gxs + a.d1;                       // [kCh][d_out]
  T* ys = gs + kCh * a.d_out;               // [kCh][d2]
  T* cy = ys + kCh * a.d2;                  // [kCh][ncy]
  T* G = cy + kCh * a.ncy;                  // [kCh][ncy]
  T* gts = G + kCh * a.ncy;                 // [kCh][nts]
  int* eids = reinterpret_cast<int*>(gts + kCh * a.nts);   // [kCh]
  const int tid = threadIdx.x;
  for (int s = blockIdx.x; s < a.N; s += gridDim.x) {
    for (int i = tid; i < a.d1; i += kThr) {
      xs[i] = to_t<T>(a.x[(size_t)s * a.d1 + i]);
      gxs[i] = T(0);
    }
    const int t_begin = a.rowptr[s], t_end = a.rowptr[s + 1];
    for (int t0 = t_begin; t0 < t_end; t0 += kCh) {
      const int cnt = min(kCh, t_end - t0);
      const int* eid = eids;
      __syncthreads();
      if (tid < cnt) eids[tid] = a.col[t0 + tid];
      for (JR it(a.d_out); it.j < cnt; it.next())
        gs[it.j * a.d_out + it.r] = to_t<T>(a.g[(size_t)a.t_dst[t0 + it.j] * a.d_out + it.r]);
      for (JR it(a.d2); it.j < cnt; it.next())
        ys[it.j * a.d2 + it.r] = to_t<T>(a.Y[(size_t)a.col[t0 + it.j] * a.d2 + it.r]);
      __syncthreads();
      chunk_cy(a, [&](int j) { return ys + j * a.d2; }, cy, cnt);
      __syncthreads();
        // per (edge, path, u): t = cy x[u], then along the weight row
        //   gW[u][w] = sum_m3 t[m3] g[w][m3],  gt[u][m3] = sum_w W[u][w] g[w][m3]
        for (JR it(a.n_pu > 0 ? a.n_pu : 1); a.n_pu > 0 && it.j < cnt; it.next()) {
          const int j = it.j, e = __ldg(a.pu_path + it.r);
          const EPath p = a.paths[e & 0xffff];
          const int u = e >> 16;
          const size_t row = (size_t)eid[j] * a.w_numel + p.woff + (size_t)u * p.mul_out;
          const T* gj = gs + j * a.d_out + p.ooff;
          with_d3(p.D3, [&](auto d3c) {
            constexpr int D3 = decltype(d3c)::value;
            T t[D3], gt[D3];
            t_row<D3>(cy + j * a.ncy + p.cyo, xs + p.off1 + u * p.D1, p.D1, t);
#pragma unroll
            for (int m3 = 0; m3 < D3; ++m3) gt[m3] = T(0);
            for (int w = 0; w < p.mul_out; w += V) {
              T wv[V], gw[V];
              ldrow<V>(a.W + row + w, wv);
#pragma unroll
              for (int c = 0; c < V; ++c) {
                gw[c] = T(0);
#pragma unroll
                for (int m3 = 0; m3 < D3; ++m3) {
                  const T gv = gj[(w + c) * D3 + m3];
                  gw[c] += t[m3] * gv;
                  gt[m3] += wv[c] * gv;
                }
              }
              strow<V>(a.gW + row + w, gw);
            }
            T* gd = gts + j * a.nts + p.tso + u * D3;
#pragma unroll
            for (int m3 = 0; m3 < D3; ++m3) gd[m3] = gt[m3];
          });
        }
      __syncthreads();
        // G[j][path][m1][m3] = sum_u x[u][m1] gt[u][m3]
        if (a.ncy > 0) {
          for (JR it(a.ncy); it.j < cnt; it.next()) {
            const int e = __ldg(a.cy_path + it.r);
            const EPath p = a.paths[e & 0xffff];
            const int m1 = (e >> 16) & 0xff, m3 = e >> 24;
            const T* gt = gts + it.j * a.nts + p.tso + m3;
            const T* xr = xs + p.off1 + m1;
            T v = T(0);
            for (int u = 0; u < p.mul1; ++u) v += xr[u * p.D1] * gt[u * p.D3];
            G[it.j * a.ncy + it.r] = v;
          }
        }
        // gx[u][m1] of every in1 block += sum over the chunk's edges and the block's paths
        for (int b = 0; b < a.n_ib; ++b) {
          const int o0 = a.ib[4 * b], o1 = a.ib[4 * b + 1], q0 = a.ib[4 * b + 2], q1 = a.ib[4 * b + 3];
          if (q0 == q1) continue;
          const int D1 = a.paths[a.plist[q0]].D1;   // every path of an in1 block shares its degree
          for (int f = o0 + tid; f < o1; f += kThr) {
            const int u = (f - o0) / D1, m1 = (f - o0) - u * D1;
            T v = T(0);
            for (int q = q0; q < q1; ++q) {
              const EPath p = a.paths[a.plist[q]];
              with_d3(p.D3, [&](auto d3c) {
                constexpr int D3 = decltype(d3c)::value;
                for (int j = 0; j < cnt; ++j) {
                  const T* c = cy + j * a.ncy + p.cyo + m1 * D3;
                  const T* gt = gts + j * a.nts + p.tso + u * D3;
#pragma unroll
                  for (int m3 = 0; m3 < D3; ++m3) v += c[m3] * gt[m3];
                }
              });
            }
            gxs[f] += v;
          }
        }
      __syncthreads();
      // gY[j][m2] of every in2 block = sum over the block's paths of C . G
      for (JR it(a.d2); it.j < cnt; it.next()) {
        const int j = it.j, col2 = it.r;
        int b = 0;
        while (b + 1 < a.n_yb && a.yb[4 * (b + 1)] <= col2) ++b;
        T v = T(0);
        for (int q = a.yb[4 * b + 2]; q < a.yb[4 * b + 3]; ++q) {
          const EPath p = a.paths[a.plist[q]];
          const int m2 = col2 - p.off2;
          const T* Gj = G + j * a.ncy + p.cyo;
          for (int m1 = 0; m1 < p.D1; ++m1)
            for (int m3 = 0; m3 < p.D3; ++m3) v += __ldg(a.C + p.coff + (m1 * p.D2 + m2) * p.D3 + m3) * Gj[m1 * p.D3 + m3];
        }
        a.gY[(size_t)eid[j] * a.d2 + col2] = v;
      }
    }
    __syncthreads();
    for (int i = tid; i < a.d1; i += kThr) a.gx[(size_t)s * a.d1 + i] = gxs[i];
    __syncthreads();
  }
}

struct EState {
  void* tables = nullptr;
  const EPath* paths = nullptr;
  const void* C = nullptr;
  const int *ob = nullptr, *ib = nullptr, *yb = nullptr, *plist = nullptr;
  const int *cy_path = nullptr, *pu_path = nullptr, *pw_path = nullptr;
  bool vec = false;
  int n_paths = 0, ncy = 0, nts = 0, n_pw = 0, nac = 0, n_pu = 0, n_ob = 0, n_ib = 0, n_yb = 0;
  size_t smem_fwd = 0, smem_bwd = 0;
};

}  // namespace uvwe_detail

using namespace uvwe_detail;

cgtp_status uvwe_create(cgtp_plan_s* plan) {
  int lmax = 0;
  for (const auto& p : plan->paths) lmax = std::max(lmax, std::max(p.l1, std::max(p.l2, p.l3)));
  if (lmax > 3) return fail(CGTP_EUNSUPPORTED, "per-edge uvw weights support l <= 3");
  std::vector<EPath> ep;
  std::vector<double> C;
  int ncy = 0, nts = 0, n_pw = 0, nac = 0, n_pu = 0;
  for (const auto& h : plan->paths) {
    EPath e{};
    e.D1 = 2 * h.l1 + 1;
    e.D2 = 2 * h.l2 + 1;
    e.D3 = 2 * h.l3 + 1;
    e.mul1 = h.mul1;
    e.mul_out = h.mul_out;
    e.off1 = h.off1;
    e.off2 = h.off2;
    e.ooff = h.ooff;
    e.woff = h.woff;
    e.coff = static_cast<int>(C.size());
    e.cyo = ncy;
    e.tso = nts;
    e.aco = nac;
    e.i1 = h.i1;
    e.i2 = h.i2;
    e.io = h.io;
    ncy += e.D1 * e.D3;
    nts += e.mul1 * e.D3;
    n_pw += e.mul_out;
    nac += e.mul_out * e.D3;
    n_pu += e.mul1;
    C.insert(C.end(), h.C.begin(), h.C.end());
    ep.push_back(e);
  }
  // blocks -> feeding paths, in path order (the order of every sum)
  std::vector<int> ob, ib, yb, plist;
  auto blocks = [&](const std::vector<Irrep>& irr, auto which, std::vector<int>& out) {
    int off = 0;
    for (size_t k = 0; k < irr.size(); ++k) {
      const int size = irr[k].mul * (2 * irr[k].l + 1);
      const int q0 = static_cast<int>(plist.size());
      for (size_t pi = 0; pi < ep.size(); ++pi)
        if (which(ep[pi]) == static_cast<int>(k)) plist.push_back(static_cast<int>(pi));
      out.insert(out.end(), {off, off + size, q0, static_cast<int>(plist.size())});
      off += size;
    }
  };
  blocks(plan->out, [](const EPath& e) { return e.io; }, ob);
  blocks(plan->in1, [](const EPath& e) { return e.i1; }, ib);
  blocks(plan->in2, [](const EPath& e) { return e.i2; }, yb);
  // path of every flattened entry of the per-edge rows the stages index
  // packed as path | sub-index << 16 (cy: path | m1 << 16 | m3 << 24).  The (path, u)
  // and (path, w) entries are ordered by output block size, so that a warp's
  // threads mostly run the same specialised code.
  if (ep.size() > 0xffff) return fail(CGTP_EUNSUPPORTED, "per-edge uvw weights: too many paths");
  std::vector<int> cy_path, pu_path, pw_path;
  bool vec = true;   // every weight-row segment a whole number of 16-byte vectors
  const int vw = plan->dtype == CGTP_F64 ? 2 : 4;
  if (plan->w_numel % vw) vec = false;
  std::vector<int> by_d3(ep.size());
  for (size_t pi = 0; pi < ep.size(); ++pi) by_d3[pi] = static_cast<int>(pi);
  std::stable_sort(by_d3.begin(), by_d3.end(), [&](int x, int y) { return ep[x].D3 < ep[y].D3; });
  for (size_t pi = 0; pi < ep.size(); ++pi) {
    const EPath& e = ep[pi];
    if (e.mul1 > 0x7fff || e.mul_out > 0x7fff)
      return fail(CGTP_EUNSUPPORTED, "per-edge uvw weights: multiplicity above 32767");
    for (int m1 = 0; m1 < e.D1; ++m1)
      for (int m3 = 0; m3 < e.D3; ++m3) cy_path.push_back(static_cast<int>(pi) | m1 << 16 | m3 << 24);
    if (e.mul_out % vw || e.woff % vw) vec = false;
  }
  for (int pi : by_d3) {
    for (int u = 0; u < ep[pi].mul1; ++u) pu_path.push_back(pi | u << 16);
    for (int w = 0; w < ep[pi].mul_out; ++w) pw_path.push_back(pi | w << 16);
  }
  const size_t es = plan->dtype == CGTP_F64 ? 8 : 4;
  EState* st = new EState();
  st->n_paths = static_cast<int>(ep.size());
  st->ncy = ncy;
  st->nts = nts;
  st->n_pw = n_pw;
  st->nac = nac;
  st->n_pu = n_pu;
  st->n_ob = static_cast<int>(ob.size() / 4);
  st->n_ib = static_cast<int>(ib.size() / 4);
  st->n_yb = static_cast<int>(yb.size() / 4);
  st->smem_fwd = es * (size_t(nac) + kCh * (size_t(plan->d1) + ncy + nts));
  st->smem_bwd = es * (2 * size_t(plan->d1) + kCh * (size_t(plan->d_out) + plan->d2 + 2 * ncy + nts)) + kCh * sizeof(int);
  if (st->smem_bwd > kSmemCap || st->smem_fwd > kSmemCap) {
    delete st;
    return fail(CGTP_EUNSUPPORTED, "per-edge uvw weights: rows too long for shared memory");
  }
  std::vector<unsigned char> buf;
  auto put = [&](const void* src, size_t bytes) {
    const size_t o = (buf.size() + 15) / 16 * 16;
    buf.resize(o + std::max<size_t>(bytes, 16));
    if (bytes) std::memcpy(buf.data() + o, src, bytes);
    return o;
  };
  const size_t o_p = put(ep.data(), ep.size() * sizeof(EPath));
  std::vector<unsigned char> cbytes(C.size() * es);
  for (size_t i = 0; i < C.size(); ++i) {
    if (es == 8) {
      std::memcpy(cbytes.data() + i * 8, &C[i], 8);
    } else {
      const float f = static_cast<float>(C[i]);
      std::memcpy(cbytes.data() + i * 4, &f, 4);
    }
  }
  const size_t o_c = put(cbytes.data(), cbytes.size());
  const size_t o_ob = put(ob.data(), ob.size() * sizeof(int));
  const size_t o_ib = put(ib.data(), ib.size() * sizeof(int));
  const size_t o_yb = put(yb.data(), yb.size() * sizeof(int));
  const size_t o_pl = put(plist.data(), plist.size() * sizeof(int));
  const size_t o_cp = put(cy_path.data(), cy_path.size() * sizeof(int));
  const size_t o_up = put(pu_path.data(), pu_path.size() * sizeof(int));
  const size_t o_wp = put(pw_path.data(), pw_path.size() * sizeof(int));
  if (cudaMalloc(&st->tables, buf.size()) != cudaSuccess) {
    delete st;
    return fail(CGTP_ENOMEM, "per-edge uvw table allocation failed");
  }
  if (cudaMemcpy(st->tables, buf.data(), buf.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(st->tables);
    delete st;
    return fail(CGTP_ECUDA, "per-edge uvw table upload failed");
  }
  plan->device_bytes += buf.size();
  auto at = [&](size_t o) { return static_cast<unsigned char*>(st->tables) + o; };
  st->paths = reinterpret_cast<const EPath*>(at(o_p));
  st->C = at(o_c);
  st->ob = reinterpret_cast<const int*>(at(o_ob));
  st->ib = reinterpret_cast<const int*>(at(o_ib));
  st->yb = reinterpret_cast<const int*>(at(o_yb));
  st->plist = reinterpret_cast<const int*>(at(o_pl));
  st->cy_path = reinterpret_cast<const int*>(at(o_cp));
  st->pu_path = reinterpret_cast<const int*>(at(o_up));
  st->pw_path = reinterpret_cast<const int*>(at(o_wp));
  st->vec = vec;
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_fwd_kernel<float, float>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_bwd_kernel<float, 1, float>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_bwd_kernel<float, 4, float>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_fwd_kernel<double, double>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_bwd_kernel<double, 1, double>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_bwd_kernel<double, 2, double>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_fwd_kernel<float, __nv_bfloat16>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_bwd_kernel<float, 1, __nv_bfloat16>));
  raise_smem_limit(reinterpret_cast<const void*>(uvwe_bwd_kernel<float, 4, __nv_bfloat16>));
  plan->uvwe = st;
  return CGTP_OK;
}

void uvwe_destroy(cgtp_plan_s* plan) {
  EState* st = static_cast<EState*>(plan->uvwe);
  if (!st) return;
  if (st->tables) cudaFree(st->tables);
  delete st;
  plan->uvwe = nullptr;
}

template <typename T, typename S>
static EArgs<T, S> e_args(const cgtp_plan_s* plan, const EState* st, const cgtp_graph_s* g) {
  EArgs<T, S> a{};
  a.N = static_cast<int>(g->N);
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.d_out = static_cast<int>(plan->d_out);
  a.w_numel = static_cast<int>(plan->w_numel);
  a.n_paths = st->n_paths;
  a.ncy = st->ncy;
  a.nts = st->nts;
  a.n_pw = st->n_pw;
  a.nac = st->nac;
  a.n_pu = st->n_pu;
  a.paths = st->paths;
  a.C = static_cast<const T*>(st->C);
  a.n_ob = st->n_ob;
  a.n_ib = st->n_ib;
  a.n_yb = st->n_yb;
  a.ob = st->ob;
  a.ib = st->ib;
  a.yb = st->yb;
  a.plist = st->plist;
  a.cy_path = st->cy_path;
  a.pu_path = st->pu_path;
  a.pw_path = st->pw_path;
  return a;
}

template <typename T, typename S = T>
static cgtp_status fwd_t(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* x, const void* Y,
                         const void* W, void* out, cudaStream_t s) {
  const EState* st = static_cast<const EState*>(plan->uvwe);
  EArgs<T, S> a = e_args<T, S>(plan, st, g);
  a.x = static_cast<const S*>(x);
  a.Y = static_cast<const S*>(Y);
  a.W = static_cast<const S*>(W);
  a.out = static_cast<T*>(out);
  a.rowptr = g->rowptr;
  a.col = g->col;
  // as many receivers in flight as fit: the forward's weight stream is contiguous
  int occ = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, uvwe_fwd_kernel<T, S>, kThr, st->smem_fwd);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g->N, (int64_t)plan->num_sms * std::max(occ, 1))));
  uvwe_fwd_kernel<T, S><<<grid, kThr, st->smem_fwd, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CGTP_OK : fail(CGTP_ECUDA, std::string("per-edge uvw forward launch: ") + cudaGetErrorString(e));
}

template <typename T, typename S = T>
static cgtp_status bwd_t(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* gout, const void* x,
                         const void* Y, const void* W, void* gx, void* gY, void* gW, cudaStream_t s) {
  const EState* st = static_cast<const EState*>(plan->uvwe);
  EArgs<T, S> a = e_args<T, S>(plan, st, g);
  a.x = static_cast<const S*>(x);
  a.Y = static_cast<const S*>(Y);
  a.W = static_cast<const S*>(W);
  a.g = static_cast<const S*>(gout);
  a.gx = static_cast<T*>(gx);
  a.gY = static_cast<T*>(gY);
  a.gW = static_cast<T*>(gW);
  a.rowptr = g->t_rowptr;
  a.col = g->t_eid;
  a.t_dst = g->t_dst;
  // as many senders in flight as fit; the backward's weight rows are scattered, so it
  // relies on occupancy rather than an L2 prefetch (with the prefetch, a full grid
  // thrashed L2: 4.1 ms; without it 3.22 ms against 3.35 ms at four CTAs per SM)
  int occ = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, uvwe_bwd_kernel<T, 1, S>, kThr, st->smem_bwd);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g->N, (int64_t)plan->num_sms * std::max(occ, 1))));
  constexpr int kVec = 16 / sizeof(T);
  const bool vec = st->vec && (reinterpret_cast<uintptr_t>(W) % 16 == 0) && (reinterpret_cast<uintptr_t>(gW) % 16 == 0);
  if (vec)
    uvwe_bwd_kernel<T, kVec, S><<<grid, kThr, st->smem_bwd, s>>>(a);
  else
    uvwe_bwd_kernel<T, 1, S><<<grid, kThr, st->smem_bwd, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CGTP_OK : fail(CGTP_ECUDA, std::string("per-edge uvw backward launch: ") + cudaGetErrorString(e));
}

cgtp_status uvwe_forward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* x, const void* Y,
                         const void* W, void* out, void* stream) {
  if (g->N == 0) return CGTP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (plan->dtype == CGTP_BF16) return fwd_t<float, __nv_bfloat16>(plan, g, x, Y, W, out, s);
  return plan->dtype == CGTP_F64 ? fwd_t<double>(plan, g, x, Y, W, out, s) : fwd_t<float>(plan, g, x, Y, W, out, s);
}

cgtp_status uvwe_backward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* gout, const void* x,
                          const void* Y, const void* W, void* gx, void* gY, void* gW, void* stream) {
  if (g->N == 0) return CGTP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (plan->dtype == CGTP_BF16) return bwd_t<float, __nv_bfloat16>(plan, g, gout, x, Y, W, gx, gY, gW, s);
  return plan->dtype == CGTP_F64 ? bwd_t<double>(plan, g, gout, x, Y, W, gx, gY, gW, s)
                                 : bwd_t<float>(plan, g, gout, x, Y, W, gx, gY, gW, s);
}

}  // namespace cgtp
