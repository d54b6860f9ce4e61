// uvu4_impl.cuh -- uvu convolution kernels with each warp's gathered operands
// staged through a private shared-memory ring by bulk asynchronous copies.
//
// Same operation and arithmetic as uvu3_impl.cuh ("An Efficient Sparse Kernel
// Generator for O(3)-Equivariant Deep Networks", Figure 4B: the CG tensor
// product fused with the receiver sum; gradients from its Abstract) and the
// same scheduling: one counter per CTA hands out (item, receiver) pairs
// item-major (forward) or (sender, item) pairs per phase (backward), so the
// warps of an SM run the same baked path code at a time.
//
// What changes is how operands arrive.  v3 loads each edge's gathered rows
// (x[src] slice, W slice, Y row; in the backward the output-gradient slice of
// the receiver) straight into registers right before using them, so every
// edge waits for an L2 round trip.  Here every warp owns a ring of S stages in
// shared memory; a stage holds SC edges of one unit.  The warp's lanes issue
// one cp.async.bulk per operand and edge (completion counted on the stage's
// mbarrier) for the stages ahead of the one being computed, so S-1 stages of
// gathers are in flight while the warp computes.  The warp is its own producer
// and consumer: a stage is refilled only after the warp has read it (program
// order, then a proxy fence), so no cross-warp synchronisation is added.
//
// Every mbarrier wait is bounded; a wait that gives up sets bit 0 of the
// plan's host-mapped error word, the warp stops computing, waits (bounded) for
// its copies still in flight and leaves the kernel; the host reports
// CGTP_ECUDA on the plan's next call.
#pragma once
#include "bulk.cuh"
#include "uvu3_impl.cuh"

namespace cgtp {
namespace uvu4_detail {
using namespace uvu3_detail;

constexpr int kV4Warps = 8;
constexpr int kV4Threads = kV4Warps * 32;

// Staging geometry of a plan (V4Ring, host-computed in build_v3).  Per edge a
// stage holds the unit's slice of the gathered operand (x in the forward, the
// output gradient in the backward: ublock * (2l+1) elements, room for the
// largest l), its weight slice (ublock elements), its harmonics row (d2
// elements; none for edge vectors) and, in the backward, its edge id; the
// backward's stage also holds the sender's x slice (first stage of a unit).
using Ring = V4Ring;

// Accumulation into gY / gx: each element gets at most one contribution per
// backward phase and the phases are separated by block barriers, so the order
// of the additions is fixed (deterministic); the reduction needs no return
// value, so the warp does not wait for the read.
__device__ __forceinline__ void gY_add(float* p, float v) { atomicAdd(p, v); }
__device__ __forceinline__ void gY_add(double* p, double v) { atomicAdd(p, v); }

template <typename T, typename S>
struct Uvu4Args {
  Uvu3Args<T, S> b;
  Ring r;
  int ublock;            // channels of an item (4 * LPE)
  int* err;              // host-mapped error word (bit 0: a staging wait gave up)
  long long wait_limit;  // polls before a staging wait gives up
};

// Warp-uniform fetch cursor (kept in shared memory, one per warp).
struct FetchState {
  int k;      // unit being fetched
  int it;     // its item
  int n;      // receiver (forward) / sender (backward)
  int e0;     // first CSR (transpose) position of the unit's edges
  int deg;    // its edge count
  int j;      // next edge offset to fetch
  int done;   // no more units in this phase
  int pad;
};

// offsets inside a stage (bytes)
template <typename S>
__device__ __forceinline__ int off_w(const Ring& r) { return r.SC * r.a_elems * (int)sizeof(S); }
template <typename S>
__device__ __forceinline__ int off_y(const Ring& r, int ublock) { return off_w<S>(r) + r.SC * ublock * (int)sizeof(S); }
template <typename S>
__device__ __forceinline__ int off_e(const Ring& r, int ublock) { return off_y<S>(r, ublock) + r.SC * r.y_elems * (int)sizeof(S); }
template <typename S>
__device__ __forceinline__ int off_x(const Ring& r, int ublock) { return off_e<S>(r, ublock) + ((r.SC * 4 + 15) & ~15); }

// Fetch the next stage of this warp into `slot`: acquire a unit when the
// current one is exhausted, then issue one bulk copy per operand and edge.
// Returns false when the warp's units are exhausted.  BWD selects the
// backward's operands (transpose edges, output-gradient slices, sender x slice).
template <bool BWD, typename T, typename S>
__device__ __forceinline__ bool v4_fetch(const S* __restrict__ x, const S* __restrict__ Y, const S* __restrict__ W,
                                      const S* __restrict__ gout, const int* __restrict__ rowptr,
                                      const int* __restrict__ col, const int* __restrict__ t_dst,
                                      const Item* __restrict__ items, const PathDev* __restrict__ paths,
                                      int d1, int d2, int d_out, int w_numel, Ring r, int ublock, int nb,
                                      int nr, int ni, int item0, int total, int* ctr, FetchState* fs,
                                      unsigned char* ring, uint64_t* bars, int4* desc, int slot) {
  const int lane = threadIdx.x & 31;
  if (fs->done) return false;
  if (fs->j >= max(fs->deg, 1)) {  // acquire the next unit
    int k = 0;
    if (lane == 0) k = atomicAdd(ctr, 1);
    k = __shfl_sync(0xffffffffu, k, 0);
    __syncwarp();
    if (k >= total) {
      if (lane == 0) fs->done = 1;
      __syncwarp();
      return false;
    }
    int it, n;
    if (BWD) {  // sender-major inside a phase
      const int sl = k / ni;
      it = item0 + (k - sl * ni);
      n = nb + sl;
    } else {    // item-major
      it = k / nr;
      n = nb + (k - it * nr);
    }
    const int e0 = __ldg(rowptr + n), deg = __ldg(rowptr + n + 1) - e0;
    if (lane == 0) {
      fs->k = k;
      fs->it = it;
      fs->n = n;
      fs->e0 = e0;
      fs->deg = deg;
      fs->j = 0;
    }
    __syncwarp();
  }
  const int j = fs->j, deg = fs->deg, e0 = fs->e0, n = fs->n, it = fs->it, k = fs->k;
  __syncwarp();  // every lane has read the cursor before lane 0 advances it
  const Item item = items[it];
  const PathDev p = paths[item.path];
  const int cnt = min(r.SC, deg - j);
  const int es = (int)sizeof(S);
  const uint32_t abytes = ublock * (BWD ? p.D3 : p.D1) * es, wbytes = ublock * es, ybytes = r.y_elems * es;
  const uint32_t xbytes = (BWD && j == 0) ? ublock * p.D1 * es : 0;
  unsigned char* st = ring + (size_t)slot * r.stage_bytes;
  if (lane == 0) {
    desc[slot] = make_int4(k, j, cnt, deg);
    bulk::mbar_arrive_expect_tx(&bars[slot], cnt * (abytes + wbytes + ybytes) + xbytes);
    fs->j = j + max(cnt, 1);  // an empty row is one (empty) stage
  }
  __syncwarp();
  if (lane < cnt) {
    int e, src_row;
    if (BWD) {
      e = __ldg(col + e0 + j + lane);         // transpose: edge id
      src_row = __ldg(t_dst + e0 + j + lane);  // its receiver
      reinterpret_cast<int*>(st + off_e<S>(r, ublock))[lane] = e;
      bulk::copy_g2s(st + lane * r.a_elems * es, gout + (size_t)src_row * d_out + p.ooff + item.u0 * p.D3, abytes,
                     &bars[slot]);
    } else {
      e = e0 + j + lane;
      src_row = __ldg(col + e);
      bulk::copy_g2s(st + lane * r.a_elems * es, x + (size_t)src_row * d1 + p.off1 + item.u0 * p.D1, abytes,
                     &bars[slot]);
    }
    bulk::copy_g2s(st + off_w<S>(r) + lane * ublock * es, W + (size_t)e * w_numel + p.woff + item.u0, wbytes,
                   &bars[slot]);
    if (r.y_elems)
      bulk::copy_g2s(st + off_y<S>(r, ublock) + lane * r.y_elems * es, Y + (size_t)e * d2, ybytes, &bars[slot]);
  }
  if (BWD && j == 0 && lane == 31)
    bulk::copy_g2s(st + off_x<S>(r, ublock), x + (size_t)n * d1 + p.off1 + item.u0 * p.D1, xbytes, &bars[slot]);
  __syncwarp();
  return true;
}

// Per-warp ring bookkeeping, warp-uniform (registers).
struct RingPos {
  int fetched;    // stages fetched so far
  int consumed;   // stages consumed
  uint32_t par;   // parity bit per slot of the phase to wait for next
  int abort;      // a wait gave up
};

// smem loads of staged operands (S storage, widened to T)
template <typename T, int N>
__device__ __forceinline__ void ldsv(const float* p, T (&v)[N]) {  // N consecutive, 16-byte aligned
#pragma unroll
  for (int i = 0; i < N / 4; ++i) {
    const float4 q = reinterpret_cast<const float4*>(p)[i];
    v[4 * i] = q.x;
    v[4 * i + 1] = q.y;
    v[4 * i + 2] = q.z;
    v[4 * i + 3] = q.w;
  }
}
template <typename T, int N>
__device__ __forceinline__ void ldsv(const double* p, T (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const double2 q = reinterpret_cast<const double2*>(p)[i];
    v[2 * i] = q.x;
    v[2 * i + 1] = q.y;
  }
}
template <typename T, int N>
__device__ __forceinline__ void ldsv(const __nv_bfloat16* p, T (&v)[N]) {  // 8-byte aligned
#pragma unroll
  for (int i = 0; i < N / 4; ++i) {
    const uint2 q = reinterpret_cast<const uint2*>(p)[i];
    v[4 * i] = T(__uint_as_float(q.x << 16));
    v[4 * i + 1] = T(__uint_as_float(q.x & 0xffff0000u));
    v[4 * i + 2] = T(__uint_as_float(q.y << 16));
    v[4 * i + 3] = T(__uint_as_float(q.y & 0xffff0000u));
  }
}
__device__ __forceinline__ float lds1(const float* p) { return *p; }
__device__ __forceinline__ double lds1(const double* p) { return *p; }
__device__ __forceinline__ float lds1(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<unsigned>(*reinterpret_cast<const unsigned short*>(p)) << 16);
}

// harmonics of edge e for one path: staged row (SH = false) or evaluated from
// the edge vector (SH = true)
template <int L2, typename T, bool SH, typename S>
__device__ __forceinline__ void stage_y(const S* ys, const T* rvec, int e, int off2, T (&yv)[2 * L2 + 1]) {
  if constexpr (SH) {
    const T* rr = rvec + 3 * (size_t)e;
    const T rx = __ldg(rr), ry = __ldg(rr + 1), rz = __ldg(rr + 2);
    const T n2 = rx * rx + ry * ry + rz * rz;
    const T inv = n2 > T(0) ? T(1) / sqrt(n2) : T(0);
    sh_block<L2, T, T>(rx * inv, ry * inv, rz * inv, yv);
  } else {
#pragma unroll
    for (int m = 0; m < 2 * L2 + 1; ++m) yv[m] = lds1(ys + off2 + m);
  }
}

// Shared prologue of both kernels: the CTA's node range, balanced by edges + rows.
__device__ __forceinline__ void cta_range(const int* rowptr, int N, int* s_range) {
  if (threadIdx.x == 0) {
    const long long tot = (long long)rowptr[N] + N;
    const long long t0 = tot * blockIdx.x / gridDim.x, t1 = tot * (blockIdx.x + 1) / gridDim.x;
    auto lb = [&](long long target) {
      int lo = 0, hi = N;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)rowptr[mid] + mid < target) lo = mid + 1; else hi = mid;
      }
      return lo;
    };
    s_range[0] = lb(t0);
    s_range[1] = (blockIdx.x + 1 == gridDim.x) ? N : lb(t1);
  }
}

// Wait for the stage at the consumer position; on give-up record the error
// (the stage's parity is left as it was, for the clean-up wait).
// The error word (host-mapped, 16 ints): [0] = 1 once a wait gave up; the first
// warp to give up records where: [1] block, [2] warp, [3] stage consumed,
// [4] stages fetched, [5] slot, [6] parity waited for, [7..8] the mbarrier's
// state word, [9..12] the stage descriptor.
__device__ __forceinline__ bool v4_wait(uint64_t* bars, RingPos& rp, int S, int* err, long long limit,
                                        const int4* desc) {
  const int slot = rp.consumed % S;
  const bool ok = bulk::mbar_wait(&bars[slot], (rp.par >> slot) & 1u, limit);
  if (ok) {
    rp.par ^= 1u << slot;
  } else {
    if ((threadIdx.x & 31) == 0) {
      if (atomicCAS(err + 1, 0, blockIdx.x + 1) == 0) {
        volatile int* e = err;
        const unsigned long long st = *reinterpret_cast<volatile unsigned long long*>(&bars[slot]);
        const int4 d = desc[slot];
        e[2] = threadIdx.x >> 5;
        e[3] = rp.consumed;
        e[4] = rp.fetched;
        e[5] = slot;
        e[6] = (rp.par >> slot) & 1u;
        e[7] = static_cast<int>(st & 0xffffffffu);
        e[8] = static_cast<int>(st >> 32);
        e[9] = d.x;
        e[10] = d.y;
        e[11] = d.z;
        e[12] = d.w;
      }
      *reinterpret_cast<volatile int*>(err) = 1;
    }
    rp.abort = 1;
  }
  return ok;
}

// After a wait gave up: bounded waits for every stage still in flight (at most
// S, each in its own slot), so no copy lands after the CTA has left.
constexpr long long kCleanupPolls = 1ll << 24;
__device__ __forceinline__ void v4_drain(uint64_t* bars, const RingPos& rp, int S) {
  for (int c = rp.consumed; c < rp.fetched; ++c)
    bulk::mbar_wait(&bars[c % S], (rp.par >> (c % S)) & 1u, kCleanupPolls);
}

// The stage at the consumer position has been read: release it and fetch ahead.
#define V4_RELEASE_AND_FETCH(BWD)                                                                              \
  do {                                                                                                         \
    __syncwarp();                                                                                              \
    bulk::fence_proxy_async();                                                                                 \
    ++rp.consumed;                                                                                             \
    while (!rp.abort && rp.fetched < rp.consumed + R.S &&                                                      \
           v4_fetch<BWD, T, S>(a.b.x, a.b.Y, a.b.W, a.b.gout, a.b.rowptr, a.b.col, a.b.t_dst, a.b.items,       \
                               a.b.paths, a.b.d1, a.b.d2, a.b.d_out, a.b.w_numel, R, a.ublock, nb, nr, ni,    \
                               item0, total, ctr, fs, ring, bars, desc, rp.fetched % R.S))                     \
      ++rp.fetched;                                                                                            \
  } while (0)

// ---------------------------------------------------------------------------
// forward: one (item, receiver) unit, its edges streamed stage by stage
// ---------------------------------------------------------------------------
template <typename T, int LPE, int L1, int L2, int L3, bool SH, typename S>
__device__ __forceinline__ void fwd4_unit(const Uvu4Args<T, S>& a, const Ring R, RingPos& rp, int nb, int nr,
                                       int ni, int item0, int total, int* ctr, FetchState* fs,
                                       unsigned char* ring, uint64_t* bars, int4* desc, int n, int deg,
                                       const PathDev& p, int u0) {
  using P = typename PairT<T>::P;
  constexpr int D1 = 2 * L1 + 1, D2 = 2 * L2 + 1, D3 = 2 * L3 + 1;
  constexpr int EPW = 32 / LPE;
  const int lane = threadIdx.x & 31, q = lane % LPE, g = lane / LPE;
  const int ub = a.ublock;
  const int u = u0 + 4 * q;
  const bool active = u < p.mul;
  P t01[D3], t23[D3];
#pragma unroll
  for (int k = 0; k < D3; ++k) t01[k] = t23[k] = P{T(0), T(0)};
  const int nst = max(1, (deg + R.SC - 1) / R.SC);
  const int ebase = SH ? __ldg(a.b.rowptr + n) : 0;  // CSR position of the receiver's first edge
  for (int st = 0; st < nst; ++st) {
    if (!v4_wait(bars, rp, R.S, a.err, a.wait_limit, desc)) return;
    const int slot = rp.consumed % R.S;
    const unsigned char* sb = ring + (size_t)slot * R.stage_bytes;
    const int4 d = desc[slot];
    const int cnt = d.z, e_first = ebase + d.y;
    const S* xs_base = reinterpret_cast<const S*>(sb);
    const S* ws_base = reinterpret_cast<const S*>(sb + off_w<S>(R));
    const S* ys_base = reinterpret_cast<const S*>(sb + off_y<S>(R, ub));
    if (active) {
      for (int j = g; j < cnt; j += 2 * EPW) {
        const int jb = j + EPW;
        const bool okb = jb < cnt;
        FwdEdge<T, D1, D2, D3> A, B;
        stage_y<L2, T, SH>(ys_base + j * R.y_elems, a.b.rvec, e_first + j, p.off2, A.yv);
        ldsv<T, 4 * D1>(xs_base + j * R.a_elems + 4 * q * D1, A.xs);
        ldsv<T, 4>(ws_base + j * ub + 4 * q, A.wv);
        const int jj = okb ? jb : j;
        stage_y<L2, T, SH>(ys_base + jj * R.y_elems, a.b.rvec, e_first + jj, p.off2, B.yv);
        ldsv<T, 4 * D1>(xs_base + jj * R.a_elems + 4 * q * D1, B.xs);
        ldsv<T, 4>(ws_base + jj * ub + 4 * q, B.wv);
        if (!okb) {
#pragma unroll
          for (int i = 0; i < 4; ++i) B.wv[i] = T(0);
        }
        fwd3_math<T, LPE, L1, L2, L3>(A, t01, t23);
        fwd3_math<T, LPE, L1, L2, L3>(B, t01, t23);
      }
    }
    V4_RELEASE_AND_FETCH(false);
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
    T* dst = a.b.out + (size_t)n * a.b.d_out + p.ooff + u * D3;
#pragma unroll
    for (int i = 0; i < 4 * D3; ++i) dst[i] = v[i];
  }
}

#define CGTP4_FWD_CASE(L1, L2, L3)                                                                           \
  case (L1)*16 + (L2)*4 + (L3):                                                                              \
    if constexpr ((L3) <= 3 && (L3) >= ((L1) > (L2) ? (L1) - (L2) : (L2) - (L1)) && (L3) <= (L1) + (L2))    \
      fwd4_unit<T, LPE, L1, L2, L3, SH, S>(a, R, rp, nb, nr, ni, item0, total, ctr, fs, ring, bars, desc, n, \
                                           d.w, p, item.u0);                                                 \
    break;

template <typename T, int LPE, typename S = T, bool SH = false>
__global__ void __launch_bounds__(kV4Threads, 1) uvu_forward4_kernel(const Uvu4Args<T, S> a) {
  extern __shared__ __align__(128) unsigned char v4_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Ring R = a.r;
  __shared__ int s_range[2];
  __shared__ int s_ctr;
  __shared__ FetchState s_fs[kV4Warps];
  cta_range(a.b.rowptr, a.b.N, s_range);
  unsigned char* ring = v4_smem + (size_t)warp * R.warp_bytes;
  int4* desc = reinterpret_cast<int4*>(ring + (size_t)R.S * R.stage_bytes);  // 16-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(desc + R.S);
  FetchState* fs = &s_fs[warp];
  if (tid == 0) s_ctr = 0;
  if (lane == 0) {
    for (int s = 0; s < R.S; ++s) bulk::mbar_init(&bars[s], 1);
    bulk::fence_mbar_init();
    *fs = FetchState{0, 0, 0, 0, 0, 1, 0, 0};
  }
  __syncthreads();
  const int nb = s_range[0], nr = s_range[1] - s_range[0];
  const int total = a.b.n_items * nr, ni = 0, item0 = 0;
  int* ctr = &s_ctr;
  RingPos rp{0, 0, 0u, 0};
  while (rp.fetched < R.S &&
         v4_fetch<false, T, S>(a.b.x, a.b.Y, a.b.W, a.b.gout, a.b.rowptr, a.b.col, a.b.t_dst, a.b.items,
                               a.b.paths, a.b.d1, a.b.d2, a.b.d_out, a.b.w_numel, R, a.ublock, nb, nr, ni, item0,
                               total, ctr, fs, ring, bars, desc, rp.fetched % R.S))
    ++rp.fetched;
  while (!rp.abort && rp.consumed < rp.fetched) {
    const int4 d = desc[rp.consumed % R.S];
    const int it = d.x / nr, n = nb + (d.x - it * nr);
    const Item item = a.b.items[it];
    const PathDev p = a.b.paths[item.path];
    switch (p.l1 * 16 + p.l2 * 4 + p.l3) {
      CGTP3_TRIPLES(CGTP4_FWD_CASE)
      default: rp.abort = 1; break;  // no code for this triple (not reachable for a qualified plan)
    }
  }
  if (rp.abort) v4_drain(bars, rp, R.S);  // copies still in flight land before the CTA leaves
}

// ---------------------------------------------------------------------------
// backward: one (sender, item) unit over the sender's out-edges, streamed
// ---------------------------------------------------------------------------
template <typename T, int LPE, int L1, int L2, int L3, bool SH, typename S>
__device__ __noinline__ void bwd4_unit(const Uvu4Args<T, S>& a, const Ring R, RingPos& rp, int nb, int nr,
                                       int ni, int item0, int total, int* ctr, FetchState* fs,
                                       unsigned char* ring, uint64_t* bars, int4* desc, int s, int deg,
                                       const PathDev& p, int u0) {
  using P = typename PairT<T>::P;
  constexpr int D1 = 2 * L1 + 1, D2 = 2 * L2 + 1, D3 = 2 * L3 + 1, NF = D1 * D3;
  constexpr int EPW = 32 / LPE;
  constexpr int HV = (D2 + LPE - 1) / LPE * LPE;
  const int lane = threadIdx.x & 31, q = lane % LPE, g = lane / LPE;
  const int ub = a.ublock;
  const int u = u0 + 4 * q;
  const bool active = u < p.mul;
  P x01[D1], x23[D1], gxa01[D1], gxa23[D1];
#pragma unroll
  for (int m = 0; m < D1; ++m) gxa01[m] = gxa23[m] = P{T(0), T(0)};
  const int nst = max(1, (deg + R.SC - 1) / R.SC);
  // the sender's slice comes with the unit's first stage
  if (!v4_wait(bars, rp, R.S, a.err, a.wait_limit, desc)) return;
  {
    T xs[4 * D1];
    const unsigned char* sb0 = ring + (size_t)(rp.consumed % R.S) * R.stage_bytes;
    if (active) {
      ldsv<T, 4 * D1>(reinterpret_cast<const S*>(sb0 + off_x<S>(R, ub)) + 4 * q * D1, xs);
    } else {
#pragma unroll
      for (int i = 0; i < 4 * D1; ++i) xs[i] = T(0);
    }
#pragma unroll
    for (int m = 0; m < D1; ++m) {
      x01[m] = P{xs[m], xs[D1 + m]};
      x23[m] = P{xs[2 * D1 + m], xs[3 * D1 + m]};
    }
  }
  for (int st = 0; st < nst; ++st) {
    if (st > 0 && !v4_wait(bars, rp, R.S, a.err, a.wait_limit, desc)) return;
    const int slot = rp.consumed % R.S;
    const unsigned char* sb = ring + (size_t)slot * R.stage_bytes;
    const int cnt = desc[slot].z;
    const S* gs_base = reinterpret_cast<const S*>(sb);
    const S* ws_base = reinterpret_cast<const S*>(sb + off_w<S>(R));
    const S* ys_base = reinterpret_cast<const S*>(sb + off_y<S>(R, ub));
    const int* eids = reinterpret_cast<const int*>(sb + off_e<S>(R, ub));
    // uniform trip count over the stage (the gY reduction shuffles across the path's lanes)
    for (int j0 = 0; j0 < cnt; j0 += EPW) {
      const int j = j0 + g;
      const bool valid = active && j < cnt;
      int e = 0;
      T yv[D2], gs[4 * D3], wv[4];
      if (valid) {
        e = eids[j];
        stage_y<L2, T, SH>(ys_base + j * R.y_elems, a.b.rvec, e, p.off2, yv);
        ldsv<T, 4>(ws_base + j * ub + 4 * q, wv);
        ldsv<T, 4 * D3>(gs_base + j * R.a_elems + 4 * q * D3, gs);
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
          T* gp = a.b.gW + (size_t)e * a.b.w_numel + p.woff + u;
          if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<float4*>(gp) = make_float4(gw[0], gw[1], gw[2], gw[3]);
          } else {
            reinterpret_cast<double2*>(gp)[0] = make_double2(gw[0], gw[1]);
            reinterpret_cast<double2*>(gp)[1] = make_double2(gw[2], gw[3]);
          }
        }
      }
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
          const int sl = q * (HV / LPE) + k;
          if (sl < D2) gY_add(a.b.gY + (size_t)e * a.b.d2 + p.off2 + sl, h[k]);
        }
      }
    }
    V4_RELEASE_AND_FETCH(true);
  }
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
    T* dst = a.b.gx + (size_t)s * a.b.d1 + p.off1 + u * D1;
#pragma unroll
    for (int i = 0; i < 4 * D1; ++i) gY_add(dst + i, v[i]);
  }
}

#define CGTP4_BWD_CASE(L1, L2, L3)                                                                           \
  case (L1)*16 + (L2)*4 + (L3):                                                                              \
    if constexpr ((L3) <= 3 && (L3) >= ((L1) > (L2) ? (L1) - (L2) : (L2) - (L1)) && (L3) <= (L1) + (L2))    \
      bwd4_unit<T, LPE, L1, L2, L3, SH, S>(a, R, rp, nb, nr, ni, item0, total, ctr, fs, ring, bars, desc, s, \
                                           d.w, p, item.u0);                                                 \
    break;

template <typename T, int LPE, typename S = T, bool SH = false>
__global__ void __launch_bounds__(kV4Threads, 1) uvu_backward4_kernel(const Uvu4Args<T, S> a) {
  extern __shared__ __align__(128) unsigned char v4_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Ring R = a.r;
  __shared__ int s_range[2];
  __shared__ int s_next[2];
  __shared__ FetchState s_fs[kV4Warps];
  cta_range(a.b.rowptr, a.b.N, s_range);
  __syncthreads();
  const int sb = s_range[0], se = s_range[1], nr = se - sb, nb = sb;
  // clear gx and gY of the CTA's senders (and their out-edges) before the first phase
  for (int s = sb + warp; s < se; s += kV4Warps) {
    for (int i = lane; i < a.b.d1; i += 32) a.b.gx[(size_t)s * a.b.d1 + i] = T(0);
    const int tb = a.b.rowptr[s], te = a.b.rowptr[s + 1];
    for (int i = lane; i < (te - tb) * a.b.d2; i += 32) {
      const int j = i / a.b.d2, c = i - j * a.b.d2;
      a.b.gY[(size_t)a.b.col[tb + j] * a.b.d2 + c] = T(0);
    }
  }
  unsigned char* ring = v4_smem + (size_t)warp * R.warp_bytes;
  int4* desc = reinterpret_cast<int4*>(ring + (size_t)R.S * R.stage_bytes);  // 16-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(desc + R.S);
  FetchState* fs = &s_fs[warp];
  if (lane == 0) {
    for (int s = 0; s < R.S; ++s) bulk::mbar_init(&bars[s], 1);
    bulk::fence_mbar_init();
  }
  RingPos rp{0, 0, 0u, 0};
  int failed = 0;
  // Items come in phases whose items share no in1 block and no in2 block, so
  // within a phase every gx / gY slice has one writer; a block barrier
  // separates the phases, and every gx / gY element receives its contributions
  // in phase order (deterministic).
  for (int ph = 0; ph < a.b.n_phases; ++ph) {
    const int item0 = a.b.phase_begin[ph], ni = a.b.phase_begin[ph + 1] - item0;
    if (tid == 0) s_next[ph & 1] = 0;
    if (lane == 0) *fs = FetchState{0, 0, 0, 0, 0, 1, 0, 0};
    __syncthreads();
    const int total = ni * nr;
    int* ctr = &s_next[ph & 1];
    if (!failed) {
      while (rp.fetched < rp.consumed + R.S &&
             v4_fetch<true, T, S>(a.b.x, a.b.Y, a.b.W, a.b.gout, a.b.rowptr, a.b.col, a.b.t_dst, a.b.items,
                                  a.b.paths, a.b.d1, a.b.d2, a.b.d_out, a.b.w_numel, R, a.ublock, nb, nr, ni,
                                  item0, total, ctr, fs, ring, bars, desc, rp.fetched % R.S))
        ++rp.fetched;
      while (!rp.abort && rp.consumed < rp.fetched) {
        const int4 d = desc[rp.consumed % R.S];
        const int sl = d.x / ni;
        const int s = nb + sl;
        const Item item = a.b.items[item0 + (d.x - sl * ni)];
        const PathDev p = a.b.paths[item.path];
        switch (p.l1 * 16 + p.l2 * 4 + p.l3) {
          CGTP3_TRIPLES(CGTP4_BWD_CASE)
          default: rp.abort = 1; break;  // no code for this triple (not reachable for a qualified plan)
        }
      }
      if (rp.abort) {  // let the copies still in flight land, then only take part in the barriers
        v4_drain(bars, rp, R.S);
        failed = 1;
      }
    }
    __syncthreads();
  }
}

}  // namespace uvu4_detail
}  // namespace cgtp
