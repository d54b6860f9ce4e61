// uvw.cu -- fully connected (uvw) CG tensor-product convolution with radial
// weights, streamed through bounded node state.
//
// "Sobek: Streaming Equivariant Tensor Product Convolutions", Abstract: the
// edge-specific weights, messages and adjoints of the conventional schedule are
// artefacts; reassociating radial projection, spherical-harmonic coupling and
// aggregation lets edge-local products be consumed into bounded receiver-side
// state, through forward and backward, keeping fully connected multiplicity
// mixing.  With W_e[path,u,w] = sum_k R[e,k] M[k,path,u,w] (never formed):
//
// forward, per receiver n (edge stage: a warp per (receiver, path, 32 channels),
// the sums in registers, written once per node):
//   S[n][k,path,u,m3] = sum_{e in row n} R[e,k] sum_m1 cy_e[path][m1,m3] x[src][u,m1]
// then a node GEMM over a chunk of receivers (M shared by all nodes):
//   out[n][i_out][w,m3] = sum_{path -> i_out} sum_{k,u} M[k,path,u,w] S[n][k,path,u,m3]
//
// backward, sender-owned over the transpose (no scatter; gR and gY take one
// atomic addition per element between block barriers, in a fixed order):
//   A[s][k,path,w,m1]  = sum_u x[s][u,m1] M[k,path,u,w]                  (node GEMM)
//   per out-edge e = (s -> d):  p_e[path,w,m1] = sum_m3 cy_e[m1,m3] g[d][w,m3]
//     H[s][k,path,w,m1] += R[e,k] p_e
//     gR[e,k]  = sum A[s][k] . p_e
//     gY[e][m2] = sum_path sum C[m1,m2,m3] (sum_w (sum_k R[e,k] A[s][k,path,w,m1]) g[d][w,m3])
//   gx[s][u,m1] = sum_{k,path,w} M[k,path,u,w] H[s][k,path,w,m1]             (node GEMM)
//   gM[k,path,u,w] += sum_{s,m1} x[s][u,m1] H[s][k,path,w,m1]   (per chunk, chunks in order)
//
// Node state lives in a scratch buffer owned by the plan and sized by a fixed
// node chunk (not by the graph): the working set is bounded whatever E is.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "internal.h"
#include "uvu3_impl.cuh"
#include "sh.cuh"

namespace cgtp {
namespace uvw_detail {

constexpr int kChunkPerSm = 128;    // default nodes per streamed chunk, per SM (cgtp_plan_set_node_chunk)
constexpr int kKB = 8;              // radial functions held in registers (K <= 8)
constexpr int kGmSplits = 16;       // split-K factor of the gM reduction over nodes

struct UvwPath {
  int l1, l2, l3, D1, D2, D3, mul1, mul_out;
  int off1, off2, ooff, woff;
  // Node state, one radial slice [k] of a node: forward S grouped by output
  // block o as [m3][paths into o: u], backward A / H grouped by in1 block as
  // [m1][paths from that block: w] (channels innermost: the edge stages' lanes
  // and the node GEMMs' rows read and write contiguous runs)
  int soff;      // forward: offset of this path's u = 0, m3 = 0 inside the slice
  int aoff;      // backward: offset of this path's w = 0, m1 = 0 inside the slice
  int sstr;      // forward: stride of m3 (the channels of every path into the block)
  int astr;      // backward: stride of m1 (the channels of every path from the in1 block)
  int i1, io;
};

struct GemmSeg {
  long long a_off, b_off;
  int K;        // <0: use the launch's node count
  int a_k, b_k;
  int b_j;      // column stride of B (may differ between the segments of a problem)
};

struct GemmProb {
  int a_base, b_base, c_base;  // which launch pointer
  int Nn;                      // rows = Nn * D (Nn < 0: the launch's node count)
  int D, J;
  long long a_off, a_n, a_m;
  int b_j, c_j;
  long long c_off, c_n, c_m;
  int beta;                    // 0 overwrite, 1 accumulate
  int seg0, seg1;
  // tile loading: 0 = a warp's lanes walk K (32 consecutive k of one row / column);
  // 1 = they walk the rows of A (cols of B) at fixed k -- for operands whose K stride is large
  unsigned char a_mode, b_mode;
  // 16-byte copies possible: the operand is contiguous along K (k stride 1) with 4-aligned row strides
  unsigned char a_vec, b_vec;
};

struct UvwState {
  std::vector<UvwPath> paths_h;
  UvwPath* paths = nullptr;
  int n_paths = 0;
  int K = 0;
  int s_slice = 0, a_slice = 0;  // elements of one radial slice of the node state
  int s_node = 0, a_node = 0;    // K * slice
  int chunk_nodes = 0;
  float* scratch = nullptr;      // [2][chunk_nodes][s_node]
  float* gm_part = nullptr;      // [kGmSplits][K][w_numel] split-K partials of gM
  Item* bwd3_items = nullptr;    // (path, 32-block of mul_out) in path order
  Item* fwd3_items = nullptr;    // (path, 32-block of mul1) in path order
  int fwd3_n_items = 0;
  int* err_dev = nullptr;        // set by a tensor-core wait that gave up
  int* err_host = nullptr;       // pinned copy, refreshed after every call (sticky error)
  int bwd3_n_items = 0;
  size_t scratch_elems = 0;
  // GEMM descriptor tables (device) per use
  GemmProb* fwd_probs = nullptr;  int fwd_np = 0;  GemmSeg* fwd_segs = nullptr;
  GemmProb* pre_probs = nullptr;  int pre_np = 0;  GemmSeg* pre_segs = nullptr;
  GemmProb* gx_probs = nullptr;   int gx_np = 0;   GemmSeg* gx_segs = nullptr;
  GemmProb* gm_probs = nullptr;   int gm_np = 0;   GemmSeg* gm_segs = nullptr;
  void* tables = nullptr;
};

// ---------------------------------------------------------------------------
// grouped GEMM on the tensor cores (tcgen05, kind::tf32, 3xTF32):
//   C[(n,m), j] (+)= sum_seg sum_k A[(n,m), k] B[k, j]
// One CTA (4 warps) computes a 128-row x 64-column tile.  Per K step of 32:
// every thread loads its share of the A and B tiles through the generic
// strided addressing of the descriptors, splits each value into a TF32 high
// part and a TF32 residual, and writes both into shared memory in the K-major
// 128-byte-swizzled layout; one thread issues hi*hi + hi*lo + lo*hi as
// tcgen05.mma into a TMEM accumulator (128 lanes x 64 columns) and commits to an
// mbarrier (waited with a bounded spin that records an error instead of
// hanging).  The epilogue reads TMEM with tcgen05.ld and scatters through the
// descriptor's (n, m, j) strides.  The three products give FP32-level accuracy.
// ---------------------------------------------------------------------------
constexpr int kTM = 128, kTN = 64, kTK = 32;
constexpr int kATile = kTM * kTK * 4, kBTile = kTN * kTK * 4;
constexpr int kTcSmem = 2 * (2 * kATile + 2 * kBTile) + 1024 + 64;  // two stages
// dynamic shared memory of a launch over np problems: the above plus the tile prefix
inline size_t gemm_smem(int np) { return kTcSmem + sizeof(int) * size_t(np + 1); }
constexpr long long kTcCleanupPolls = 1ll << 24;                     // bounded clean-up wait

struct GemmLaunch {
  const float* ptr[6];
  int nodes;  // node count of this launch (chunk)
  int nprob;
  const GemmProb* probs;
  const GemmSeg* segs;
  // split-K over node-sized segments (K < 0): blockIdx.y takes node slice
  // [y*ceil(nodes/splits), ...) and writes its partial to C + y*c_split_stride
  int splits;
  long long c_split_stride;
  int* err;  // set when a tensor-core wait gives up
  long long wait_limit;  // polls before a tensor-core wait gives up
  int tiles;             // tiles of the launch (a persistent CTA takes every gridDim.x-th)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// byte offset of element (row r, k) in a K-major tile of 128-byte rows, 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int k) {
  const uint32_t chunk = (uint32_t)(k >> 2) ^ (uint32_t)(r & 7);
  return (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u + chunk * 16u + (uint32_t)(k & 3) * 4u;
}
// shared-memory matrix descriptor: start >> 4, leading offset 16 B, stride 1024 B
// (8 rows x 128 B), descriptor version 1, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ float tf32_round(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
__device__ __forceinline__ void mma_tf32(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
               ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// row r of a problem -> (node n, component m) for rows of D components: the block
// dimensions 2l+1 (l <= 3) as compile-time divisors (a multiply and a shift)
__device__ __forceinline__ int div_rows(int r, int D) {
  switch (D) {
    case 1: return r;
    case 3: return r / 3;
    case 5: return r / 5;
    case 7: return r / 7;
    default: return r / D;
  }
}

// bounded wait on an mbarrier phase (false: gave up)
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, long long limit) {
  for (long long it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    if (done) return true;
  }
  return false;
}

// Two shared-memory stages: while the tensor core runs the MMAs of K step i
// (stage i % 2, committed to that stage's mbarrier), the threads load and split
// step i + 1 into the other stage; a stage is overwritten only after the commit
// of the MMAs that read it (step i - 1) has arrived.
constexpr int kTcWarps = 8;  // loaders; warp w % 4 reads TMEM lanes 32 (w % 4).., columns half w / 4

__global__ void __launch_bounds__(kTcWarps * 32, 2) grouped_gemm_tc_kernel(const GemmLaunch L) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  constexpr int kStage = 2 * kATile + 2 * kBTile;
  uint64_t* mbar = (uint64_t*)(sm + 2 * kStage);         // one per stage
  uint32_t* tmem_holder = (uint32_t*)(sm + 2 * kStage + 16);
  int* t0 = reinterpret_cast<int*>(sm + 2 * kStage + 64);  // [nprob + 1]: first tile of each problem
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < L.nprob; i += kTcWarps * 32) {
    const GemmProb& Q = L.probs[i];
    const int rows = (Q.Nn < 0 ? L.nodes : Q.Nn) * Q.D;
    t0[i + 1] = ((rows + kTM - 1) / kTM) * ((Q.J + kTN - 1) / kTN);
  }
  __syncthreads();
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar[1])));
    asm volatile("fence.mbarrier_init.release.cluster;");
    t0[0] = 0;
    for (int i = 0; i < L.nprob; ++i) t0[i + 1] += t0[i];
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)), "r"(64));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = *tmem_holder;
  const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kTN >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);
  uint32_t phase = 0;   // bit s: parity of stage s's next commit
  uint32_t pend = 0;    // bit s: stage s has a commit not yet waited for
  int issued = 0;       // K steps whose MMAs were committed (over all tiles of this CTA): picks the stage
  bool ok = true;
  const int split = blockIdx.y;
  const int slice = (L.nodes + L.splits - 1) / L.splits;
  // persistent: this CTA takes tiles blockIdx.x, + gridDim.x, ... of the launch
  for (int tile_g = blockIdx.x; tile_g < L.tiles && ok; tile_g += gridDim.x) {
  // locate the tile's problem (uniform over the CTA): binary search of the tile prefix
  if (tile_g >= t0[L.nprob]) break;
  int pi = 0;
  {
    int hi = L.nprob - 1;
    while (pi < hi) {  // last problem whose first tile is <= tile_g
      const int mid = (pi + hi + 1) >> 1;
      if (t0[mid] <= tile_g) pi = mid; else hi = mid - 1;
    }
  }
  const GemmProb P = L.probs[pi];
  const int ntc = (P.J + kTN - 1) / kTN, rt = (tile_g - t0[pi]) / ntc, ct = tile_g - t0[pi] - rt * ntc;
  const int rows = (P.Nn < 0 ? L.nodes : P.Nn) * P.D;
  const float* A = L.ptr[P.a_base];
  const float* B = L.ptr[P.b_base];
  float* C = const_cast<float*>(L.ptr[P.c_base]);
  if (L.splits > 1) C += split * L.c_split_stride;
  const int r0 = rt * kTM, c0 = ct * kTN;
  // this thread stages column k = lane of rows warp + 8 t (A) and of columns warp + 8 t (B)
  constexpr int kAR = kTM / kTcWarps, kBC = kTN / kTcWarps;
  // value t of this thread: mode 0 row warp + 8 t, k = lane; mode 1 row (t % 4) 32 + lane,
  // k = warp + 8 (t / 4) for A (B: column (t % 2) 32 + lane, k = warp + 8 (t / 2))
  const bool amode = P.a_mode != 0, bmode = P.b_mode != 0;
  int aoff[kAR];
#pragma unroll
  for (int t = 0; t < kAR; ++t) {
    const int rl = amode ? (t & 3) * 32 + lane : warp + kTcWarps * t;
    const int r = r0 + rl;
    const int n = r < rows ? div_rows(r, P.D) : 0, m = r < rows ? r - n * P.D : 0;
    aoff[t] = r < rows ? (int)(n * P.a_n + m * P.a_m) : -1;
  }
  bool first = true;
  // K steps of all segments as one sequence; the loads of step i + 1 are issued
  // before step i is split and stored, so they are in flight during that work
  struct Step {
    int sg, k0, ke, a_k, b_k, b_j;
    const float* Ab;
    const float* Bb;
  };
  auto seg_from = [&](Step& st, int sg) {  // first non-empty segment at or after sg
    for (; sg < P.seg1; ++sg) {
      const GemmSeg S = L.segs[sg];
      int kb = 0, ke = S.K < 0 ? L.nodes : S.K;
      if (S.K < 0 && L.splits > 1) {
        kb = min(L.nodes, split * slice);
        ke = min(L.nodes, kb + slice);
      }
      if (kb < ke) {
        st = Step{sg, kb, ke, S.a_k, S.b_k, S.b_j, A + P.a_off + S.a_off, B + S.b_off};
        return true;
      }
    }
    return false;
  };
  auto load_step = [&](const Step& st, float (&av)[kAR], float (&bv)[kBC]) {
#pragma unroll
    for (int t = 0; t < kAR; ++t) {
      const int k = st.k0 + (amode ? warp + kTcWarps * (t >> 2) : lane);
      av[t] = (k < st.ke && aoff[t] >= 0) ? __ldg(st.Ab + aoff[t] + (long long)k * st.a_k) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < kBC; ++t) {
      const int k = st.k0 + (bmode ? warp + kTcWarps * (t >> 1) : lane);
      const int c = c0 + (bmode ? (t & 1) * 32 + lane : warp + kTcWarps * t);
      bv[t] = (k < st.ke && c < P.J) ? __ldg(st.Bb + (long long)k * st.b_k + (long long)c * st.b_j) : 0.f;
    }
  };
  Step cur;
  bool have = seg_from(cur, P.seg0);
  float av[kAR], bv[kBC];
  if (have) load_step(cur, av, bv);
  while (have && ok) {
    Step nxt = cur;
    nxt.k0 += kTK;
    const bool have_next = nxt.k0 < nxt.ke || seg_from(nxt, cur.sg + 1);
    float an[kAR], bn[kBC];
    if (have_next) load_step(nxt, an, bn);
    {
      const int st = issued & 1;
      unsigned char* a_hi = sm + st * kStage;
      unsigned char* a_lo = a_hi + kATile;
      unsigned char* b_hi = a_hi + 2 * kATile;
      unsigned char* b_lo = b_hi + kBTile;
      if ((pend >> st) & 1u) {  // the MMAs of step issued - 2 read this stage
        const bool done = tc_wait(&mbar[st], (phase >> st) & 1u, L.wait_limit);
        asm volatile("tcgen05.fence::after_thread_sync;");
        if (__syncthreads_or(!done)) {
          ok = false;
          break;
        }
        phase ^= 1u << st;
        pend &= ~(1u << st);
      }
#pragma unroll
      for (int t = 0; t < kAR; ++t) {
        const int rr = amode ? (t & 3) * 32 + lane : warp + kTcWarps * t;
        const int kk = amode ? warp + kTcWarps * (t >> 2) : lane;
        const float hi = tf32_round(av[t]);
        *(float*)(a_hi + sw128(rr, kk)) = hi;
        *(float*)(a_lo + sw128(rr, kk)) = tf32_round(av[t] - hi);
      }
#pragma unroll
      for (int t = 0; t < kBC; ++t) {
        const int jj = bmode ? (t & 1) * 32 + lane : warp + kTcWarps * t;
        const int kk = bmode ? warp + kTcWarps * (t >> 1) : lane;
        const float hi = tf32_round(bv[t]);
        *(float*)(b_hi + sw128(jj, kk)) = hi;
        *(float*)(b_lo + sw128(jj, kk)) = tf32_round(bv[t] - hi);
      }
      asm volatile("fence.proxy.async.shared::cta;");
      __syncthreads();
      if (tid == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t ah = smem_u32(a_hi), al = smem_u32(a_lo), bh = smem_u32(b_hi), bl = smem_u32(b_lo);
#pragma unroll
        for (int ks = 0; ks < kTK / 8; ++ks) {
          const uint32_t off = ks * 32;  // 8 TF32 values along K
          mma_tf32(tmem, sdesc(ah + off), sdesc(bh + off), idesc, first ? 0u : 1u);
          mma_tf32(tmem, sdesc(ah + off), sdesc(bl + off), idesc, 1u);
          mma_tf32(tmem, sdesc(al + off), sdesc(bh + off), idesc, 1u);
          first = false;
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&mbar[st])));
      }
      first = false;
      pend |= 1u << st;
      ++issued;
    }
#pragma unroll
    for (int t = 0; t < kAR; ++t) av[t] = an[t];
#pragma unroll
    for (int t = 0; t < kBC; ++t) bv[t] = bn[t];
    cur = nxt;
    have = have_next;
  }
  // the tile's last commits (at most two outstanding, one per stage) before TMEM is read
  if (ok) {
    for (int st = 0; st < 2; ++st) {
      if (!((pend >> st) & 1u)) continue;
      const bool done = tc_wait(&mbar[st], (phase >> st) & 1u, L.wait_limit);
      if (__syncthreads_or(!done)) {
        ok = false;
        break;
      }
      phase ^= 1u << st;
      pend &= ~(1u << st);
    }
    asm volatile("tcgen05.fence::after_thread_sync;");
  }
  if (!ok) break;
  // epilogue: warp w owns TMEM lanes (tile rows) 32 (w % 4) .. + 31 and the column half w / 4
  const int quarter = warp & 3, chalf = warp >> 2;
  const int r = r0 + 32 * quarter + lane;
  const bool rok = r < rows;
  const int n = rok ? div_rows(r, P.D) : 0, m = rok ? r - n * P.D : 0;
  float* crow = C + P.c_off + n * P.c_n + m * P.c_m;
  const bool vec = P.c_j == 1 && ((reinterpret_cast<uintptr_t>(crow + c0)) & 15u) == 0;
  const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16);
#pragma unroll
  for (int cc = chalf * (kTN / 2); cc < (chalf + 1) * (kTN / 2); cc += 16) {
    uint32_t v[16];
    if (!first) {
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                   : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                     "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                   : "r"(taddr + cc));
      asm volatile("tcgen05.wait::ld.sync.aligned;");
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0u;  // empty K range: the product is zero
    }
    if (vec) {  // contiguous 16-byte aligned columns: four at a time
#pragma unroll
      for (int j = 0; j < 16; j += 4) {
        const int c = c0 + cc + j;
        if (rok && c + 3 < P.J) {
          float4* dst = reinterpret_cast<float4*>(crow + c);
          float4 val = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                   __uint_as_float(v[j + 3]));
          if (P.beta) {
            const float4 o = *dst;
            val.x += o.x;
            val.y += o.y;
            val.z += o.z;
            val.w += o.w;
          }
          *dst = val;
        } else {
          for (int q = 0; q < 4; ++q)
            if (rok && c + q < P.J) {
              float* d = crow + c + q;
              *d = P.beta ? *d + __uint_as_float(v[j + q]) : __uint_as_float(v[j + q]);
            }
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + cc + j;
        if (rok && c < P.J) {
          float* dst = crow + (long long)c * P.c_j;
          const float val = __uint_as_float(v[j]);
          *dst = P.beta ? *dst + val : val;
        }
      }
    }
  }
  // every thread's TMEM reads are done before the next tile's MMAs overwrite the accumulator
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  }  // tiles
  if (!ok) {  // a tensor-core wait gave up: record, let the MMAs in flight finish (bounded), clean up
    if (tid == 0) atomicOr(L.err, 1);
    for (int st = 0; st < 2; ++st)
      if ((pend >> st) & 1u) tc_wait(&mbar[st], (phase >> st) & 1u, kTcCleanupPolls);
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(64));
}

__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cpa_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// gM (+)= sum over the split-K partials, in split order (deterministic)
__global__ void splitk_reduce_kernel(float* __restrict__ gM, const float* __restrict__ part, int splits,
                                     long long n, int accumulate) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    float v = accumulate ? gM[i] : 0.f;
    for (int s = 0; s < splits; ++s) v += part[s * n + i];
    gM[i] = v;
  }
}

// ---------------------------------------------------------------------------
// edge stages
// ---------------------------------------------------------------------------
// Gaussian radial basis of the edge length d: R_k = exp(-gamma (d - lo - k step)^2)
struct Rbf {
  float lo, step, gamma;
};
__device__ __forceinline__ float rbf_k(const Rbf& b, float d, int k) {
  const float t = d - (b.lo + k * b.step);
  return expf(-b.gamma * t * t);
}

// ---------------------------------------------------------------------------
// backward edge stage (sender-owned)
// ---------------------------------------------------------------------------
// Sum eight values over the 32 lanes; lane l ends with the total of value
// (l >> 2) & 7.
__device__ __forceinline__ float reduce8(float (&v)[8], int lane) {
#pragma unroll
  for (int o = 16, n = 8; o >= 4; o >>= 1, n >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i < n / 2) {
        const float send = up ? v[i] : v[i + n / 2];
        const float keep = up ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  float r = v[0];
  r += __shfl_xor_sync(0xffffffffu, r, 2);
  r += __shfl_xor_sync(0xffffffffu, r, 1);
  return r;
}

// ---------------------------------------------------------------------------
// backward edge stage, warp-autonomous and path-major: the warps of a CTA take
// (sender, item) units of the CTA's edge-balanced sender range from a shared
// counter; a unit is (sender, path, 32 output channels w), lanes <-> w.
// A[s][k][path][w][m1] and the accumulating H[s][k][path][w][m1] of the unit
// stay in registers; the CG nonzeros of (l1, l2, l3) are compiled in, so
//   p_e[m1]  = sum_{m2,m3} C Y[e][m2] g[d][w][m3]
//   h[m2]    = sum_{m1,m3} C ar[m1] g[d][w][m3],  ar[m1] = sum_k R[e,k] A[k][m1]
// and only gR (K values) and h (2l2+1 values) cross the 32 lanes; they are added
// with one atomic per element per item, items separated by block barriers, so
// every element's additions come in item order (deterministic).
// ---------------------------------------------------------------------------
struct Bwd3Args {
  const float* Y;      // edge-vector mode: the vectors [E,3]
  const float* R;
  Rbf rbf;
  const float* g;
  const float* Astate;  // [chunk][K][s_slice]
  float* Hstate;        // [chunk][K][s_slice]
  float* gY;
  float* gR;
  const int* t_rowptr;
  const int* t_eid;
  const int* t_dst;
  int n0, n1;
  int d2, d_out, K, s_node, s_slice;
  const UvwPath* paths;
  const Item* items;    // (path, w0), path order
  int n_items;
  int idx_cap;          // ints of dynamic shared memory for the CTA's transpose slice
};

// Per-warp ring of staged edge operands: stage j holds, for one edge of the
// unit, the 32 * D3 output-gradient values of the unit's w range, then (at
// kRingY) the path's harmonics (or the edge vector) and (at kRingR) the K
// radial values.  Copies are 4-byte cp.async issued kRingDepth - 1 edges ahead
// of the edge being computed, so the warp keeps that many edges' gathers in
// flight without holding them in registers.
constexpr int kRingDepth = 4;
constexpr int kRingY = 32 * 7;               // 32 lanes x D3 (l3 <= 3)
constexpr int kRingR = kRingY + 8;
constexpr int kRingStage = kRingR + kKB;     // floats per stage
constexpr int kRingWarp = kRingDepth * kRingStage;

__device__ __forceinline__ void cp_async4(float* s, const float* g) {
  const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(s));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(sa), "l"(g) : "memory");
}

template <int L1, int L2, int L3, bool SH>
__device__ __noinline__ void uvw_bwd3_unit(const float* __restrict__ Yp, const float* __restrict__ Rp, Rbf rbf,
                                           const float* __restrict__ gp_, const float* __restrict__ Astate,
                                           float* __restrict__ Hstate, float* __restrict__ gY,
                                           float* __restrict__ gR, const int* __restrict__ t_eid,
                                           const int* __restrict__ t_dst, int tb, int te, size_t node_off,
                                           int d2, int d_out, int K, int s_slice, int off2, int ooff,
                                           int aoff, int astr, int mul_out, int w0, int lane, float* ring) {
  constexpr int D1 = 2 * L1 + 1, D2 = 2 * L2 + 1, D3 = 2 * L3 + 1;
  constexpr int NY = SH ? 3 : D2;
  const int w = w0 + lane;
  const bool active = w < mul_out;
  const int n_g = min(32, mul_out - w0) * D3;  // in-bounds gradient values of the unit's w range
  float A[kKB][D1], H[kKB][D1];
  const float* As = Astate + node_off + aoff + w;
#pragma unroll
  for (int k = 0; k < kKB; ++k)
#pragma unroll
    for (int m = 0; m < D1; ++m) {
      A[k][m] = (active && k < K) ? __ldg(As + k * s_slice + m * astr) : 0.f;
      H[k][m] = 0.f;
    }
  // stage edge t into ring slot `slot`; one commit group per call (empty past te)
  auto issue = [&](int t, int slot) {
    if (t < te) {
      const int e = t_eid[t], d = t_dst[t];
      float* st = ring + slot * kRingStage;
      const float* gsrc = gp_ + (size_t)d * d_out + ooff + w0 * D3;
#pragma unroll
      for (int j = 0; j < D3; ++j)
        if (j * 32 + lane < n_g) cp_async4(st + j * 32 + lane, gsrc + j * 32 + lane);
      if (lane < NY)
        cp_async4(st + kRingY + lane, SH ? Yp + 3 * (size_t)e + lane : Yp + (size_t)e * d2 + off2 + lane);
      else if (!SH && lane >= 8 && lane < 8 + K)
        cp_async4(st + kRingR + lane - 8, Rp + (size_t)e * K + lane - 8);
    }
    cpa_commit();
  };
#pragma unroll
  for (int i = 0; i < kRingDepth - 1; ++i) issue(tb + i, i);
  int slot = 0;
  for (int t = tb; t < te; ++t) {
    // edge t's group is complete once at most kRingDepth - 2 younger groups are pending;
    // the warp barrier also ends every lane's reads of the slot refilled below
    cpa_wait<kRingDepth - 2>();
    __syncwarp();
    issue(t + kRingDepth - 1, slot == 0 ? kRingDepth - 1 : slot - 1);
    const float* st = ring + slot * kRingStage;
    slot = slot + 1 == kRingDepth ? 0 : slot + 1;
    const int e = t_eid[t];
    float yv[D2], r[kKB], gv[D3];
    if constexpr (SH) {  // the edge vector: harmonics and radial basis evaluated here
      const float rx = st[kRingY], ry = st[kRingY + 1], rz = st[kRingY + 2];
      const float dd = sqrtf(rx * rx + ry * ry + rz * rz), inv = dd > 0.f ? 1.f / dd : 0.f;
      sh_block<L2, float, float>(rx * inv, ry * inv, rz * inv, yv);
#pragma unroll
      for (int k = 0; k < kKB; ++k) r[k] = (k < K) ? rbf_k(rbf, dd, k) : 0.f;
    } else {
#pragma unroll
      for (int m = 0; m < D2; ++m) yv[m] = st[kRingY + m];
#pragma unroll
      for (int k = 0; k < kKB; ++k) r[k] = (k < K) ? st[kRingR + k] : 0.f;
    }
#pragma unroll
    for (int m = 0; m < D3; ++m) gv[m] = active ? st[lane * D3 + m] : 0.f;
    float pe[D1];
#pragma unroll
    for (int m = 0; m < D1; ++m) pe[m] = 0.f;
    CGB<L1, L2, L3>::each([&](int m1, int m2, int m3, double c) { pe[m1] += float(c) * yv[m2] * gv[m3]; });
    float gr[kKB], ar[D1];
#pragma unroll
    for (int m = 0; m < D1; ++m) ar[m] = 0.f;
#pragma unroll
    for (int k = 0; k < kKB; ++k) {
      float dot = 0.f;
#pragma unroll
      for (int m = 0; m < D1; ++m) {
        H[k][m] += r[k] * pe[m];
        dot += A[k][m] * pe[m];
        ar[m] += r[k] * A[k][m];
      }
      gr[k] = dot;
    }
    float h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = 0.f;
    CGB<L1, L2, L3>::each([&](int m1, int m2, int m3, double c) { h[m2] += float(c) * ar[m1] * gv[m3]; });
    const float grt = reduce8(gr, lane);   // lane holds the total of index (lane >> 2) & 7
    const float ht = reduce8(h, lane);
    const int idx = (lane >> 2) & 7;
    // one contribution per (edge, item); items are separated by block barriers, so
    // every element's additions come in item order (deterministic) and nothing is read back
    if ((lane & 3) == 0) {
      if (idx < K) atomicAdd(gR + (size_t)e * K + idx, grt);
      if (idx < D2) atomicAdd(gY + (size_t)e * d2 + off2 + idx, ht);
    }
  }
  __syncwarp();  // the ring is reused by the warp's next unit
  if (active) {
    float* Hs = Hstate + node_off + aoff + w;
#pragma unroll
    for (int k = 0; k < kKB; ++k)
      if (k < K)
#pragma unroll
        for (int m = 0; m < D1; ++m) Hs[k * s_slice + m * astr] = H[k][m];
  }
}

#define UVW3_BWD_CASE(L1, L2, L3)                                                                  \
  case (L1)*16 + (L2)*4 + (L3):                                                                    \
    if constexpr ((L3) <= 3 && (L3) >= ((L1) > (L2) ? (L1) - (L2) : (L2) - (L1)) && (L3) <= (L1) + (L2)) \
      uvw_bwd3_unit<L1, L2, L3, SH>(a.Y, a.R, a.rbf, a.g, a.Astate, a.Hstate, a.gY, a.gR, eidp, dstp,           \
                                rp[s], rp[s + 1], (size_t)(s - a.n0) * a.s_node, a.d2, a.d_out, a.K,  \
                                a.s_slice, p.off2, p.ooff, p.aoff, p.astr, p.mul_out, item.u0, lane, ring); \
    break;

constexpr int kBwd3Warps = 16;

constexpr int kBwd3IdxInts = 16384;  // shared memory for the CTA's transpose slice (ids + receivers)
constexpr int kBwd3RingBytes = kBwd3Warps * kRingWarp * int(sizeof(float));

template <bool SH>
__global__ void __launch_bounds__(kBwd3Warps * 32, 1) uvw_bwd_edge3_kernel(const Bwd3Args a) {
  extern __shared__ int bwd3_idx[];  // [idx_cap] transpose slice, then the warps' edge rings
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* ring = reinterpret_cast<float*>(bwd3_idx + a.idx_cap) + warp * kRingWarp;
  __shared__ int s_range[2];
  const int* rp = a.t_rowptr;
  if (tid == 0) {
    const long long base = (long long)rp[a.n0] + a.n0, total = (long long)rp[a.n1] + a.n1 - base;
    const long long t0 = base + total * blockIdx.x / gridDim.x, t1 = base + total * (blockIdx.x + 1) / gridDim.x;
    auto lb = [&](long long target) {
      int lo = a.n0, hi = a.n1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)rp[mid] + mid < target) lo = mid + 1; else hi = mid;
      }
      return lo;
    };
    s_range[0] = lb(t0);
    s_range[1] = (blockIdx.x + 1 == gridDim.x) ? a.n1 : lb(t1);
  }
  __syncthreads();
  const int sb = s_range[0], se = s_range[1];
  // the CTA's transpose slice in shared memory when it fits: no index load from
  // global memory in front of an edge's gathers
  const int tp0 = rp[sb], tp1 = rp[se];
  const int* eidp = a.t_eid;
  const int* dstp = a.t_dst;
  if (tp1 - tp0 <= a.idx_cap / 2) {
    for (int i = tid; i < tp1 - tp0; i += kBwd3Warps * 32) {
      bwd3_idx[i] = __ldg(a.t_eid + tp0 + i);
      bwd3_idx[a.idx_cap / 2 + i] = __ldg(a.t_dst + tp0 + i);
    }
    eidp = bwd3_idx - tp0;
    dstp = bwd3_idx + a.idx_cap / 2 - tp0;
  }
  // clear gY and gR of the CTA's senders' out-edges before the first path
  for (int s = sb + warp; s < se; s += kBwd3Warps)
    for (int t = rp[s]; t < rp[s + 1]; ++t) {
      const int e = a.t_eid[t];
      for (int i = lane; i < a.d2; i += 32) a.gY[(size_t)e * a.d2 + i] = 0.f;
      for (int i = lane; i < a.K; i += 32) a.gR[(size_t)e * a.K + i] = 0.f;
    }
  // path-major (one hot instruction stream per SM); inside a path, warps take
  // senders one at a time from a shared counter, and block barriers between
  // paths order every row's path contributions (deterministic, race-free)
  __shared__ int s_next[2];
  for (int it = 0; it < a.n_items; ++it) {
    const Item item = a.items[it];
    const UvwPath p = a.paths[item.path];
    if (tid == 0) s_next[it & 1] = sb;
    __syncthreads();
    for (;;) {
      int s = 0;
      if (lane == 0) s = atomicAdd(&s_next[it & 1], 1);
      s = __shfl_sync(0xffffffffu, s, 0);
      if (s >= se) break;
      switch (p.l1 * 16 + p.l2 * 4 + p.l3) {
        CGTP3_TRIPLES(UVW3_BWD_CASE)
        default: break;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// forward edge stage, warp-autonomous: a unit is (receiver n, path, 32
// channels u), lanes <-> u.  Over n's in-edges, lane u sums
//   S[k][m3] = sum_e R[e,k] t_e[m3],  t_e[m3] = sum_{m1} cy_e[m1,m3] x[src e][u,m1],
//   cy_e[m1,m3] = sum_{m2} C[m1,m2,m3] Y[e][m2]   (compiled-in nonzeros)
// in registers, with the edge operands staged through the warp's cp.async ring,
// and writes its K x D3 values of the node state once.  Every unit writes
// distinct state entries, so no reduction crosses warps; the warps of a CTA
// take (path, receiver) units from one counter in path-major order, which keeps
// them on one path's code at a time.
// ---------------------------------------------------------------------------
struct Fwd3Args {
  const float* x;
  const float* Y;       // edge-vector mode: the vectors [E,3]
  const float* R;
  Rbf rbf;
  float* state;         // [chunk][K][s_slice]
  const int* rowptr;
  const int* col;
  int n0, n1;
  int d1, d2, K, s_node, s_slice;
  const UvwPath* paths;
  const Item* items;    // (path, u0), path order
  int n_items;
  int idx_cap;          // ints of dynamic shared memory for the CTA's CSR column slice
};

template <int L1, int L2, int L3, bool SH>
__device__ __noinline__ void uvw_fwd3_unit(const float* __restrict__ x, const float* __restrict__ Yp,
                                           const float* __restrict__ Rp, Rbf rbf, float* __restrict__ Sn,
                                           const int* __restrict__ col, int eb, int ee, int d1, int d2, int K,
                                           int s_slice, int off1, int off2, int soff, int sstr, int mul1,
                                           int u0, int lane, float* ring) {
  constexpr int D1 = 2 * L1 + 1, D2 = 2 * L2 + 1, D3 = 2 * L3 + 1;
  constexpr int NY = SH ? 3 : D2;
  const int u = u0 + lane;
  const bool active = u < mul1;
  const int n_x = min(32, mul1 - u0) * D1;  // in-bounds feature values of the unit's u range
  float S[kKB][D3];
#pragma unroll
  for (int k = 0; k < kKB; ++k)
#pragma unroll
    for (int m = 0; m < D3; ++m) S[k][m] = 0.f;
  auto issue = [&](int t, int slot) {
    if (t < ee) {
      float* st = ring + slot * kRingStage;
      const float* xsrc = x + (size_t)col[t] * d1 + off1 + u0 * D1;
#pragma unroll
      for (int j = 0; j < D1; ++j)
        if (j * 32 + lane < n_x) cp_async4(st + j * 32 + lane, xsrc + j * 32 + lane);
      if (lane < NY)
        cp_async4(st + kRingY + lane, SH ? Yp + 3 * (size_t)t + lane : Yp + (size_t)t * d2 + off2 + lane);
      else if (!SH && lane >= 8 && lane < 8 + K)
        cp_async4(st + kRingR + lane - 8, Rp + (size_t)t * K + lane - 8);
    }
    cpa_commit();
  };
#pragma unroll
  for (int i = 0; i < kRingDepth - 1; ++i) issue(eb + i, i);
  int slot = 0;
  for (int t = eb; t < ee; ++t) {
    cpa_wait<kRingDepth - 2>();
    __syncwarp();
    issue(t + kRingDepth - 1, slot == 0 ? kRingDepth - 1 : slot - 1);
    const float* st = ring + slot * kRingStage;
    slot = slot + 1 == kRingDepth ? 0 : slot + 1;
    float yv[D2], r[kKB], xv[D1];
    if constexpr (SH) {
      const float rx = st[kRingY], ry = st[kRingY + 1], rz = st[kRingY + 2];
      const float dd = sqrtf(rx * rx + ry * ry + rz * rz), inv = dd > 0.f ? 1.f / dd : 0.f;
      sh_block<L2, float, float>(rx * inv, ry * inv, rz * inv, yv);
#pragma unroll
      for (int k = 0; k < kKB; ++k) r[k] = (k < K) ? rbf_k(rbf, dd, k) : 0.f;
    } else {
#pragma unroll
      for (int m = 0; m < D2; ++m) yv[m] = st[kRingY + m];
#pragma unroll
      for (int k = 0; k < kKB; ++k) r[k] = (k < K) ? st[kRingR + k] : 0.f;
    }
#pragma unroll
    for (int m = 0; m < D1; ++m) xv[m] = active ? st[lane * D1 + m] : 0.f;
    float cy[D1][D3];
#pragma unroll
    for (int i = 0; i < D1; ++i)
#pragma unroll
      for (int m = 0; m < D3; ++m) cy[i][m] = 0.f;
    CGB<L1, L2, L3>::each([&](int m1, int m2, int m3, double c) { cy[m1][m3] += float(c) * yv[m2]; });
    float t3[D3];
#pragma unroll
    for (int m = 0; m < D3; ++m) {
      t3[m] = 0.f;
#pragma unroll
      for (int i = 0; i < D1; ++i)
        if ((CGB<L1, L2, L3>::mask >> (i * D3 + m)) & 1ull) t3[m] += cy[i][m] * xv[i];
    }
#pragma unroll
    for (int k = 0; k < kKB; ++k)
#pragma unroll
      for (int m = 0; m < D3; ++m) S[k][m] += r[k] * t3[m];
  }
  __syncwarp();  // the ring is reused by the warp's next unit
  if (active) {
    float* sp = Sn + soff + u;
#pragma unroll
    for (int k = 0; k < kKB; ++k)
      if (k < K)
#pragma unroll
        for (int m = 0; m < D3; ++m) sp[k * s_slice + m * sstr] = S[k][m];
  }
}

#define UVW3_FWD_CASE(L1, L2, L3)                                                                  \
  case (L1)*16 + (L2)*4 + (L3):                                                                    \
    if constexpr ((L3) <= 3 && (L3) >= ((L1) > (L2) ? (L1) - (L2) : (L2) - (L1)) && (L3) <= (L1) + (L2)) \
      uvw_fwd3_unit<L1, L2, L3, SH>(a.x, a.Y, a.R, a.rbf, a.state + (size_t)(n - a.n0) * a.s_node, colp,      \
                                a.rowptr[n], a.rowptr[n + 1], a.d1, a.d2, a.K, a.s_slice, p.off1, p.off2, \
                                p.soff, p.sstr, p.mul1, item.u0, lane, ring);                   \
    break;

template <bool SH>
__global__ void __launch_bounds__(kBwd3Warps * 32, 1) uvw_fwd_edge3_kernel(const Fwd3Args a) {
  extern __shared__ int fwd3_idx[];  // [idx_cap] CSR column slice, then the warps' edge rings
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* ring = reinterpret_cast<float*>(fwd3_idx + a.idx_cap) + warp * kRingWarp;
  __shared__ int s_range[2];
  __shared__ int s_next;
  const int* rp = a.rowptr;
  if (tid == 0) {  // edge-balanced receiver range (edges + one per node)
    const long long base = (long long)rp[a.n0] + a.n0, total = (long long)rp[a.n1] + a.n1 - base;
    const long long t0 = base + total * blockIdx.x / gridDim.x, t1 = base + total * (blockIdx.x + 1) / gridDim.x;
    auto lb = [&](long long target) {
      int lo = a.n0, hi = a.n1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)rp[mid] + mid < target) lo = mid + 1; else hi = mid;
      }
      return lo;
    };
    s_range[0] = lb(t0);
    s_range[1] = (blockIdx.x + 1 == gridDim.x) ? a.n1 : lb(t1);
    s_next = 0;
  }
  __syncthreads();
  const int rb = s_range[0], re = s_range[1], nr = re - rb;
  const int ep0 = rp[rb], ep1 = rp[re];
  const int* colp = a.col;
  if (ep1 - ep0 <= a.idx_cap) {
    for (int i = tid; i < ep1 - ep0; i += kBwd3Warps * 32) fwd3_idx[i] = __ldg(a.col + ep0 + i);
    colp = fwd3_idx - ep0;
  }
  __syncthreads();
  const long long n_units = (long long)nr * a.n_items;
  for (;;) {
    int k = 0;
    if (lane == 0) k = atomicAdd(&s_next, 1);
    k = __shfl_sync(0xffffffffu, k, 0);
    if (k >= n_units) break;
    const Item item = a.items[k / nr];
    const int n = rb + k % nr;
    const UvwPath p = a.paths[item.path];
    switch (p.l1 * 16 + p.l2 * 4 + p.l3) {
      CGTP3_TRIPLES(UVW3_FWD_CASE)
      default: break;
    }
  }
}

}  // namespace uvw_detail

using namespace uvw_detail;

cgtp_status uvw_create(cgtp_plan_s* plan) {
  UvwState* st = new UvwState();
  plan->uvw = st;
  st->K = plan->radial_k;
  if (st->K > kKB) return fail(CGTP_EUNSUPPORTED, "uvw supports radial_k <= 8");
  int lmax = 0;
  for (const auto& p : plan->paths) lmax = std::max(lmax, std::max(p.l1, std::max(p.l2, p.l3)));
  if (lmax > 3) return fail(CGTP_EUNSUPPORTED, "uvw supports l <= 3");
  // state slices: forward per output block o [m3][u of every path into o];
  // backward per in1 block b [m1][w of every path from b]
  const int n_out_blocks = static_cast<int>(plan->out.size()), n_in1_blocks = static_cast<int>(plan->in1.size());
  std::vector<int> U(n_out_blocks, 0), Wb(n_in1_blocks, 0), cu(plan->paths.size()), cw(plan->paths.size());
  for (size_t i = 0; i < plan->paths.size(); ++i) {
    const auto& q = plan->paths[i];
    cu[i] = U[q.io];
    U[q.io] += q.mul1;
    cw[i] = Wb[q.i1];
    Wb[q.i1] += q.mul_out;
  }
  std::vector<int> obase(n_out_blocks, 0), ibase(n_in1_blocks, 0);
  int soff = 0, aoff = 0;
  for (int o = 0; o < n_out_blocks; ++o) {
    obase[o] = soff;
    soff += U[o] * (2 * plan->out[o].l + 1);
  }
  for (int b = 0; b < n_in1_blocks; ++b) {
    ibase[b] = aoff;
    aoff += Wb[b] * (2 * plan->in1[b].l + 1);
  }
  for (size_t i = 0; i < plan->paths.size(); ++i) {
    const auto& q = plan->paths[i];
    UvwPath u{};
    u.l1 = q.l1;
    u.l2 = q.l2;
    u.l3 = q.l3;
    u.D1 = 2 * q.l1 + 1;
    u.D2 = 2 * q.l2 + 1;
    u.D3 = 2 * q.l3 + 1;
    u.mul1 = q.mul1;
    u.mul_out = q.mul_out;
    u.off1 = q.off1;
    u.off2 = q.off2;
    u.ooff = q.ooff;
    u.woff = q.woff;
    u.soff = obase[q.io] + cu[i];
    u.aoff = ibase[q.i1] + cw[i];
    u.sstr = U[q.io];
    u.astr = Wb[q.i1];
    u.i1 = q.i1;
    u.io = q.io;
    st->paths_h.push_back(u);
  }
  st->n_paths = static_cast<int>(plan->paths.size());
  st->s_slice = std::max(soff, aoff);
  st->s_node = st->K * st->s_slice;
  // ---- GEMM descriptors -------------------------------------------------
  // launch pointers: 0 = node state chunk, 1 = M, 2 = out / gx chunk rows,
  //                  3 = x chunk rows, 4 = gM, 5 = second node state chunk
  const int Kr = st->K;
  const long long wn = plan->w_numel;
  std::vector<GemmProb> fp, pp, xp, mp;
  std::vector<GemmSeg> fs, ps, xs, ms;
  const int n_out = static_cast<int>(plan->out.size());
  int oo = 0;
  std::vector<int> out_off;
  for (const auto& o : plan->out) {
    out_off.push_back(oo);
    oo += o.mul * (2 * o.l + 1);
  }
  // forward: one problem per output block, K over (k, path -> block), rows (n, m3), cols w
  for (int o = 0; o < n_out; ++o) {
    GemmProb P{};
    P.a_base = 0; P.b_base = 1; P.c_base = 2;
    P.Nn = -1;
    P.D = 2 * plan->out[o].l + 1;
    P.J = plan->out[o].mul;
    P.a_off = 0; P.a_n = st->s_node; P.a_m = U[o];   // S rows (n, m3): channels contiguous
    P.b_j = 1;
    P.c_off = out_off[o]; P.c_n = plan->d_out; P.c_m = 1; P.c_j = P.D;
    P.beta = 0;
    P.seg0 = int(fs.size());
    for (int k = 0; k < Kr; ++k)
      for (const auto& q : st->paths_h)
        if (q.io == o) {
          GemmSeg S{};
          S.a_off = (long long)k * st->s_slice + q.soff;
          S.b_off = (long long)k * wn + q.woff;
          S.K = q.mul1;
          S.a_k = 1;
          S.b_k = q.mul_out;
          S.b_j = 1;
          fs.push_back(S);
        }
    P.seg1 = int(fs.size());
    if (P.seg1 > P.seg0) fp.push_back(P);
  }
  // backward pre-GEMM: A[s][k][path][w][m1] = sum_u x[s][u,m1] M[k,path,u,w]
  for (int k = 0; k < Kr; ++k)
    for (const auto& q : st->paths_h) {
      GemmProb P{};
      P.a_base = 3; P.b_base = 1; P.c_base = 0;
      P.Nn = -1; P.D = q.D1; P.J = q.mul_out;
      P.a_off = q.off1; P.a_n = plan->d1; P.a_m = 1;
      P.b_j = 1;
      P.c_off = (long long)k * st->s_slice + q.aoff; P.c_n = st->s_node; P.c_m = q.astr; P.c_j = 1;
      P.beta = 0;
      P.seg0 = int(ps.size());
      GemmSeg S{};
      S.a_off = 0; S.b_off = (long long)k * wn + q.woff; S.K = q.mul1; S.a_k = q.D1; S.b_k = q.mul_out;
      S.b_j = 1;
      ps.push_back(S);
      P.seg1 = int(ps.size());
      pp.push_back(P);
    }
  // backward gx: per in1 block, rows (s, m1), cols u, K over (k, path with that block) of w
  int o1 = 0;
  for (int i1 = 0; i1 < (int)plan->in1.size(); ++i1) {
    const auto& b = plan->in1[i1];
    GemmProb P{};
    P.a_base = 5; P.b_base = 1; P.c_base = 2;
    P.Nn = -1; P.D = 2 * b.l + 1; P.J = b.mul;
    P.a_off = 0; P.a_n = st->s_node; P.a_m = Wb[i1];  // H rows (s, m1): channels contiguous
    P.c_off = o1; P.c_n = plan->d1; P.c_m = 1; P.c_j = P.D;
    P.beta = 0;
    P.seg0 = int(xs.size());
    for (int k = 0; k < Kr; ++k)
      for (const auto& q : st->paths_h)
        if (q.i1 == i1) {
          GemmSeg S{};
          S.a_off = (long long)k * st->s_slice + q.aoff;
          S.b_off = (long long)k * wn + q.woff;  // B[w][u] = M[k][woff + u*mul_out + w]
          S.K = q.mul_out; S.a_k = 1; S.b_k = 1;
          S.b_j = q.mul_out;  // B[w][u] = M[k][woff + u*mul_out + w]
          xs.push_back(S);
        }
    P.seg1 = int(xs.size());
    if (P.seg1 > P.seg0) xp.push_back(P);
    o1 += b.mul * (2 * b.l + 1);
  }
  // backward gM: per (k, path): rows u (Nn = mul1, D = 1), cols w, K over (m1, s in chunk)
  for (int k = 0; k < Kr; ++k)
    for (const auto& q : st->paths_h) {
      GemmProb P{};
      P.a_base = 3; P.b_base = 5; P.c_base = 4;
      P.Nn = q.mul1; P.D = 1; P.J = q.mul_out;
      P.a_off = q.off1; P.a_n = q.D1; P.a_m = 0;
      P.b_j = 1;
      P.c_off = (long long)k * wn + q.woff; P.c_n = q.mul_out; P.c_m = 0; P.c_j = 1;
      P.beta = 0;  // writes a split-K partial; splitk_reduce_kernel accumulates into gM
      P.seg0 = int(ms.size());
      for (int m1 = 0; m1 < q.D1; ++m1) {
        GemmSeg S{};
        S.a_off = m1; S.b_off = (long long)k * st->s_slice + q.aoff + (long long)m1 * q.astr;
        S.K = -1; S.a_k = plan->d1; S.b_k = st->s_node;
        S.b_j = 1;
        ms.push_back(S);
      }
      P.seg1 = int(ms.size());
      mp.push_back(P);
    }
  // tile-loading mode per problem from its segments' strides: lanes walk K when the
  // K stride is small, the rows of A / columns of B when those are contiguous instead
  auto set_modes = [](std::vector<GemmProb>& probs, const std::vector<GemmSeg>& segs) {
    for (auto& P : probs) {
      if (P.seg1 <= P.seg0) continue;
      const GemmSeg& S = segs[P.seg0];
      const long long row_stride = P.D > 1 ? P.a_m : P.a_n;
      P.a_mode = (S.a_k > 32 && row_stride < S.a_k) ? 1 : 0;
      P.b_mode = (S.b_j == 1 && S.b_k != 1) ? 1 : 0;
      bool av = P.a_n % 4 == 0 && (P.D == 1 || P.a_m % 4 == 0), bv = true;
      for (int g = P.seg0; g < P.seg1; ++g) {
        av = av && segs[g].a_k == 1;
        bv = bv && segs[g].b_k == 1 && segs[g].b_j % 4 == 0;
      }
      P.a_vec = av ? 1 : 0;
      P.b_vec = bv ? 1 : 0;
    }
  };
  set_modes(fp, fs);
  set_modes(pp, ps);
  set_modes(xp, xs);
  set_modes(mp, ms);
  // upload descriptor tables
  std::vector<unsigned char> buf;
  auto put = [&](const void* src, size_t bytes) {
    size_t o = (buf.size() + 15) / 16 * 16;
    buf.resize(o + bytes);
    if (bytes) memcpy(buf.data() + o, src, bytes);
    return o;
  };
  const size_t o_paths = put(st->paths_h.data(), st->paths_h.size() * sizeof(UvwPath));
  const size_t o_fp = put(fp.data(), fp.size() * sizeof(GemmProb));
  const size_t o_fs = put(fs.data(), fs.size() * sizeof(GemmSeg));
  const size_t o_pp = put(pp.data(), pp.size() * sizeof(GemmProb));
  const size_t o_ps = put(ps.data(), ps.size() * sizeof(GemmSeg));
  const size_t o_xp = put(xp.data(), xp.size() * sizeof(GemmProb));
  const size_t o_xs = put(xs.data(), xs.size() * sizeof(GemmSeg));
  const size_t o_mp = put(mp.data(), mp.size() * sizeof(GemmProb));
  const size_t o_ms = put(ms.data(), ms.size() * sizeof(GemmSeg));
  std::vector<Item> b3;
  for (int p = 0; p < st->n_paths; ++p)
    for (int w0 = 0; w0 < st->paths_h[p].mul_out; w0 += 32) b3.push_back({p, w0});
  const size_t o_b3 = put(b3.data(), b3.size() * sizeof(Item));
  std::vector<Item> f3;
  for (int p = 0; p < st->n_paths; ++p)
    for (int u0 = 0; u0 < st->paths_h[p].mul1; u0 += 32) f3.push_back({p, u0});
  const size_t o_f3 = put(f3.data(), f3.size() * sizeof(Item));
  if (cudaMalloc(&st->tables, buf.size()) != cudaSuccess) return fail(CGTP_ENOMEM, "uvw tables");
  plan->device_bytes += buf.size();
  cudaMemcpy(st->tables, buf.data(), buf.size(), cudaMemcpyHostToDevice);
  auto at = [&](size_t o) { return static_cast<unsigned char*>(st->tables) + o; };
  st->paths = reinterpret_cast<UvwPath*>(at(o_paths));
  st->fwd_probs = reinterpret_cast<GemmProb*>(at(o_fp)); st->fwd_np = int(fp.size());
  st->fwd_segs = reinterpret_cast<GemmSeg*>(at(o_fs));
  st->pre_probs = reinterpret_cast<GemmProb*>(at(o_pp)); st->pre_np = int(pp.size());
  st->pre_segs = reinterpret_cast<GemmSeg*>(at(o_ps));
  st->gx_probs = reinterpret_cast<GemmProb*>(at(o_xp)); st->gx_np = int(xp.size());
  st->gx_segs = reinterpret_cast<GemmSeg*>(at(o_xs));
  st->gm_probs = reinterpret_cast<GemmProb*>(at(o_mp)); st->gm_np = int(mp.size());
  st->gm_segs = reinterpret_cast<GemmSeg*>(at(o_ms));
  st->bwd3_items = reinterpret_cast<Item*>(at(o_b3));
  st->bwd3_n_items = int(b3.size());
  st->fwd3_items = reinterpret_cast<Item*>(at(o_f3));
  st->fwd3_n_items = int(f3.size());
  // node-state scratch: two chunks of state (forward S; backward A and H), addressed
  // with 32-bit element offsets inside a chunk
  st->chunk_nodes = kChunkPerSm * std::max(1, plan->num_sms);
  while ((long long)st->chunk_nodes * st->s_node >= (1ll << 31) && st->chunk_nodes > 1) st->chunk_nodes /= 2;
  st->scratch_elems = size_t(2) * st->chunk_nodes * st->s_node;
  if (cudaMalloc(&st->scratch, st->scratch_elems * sizeof(float)) != cudaSuccess)
    return fail(CGTP_ENOMEM, "uvw node-state scratch allocation failed");
  if (cudaMalloc(&st->gm_part, sizeof(float) * kGmSplits * st->K * plan->w_numel) != cudaSuccess)
    return fail(CGTP_ENOMEM, "uvw gM partial allocation failed");
  if (cudaMalloc(&st->err_dev, sizeof(int)) != cudaSuccess ||
      cudaHostAlloc(&st->err_host, sizeof(int), cudaHostAllocDefault) != cudaSuccess)
    return fail(CGTP_ENOMEM, "uvw error flag allocation failed");
  plan->device_bytes += st->scratch_elems * sizeof(float) + sizeof(float) * kGmSplits * st->K * plan->w_numel +
                        sizeof(int);
  cudaMemset(st->err_dev, 0, sizeof(int));
  *st->err_host = 0;
  const int np_max = std::max(std::max(st->fwd_np, st->pre_np), std::max(st->gx_np, st->gm_np));
  if (gemm_smem(np_max) > 113 * 1024)  // two CTAs per SM
    return fail(CGTP_EUNSUPPORTED, "uvw plan has too many GEMM problems for the tile table");
  if (cudaFuncSetAttribute(grouped_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(gemm_smem(np_max))) != cudaSuccess)
    return fail(CGTP_ECUDA, "tensor-core GEMM shared memory attribute rejected");
  return CGTP_OK;
}

void uvw_destroy(cgtp_plan_s* plan) {
  UvwState* st = static_cast<UvwState*>(plan->uvw);
  if (!st) return;
  if (st->tables) cudaFree(st->tables);
  if (st->scratch) cudaFree(st->scratch);
  if (st->gm_part) cudaFree(st->gm_part);
  if (st->err_dev) cudaFree(st->err_dev);
  if (st->err_host) cudaFreeHost(st->err_host);
  delete st;
  plan->uvw = nullptr;
}

namespace {
cgtp_status launch_gemm(const GemmProb* probs_dev, int np, const GemmSeg* segs,
                        const float* const ptr[6], int nodes, int tiles, cudaStream_t s, int* err,
                        long long wait_limit, int splits = 1, long long c_split_stride = 0) {
  GemmLaunch L{};
  for (int i = 0; i < 6; ++i) L.ptr[i] = ptr[i];
  L.nodes = nodes;
  L.nprob = np;
  L.probs = probs_dev;
  L.segs = segs;
  L.splits = splits;
  L.c_split_stride = c_split_stride;
  L.err = err;
  L.wait_limit = wait_limit;
  L.tiles = tiles;
  int dev = 0, nsm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::max(1, std::min(tiles, 2 * nsm));  // two CTAs per SM, persistent
  grouped_gemm_tc_kernel<<<dim3(grid, splits), kTcWarps * 32, gemm_smem(np), s>>>(L);
  return cudaGetLastError() == cudaSuccess ? CGTP_OK : fail(CGTP_ECUDA, "uvw gemm launch failed");
}

// tiles of a descriptor set for `nodes` nodes (host copy of the descriptors needed)
int count_tiles(const std::vector<std::pair<int, int>>& rows_cols) {
  int t = 0;
  for (auto& rc : rows_cols) t += ((rc.first + kTM - 1) / kTM) * ((rc.second + kTN - 1) / kTN);
  return t;
}
}  // namespace

// Host mirrors of the GEMM shapes (rows per node, cols, fixed rows) to size the grids.
static int tiles_for(const cgtp_plan_s* plan, const UvwState* st, int which, int nodes) {
  std::vector<std::pair<int, int>> rc;
  if (which == 0) {
    for (size_t o = 0; o < plan->out.size(); ++o) {
      bool any = false;
      for (const auto& q : st->paths_h) any |= (q.io == int(o));
      if (any) rc.push_back({nodes * (2 * plan->out[o].l + 1), plan->out[o].mul});
    }
  } else if (which == 1) {
    for (int k = 0; k < st->K; ++k)
      for (const auto& q : st->paths_h) rc.push_back({nodes * q.D1, q.mul_out});
  } else if (which == 2) {
    for (size_t i1 = 0; i1 < plan->in1.size(); ++i1) {
      bool any = false;
      for (const auto& q : st->paths_h) any |= (q.i1 == int(i1));
      if (any) rc.push_back({nodes * (2 * plan->in1[i1].l + 1), plan->in1[i1].mul});
    }
  } else {
    for (int k = 0; k < st->K; ++k)
      for (const auto& q : st->paths_h) rc.push_back({q.mul1, q.mul_out});
  }
  return count_tiles(rc);
}

cgtp_status uvw_set_chunk(cgtp_plan_s* plan, int nodes) {
  UvwState* st = static_cast<UvwState*>(plan->uvw);
  // the kernels address one chunk's node state with 32-bit element offsets
  if ((long long)nodes * st->s_node >= (1ll << 31))
    return fail(CGTP_EINVAL, "uvw node chunk too large: chunk x node-state size must stay below 2^31 elements");
  const size_t elems = size_t(2) * nodes * st->s_node;
  float* p = nullptr;
  if (cudaMalloc(&p, elems * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    return fail(CGTP_ENOMEM, "uvw node-state scratch allocation failed");
  }
  cudaFree(st->scratch);  // waits for the work that used the old buffer
  plan->device_bytes = plan->device_bytes - st->scratch_elems * sizeof(float) + elems * sizeof(float);
  st->scratch = p;
  st->scratch_elems = elems;
  st->chunk_nodes = nodes;
  return CGTP_OK;
}

int uvw_chunk(const cgtp_plan_s* plan) { return static_cast<const UvwState*>(plan->uvw)->chunk_nodes; }

static cgtp_status sticky_error(const UvwState* st) {
  if (*st->err_host)
    return fail(CGTP_ECUDA, "a tensor-core wait gave up in an earlier uvw call on this plan");
  return CGTP_OK;
}
static void refresh_error(const UvwState* st, cudaStream_t s) {
  cudaMemcpyAsync(st->err_host, st->err_dev, sizeof(int), cudaMemcpyDeviceToHost, s);
}

static Rbf make_rbf(int K, double lo, double hi) {
  const double step = K > 1 ? (hi - lo) / (K - 1) : (hi - lo);
  return Rbf{static_cast<float>(lo), static_cast<float>(step), static_cast<float>(1.0 / (step * step))};
}

cgtp_status uvw_forward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* x,
                        const void* Y, const void* R, const void* M, void* out, void* stream,
                        const void* rvec, double rbf_lo, double rbf_hi) {
  const UvwState* st = static_cast<const UvwState*>(plan->uvw);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cgtp_status e = sticky_error(st)) return e;
  if ((long long)st->chunk_nodes * st->fwd3_n_items >= (1ll << 31))
    return fail(CGTP_EUNSUPPORTED, "uvw forward: node chunk x channel blocks exceeds the 32-bit unit counter");
  Fwd3Args a{};
  a.x = static_cast<const float*>(x);
  a.Y = static_cast<const float*>(rvec ? rvec : Y);
  a.R = static_cast<const float*>(R);
  a.rbf = make_rbf(st->K, rbf_lo, rbf_hi);
  a.state = st->scratch;
  a.rowptr = g->rowptr;
  a.col = g->col;
  a.d1 = static_cast<int>(plan->d1);
  a.d2 = static_cast<int>(plan->d2);
  a.K = st->K;
  a.s_node = st->s_node;
  a.s_slice = st->s_slice;
  a.paths = st->paths;
  a.items = st->fwd3_items;
  a.n_items = st->fwd3_n_items;
  const void* kf = rvec ? reinterpret_cast<const void*>(uvw_fwd_edge3_kernel<true>)
                        : reinterpret_cast<const void*>(uvw_fwd_edge3_kernel<false>);
  const int cap = smem_cap_cached(kf);
  if (cap < kBwd3RingBytes) return fail(CGTP_ECUDA, "uvw forward edge stage: shared memory below its edge rings");
  a.idx_cap = cap >= int(kBwd3IdxInts * sizeof(int)) + kBwd3RingBytes ? kBwd3IdxInts : 0;
  const size_t fsz = size_t(a.idx_cap) * sizeof(int) + kBwd3RingBytes;
  for (int64_t n0 = 0; n0 < g->N; n0 += st->chunk_nodes) {
    const int n1 = static_cast<int>(std::min<int64_t>(g->N, n0 + st->chunk_nodes));
    a.n0 = static_cast<int>(n0);
    a.n1 = n1;
    const int nodes = n1 - a.n0;
    const int grid = std::min(nodes, plan->num_sms);
    if (rvec)
      uvw_fwd_edge3_kernel<true><<<grid, kBwd3Warps * 32, fsz, s>>>(a);
    else
      uvw_fwd_edge3_kernel<false><<<grid, kBwd3Warps * 32, fsz, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return fail(CGTP_ECUDA, "uvw forward edge stage launch failed");
    const float* ptr[6] = {st->scratch, static_cast<const float*>(M),
                           static_cast<float*>(out) + (size_t)n0 * plan->d_out, nullptr, nullptr, nullptr};
    cgtp_status r = launch_gemm(st->fwd_probs, st->fwd_np, st->fwd_segs, ptr, nodes,
                                tiles_for(plan, st, 0, nodes), s, st->err_dev, plan->wait_limit);
    if (r != CGTP_OK) return r;
  }
  refresh_error(st, s);
  return CGTP_OK;
}

cgtp_status uvw_backward(const cgtp_plan_s* plan, const cgtp_graph_s* g, const void* gout,
                         const void* x, const void* Y, const void* R, const void* M, void* gx,
                         void* gY, void* gR, void* gM, void* stream, const void* rvec, double rbf_lo,
                         double rbf_hi) {
  const UvwState* st = static_cast<const UvwState*>(plan->uvw);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cgtp_status e = sticky_error(st)) return e;
  float* Abuf = st->scratch;
  float* Hbuf = st->scratch + (size_t)st->chunk_nodes * st->s_node;
  bool first = true;
  for (int64_t n0 = 0; n0 < g->N; n0 += st->chunk_nodes) {
    const int n1 = static_cast<int>(std::min<int64_t>(g->N, n0 + st->chunk_nodes));
    const int nodes = n1 - static_cast<int>(n0);
    const float* xrows = static_cast<const float*>(x) + (size_t)n0 * plan->d1;
    const float* pre[6] = {Abuf, static_cast<const float*>(M), nullptr, xrows, nullptr, nullptr};
    cgtp_status r = launch_gemm(st->pre_probs, st->pre_np, st->pre_segs, pre, nodes,
                                tiles_for(plan, st, 1, nodes), s, st->err_dev, plan->wait_limit);
    if (r != CGTP_OK) return r;
    Bwd3Args b{};
    b.Y = static_cast<const float*>(rvec ? rvec : Y);
    b.R = static_cast<const float*>(R);
    b.rbf = make_rbf(st->K, rbf_lo, rbf_hi);
    b.g = static_cast<const float*>(gout);
    b.Astate = Abuf;
    b.Hstate = Hbuf;
    b.gY = static_cast<float*>(gY);
    b.gR = static_cast<float*>(gR);
    b.t_rowptr = g->t_rowptr;
    b.t_eid = g->t_eid;
    b.t_dst = g->t_dst;
    b.n0 = static_cast<int>(n0);
    b.n1 = n1;
    b.d2 = static_cast<int>(plan->d2);
    b.d_out = static_cast<int>(plan->d_out);
    b.K = st->K;
    b.s_node = st->s_node;
    b.s_slice = st->s_slice;
    b.paths = st->paths;
    b.items = st->bwd3_items;
    b.n_items = st->bwd3_n_items;
    const int grid = std::min(nodes, plan->num_sms);
    const void* kb = rvec ? reinterpret_cast<const void*>(uvw_bwd_edge3_kernel<true>)
                          : reinterpret_cast<const void*>(uvw_bwd_edge3_kernel<false>);
    const int cap = smem_cap_cached(kb);
    if (cap < kBwd3RingBytes) return fail(CGTP_ECUDA, "uvw backward edge stage: shared memory below its edge rings");
    b.idx_cap = cap >= int(kBwd3IdxInts * sizeof(int)) + kBwd3RingBytes ? kBwd3IdxInts : 0;
    const size_t isz = size_t(b.idx_cap) * sizeof(int) + kBwd3RingBytes;
    if (rvec)
      uvw_bwd_edge3_kernel<true><<<grid, kBwd3Warps * 32, isz, s>>>(b);
    else
      uvw_bwd_edge3_kernel<false><<<grid, kBwd3Warps * 32, isz, s>>>(b);
    if (cudaGetLastError() != cudaSuccess) return fail(CGTP_ECUDA, "uvw backward edge stage launch failed");
    const float* post[6] = {nullptr, static_cast<const float*>(M),
                            static_cast<float*>(gx) + (size_t)n0 * plan->d1, xrows,
                            static_cast<float*>(gM), Hbuf};
    r = launch_gemm(st->gx_probs, st->gx_np, st->gx_segs, post, nodes, tiles_for(plan, st, 2, nodes), s, st->err_dev, plan->wait_limit);
    if (r != CGTP_OK) return r;
    // gM over this chunk's senders: split-K partials, then an ordered reduction
    const float* postp[6] = {post[0], post[1], post[2], post[3], st->gm_part, post[5]};
    const int splits = std::min(kGmSplits, std::max(1, nodes / 64));
    const long long n_gm = (long long)st->K * plan->w_numel;
    r = launch_gemm(st->gm_probs, st->gm_np, st->gm_segs, postp, nodes, tiles_for(plan, st, 3, nodes), s, st->err_dev,
                    plan->wait_limit, splits, n_gm);
    if (r != CGTP_OK) return r;
    splitk_reduce_kernel<<<std::min<long long>((n_gm + 255) / 256, 4096), 256, 0, s>>>(
        static_cast<float*>(gM), st->gm_part, splits, n_gm, first ? 0 : 1);
    if (cudaGetLastError() != cudaSuccess) return fail(CGTP_ECUDA, "uvw gM reduction launch failed");
    first = false;
  }
  refresh_error(st, s);
  if (g->N == 0) cudaMemsetAsync(gM, 0, sizeof(float) * plan->w_numel * st->K, s);
  return CGTP_OK;
}

}  // namespace cgtp
