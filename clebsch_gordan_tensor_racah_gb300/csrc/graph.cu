// graph.cu -- CSR validation and the sender transpose, on the device.
//
// "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
// Figure 4B: the convolution sums edge messages into the receiving node, so
// the forward pass walks the receiver-sorted CSR.  The gradient with respect to
// the node features belongs to the sender; the backward pass walks the
// transpose: t_rowptr (prefix sum of out-degrees), t_eid (CSR positions
// grouped by sender, ascending inside each sender -- a stable sort by sender)
// and t_dst (receiver of each such edge).
//
// Steps: (1) check rowptr[0] = 0, rowptr[N] = E, rowptr monotone, 0 <= col < N;
// (2) out-degree histogram (integer atomics: the counts are exact);
// (3) exclusive scan -> t_rowptr; (4) scatter positions into their sender
// segment (integer atomics pick slots in arbitrary order); (5) sort each
// segment ascending, which makes the result unique and bit-exact; (6) t_dst by
// binary search of rowptr.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <mutex>
#include <string>

#include "internal.h"

namespace cgtp {

namespace {

constexpr int kSortWarp = 1024;      // segments up to this length: one warp, rank sort
constexpr int kSortBlock = 32768;    // longer segments up to this: one CTA, bitonic
constexpr int kScanTile = 1024;

enum : int { kBadRow0 = 1, kBadRowN = 2, kNotMonotone = 4, kBadCol = 8, kTooLong = 16 };

__global__ void csr_check_kernel(const int* rowptr, const int* col, int N, int E, int* flag) {
  int bits = 0;
  const int total = max(N + 1, E);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    if (i <= N) {
      const int r = rowptr[i];
      if (i == 0 && r != 0) bits |= kBadRow0;
      if (i == N && r != E) bits |= kBadRowN;
      if (i < N && r > rowptr[i + 1]) bits |= kNotMonotone;
    }
    if (i < E) {
      const int c = col[i];
      if (c < 0 || c >= N) bits |= kBadCol;
    }
  }
  if (bits) atomicOr(flag, bits);
}

__global__ void histogram_kernel(const int* col, int E, int* counts) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < E; i += gridDim.x * blockDim.x)
    atomicAdd(&counts[col[i]], 1);
}

// Tile-wise exclusive scan: out[i] = sum of in[<i] inside the tile; tile total to sums.
__global__ void scan_tiles_kernel(const int* in, int n, int* out, int* sums) {
  __shared__ int s[kScanTile];
  const int base = blockIdx.x * kScanTile;
  for (int i = threadIdx.x; i < kScanTile; i += blockDim.x)
    s[i] = (base + i < n) ? in[base + i] : 0;
  __syncthreads();
  for (int off = 1; off < kScanTile; off <<= 1) {  // Hillis-Steele inclusive
    int v[kScanTile / 256];
    for (int k = 0; k < kScanTile / 256; ++k) {
      const int i = threadIdx.x + k * 256;
      v[k] = (i >= off) ? s[i - off] : 0;
    }
    __syncthreads();
    for (int k = 0; k < kScanTile / 256; ++k) s[threadIdx.x + k * 256] += v[k];
    __syncthreads();
  }
  for (int i = threadIdx.x; i < kScanTile; i += blockDim.x)
    if (base + i < n) out[base + i] = (i == 0) ? 0 : s[i - 1];
  if (threadIdx.x == 0) sums[blockIdx.x] = s[kScanTile - 1];
}

// Sequential exclusive scan of the tile sums (one thread; tiles are few).
__global__ void scan_sums_kernel(int* sums, int ntiles, int* total_out) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    int acc = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int v = sums[t];
      sums[t] = acc;
      acc += v;
    }
    *total_out = acc;
  }
}

__global__ void add_offsets_kernel(int* out, int n, const int* sums) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] += sums[i / kScanTile];
}

__global__ void scatter_kernel(const int* col, int E, int* cursor, int* t_eid) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < E; i += gridDim.x * blockDim.x) {
    const int pos = atomicAdd(&cursor[col[i]], 1);
    t_eid[pos] = i;
  }
}

// One warp per segment of length <= kSortWarp: rank sort (values are distinct).
__global__ void sort_short_kernel(const int* t_rowptr, int N, int* t_eid, int* flag) {
  __shared__ int buf[4][kSortWarp];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nw = gridDim.x * 4;
  for (int s = blockIdx.x * 4 + w; s < N; s += nw) {
    const int b = t_rowptr[s], len = t_rowptr[s + 1] - b;
    if (len <= 1) continue;
    if (len > kSortWarp) {
      if (len > kSortBlock && lane == 0) atomicOr(flag, kTooLong);
      continue;
    }
    for (int i = lane; i < len; i += 32) buf[w][i] = t_eid[b + i];
    __syncwarp();
    for (int i = lane; i < len; i += 32) {
      const int v = buf[w][i];
      int r = 0;
      for (int k = 0; k < len; ++k) r += (buf[w][k] < v);
      t_eid[b + r] = v;
    }
    __syncwarp();
  }
}

// One CTA per segment of length in (kSortWarp, kSortBlock]: bitonic sort in shared memory.
__global__ void sort_long_kernel(const int* t_rowptr, int N, int* t_eid) {
  extern __shared__ int sbuf[];
  for (int s = blockIdx.x; s < N; s += gridDim.x) {
    const int b = t_rowptr[s], len = t_rowptr[s + 1] - b;
    if (len <= kSortWarp || len > kSortBlock) continue;
    int n2 = 1;
    while (n2 < len) n2 <<= 1;
    for (int i = threadIdx.x; i < n2; i += blockDim.x) sbuf[i] = (i < len) ? t_eid[b + i] : INT_MAX;
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = threadIdx.x; i < n2; i += blockDim.x) {
          const int p = i ^ j;
          if (p > i) {
            const bool asc = (i & k) == 0;
            const int a = sbuf[i], c = sbuf[p];
            if ((a > c) == asc) {
              sbuf[i] = c;
              sbuf[p] = a;
            }
          }
        }
        __syncthreads();
      }
    for (int i = threadIdx.x; i < len; i += blockDim.x) t_eid[b + i] = sbuf[i];
    __syncthreads();
  }
}

__global__ void dst_kernel(const int* rowptr, int N, const int* t_eid, int E, int* t_dst) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < E; i += gridDim.x * blockDim.x) {
    const int p = t_eid[i];
    int lo = 0, hi = N;  // last n with rowptr[n] <= p
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (rowptr[mid] <= p)
        lo = mid;
      else
        hi = mid;
    }
    t_dst[i] = lo;
  }
}

}  // namespace

cgtp_status graph_build(cgtp_graph_s* g, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = static_cast<int>(g->N), E = static_cast<int>(g->E);
  int* scratch = nullptr;  // flag | total | counts/cursor [N+1] | tile sums
  const int ntiles = (N + 1 + kScanTile - 1) / kScanTile;
  const size_t words = 2 + static_cast<size_t>(N + 1) + ntiles;
  if (cudaMalloc(&scratch, words * sizeof(int)) != cudaSuccess)
    return fail(CGTP_ENOMEM, "graph scratch allocation failed");
  int* flag = scratch;
  int* total = scratch + 1;
  int* counts = scratch + 2;
  int* sums = counts + (N + 1);
  cudaMemsetAsync(scratch, 0, words * sizeof(int), st);
  const int threads = 256;
  auto blocks = [](int64_t n) { return static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096)); };
  csr_check_kernel<<<std::max(1, blocks(std::max(N + 1, E))), threads, 0, st>>>(g->rowptr, g->col, N, E, flag);
  int hflag = 0;
  cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, st);
  cudaError_t err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) {
    cudaFree(scratch);
    return fail(CGTP_ECUDA, std::string("graph check: ") + cudaGetErrorString(err));
  }
  if (hflag) {
    cudaFree(scratch);
    std::string why;
    if (hflag & kBadRow0) why += " rowptr[0] != 0;";
    if (hflag & kBadRowN) why += " rowptr[N] != E;";
    if (hflag & kNotMonotone) why += " rowptr not monotone;";
    if (hflag & kBadCol) why += " col out of [0, N);";
    return fail(CGTP_EGRAPH, "invalid CSR:" + why);
  }
  if (E > 0) histogram_kernel<<<blocks(E), threads, 0, st>>>(g->col, E, counts);
  // counts[N] = 0 -> exclusive scan over N+1 entries gives t_rowptr with t_rowptr[N] = E
  scan_tiles_kernel<<<ntiles, 256, 0, st>>>(counts, N + 1, g->t_rowptr, sums);
  scan_sums_kernel<<<1, 32, 0, st>>>(sums, ntiles, total);
  add_offsets_kernel<<<blocks(N + 1), threads, 0, st>>>(g->t_rowptr, N + 1, sums);
  if (E > 0) {
    cudaMemcpyAsync(counts, g->t_rowptr, sizeof(int) * (N + 1), cudaMemcpyDeviceToDevice, st);
    scatter_kernel<<<blocks(E), threads, 0, st>>>(g->col, E, counts, g->t_eid);
    sort_short_kernel<<<std::max(1, std::min((N + 3) / 4, 4096)), 128, 0, st>>>(g->t_rowptr, N, g->t_eid, flag);
    const size_t lsm = kSortBlock * sizeof(int);
    err = cudaFuncSetAttribute(sort_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lsm);
    if (err != cudaSuccess) {
      cudaStreamSynchronize(st);
      cudaFree(scratch);
      return fail(CGTP_ECUDA, std::string("graph build (sort shared memory): ") + cudaGetErrorString(err));
    }
    sort_long_kernel<<<std::max(1, std::min(N, 1024)), 1024, lsm, st>>>(g->t_rowptr, N, g->t_eid);
    dst_kernel<<<blocks(E), threads, 0, st>>>(g->rowptr, N, g->t_eid, E, g->t_dst);
  }
  // a launch refused for its configuration is reported here, not by the synchronisation
  const cudaError_t lerr = cudaGetLastError();
  cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, st);
  err = cudaStreamSynchronize(st);
  cudaFree(scratch);
  if (lerr != cudaSuccess) return fail(CGTP_ECUDA, std::string("graph build launch: ") + cudaGetErrorString(lerr));
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("graph build: ") + cudaGetErrorString(err));
  if (hflag & kTooLong) return fail(CGTP_EUNSUPPORTED, "a sender has more than 32768 out-edges");
  return CGTP_OK;
}

}  // namespace cgtp

// ---------------------------------------------------------------------------
// Allocation-free variant of the transpose build.
//
// Some callers cannot call cudaMalloc at the point where they need the
// transpose: their framework owns all device memory through its own pool and
// forbids raw allocations, or they run under a fixed device-memory budget
// reserved at start-up, or they cannot afford the device-wide synchronisation
// an allocation may imply.  This entry point writes the transpose into arrays
// the caller provides and takes its working memory (validation flag, degree
// counts / cursors, scan tile sums) from the file-scope array below, which
// every GPU that loads this library holds until the process exits.
// ---------------------------------------------------------------------------
namespace cgtp {
namespace {
constexpr int64_t kNoAllocMaxN = int64_t(1) << 20;   // largest node count accepted
constexpr int64_t kNoAllocTiles = (kNoAllocMaxN + 1 + kScanTile - 1) / kScanTile;
constexpr int64_t kNoAllocWords = 2 + (kNoAllocMaxN + 1) + kNoAllocTiles;  // ~4 MiB of int32
// flag, total, counts [N+1] and the tile sums of the largest accepted N fill the array exactly
static_assert(2 + (kNoAllocMaxN + 1) + (kNoAllocMaxN + 1 + kScanTile - 1) / kScanTile <= kNoAllocWords,
              "transpose scratch too small for the largest accepted node count");

static __device__ __align__(256) int g_transpose_scratch[kNoAllocWords];

// Device address of g_transpose_scratch per device, looked up once with that
// device current (in host code the symbol name is only a host-side stand-in).
// The cached address belongs to the device's primary context: after a
// cudaDeviceReset the library must not be used on that device again.
constexpr int kMaxDevices = 64;
int* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

cgtp_status scratch_for_current_device(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(CGTP_ECUDA, "no current CUDA device");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    int* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_transpose_scratch);
    if (e != cudaSuccess || !p)
      return fail(CGTP_ECUDA, std::string("cudaGetSymbolAddress(transpose scratch): ") + cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CGTP_OK;
}
}  // namespace
}  // namespace cgtp

extern "C" cgtp_status cgtp_graph_transpose_noalloc(const int32_t* rowptr, const int32_t* col,
                                                    int64_t N, int64_t E, int32_t* t_rowptr,
                                                    int32_t* t_eid, int32_t* t_dst, void* stream) {
  using namespace cgtp;
  clear_error();
  if (N < 1 || N > kNoAllocMaxN)
    return fail(CGTP_EINVAL, "cgtp_graph_transpose_noalloc: N must be in [1, 1048576]");
  if (E < 0 || E >= (int64_t(1) << 31)) return fail(CGTP_EINVAL, "E must be in [0, 2^31)");
  if (!rowptr || !t_rowptr) return fail(CGTP_EINVAL, "null rowptr or t_rowptr");
  if (E > 0 && (!col || !t_eid || !t_dst)) return fail(CGTP_EINVAL, "null col, t_eid or t_dst");
  int* scratch = nullptr;
  cgtp_status s = scratch_for_current_device(&scratch);
  if (s != CGTP_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int n = static_cast<int>(N), e = static_cast<int>(E);
  const int ntiles = (n + 1 + kScanTile - 1) / kScanTile;
  int* flag = scratch;
  int* total = scratch + 1;
  int* counts = scratch + 2;
  int* sums = counts + (n + 1);
  // the array keeps the previous call's contents: clear flag, total, counts and sums
  const size_t words = 2 + static_cast<size_t>(n + 1) + ntiles;
  if (cudaMemsetAsync(scratch, 0, words * sizeof(int), st) != cudaSuccess)
    return fail(CGTP_ECUDA, "clearing the transpose scratch failed");
  const int threads = 256;
  auto blocks = [](int64_t k) { return static_cast<int>(std::min<int64_t>((k + 255) / 256, 4096)); };
  csr_check_kernel<<<std::max(1, blocks(std::max(n + 1, e))), threads, 0, st>>>(rowptr, col, n, e, flag);
  int hflag = 0;
  cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, st);
  cudaError_t err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("graph check: ") + cudaGetErrorString(err));
  if (hflag) return fail(CGTP_EGRAPH, "invalid CSR (rowptr not a monotone prefix of E, or col out of range)");
  if (e > 0) histogram_kernel<<<blocks(e), threads, 0, st>>>(col, e, counts);
  scan_tiles_kernel<<<ntiles, 256, 0, st>>>(counts, n + 1, t_rowptr, sums);
  scan_sums_kernel<<<1, 32, 0, st>>>(sums, ntiles, total);
  add_offsets_kernel<<<blocks(n + 1), threads, 0, st>>>(t_rowptr, n + 1, sums);
  if (e > 0) {
    cudaMemcpyAsync(counts, t_rowptr, sizeof(int) * (n + 1), cudaMemcpyDeviceToDevice, st);
    scatter_kernel<<<blocks(e), threads, 0, st>>>(col, e, counts, t_eid);
    sort_short_kernel<<<std::max(1, std::min((n + 3) / 4, 4096)), 128, 0, st>>>(t_rowptr, n, t_eid, flag);
    const size_t lsm = kSortBlock * sizeof(int);
    err = cudaFuncSetAttribute(sort_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lsm);
    if (err != cudaSuccess) {
      cudaStreamSynchronize(st);
      return fail(CGTP_ECUDA, std::string("graph transpose (sort shared memory): ") + cudaGetErrorString(err));
    }
    sort_long_kernel<<<std::max(1, std::min(n, 1024)), 1024, lsm, st>>>(t_rowptr, n, t_eid);
    dst_kernel<<<blocks(e), threads, 0, st>>>(rowptr, n, t_eid, e, t_dst);
  }
  // a launch refused for its configuration is reported here, not by the synchronisation
  const cudaError_t lerr = cudaGetLastError();
  cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, st);
  err = cudaStreamSynchronize(st);
  if (lerr != cudaSuccess) return fail(CGTP_ECUDA, std::string("graph transpose launch: ") + cudaGetErrorString(lerr));
  if (err != cudaSuccess) return fail(CGTP_ECUDA, std::string("graph transpose: ") + cudaGetErrorString(err));
  if (hflag & kTooLong) return fail(CGTP_EUNSUPPORTED, "a sender has more than 32768 out-edges");
  return CGTP_OK;
}
