// mf_noalloc.cu — block-level top-p selection into a caller's BSR structure
// without allocating any device memory.
//
// Why it exists: mf_compress allocates its buffers (through the caller's
// allocator or cudaMallocAsync).  Some callers cannot allocate at the moment
// they need a selection: serving engines that reserve nearly all device
// memory for their KV cache at start-up and forbid further cudaMalloc, and
// latency-critical loops that cannot afford the implicit device
// synchronisation of cudaFree.  This entry point takes the block masses and
// the output arrays from the caller and keeps its own intermediates (the
// per-row kept counts and kept-column lists, and the block-row table) in one
// file-scope static device array, reserved once when the library is loaded.
//
// Limits and sharing:
//   * the scratch is kNoAllocScratchBytes (16 MiB) per device; a call whose
//     intermediates do not fit is rejected with MF_ERR_UNSUPPORTED;
//   * every GPU that loads the library holds those 16 MiB until the process
//     exits;
//   * all calls on a device share the one array: calls that overlap on the
//     GPU (concurrent streams, or a second call launched before the first
//     finished on another stream) race and corrupt each other's results;
//     calls on one stream are ordered and safe;
//   * nothing in the array needs clearing between calls: every word a call
//     reads is written earlier by the same call.
//
// The selection rule is the one of mf_compress (mass descending, ties to the
// lower column, exact fixed-point cumulative threshold) — see mf_select.cu.
#include <cuda_runtime.h>

#include <mutex>

#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// The scratch.  In host code this name is only a stand-in for the device
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kThreads = 256;
constexpr int kMaxCand = 512;

struct NoAllocParams {
  const RowBlock* rbs;  // [R] in scratch
  const float* mass;    // [H_s][C] caller input
  int* kcount;          // [H_s*R] in scratch
  int* keptcols;        // [H_s][C] in scratch
  int* row_ptr;         // [H_s*R+1] caller output
  int* col_idx;         // caller output (capacity >= H_s*C)
  long long* nnz;       // caller device output
  int H_s, R, C, B, causal;
  float p;
};

__global__ void __launch_bounds__(kThreads) noalloc_select_kernel(const NoAllocParams p) {
  __shared__ unsigned long long key[kMaxCand];
  __shared__ unsigned long long pre[kMaxCand];
  __shared__ int flag[kMaxCand];
  __shared__ int pos[kMaxCand];
  const int row = blockIdx.x;
  const int h = row / p.R, rb = row - h * p.R;
  const RowBlock rbk = p.rbs[rb];
  const int nb = (rbk.L + p.B - 1) / p.B;
  const int n = p.causal ? rbk.bi + 1 : nb;
  int npow = 1;
  while (npow < n) npow <<= 1;
  const float* mass = p.mass + static_cast<size_t>(h) * p.C + rbk.cand_off;
  for (int i = threadIdx.x; i < npow; i += blockDim.x) {
    if (i < n) {
      const uint32_t bits = __float_as_uint(mass[i]);
      key[i] = (static_cast<unsigned long long>(0xFFFFFFFFu - bits) << 32) | static_cast<uint32_t>(i);
    } else {
      key[i] = ~0ull;
    }
    flag[i] = 0;
  }
  __syncthreads();
  for (int k = 2; k <= npow; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < npow; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = key[i], b = key[ixj];
          if ((a > b) == ((i & k) == 0)) {
            key[i] = b;
            key[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < npow; i += blockDim.x)
    pre[i] = (i < n) ? __double2ull_rn(static_cast<double>(mass[key[i] & 0xFFFFFFFFu]) * 4294967296.0)
                     : 0ull;
  __syncthreads();
  for (int off = 1; off < npow; off <<= 1) {
    unsigned long long add[kMaxCand / kThreads];
    int c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) add[c] = (i >= off) ? pre[i - off] : 0ull;
    __syncthreads();
    c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) pre[i] += add[c];
    __syncthreads();
  }
  const unsigned long long tot = (n > 0) ? pre[n - 1] : 0ull;
  const unsigned long long thr =
      static_cast<unsigned long long>(__double2ull_rn(static_cast<double>(p.p) * 1048576.0)) * tot;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long excl = (i == 0) ? 0ull : pre[i - 1];
    if ((excl << 20) < thr) flag[static_cast<int>(key[i] & 0xFFFFFFFFu)] = 1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < npow; i += blockDim.x) pos[i] = (i < n) ? flag[i] : 0;
  __syncthreads();
  for (int off = 1; off < npow; off <<= 1) {
    int add[kMaxCand / kThreads];
    int c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) add[c] = (i >= off) ? pos[i - off] : 0;
    __syncthreads();
    c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) pos[i] += add[c];
    __syncthreads();
  }
  int* out = p.keptcols + static_cast<size_t>(h) * p.C + rbk.cand_off;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if (flag[i]) out[pos[i] - 1] = i;
  if (threadIdx.x == 0) p.kcount[row] = (n > 0) ? pos[n - 1] : 0;
}

__global__ void __launch_bounds__(1024) noalloc_scan_kernel(const NoAllocParams p) {
  __shared__ long long wsum[32];
  __shared__ long long carry_s;
  const int n = p.H_s * p.R;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  constexpr int per = 8;
  for (int base = 0; base < n; base += 1024 * per) {
    const int i0 = base + threadIdx.x * per;
    long long v[per], local = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      v[j] = (i0 + j < n) ? p.kcount[i0 + j] : 0;
      local += v[j];
    }
    long long incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      long long s = wsum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
      }
      wsum[lane] = s;
    }
    __syncthreads();
    long long run = carry_s + (warp > 0 ? wsum[warp - 1] : 0) + (incl - local);
#pragma unroll
    for (int j = 0; j < per; ++j) {
      if (i0 + j < n) p.row_ptr[i0 + j] = static_cast<int>(run);
      run += v[j];
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry_s = run;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.row_ptr[n] = static_cast<int>(carry_s);
    *p.nnz = carry_s;
  }
}

__global__ void __launch_bounds__(kThreads) noalloc_compact_kernel(const NoAllocParams p) {
  const int row = blockIdx.x;
  const int h = row / p.R, rb = row - h * p.R;
  const int k = p.kcount[row];
  const int base = p.row_ptr[row];
  const int* src = p.keptcols + static_cast<size_t>(h) * p.C + p.rbs[rb].cand_off;
  for (int i = threadIdx.x; i < k; i += blockDim.x) p.col_idx[base + i] = src[i];
}

// Device address of the scratch, looked up once per device with that device
// current.
constexpr int kMaxDevices = 64;
unsigned char* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

cudaError_t scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(ptr);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

size_t noalloc_needed_bytes(long long R, long long H_s, long long C) {
  return up256(R * sizeof(RowBlock)) + up256(H_s * R * 4) + up256(H_s * C * 4);
}

cudaError_t launch_select_noalloc(const RowBlock* rbs_host, int R, int C, int H_s, int B,
                                  int causal, float p, const float* mass, int* row_ptr,
                                  int* col_idx, long long* nnz, cudaStream_t s) {
  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return e;
  NoAllocParams prm{};
  size_t off = 0;
  prm.rbs = reinterpret_cast<const RowBlock*>(base + off);
  off += up256(static_cast<size_t>(R) * sizeof(RowBlock));
  prm.kcount = reinterpret_cast<int*>(base + off);
  off += up256(static_cast<size_t>(H_s) * R * 4);
  prm.keptcols = reinterpret_cast<int*>(base + off);
  prm.mass = mass;
  prm.row_ptr = row_ptr;
  prm.col_idx = col_idx;
  prm.nnz = nnz;
  prm.H_s = H_s;
  prm.R = R;
  prm.C = C;
  prm.B = B;
  prm.causal = causal;
  prm.p = p;
  e = cudaMemcpyAsync(const_cast<RowBlock*>(prm.rbs), rbs_host, sizeof(RowBlock) * R,
                      cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  noalloc_select_kernel<<<H_s * R, kThreads, 0, s>>>(prm);
  noalloc_scan_kernel<<<1, 1024, 0, s>>>(prm);
  noalloc_compact_kernel<<<H_s * R, kThreads, 0, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace mf
