// mf_select.cu — Attention State Compressor, step 2 (block selection) and the
// BSR bookkeeping around it.
//
// Block-level top-p ("Accelerating Cross-Model LLM Inference via Attention
// Map Reuse", section "Practical Implementation Details" and bold header 3:
// keep the blocks needed to reach cumulative probability p): per (head,
// block-row), candidates are sorted by mass descending with ties to the lower
// block column, and the shortest prefix whose cumulative mass reaches p of the
// row total is kept.  The cumulative sum and the comparison are done exactly
// in 64-bit fixed point so the decision is independent of summation order:
//   q_b = rint(mass_b * 2^32), Tot = sum_b q_b, P_q = rint(p * 2^20),
//   keep the smallest k with 2^20 * sum_{t<k} q_(t) >= P_q * Tot.
// (Every mass is <= B <= 128, so Tot < 2^40 and both sides stay below 2^60.)
//
// Kernels here:
//   select_kernel   one CTA per BSR row: bitonic sort of the candidates in
//                   shared memory, fixed-point prefix sum, kept list ascending
//   scan_kernel     row_ptr = exclusive scan of the kept counts (single CTA,
//                   warp-aggregated: per-thread serial chunk, warp shuffles,
//                   one shared-memory pass over warp totals)
//   union_kernel    per block-row, the ascending union over sender heads of
//                   the kept block columns (the retrieval's iteration list)
//                   and the kept-tile table re-indexed by union position
#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kSelThreads = 256;
constexpr int kMaxCand = 512;  // >= 256 blocks per row (non-causal worst case)

__global__ void __launch_bounds__(kSelThreads) select_kernel(const CompressParams p) {
  __shared__ unsigned long long key[kMaxCand];
  __shared__ unsigned long long pre[kMaxCand];
  __shared__ int flag[kMaxCand];
  const int row = blockIdx.x;            // h * R + rb
  const int h = row / p.R, rb = row - h * p.R;
  const RowBlock rbk = p.rbs[rb];
  const int nb = (rbk.L + p.B - 1) / p.B;
  const int n = p.causal ? rbk.bi + 1 : nb;
  int npow = 1;
  while (npow < n) npow <<= 1;
  const float* mass = p.mass + static_cast<size_t>(h) * p.C + rbk.cand_off;

  for (int i = threadIdx.x; i < npow; i += blockDim.x) {
    if (i < n) {
      const uint32_t bits = __float_as_uint(mass[i]);  // masses are >= 0
      key[i] = (static_cast<unsigned long long>(0xFFFFFFFFu - bits) << 32) | static_cast<uint32_t>(i);
    } else {
      key[i] = ~0ull;
    }
    flag[i] = 0;
  }
  __syncthreads();
  // bitonic sort, ascending key == mass descending, column ascending
  for (int k = 2; k <= npow; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < npow; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = key[i], b = key[ixj];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            key[i] = b;
            key[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // fixed-point values in sorted order and their inclusive prefix sum
  for (int i = threadIdx.x; i < npow; i += blockDim.x) {
    unsigned long long q = 0;
    if (i < n) {
      const int bj = static_cast<int>(key[i] & 0xFFFFFFFFu);
      q = __double2ull_rn(static_cast<double>(mass[bj]) * 4294967296.0);
    }
    pre[i] = q;
  }
  __syncthreads();
  for (int off = 1; off < npow; off <<= 1) {
    unsigned long long add[kMaxCand / kSelThreads];
    int c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) add[c] = (i >= off) ? pre[i - off] : 0ull;
    __syncthreads();
    c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) pre[i] += add[c];
    __syncthreads();
  }
  const unsigned long long tot = (n > 0) ? pre[n - 1] : 0ull;
  const unsigned long long thr = static_cast<unsigned long long>(
      __double2ull_rn(static_cast<double>(p.p) * 1048576.0)) * tot;
  // position i is kept iff its exclusive prefix is still below the threshold
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long excl = (i == 0) ? 0ull : pre[i - 1];
    if ((excl << 20) < thr) flag[static_cast<int>(key[i] & 0xFFFFFFFFu)] = 1;
  }
  __syncthreads();
  // compact kept columns in ascending order (n <= 512: one thread per pair)
  __shared__ int pos[kMaxCand];
  for (int i = threadIdx.x; i < npow; i += blockDim.x) pos[i] = (i < n) ? flag[i] : 0;
  __syncthreads();
  for (int off = 1; off < npow; off <<= 1) {
    int add[kMaxCand / kSelThreads];
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

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) scan_kernel(const CompressParams p) {
  __shared__ long long wsum[kScanThreads / 32];
  __shared__ long long carry_s;
  const int n = p.H_s * p.R;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  // process in rounds of kScanThreads * per-thread chunk
  const int per = 8;
  for (int base = 0; base < n; base += kScanThreads * per) {
    const int i0 = base + threadIdx.x * per;
    long long v[per];
    long long local = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      v[j] = (i0 + j < n) ? p.kcount[i0 + j] : 0;
      local += v[j];
    }
    // warp-level inclusive scan of per-thread totals
    long long incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      long long w = wsum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    long long run = carry_s + (warp > 0 ? wsum[warp - 1] : 0) + (incl - local);
#pragma unroll
    for (int j = 0; j < per; ++j) {
      if (i0 + j < n) p.row_ptr[i0 + j] = static_cast<int>(run);
      run += v[j];
    }
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) carry_s = run;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.row_ptr[n] = static_cast<int>(carry_s);
    *p.nnz_out = carry_s;
  }
}

// One CTA per global block-row: union over heads of the kept columns.
__global__ void __launch_bounds__(256) union_kernel(const CompressParams p) {
  __shared__ int flag[kMaxCand];
  __shared__ int pos[kMaxCand];
  const int rb = blockIdx.x;
  const RowBlock rbk = p.rbs[rb];
  const int nb = (rbk.L + p.B - 1) / p.B;
  const int n = p.causal ? rbk.bi + 1 : nb;
  int npow = 1;
  while (npow < n) npow <<= 1;
  for (int i = threadIdx.x; i < npow; i += blockDim.x) {
    int f = 0;
    if (i < n) {
      const int* t = p.tile_of + static_cast<size_t>(rbk.cand_off + i) * p.H_s;
      for (int hh = 0; hh < p.H_s; ++hh) f |= (t[hh] >= 0);
    }
    flag[i] = f;
    pos[i] = f;
  }
  __syncthreads();
  for (int off = 1; off < npow; off <<= 1) {
    int add[kMaxCand / 256];
    int c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) add[c] = (i >= off) ? pos[i - off] : 0;
    __syncthreads();
    c = 0;
    for (int i = threadIdx.x; i < npow; i += blockDim.x, ++c) pos[i] += add[c];
    __syncthreads();
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if (flag[i]) p.union_list[rbk.cand_off + pos[i] - 1] = i;
  if (threadIdx.x == 0) p.union_cnt[rb] = (n > 0) ? pos[n - 1] : 0;
  // the kept tiles again, in union order, so that a consumer walking the
  // union needs one independent load per block instead of two dependent ones
  for (int x = threadIdx.x; x < n * p.H_s; x += blockDim.x) {
    const int i = x / p.H_s, hh = x - i * p.H_s;
    if (flag[i])
      p.utile[static_cast<size_t>(rbk.cand_off + pos[i] - 1) * p.H_s + hh] =
          p.tile_of[static_cast<size_t>(rbk.cand_off + i) * p.H_s + hh];
  }
}

// One thread waits on an mbarrier that expects one arrival nobody makes; the
// bounded wait gives up after `limit_ns` and records the timeout.
__global__ void selftest_wait_kernel(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  mbar_wait(b, 0, err, limit_ns);
}

}  // namespace

cudaError_t launch_selftest_wait(int* err, unsigned long long limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 1, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_select(const CompressParams& p, cudaStream_t s) {
  select_kernel<<<p.H_s * p.R, kSelThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_scan(const CompressParams& p, cudaStream_t s) {
  scan_kernel<<<1, kScanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_union(const CompressParams& p, cudaStream_t s) {
  union_kernel<<<p.R, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mf
