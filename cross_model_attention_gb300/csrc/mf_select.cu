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
//   select_kernel   one warp per BSR row: bitonic sort of the candidates in
//                   registers, fixed-point prefix sum by warp shuffles, kept
//                   list ascending by ballots and as an 8-word bit mask of
//                   the row; every candidate's tile index is reset to -1
//                   (the pack kernel fills in the kept ones).  The
//                   last CTA to finish computes row_ptr = exclusive scan of
//                   the kept counts (warp-aggregated: per-thread serial chunk,
//                   warp shuffles, one shared-memory pass over warp totals)
//   union_kernel    per block-row, the ascending union over sender heads of
//                   the kept block columns (the retrieval's iteration list)
//                   and the kept-tile table re-indexed by union position
#include "mf_internal.cuh"
#include "mf_ptx.cuh"
#include "mf_select_common.cuh"

namespace mf {
namespace {

constexpr int kSelThreads = 256;
constexpr int kMaxCand = 512;  // >= 256 blocks per row (non-causal worst case)

// Eight BSR rows per CTA (one per warp); the last CTA to finish also scans.
template <int E>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const CompressParams p) {
  constexpr int N = 32 * E;
  __shared__ int flag_s[kSelThreads / 32][N];
  const int warp = threadIdx.x >> 5;
  const int row = blockIdx.x * (kSelThreads / 32) + warp;  // h * R + rb
  if (row < p.H_s * p.R) select_row<E>(p, row, flag_s[warp]);
  // the last CTA to finish turns the kept counts into row_ptr
  __shared__ int last_s;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_s = (atomicAdd(p.sel_done, 1) == static_cast<int>(gridDim.x) - 1);
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  scan_counts<kSelThreads>(p);
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
  const int rows = p.H_s * p.R;
  const dim3 grid((rows + kSelThreads / 32 - 1) / (kSelThreads / 32));
  if (p.max_cand <= 32) select_kernel<1><<<grid, kSelThreads, 0, s>>>(p);
  else if (p.max_cand <= 64) select_kernel<2><<<grid, kSelThreads, 0, s>>>(p);
  else if (p.max_cand <= 128) select_kernel<4><<<grid, kSelThreads, 0, s>>>(p);
  else if (p.max_cand <= 256) select_kernel<8><<<grid, kSelThreads, 0, s>>>(p);
  else return cudaErrorInvalidValue;  // at most 256 blocks per sequence
  return cudaGetLastError();
}

cudaError_t launch_union(const CompressParams& p, cudaStream_t s) {
  union_kernel<<<p.R, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mf
