// mf_select_common.cuh — block-level top-p of one BSR row by one warp, and
// the row_ptr scan by one CTA (the selection kernel's building blocks).
//
// "Accelerating Cross-Model LLM Inference via Attention Map Reuse", section
// "Practical Implementation Details", bold header 3: per (head, block-row),
// keep the fewest blocks of largest mass whose sum reaches p of the row's
// total; ties go to the lower column, and the cumulative test is done in
// exact fixed point (mass * 2^32 rounded, threshold rint(p * 2^20) * total),
// so the result does not depend on the order of the additions.
#pragma once
#include <cstdint>

#include "mf_internal.cuh"

namespace mf {

// 64-bit shuffle (two 32-bit halves).
__device__ __forceinline__ unsigned long long shfl_xor64(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}
__device__ __forceinline__ unsigned long long shfl_up64(unsigned long long v, int d) {
  const uint32_t lo = __shfl_up_sync(0xffffffffu, static_cast<uint32_t>(v), d);
  const uint32_t hi = __shfl_up_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), d);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// One warp per BSR row (h, block-row); a CTA of 8 warps takes 8 rows.  The
// row's candidates (at most 32 * E) are held E per lane, element i = lane*E +
// e: 64-bit keys (inverted mass bits, column) are bitonic-sorted ascending in
// registers (shuffles across lanes, compare-exchange within a lane), then the
// fixed-point values in sorted order are prefix-summed with warp shuffles and
// the kept columns are compacted in ascending order with ballots.
template <int E>
__device__ __forceinline__ void select_row(const CompressParams& p, int row, int* flag) {
  constexpr int N = 32 * E;
  const int lane = threadIdx.x & 31;
  const int h = row / p.R, rb = row - h * p.R;
  const RowBlock rbk = p.rbs[rb];
  const int nb = (rbk.L + p.B - 1) / p.B;
  const int n = p.causal ? rbk.bi + 1 : nb;
  const float* mass = p.mass + static_cast<size_t>(h) * p.C + rbk.cand_off;
  for (int i = lane; i < n; i += 32) p.tile_of[static_cast<size_t>(rbk.cand_off + i) * p.H_s + h] = -1;

  unsigned long long key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane * E + e;
    if (i < n) {
      const uint32_t bits = __float_as_uint(mass[i]);  // masses are >= 0
      key[e] = (static_cast<unsigned long long>(0xFFFFFFFFu - bits) << 32) | static_cast<uint32_t>(i);
    } else {
      key[e] = ~0ull;
    }
  }
  for (int c = lane; c < N; c += 32) flag[c] = 0;
  // bitonic sort, ascending key == mass descending, column ascending
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = lane * E + e;
          const unsigned long long other = shfl_xor64(key[e], j / E);
          const bool up = (i & k) == 0, lower = (i & j) == 0;
          key[e] = (lower == up) ? (key[e] < other ? key[e] : other)
                                 : (key[e] < other ? other : key[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (e & j) continue;
          const int i = lane * E + e;
          const bool up = (i & k) == 0;
          const unsigned long long a = key[e], b = key[e | j];
          if ((a > b) == up) {
            key[e] = b;
            key[e | j] = a;
          }
        }
      }
    }
  }
  // fixed-point values in sorted order; inclusive prefix within the lane,
  // exclusive prefix of the lane totals across the warp
  unsigned long long incl[E];
  unsigned long long run = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    unsigned long long q = 0;
    if (key[e] != ~0ull) {
      const int bj = static_cast<int>(key[e] & 0xFFFFFFFFu);
      q = __double2ull_rn(static_cast<double>(mass[bj]) * 4294967296.0);
    }
    run += q;
    incl[e] = run;
  }
  unsigned long long scan = run;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long y = shfl_up64(scan, d);
    if (lane >= d) scan += y;
  }
  const unsigned long long lane_base = scan - run;  // exclusive over lanes
  const uint32_t tot_lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(scan), 31);
  const uint32_t tot_hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(scan >> 32), 31);
  const unsigned long long tot = (static_cast<unsigned long long>(tot_hi) << 32) | tot_lo;
  const unsigned long long thr = static_cast<unsigned long long>(
      __double2ull_rn(static_cast<double>(p.p) * 1048576.0)) * tot;
  __syncwarp();
  // position i is kept iff its exclusive prefix is still below the threshold
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (key[e] == ~0ull) continue;
    const unsigned long long excl = lane_base + (e == 0 ? 0ull : incl[e - 1]);
    if ((excl << 20) < thr) flag[static_cast<int>(key[e] & 0xFFFFFFFFu)] = 1;
  }
  __syncwarp();
  // compact the kept columns in ascending order
  int* out = p.keptcols + static_cast<size_t>(h) * p.C + rbk.cand_off;
  int cnt = 0;
  for (int c0 = 0; c0 < n; c0 += 32) {
    const int bj = c0 + lane;
    const bool f = (bj < n) && flag[bj];
    const uint32_t m = __ballot_sync(0xffffffffu, f);
    if (f) out[cnt + __popc(m & ((1u << lane) - 1u))] = bj;
    // the row's kept columns as a bit mask of 8 words
    if (lane == 0 && p.kmask) p.kmask[static_cast<size_t>(row) * 8 + (c0 >> 5)] = m;
    cnt += __popc(m);
  }
  if (lane == 0) {
    p.kcount[row] = cnt;
    if (p.kmask)
      for (int w = (n + 31) >> 5; w < 8; ++w) p.kmask[static_cast<size_t>(row) * 8 + w] = 0u;
  }
}

// row_ptr = exclusive scan of the kept counts, by one CTA of NT threads.
template <int NT>
__device__ __forceinline__ void scan_counts(const CompressParams& p) {
  constexpr int kScanThreads = NT;
  __shared__ long long wsum[kScanThreads / 32];
  __shared__ long long carry_s;
  if (threadIdx.x == 0 && p.pack_ctr) *p.pack_ctr = 0;  // the pack kernel's item counter
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
      constexpr int kWarps = kScanThreads / 32;
      long long w = (lane < kWarps) ? wsum[lane] : 0;
#pragma unroll
      for (int off = 1; off < kWarps; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      if (lane < kWarps) wsum[lane] = w;  // inclusive over warps
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

}  // namespace mf
