// mf_stats_common.cuh — helpers of the statistics kernels (mf_stats_tc.cu,
// mf_stats2_tc.cu): the item decode of the two-CTA kernel, the cross-lane sum
// of 32 per-lane vectors and the in-place rescale of a warp's TMEM partials.
#pragma once
#include <cstdint>

#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {

// The (128-row tile, head) of item idx: through the handle's statistics order
// table when there is one (sequence by sequence, heads in chunks whose keys fit
// in L2, heaviest tiles first within a chunk), else tile-major.
__device__ __forceinline__ void item_tile_head(const CompressParams& p, int idx, int& ti, int& h) {
  if (p.stats_items) {
    const int it = p.stats_items[idx];
    ti = it >> 8;
    h = it & 255;
  } else {
    ti = idx / p.H_s;
    h = idx % p.H_s;
  }
}

// Sum v[0..31] across the 32 lanes; on return lane l holds the total of
// element l.  31 shuffles instead of 32*5.
__device__ __forceinline__ float transpose_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

__device__ __forceinline__ void rescale_parts(uint32_t taddr, int ncols, float alpha) {
  int c = 0;
  for (; c + 16 <= ncols; c += 16) {
    uint32_t v[16];
    tmem_ld16(taddr + c, v);
    tc_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr + c),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
  }
  for (; c < ncols; ++c) {
    uint32_t v;
    tmem_ld1(taddr + c, v);
    tc_wait_ld();
    tmem_st1(taddr + c, __float_as_uint(__uint_as_float(v) * alpha));
  }
  tc_wait_st();
}

}  // namespace mf
