// mf_calibrate.cu — Gram matrices of the head-map calibration, sm_103a.
//
// "Accelerating Cross-Model LLM Inference via Attention Map Reuse", section
// "MapFlow System Design", item 3: the receiver's attention map of a reused
// layer is a linear transformation of the mapped sender layer's head maps,
// with the weights fitted offline.  Reading: least squares over every map
// entry, with each map as its BSR stores it (dropped blocks are zero), i.e.
// the normal equations G W^T = C^T with
//   G[h][h'] = sum over entries of P_h * P_h'   (sender heads h, h')
//   C[i][h]  = sum over entries of A_i * P_h    (receiver heads i)
// Both are blocks of the Gram matrix X X^T of the stacked rows X = [sender
// heads; receiver heads] (at most 96) over all map entries, a dense
// contraction with the entries as the reduction dimension.
//
// calib_gram_tc_kernel: persistent CTAs walk the candidate blocks (both BSRs
// share one block grid).  Four loader warps gather, per stage, 64 entries of
// every row (the row's kept tile, or zeros where the head dropped the block)
// with 16-byte cp.async into a 128-row, 128-byte-swizzled K-major tile; one
// thread issues tcgen05.mma M=128, N=rows (rounded up to 16), K=16 with that
// one tile as both operands, accumulating X X^T in TMEM (fp32) across all of
// the CTA's blocks.  The epilogue writes the CTA's partial matrix;
// calib_reduce_kernel sums the partials in a fixed order in fp64.
#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kNR = kCalibRows;            // rows of the Gram matrix (sender + receiver heads)
constexpr int kStages = 6;
constexpr int kStageBytes = 128 * 128;     // 128 rows x 64 bf16, 128-byte swizzle
constexpr int kLoaders = 128;              // warps 0..3
constexpr int kThreads = kLoaders + 32;    // + the MMA warp
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarDone = 2 * kStages, kNumBars = 2 * kStages + 1;
constexpr int kOffTix = kStages * kStageBytes;
constexpr int kOffBars = kOffTix + kNR * 4;
constexpr int kOffSlot = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffSlot + 16 + 1024;  // + alignment slack
static_assert(kOffBars % 8 == 0, "mbarriers are 8-byte aligned");

__global__ void __launch_bounds__(kThreads) calib_gram_tc_kernel(const CalibParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  int* tix = reinterpret_cast<int*>(smem + kOffTix);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  auto bar = [&](int i) { return sb + kOffBars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nr = p.H_s + p.H_r;
  const int npad = ((nr + 15) / 16) * 16;
  const int BB = p.B * p.B;
  const int per_block = BB / 64;  // stages per candidate block
  const int n_my = (p.C > static_cast<int>(blockIdx.x)) ? (p.C - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int n_stages = n_my * per_block;

  // rows no head fills stay zero in every stage (finite padding rows)
  for (int i = threadIdx.x; i < kStages * kStageBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), kLoaders);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    mbar_init(bar(kBarDone), 1);
    fence_mbar_init();
  }
  fence_async_smem();
  if (warp == 0) tmem_alloc(smem_u32(tslot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp < 4) {
    // ------------------------------------------------------------ loaders
    bool ok = true;
    int u = 0;
    for (int c = blockIdx.x; ok && c < p.C; c += gridDim.x) {
      named_bar(1, kLoaders);  // every copy of the previous block is issued
      if (threadIdx.x < nr) {
        const int r = threadIdx.x;
        tix[r] = (r < p.H_s) ? p.s_tile_of[static_cast<size_t>(c) * p.H_s + r]
                             : p.r_tile_of[static_cast<size_t>(c) * p.H_r + (r - p.H_s)];
      }
      named_bar(1, kLoaders);
      for (int s = 0; s < per_block; ++s, ++u) {
        const int st = u % kStages;
        int good = 1;
        if (lane == 0) good = mbar_wait(bar(kBarEmpty + st), ((u / kStages) & 1) ^ 1, p.err) ? 1 : 0;
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        const uint32_t dst0 = sb + st * kStageBytes;
        for (int i = threadIdx.x; i < nr * 8; i += kLoaders) {
          const int r = i >> 3, ch = i & 7;
          const int t = tix[r];
          const uint16_t* base = (r < p.H_s) ? p.s_values : p.r_values;
          const uint16_t* src = base + static_cast<size_t>(t >= 0 ? t : 0) * BB + s * 64 + ch * 8;
          cp_async16(dst0 + sw128_off(r, ch), src, t >= 0 ? 16u : 0u);  // a dropped head is zero
        }
        cp_async_arrive(bar(kBarFull + st));
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (lane == 0 && n_stages > 0) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, npad, false, false);
    for (int u = 0; u < n_stages; ++u) {
      const int st = u % kStages;
      if (!mbar_wait(bar(kBarFull + st), (u / kStages) & 1, p.err)) break;
      fence_async_smem();  // the tile was written by cp.async (generic proxy)
      tc_fence_after();
      const uint32_t a = sb + st * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t d = sdesc_sw128(a + kk * 32, 16, 1024);
        tc_mma(tmem, d, d, idesc, (u > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(bar(kBarEmpty + st));
    }
    tc_commit(bar(kBarDone));  // arrives once every MMA issued above is complete
  }

  if (warp < 4) {
    // ----------------------------------------- epilogue: TMEM -> partials
    float* out = p.partial + static_cast<size_t>(blockIdx.x) * kNR * kNR;
    const int row = warp * 32 + lane;
    bool have = n_stages > 0;
    if (have) {
      int good = 1;
      if (lane == 0) good = mbar_wait(bar(kBarDone), 0, p.err) ? 1 : 0;
      have = __shfl_sync(0xffffffffu, good, 0) != 0;
    }
    tc_fence_after();
    for (int c0 = 0; c0 < npad; c0 += 32) {
      uint32_t x[32];
      if (have) {
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, x);
        tc_wait_ld();
      }
      if (row < nr) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < nr) out[row * kNR + c0 + j] = have ? __uint_as_float(x[j]) : 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// G[i][j] = sum over CTAs b (in order) of partial[b][i][j], in fp64.
__global__ void __launch_bounds__(256) calib_reduce_kernel(const float* __restrict__ partial, int grid, int n,
                                                           double* __restrict__ G) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * n) return;
  const int i = idx / n, j = idx - i * n;
  double acc = 0.0;
  for (int b = 0; b < grid; ++b) acc += static_cast<double>(partial[(static_cast<size_t>(b) * kNR + i) * kNR + j]);
  G[idx] = acc;
}

}  // namespace

int calib_grid(int C) {
  int sms = 0;
  if (sm_count(&sms) != cudaSuccess || sms < 1) sms = 1;
  return std::max(1, std::min(C, 2 * sms));
}

cudaError_t launch_calib_gram(const CalibParams& p, int grid, double* G, cudaStream_t s) {
  if (p.B * p.B % 64 != 0 || p.H_s + p.H_r > kNR) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(calib_gram_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  calib_gram_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = p.H_s + p.H_r;
  calib_reduce_kernel<<<(n * n + 255) / 256, 256, 0, s>>>(p.partial, grid, n, G);
  return cudaGetLastError();
}

}  // namespace mf
