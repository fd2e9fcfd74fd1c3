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
// This kernel accumulates the Gram matrix of the stacked rows [sender heads;
// receiver heads] over the candidate blocks (both BSRs share one block grid);
// the host sums the CTAs' partials in fp64 and solves the small system.
//
// CTA = persistent walker of candidate blocks.  Per block, the tiles of every
// row (the block's kept tile, or zeros where the head dropped it) come through
// shared memory 512 elements at a time, transposed to [element][row] so that
// each thread's reads are contiguous; each of the 256 threads accumulates a
// 6 x 6 patch of the (up to) 96 x 96 Gram matrix in fp32 registers.
#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kNR = kCalibRows;  // rows of the Gram matrix (sender + receiver heads)
constexpr int kChunk = 512;      // block elements per pass
constexpr int kThreads = 256;    // 16 x 16 patches of 6 x 6
constexpr int kPatch = 6;
static_assert(16 * kPatch == kNR, "patch grid covers the rows");

__global__ void __launch_bounds__(kThreads) calib_gram_kernel(const CalibParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);             // [kChunk][kNR] bf16 bits
  int* tix = reinterpret_cast<int*>(smem_raw + kChunk * kNR * 2);   // [kNR] tile of each row
  const int nr = p.H_s + p.H_r;
  const int r0 = kPatch * (threadIdx.x / 16), c0 = kPatch * (threadIdx.x % 16);
  const int BB = p.B * p.B;
  float acc[kPatch][kPatch];
#pragma unroll
  for (int i = 0; i < kPatch; ++i)
#pragma unroll
    for (int j = 0; j < kPatch; ++j) acc[i][j] = 0.f;

  for (int c = blockIdx.x; c < p.C; c += gridDim.x) {
    __syncthreads();  // the previous block's tiles are consumed
    for (int r = threadIdx.x; r < kNR; r += kThreads) {
      int t = -1;
      if (r < p.H_s) t = p.s_tile_of[static_cast<size_t>(c) * p.H_s + r];
      else if (r < nr) t = p.r_tile_of[static_cast<size_t>(c) * p.H_r + (r - p.H_s)];
      tix[r] = t;
    }
    __syncthreads();
    for (int e0 = 0; e0 < BB; e0 += kChunk) {
      if (e0 > 0) __syncthreads();  // the previous chunk is consumed
      // 16-byte loads: consecutive threads take consecutive rows of one
      // 8-element group, so the transposed shared-memory stores do not collide
      for (int idx = threadIdx.x; idx < kNR * (kChunk / 8); idx += kThreads) {
        const int r = idx % kNR, q = idx / kNR;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        const int t = tix[r];
        if (t >= 0) {
          const uint16_t* src = ((r < p.H_s) ? p.s_values : p.r_values) + static_cast<size_t>(t) * BB + e0 + q * 8;
          v = *reinterpret_cast<const uint4*>(src);
        }
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xs[(q * 8 + 2 * j) * kNR + r] = static_cast<uint16_t>(w[j] & 0xFFFFu);
          xs[(q * 8 + 2 * j + 1) * kNR + r] = static_cast<uint16_t>(w[j] >> 16);
        }
      }
      __syncthreads();
#pragma unroll 4
      for (int k = 0; k < kChunk; ++k) {
        const uint32_t* row = reinterpret_cast<const uint32_t*>(xs + k * kNR);
        float a[kPatch], b[kPatch];
#pragma unroll
        for (int i = 0; i < kPatch; i += 2) {
          const uint32_t wa = row[(r0 + i) >> 1], wb = row[(c0 + i) >> 1];
          a[i] = bf16lo(wa);
          a[i + 1] = bf16hi(wa);
          b[i] = bf16lo(wb);
          b[i + 1] = bf16hi(wb);
        }
#pragma unroll
        for (int i = 0; i < kPatch; ++i)
#pragma unroll
          for (int j = 0; j < kPatch; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
    }
  }
  float* out = p.partial + static_cast<size_t>(blockIdx.x) * kNR * kNR;
#pragma unroll
  for (int i = 0; i < kPatch; ++i)
#pragma unroll
    for (int j = 0; j < kPatch; ++j) out[(r0 + i) * kNR + c0 + j] = acc[i][j];
}

}  // namespace

int calib_grid() {
  int sms = 0;
  if (sm_count(&sms) != cudaSuccess || sms < 1) sms = 1;
  return 2 * sms;
}

cudaError_t launch_calib_gram(const CalibParams& p, int grid, cudaStream_t s) {
  const int smem = kChunk * kNR * 2 + kNR * 4;
  cudaError_t e = cudaFuncSetAttribute(calib_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  calib_gram_kernel<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mf
