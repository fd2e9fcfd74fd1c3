// mf_f32.cu — fp32 inputs: compressor statistics, BSR pack and retrieval on
// CUDA cores.
//
// The tensor-core path is bf16; an fp32 sender (Q, K) or receiver (V, W, O)
// keeps fp32 arithmetic end to end (TF32 would lose ~1e-3 on the logits), so
// these kernels use plain fp32 FMA.  The method is the same as the bf16 path
// ("Accelerating Cross-Model LLM Inference via Attention Map Reuse",
// "Practical Implementation Details"; "北大MapFlow：注意力图跨模型复用，
// prefill延迟降15%–20%", paragraphs "其一" and "其三"); the BSR tiles are bf16
// in both paths.
//
//   stats_f32   CTA = (block-row, head), one thread per query row: online
//               max/sum over the visible keys, then a second pass for the
//               exact block masses
//   pack_f32    CTA = (block-row, head): recompute and store the kept tiles
//   retrieve_f32 CTA = (block-row, receiver head): per union block, A_hat in
//               shared memory (fp32), then O += A_hat . V
#include <cmath>
#include <type_traits>

#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

template <int D, int BLK>
__global__ void __launch_bounds__(BLK) stats_f32_kernel(const CompressParams p,
                                                        const float* __restrict__ q,
                                                        const float* __restrict__ k) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && p.sel_done) *p.sel_done = 0;
  __shared__ float sk[BLK * D];
  __shared__ float red[BLK];
  const int rb = blockIdx.x, h = blockIdx.y;
  const int hk = h / (p.H_s / p.H_ks);
  const RowBlock rbk = p.rbs[rb];
  const int row = threadIdx.x;
  const int il = rbk.bi * BLK + row;
  const bool ok = il < rbk.L;
  const int nb = (rbk.L + BLK - 1) / BLK;
  const int ncand = p.causal ? rbk.bi + 1 : nb;
  const float scale = rsqrtf(static_cast<float>(D));
  float qr[D];
#pragma unroll
  for (int c = 0; c < D; ++c)
    qr[c] = ok ? q[(static_cast<size_t>(rbk.seq_start + il) * p.H_s + h) * D + c] : 0.f;
  auto load_k = [&](int bj) {
    __syncthreads();
    for (int e = threadIdx.x; e < BLK * D; e += BLK) {
      const int r = e / D, c = e - r * D;
      const int j = bj * BLK + r;
      sk[e] = (j < rbk.L) ? k[(static_cast<size_t>(rbk.seq_start + j) * p.H_ks + hk) * D + c] : 0.f;
    }
    __syncthreads();
  };
  auto logit = [&](int c) {
    float s = 0.f;
#pragma unroll
    for (int t = 0; t < D; ++t) s = fmaf(qr[t], sk[c * D + t], s);
    return s * scale;
  };
  float m = -INFINITY, l = 0.f;
  for (int bj = 0; bj < ncand; ++bj) {
    load_k(bj);
    for (int c = 0; c < BLK; ++c) {
      const int j = bj * BLK + c;
      if (ok && j < rbk.L && (!p.causal || j <= il)) {
        const float s = logit(c);
        if (s > m) {
          l = l * expf(m - s) + 1.f;
          m = s;
        } else {
          l += expf(s - m);
        }
      }
    }
  }
  const float invl = (ok && l > 0.f) ? 1.f / l : 0.f;
  for (int bj = 0; bj < ncand; ++bj) {
    load_k(bj);
    float bs = 0.f;
    for (int c = 0; c < BLK; ++c) {
      const int j = bj * BLK + c;
      if (ok && j < rbk.L && (!p.causal || j <= il)) bs += expf(logit(c) - m) * invl;
    }
    red[row] = bs;
    __syncthreads();
    if (row == 0) {
      float t = 0.f;
      for (int r = 0; r < BLK; ++r) t += red[r];
      p.mass[static_cast<size_t>(h) * p.C + rbk.cand_off + bj] = t;
    }
  }
  if (ok) {
    const size_t o = static_cast<size_t>(h) * p.T + rbk.seq_start + il;
    p.row_max[o] = m;
    p.row_sum[o] = l;
  }
}

template <int D, int BLK>
__global__ void __launch_bounds__(BLK) pack_f32_kernel(const CompressParams p,
                                                       const float* __restrict__ q,
                                                       const float* __restrict__ k,
                                                       __nv_bfloat16* __restrict__ values) {
  __shared__ float sk[BLK * D];
  const int rb = blockIdx.x, h = blockIdx.y;
  const int hk = h / (p.H_s / p.H_ks);
  const RowBlock rbk = p.rbs[rb];
  const int row = threadIdx.x;
  const int il = rbk.bi * BLK + row;
  const bool ok = il < rbk.L;
  const int brow = h * p.R + rb;
  const int kc = p.kcount[brow];
  const int base = p.row_ptr[brow];
  const int* kl = p.keptcols + static_cast<size_t>(h) * p.C + rbk.cand_off;
  const float scale = rsqrtf(static_cast<float>(D));
  float qr[D];
#pragma unroll
  for (int c = 0; c < D; ++c)
    qr[c] = ok ? q[(static_cast<size_t>(rbk.seq_start + il) * p.H_s + h) * D + c] : 0.f;
  float m = 0.f, invl = 0.f;
  if (ok) {
    const size_t o = static_cast<size_t>(h) * p.T + rbk.seq_start + il;
    m = p.row_max[o];
    invl = 1.f / p.row_sum[o];
  }
  for (int t = 0; t < kc; ++t) {
    const int bj = kl[t];
    if (row == 0) {
      p.col_idx[base + t] = bj;
      p.tile_of[static_cast<size_t>(rbk.cand_off + bj) * p.H_s + h] = base + t;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < BLK * D; e += BLK) {
      const int r = e / D, c = e - r * D;
      const int j = bj * BLK + r;
      sk[e] = (j < rbk.L) ? k[(static_cast<size_t>(rbk.seq_start + j) * p.H_ks + hk) * D + c] : 0.f;
    }
    __syncthreads();
    __nv_bfloat16* dst = values + (static_cast<size_t>(base + t) * BLK + row) * BLK;
    for (int c = 0; c < BLK; ++c) {
      const int j = bj * BLK + c;
      float v = 0.f;
      if (ok && j < rbk.L && (!p.causal || j <= il)) {
        float s = 0.f;
#pragma unroll
        for (int tt = 0; tt < D; ++tt) s = fmaf(qr[tt], sk[c * D + tt], s);
        v = expf(s * scale - m) * invl;
      }
      dst[c] = __float2bfloat16_rn(v);
    }
  }
}

template <int D, int BLK>
__global__ void __launch_bounds__(256) retrieve_f32_kernel(const RetrieveParams p,
                                                           const uint16_t* __restrict__ values,
                                                           const float* __restrict__ v,
                                                           float* __restrict__ o) {
  extern __shared__ float sa[];  // A_hat tile [BLK][BLK]
  constexpr int kPer = BLK * D / 256;
  const int rb = blockIdx.x, i = blockIdx.y;
  const RowBlock rbk = p.rbs[rb];
  const int hpg = p.H_r / p.H_kv;
  const int g = i / hpg;
  const int nu = p.union_cnt[rb];
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int u = 0; u < nu; ++u) {
    const int bj = p.union_list[rbk.cand_off + u];
    const int* trow = p.tile_of + static_cast<size_t>(rbk.cand_off + bj) * p.H_s;
    __syncthreads();
    for (int e = threadIdx.x; e < BLK * BLK; e += 256) {
      float a = 0.f;
      for (int hh = 0; hh < p.H_s; ++hh) {
        const int tix = trow[hh];
        if (tix >= 0) {
          const uint32_t bits = values[static_cast<size_t>(tix) * BLK * BLK + e];
          a = fmaf(p.W[static_cast<size_t>(i) * p.H_s + hh], __uint_as_float(bits << 16), a);
        }
      }
      sa[e] = a;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int idx = threadIdx.x + 256 * e;
      const int r = idx / D, dd = idx - r * D;
      float s = acc[e];
      for (int c = 0; c < BLK; ++c) {
        const int j = bj * BLK + c;
        const float vv = (j < rbk.L) ? v[(static_cast<size_t>(rbk.seq_start + j) * p.H_kv + g) * D + dd] : 0.f;
        s = fmaf(sa[r * BLK + c], vv, s);
      }
      acc[e] = s;
    }
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int idx = threadIdx.x + 256 * e;
    const int r = idx / D, dd = idx - r * D;
    const int il = rbk.bi * BLK + r;
    if (il < rbk.L) o[(static_cast<size_t>(rbk.seq_start + il) * p.H_r + i) * D + dd] = acc[e];
  }
}

template <typename F>
cudaError_t dispatch(int d, int B, F&& f) {
  if (d == 64 && B == 64) return f(std::integral_constant<int, 64>{}, std::integral_constant<int, 64>{});
  if (d == 64 && B == 128) return f(std::integral_constant<int, 64>{}, std::integral_constant<int, 128>{});
  if (d == 128 && B == 64) return f(std::integral_constant<int, 128>{}, std::integral_constant<int, 64>{});
  if (d == 128 && B == 128) return f(std::integral_constant<int, 128>{}, std::integral_constant<int, 128>{});
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_stats_f32(const CompressParams& p, const float* q, const float* k,
                             cudaStream_t s) {
  return dispatch(p.d, p.B, [&](auto Dc, auto Bc) {
    constexpr int D = decltype(Dc)::value, BLK = decltype(Bc)::value;
    if (sizeof(float) * (BLK * D + BLK) > 48 * 1024) return cudaErrorInvalidValue;
    stats_f32_kernel<D, BLK><<<dim3(p.R, p.H_s), BLK, 0, s>>>(p, q, k);
    return cudaGetLastError();
  });
}

cudaError_t launch_pack_f32(const CompressParams& p, const float* q, const float* k,
                            uint16_t* values, cudaStream_t s) {
  return dispatch(p.d, p.B, [&](auto Dc, auto Bc) {
    constexpr int D = decltype(Dc)::value, BLK = decltype(Bc)::value;
    if (sizeof(float) * BLK * D > 48 * 1024) return cudaErrorInvalidValue;
    pack_f32_kernel<D, BLK><<<dim3(p.R, p.H_s), BLK, 0, s>>>(
        p, q, k, reinterpret_cast<__nv_bfloat16*>(values));
    return cudaGetLastError();
  });
}

cudaError_t launch_retrieve_f32(const RetrieveParams& p, const uint16_t* values, const float* v,
                                float* o, cudaStream_t s) {
  return dispatch(p.d, p.B, [&](auto Dc, auto Bc) {
    constexpr int D = decltype(Dc)::value, BLK = decltype(Bc)::value;
    const int smem = BLK * BLK * 4;
    auto kern = retrieve_f32_kernel<D, BLK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(p.R, p.H_r), 256, smem, s>>>(p, values, v, o);
    return cudaGetLastError();
  });
}

}  // namespace mf
