// mf_retrieve_cl.cu — fused Attention Retrieval with the head combine on the
// tensor cores, one 8-CTA thread-block cluster per 64 query rows (receivers
// with 8 KV heads), bf16, sm_103a.
//
// What it computes is the fused retrieval of "Accelerating Cross-Model LLM
// Inference via Attention Map Reuse" (section "Practical Implementation
// Details", bold header 4; head mapping per "MapFlow System Design" item 3) as
// the news article "北大MapFlow：注意力图跨模型复用，prefill延迟降15%–20%"
// describes it in paragraph "其三": read the sparse blocks, combine the sender
// heads on chip, multiply by the receiver's V and accumulate the output:
//   O_i[rows] = sum_bj ( sum_h W[i,h] P_h[rows, bj] ) V_g(i)[bj].
//
// Work split.  The head combine costs H_r multiply-adds per sender-tile
// element, too many for the CUDA cores at HBM speed, and one block-row's O
// accumulators (32 heads x 64 rows x d fp32) are four times the tensor memory
// of one SM.  So the 8 CTAs of a cluster split the 64 rows two ways:
//   * combine: CTA c takes rows 8c..8c+7 of every kept tile of the block-row
//     (TMA gather of 128-byte tile rows into a head-interleaved, MN-major
//     operand; absent heads read an all-zero tile) and computes
//     A_hat[elem, i] for ALL receiver heads with tcgen05 (M = 128 elements,
//     N = 32 heads, K = sender heads; W^T in bf16 as the B operand);
//   * exchange: each CTA converts its A_hat rows to bf16 and writes them, over
//     distributed shared memory, into the operand buffer of the CTA that owns
//     head i (CTA c owns KV group c and its H_r/8 heads);
//   * A_hat . V: each CTA multiplies its heads' A_hat (two heads stacked per
//     128-row tile) by V_c with tcgen05 into TMEM, accumulating over blocks.
// Every sender-tile byte is read from HBM once and from shared memory once.
//
// Warp roles (192 threads): warp 0 TMA (V tile, P gathers), warp 1 tcgen05
// issue (combine of block u and A_hat.V of block u-1 interleaved), warps 2-5
// convert/exchange and the epilogue.  All waits are bounded.
#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kCS = 8;          // CTAs per cluster = receiver KV groups
constexpr int kThreads = 192;
constexpr int kPStages = 2;
constexpr int kNComb = 32;      // receiver heads per combine MMA (padded)

struct ClLayout {
  int hpad, prow, pstage, pairs, abuf, vbytes, nv;
  int off_p, off_a, off_v, off_w, off_bar, bytes;
  __host__ __device__ ClLayout(int D, int Hs, int hpc) {
    hpad = (Hs + 15) / 16 * 16;
    prow = hpad * 128;
    pstage = 8 * prow;
    pairs = (hpc + 1) / 2;
    abuf = pairs * 16384;
    vbytes = 64 * D * 2;
    const int base = kPStages * pstage + 2 * abuf + 4096;
    nv = (base + 2 * vbytes + 2048 <= 226 * 1024) ? 2 : 1;
    off_p = 0;
    off_a = off_p + kPStages * pstage;
    off_v = off_a + 2 * abuf;
    off_w = off_v + nv * vbytes;
    off_bar = off_w + 4096;
    bytes = off_bar + 24 * 8 + 64 + 1024;
  }
};

// barrier indices
enum : int {
  kBarPFull = 0, kBarPEmpty = 2, kBarVFull = 4, kBarVEmpty = 6, kBarDFull = 8, kBarDEmpty = 10,
  kBarAFull = 12, kBarAFree = 14, kBarO = 16, kNumBars = 17
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err, bool cluster) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0)
    ok = (cluster ? mbar_wait_cluster(bar, parity, err) : mbar_wait(bar, parity, err)) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) {
    if (cluster) mbar_try_cluster(bar, parity);
    else mbar_try(bar, parity);
  }
  __syncwarp();
  return ok != 0;
}

// 8x8 transpose of 32-bit words across the 8 lanes of an aligned lane group:
// on entry lane q holds row q (w[0..7]); on exit it holds column q.
__device__ __forceinline__ void transpose8(uint32_t* w) {
  const int q = threadIdx.x & 7;
#pragma unroll
  for (int s = 4; s >= 1; s >>= 1) {
    const bool up = (q & s) != 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (e & s) continue;
      const uint32_t send = up ? w[e] : w[e | s];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, s);
      if (up) w[e] = recv;
      else w[e | s] = recv;
    }
  }
}

template <int D, int BLK>
__global__ void __launch_bounds__(kThreads, 1)
    retrieve_cl_kernel(const __grid_constant__ CUtensorMap tp, const __grid_constant__ CUtensorMap tv,
                       const RetrieveParams p, __nv_bfloat16* __restrict__ o) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const int hpc = p.H_r / kCS;
  const ClLayout lay(D, p.H_s, hpc);
  const RowSlab slab = p.slabs[blockIdx.x / kCS];
  const RowBlock rbk = p.rbs[slab.rb];
  constexpr int kSub = BLK / 64;
  const int n_sub = p.union_cnt[slab.rb] * kSub;
  const int row0 = rbk.bi * BLK + slab.half * 64;
  const int g = static_cast<int>(crank);
  auto bar = [&](int i) { return sb + lay.off_bar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.off_bar + kNumBars * 8);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + lay.off_bar + kNumBars * 8 + 16);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarPFull + s), 1);
      mbar_init(bar(kBarPEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
      mbar_init(bar(kBarDFull + s), 1);
      mbar_init(bar(kBarDEmpty + s), 4);
      mbar_init(bar(kBarAFull + s), kCS * 4);
      mbar_init(bar(kBarAFree + s), kCS);
    }
    mbar_init(bar(kBarO), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // W^T as the combine's B operand: row n = receiver head (32 rows), 64 bf16
  // sender-head slots per row, 128-byte swizzle; zero beyond H_r / H_s.
  for (int t = threadIdx.x; t < kNComb * 64; t += kThreads) {
    const int n = t >> 6, k = t & 63;
    const float wv = (n < p.H_r && k < p.H_s) ? p.W[static_cast<size_t>(n) * p.H_s + k] : 0.f;
    *reinterpret_cast<__nv_bfloat16*>(smem + lay.off_w + sw128_off(n, k >> 3) + (k & 7) * 2) =
        __float2bfloat16_rn(wv);
  }
  fence_async_smem();
  if (warp == 1) tmem_alloc(smem_u32(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // barrier inits visible to the whole cluster
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int nq = lay.hpad / 4;
    bool ok = true;
    for (int u = 0; ok && u < n_sub; ++u) {
      const int ue = u / kSub, cs = u - ue * kSub;
      const int bj = p.union_list[rbk.cand_off + ue];
      const int vs = (lay.nv == 2) ? (u & 1) : 0;
      const uint32_t vph = (lay.nv == 2) ? ((u >> 1) & 1) : (u & 1);
      const int st = u & 1;
      const uint32_t ph = (u >> 1) & 1;
      // P gathers of block u first: the tcgen05 issuer combines block u
      // before it multiplies block u-1, which is what frees a single V stage
      int good = 1;
      if (lane == 0) {
        good = mbar_wait(bar(kBarPEmpty + st), ph ^ 1, p.err) ? 1 : 0;
        if (good) mbar_arrive_tx(bar(kBarPFull + st), lay.pstage);
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) {
        ok = false;
        break;
      }
      if (lane < nq) {
        const int* trow = p.tile_of + static_cast<size_t>(rbk.cand_off + bj) * p.H_s;
        int y[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int h = 4 * lane + t;
          const int tix = (h < p.H_s) ? trow[h] : -1;
          y[t] = (tix >= 0 ? tix : p.zero_tile) * BLK + slab.half * 64 + 8 * g;
        }
        const uint32_t dst = sb + lay.off_p + st * lay.pstage + (lane >> 1) * 1024 + (lane & 1) * 512;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          tma_gather4(dst + r * lay.prow, &tp, cs * 64, y[0] + r, y[1] + r, y[2] + r, y[3] + r,
                      bar(kBarPFull + st));
      }
      __syncwarp();
      if (lane == 0) {
        good = mbar_wait(bar(kBarVEmpty + vs), vph ^ 1, p.err) ? 1 : 0;
        if (good) {
          mbar_arrive_tx(bar(kBarVFull + vs), lay.vbytes);
          const int tok0 = rbk.seq_start + bj * BLK + cs * 64;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sb + lay.off_v + vs * lay.vbytes + c * 8192, &tv, g * D + c * 64, tok0,
                        bar(kBarVFull + vs));
        }
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) {
        ok = false;
        break;
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_comb = idesc_bf16_f32(128, kNComb, true, false);
      constexpr uint32_t idesc_av = idesc_bf16_f32(128, 64, false, true);
      const int ksteps = lay.hpad / 16;
      bool ok = true;
      for (int step = 0; ok && step <= n_sub; ++step) {
        if (step < n_sub) {
          const int u = step, st = u & 1, b = u & 1;
          const uint32_t ph = (u >> 1) & 1;
          if (!mbar_wait(bar(kBarPFull + st), ph, p.err) ||
              !mbar_wait(bar(kBarDEmpty + b), ph ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t pbase = sb + lay.off_p + st * lay.pstage;
          const uint32_t wbase = sb + lay.off_w;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            for (int ks = 0; ks < ksteps; ++ks) {
              const uint64_t ad = sdesc_sw128(pbase + 2 * k * lay.prow + ks * 2048, lay.prow, 1024);
              const uint64_t bd = sdesc_sw128(wbase + ks * 32, 16, 1024);
              tc_mma(tmem + b * 128 + k * kNComb, ad, bd, idesc_comb, ks > 0 ? 1u : 0u);
            }
          }
          tc_commit(bar(kBarPEmpty + st));
          tc_commit(bar(kBarDFull + b));
        }
        if (step >= 1) {
          const int u = step - 1, ab = u & 1;
          const uint32_t aph = (u >> 1) & 1;
          const int vs = (lay.nv == 2) ? (u & 1) : 0;
          const uint32_t vph = (lay.nv == 2) ? ((u >> 1) & 1) : (u & 1);
          if (!mbar_wait_cluster(bar(kBarAFull + ab), aph, p.err) ||
              !mbar_wait(bar(kBarVFull + vs), vph, p.err)) {
            ok = false;
            break;
          }
          fence_async_smem();  // A_hat arrived through generic (remote) stores
          tc_fence_after();
          const uint32_t abase = sb + lay.off_a + ab * lay.abuf;
          const uint32_t vbase = sb + lay.off_v + vs * lay.vbytes;
          for (int pr = 0; pr < lay.pairs; ++pr) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint64_t ad = sdesc_sw128(abase + pr * 16384 + s * 32, 16, 1024);
#pragma unroll
              for (int c = 0; c < D / 64; ++c) {
                const uint64_t bd = sdesc_sw128(vbase + c * 8192 + s * 2048, 8192, 1024);
                tc_mma(tmem + 256 + pr * D + c * 64, ad, bd, idesc_av, (u > 0 || s > 0) ? 1u : 0u);
              }
            }
          }
          tc_commit(bar(kBarVEmpty + vs));
          if (u + 2 < n_sub) tc_commit_mc(bar(kBarAFree + ab), 0xFF);
        }
      }
      if (!ok) *abort_flag = 1;
      tc_commit(bar(kBarO));
    }
  } else {
    // ------------------------------------------------- convert + exchange
    const int wq = warp & 3;
    const int q = lane & 7;
    const int grp = 4 * (wq & 1) + (lane >> 3);  // 16-byte chunk (8 columns) of this lane group
    const uint32_t tq = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    bool ok = true;
    for (int u = 0; ok && u < n_sub; ++u) {
      const int b = u & 1, ab = u & 1;
      const uint32_t ph = (u >> 1) & 1;
      if (!warp_wait(bar(kBarDFull + b), ph, p.err, false)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_ld32(tq + b * 128 + k * kNComb, v[k]);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarDEmpty + b));
      if (!warp_wait(bar(kBarAFree + ab), ph ^ 1, p.err, true)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = 2 * k + (wq >> 1);  // combine row within this CTA's 8 rows
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w[j] = pack_bf16x2(__uint_as_float(v[k][2 * j]), __uint_as_float(v[k][2 * j + 1]));
        transpose8(w);
        transpose8(w + 8);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const uint32_t* x = w + 8 * blk;
          const int wi = q + 8 * blk;  // word index: heads 2wi, 2wi+1
          const uint4 lo = make_uint4(prmt(x[0], x[1], 0x5410), prmt(x[2], x[3], 0x5410),
                                      prmt(x[4], x[5], 0x5410), prmt(x[6], x[7], 0x5410));
          const uint4 hi = make_uint4(prmt(x[0], x[1], 0x7632), prmt(x[2], x[3], 0x7632),
                                      prmt(x[4], x[5], 0x7632), prmt(x[6], x[7], 0x7632));
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int hh = 2 * wi + e;
            if (hh < p.H_r) {
              const int own = hh / hpc, t = hh - own * hpc;
              const int R = (t & 1) * 64 + 8 * g + r;
              const uint32_t off = lay.off_a + ab * lay.abuf + (t >> 1) * 16384 + sw128_off(R, grp);
              st_cluster_v4(mapa(sb + off, own), e ? hi : lo);
            }
          }
        }
      }
      __syncwarp();
      if (lane < kCS) mbar_arrive_remote(mapa(bar(kBarAFull + ab), lane));
    }
    if (!ok) *abort_flag = 1;
    // -------------------------------------------------------- epilogue
    const int L = wq * 32 + lane;  // TMEM lane: head 2pr + L/64, row L%64
    const int r = L & 63;
    const int rloc = row0 + r;
    const bool row_ok = rloc < rbk.L;
    const bool have = n_sub > 0 && ok;
    if (have) warp_wait(bar(kBarO), 0, p.err, false);
    tc_fence_after();
    for (int pr = 0; pr < lay.pairs; ++pr) {
      const int t = 2 * pr + (L >> 6);
      const bool write = row_ok && t < hpc && *abort_flag == 0;
      __nv_bfloat16* dst = o + (static_cast<size_t>(rbk.seq_start + rloc) * p.H_r + g * hpc + t) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t x[32];
        if (have) {
          tmem_ld32(tq + 256 + pr * D + c0, x);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = 0u;
        }
        if (write) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w4;
            w4.x = pack_bf16x2(__uint_as_float(x[e + 0]), __uint_as_float(x[e + 1]));
            w4.y = pack_bf16x2(__uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
            w4.z = pack_bf16x2(__uint_as_float(x[e + 4]), __uint_as_float(x[e + 5]));
            w4.w = pack_bf16x2(__uint_as_float(x[e + 6]), __uint_as_float(x[e + 7]));
            *reinterpret_cast<uint4*>(dst + c0 + e) = w4;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while a peer may still touch its shared memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int BLK>
cudaError_t launch_cl_t(const RetrieveParams& p, const CUtensorMap& tp, const CUtensorMap& tv,
                        void* o, cudaStream_t s) {
  auto kern = retrieve_cl_kernel<D, BLK>;
  const ClLayout lay(D, p.H_s, p.H_r / kCS);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_slabs * kCS, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = lay.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tp, tv, p, static_cast<__nv_bfloat16*>(o));
}

}  // namespace

bool retrieve_cluster_supported(int H_s, int H_r, int H_kv, int d, int B) {
  return H_kv == kCS && H_r % kCS == 0 && H_r / kCS <= 4 && H_r <= kNComb && H_s <= 64 &&
         (d == 64 || d == 128) && (B == 64 || B == 128);
}

cudaError_t launch_retrieve_cluster(const RetrieveParams& p, const CUtensorMap& tp,
                                    const CUtensorMap& tv, void* o, cudaStream_t s) {
  if (p.d == 128 && p.B == 64) return launch_cl_t<128, 64>(p, tp, tv, o, s);
  if (p.d == 128 && p.B == 128) return launch_cl_t<128, 128>(p, tp, tv, o, s);
  if (p.d == 64 && p.B == 64) return launch_cl_t<64, 64>(p, tp, tv, o, s);
  if (p.d == 64 && p.B == 128) return launch_cl_t<64, 128>(p, tp, tv, o, s);
  return cudaErrorInvalidValue;
}

}  // namespace mf
