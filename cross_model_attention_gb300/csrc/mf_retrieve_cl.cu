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
//     (copied into a head-interleaved, MN-major operand; absent heads are
//     zero-filled) and computes
//     A_hat[elem, i] for ALL receiver heads with tcgen05 (M = 128 elements,
//     N = 32 heads, K = sender heads; W^T in bf16 as the B operand);
//   * exchange: each CTA converts its A_hat rows to bf16 and writes them, over
//     distributed shared memory, into the operand buffer of the CTA that owns
//     head i (CTA c owns KV group c and its H_r/8 heads);
//   * A_hat . V: each CTA multiplies its heads' A_hat (two heads stacked per
//     128-row tile) by V_c with tcgen05 into TMEM, accumulating over blocks.
// Every sender-tile byte is read from HBM once and from shared memory once.
//
// Warp roles (480 threads): warp 0 TMA of V tiles, warps 11-14 copy the
// sender rows with 16-byte cp.async straight into the swizzled,
// head-interleaved operand layout (one TMA gather per four 128-byte rows
// issues too slowly to keep up), warp 1 issues the combine MMAs, warps 2-9
// convert/exchange (two per TMEM lane quadrant) and run the epilogue, warp 10
// issues the A_hat.V MMAs — separate issuers so the combine runs ahead while
// the exchange of earlier blocks is in flight.  The
// exchange uses st.async: each 16-byte store counts its bytes on the owner's
// mbarrier, which the owner arms with the bytes it expects per block.  All
// waits are bounded.
#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kCS = 8;          // CTAs per cluster = receiver KV groups
constexpr int kThreads = 480;  // warp 0 V TMA, 1 combine MMA, 2-9 convert, 10 A_hat.V MMA, 11-14 P copies
constexpr int kPThreads = 128;  // P copy threads (warps 11-14)
constexpr int kPSlots = 6;      // P ring: 16-head slices of 8 rows x 64 columns (16 KB)
constexpr int kSliceBytes = 8 * 16 * 128;
constexpr int kMaxUnion = 256;
constexpr int kNComb = 32;      // receiver heads per combine MMA (padded)

struct ClLayout {
  int hpad, nslice, pairs, abuf, vbytes, nv;
  int off_p, off_a, off_v, off_w, off_u, off_bar, bytes;
  __host__ __device__ ClLayout(int D, int Hs, int hpc) {
    hpad = (Hs + 15) / 16 * 16;
    nslice = hpad / 16;
    pairs = (hpc + 1) / 2;
    abuf = pairs * 16384;
    vbytes = 64 * D * 2;
    const int base = kPSlots * kSliceBytes + 2 * abuf + 4096 + kMaxUnion * 4;
    nv = (base + 2 * vbytes + 2048 <= 226 * 1024) ? 2 : 1;
    off_p = 0;
    off_a = off_p + kPSlots * kSliceBytes;
    off_v = off_a + 2 * abuf;
    off_w = off_v + nv * vbytes;
    off_u = off_w + 4096;
    off_bar = off_u + kMaxUnion * 4;
    bytes = off_bar + 32 * 8 + 64 + 1024;
  }
};

// barrier indices
enum : int {
  kBarVFull = 0, kBarVEmpty = 2, kBarDFull = 4, kBarDEmpty = 6, kBarAFull = 8, kBarAFree = 10,
  kBarO = 12, kBarPFull = 13, kBarPEmpty = 13 + kPSlots, kNumBars = 13 + 2 * kPSlots
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
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(bar(kBarPFull + s), kPThreads);
      mbar_init(bar(kBarPEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
      mbar_init(bar(kBarDFull + s), 1);
      mbar_init(bar(kBarDEmpty + s), 8);
      mbar_init(bar(kBarAFull + s), 1);  // the owner's arm + st.async bytes
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
  // ascending union of the kept block columns of this block-row
  int* s_union = reinterpret_cast<int*>(smem + lay.off_u);
  for (int t = threadIdx.x; t < n_sub / kSub; t += kThreads) s_union[t] = p.union_list[rbk.cand_off + t];
  fence_async_smem();
  if (warp == 1) tmem_alloc(smem_u32(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // barrier inits visible to the whole cluster
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);

  if (warp == 0) {
    // ------------------------------------------------------ V tile producer
    if (lane == 0) {
      bool ok = true;
      for (int u = 0; ok && u < n_sub; ++u) {
        const int ue = u / kSub, cs = u - ue * kSub;
        const int bj = s_union[ue];
        const int vs = (lay.nv == 2) ? (u & 1) : 0;
        const uint32_t vph = (lay.nv == 2) ? ((u >> 1) & 1) : (u & 1);
        if (!mbar_wait(bar(kBarVEmpty + vs), vph ^ 1, p.err)) {
          ok = false;
          break;
        }
        mbar_arrive_tx(bar(kBarVFull + vs), lay.vbytes);
        const int tok0 = rbk.seq_start + bj * BLK + cs * 64;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + lay.off_v + vs * lay.vbytes + c * 8192, &tv, g * D + c * 64, tok0,
                      bar(kBarVFull + vs));
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp >= 11) {
    // ------------------------------------------------------ P row producer
    // Thread t copies, for slice-local head h = t/8 and 16-byte chunk
    // cg = t%8, rows 8g..8g+7 of that head's kept tile (64 columns of this
    // sub-block) into the slice layout [row 8][head group 2][8 heads][128 B]
    // with the 128-byte swizzle; a dropped or padded head is zero-filled.
    const int t = threadIdx.x - 11 * 32;
    const int hl = t >> 3, cg = t & 7;
    const uint32_t dst0 = sb + lay.off_p + (hl >> 3) * 1024 + sw128_off(hl & 7, cg);
    const size_t row_bytes = static_cast<size_t>(BLK) * 2;
    const char* vbase = reinterpret_cast<const char*>(p.values);
    int tix[4], nxt[4];
    auto fetch = [&](int u, int (&o4)[4]) {
      const int bj = s_union[u / kSub];
      const int* trow = p.tile_of + static_cast<size_t>(rbk.cand_off + bj) * p.H_s;
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        const int h = sl * 16 + hl;
        o4[sl] = (sl < lay.nslice && h < p.H_s) ? trow[h] : -1;
      }
    };
    if (n_sub > 0) fetch(0, nxt);
    bool ok = true;
    int slot = 0;
    for (int u = 0; ok && u < n_sub; ++u) {
      const int cs = u % kSub;
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) tix[sl] = nxt[sl];
      if (u + 1 < n_sub) fetch(u + 1, nxt);
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        if (sl >= lay.nslice || !ok) continue;
        const int st = slot % kPSlots;
        const uint32_t ph = (slot / kPSlots) & 1;
        ++slot;
        int good = 1;
        if (lane == 0) good = mbar_wait(bar(kBarPEmpty + st), ph ^ 1, p.err) ? 1 : 0;
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          continue;
        }
        const int tt = tix[sl];
        const char* src = vbase + (static_cast<size_t>(tt >= 0 ? tt : 0) * BLK + slab.half * 64 + 8 * g) * row_bytes +
                          cs * 128 + cg * 16;
        const uint32_t nbytes = tt >= 0 ? 16u : 0u;
        const uint32_t dst = dst0 + st * kSliceBytes;
#pragma unroll
        for (int r = 0; r < 8; ++r) cp_async16(dst + r * 2048, src + r * row_bytes, nbytes);
        cp_async_arrive(bar(kBarPFull + st));
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (warp == 1) {
    // ------------------------------------------------- combine MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_comb = idesc_bf16_f32(128, kNComb, true, false);
      bool ok = true;
      int slot = 0;
      for (int u = 0; ok && u < n_sub; ++u) {
        const int b = u & 1;
        const uint32_t ph = (u >> 1) & 1;
        if (!mbar_wait(bar(kBarDEmpty + b), ph ^ 1, p.err)) {
          ok = false;
          break;
        }
        const uint32_t wbase = sb + lay.off_w;
        for (int sl = 0; sl < lay.nslice; ++sl, ++slot) {
          const int st = slot % kPSlots;
          if (!mbar_wait(bar(kBarPFull + st), (slot / kPSlots) & 1, p.err)) {
            ok = false;
            break;
          }
          fence_async_smem();  // rows were written by cp.async (generic proxy)
          tc_fence_after();
          const uint32_t pbase = sb + lay.off_p + st * kSliceBytes;
          const uint64_t bd = sdesc_sw128(wbase + sl * 32, 16, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // rows 2k, 2k+1 of the slice: LBO = row stride (2 KB), SBO = head group (1 KB)
            const uint64_t ad = sdesc_sw128(pbase + 2 * k * 2048, 2048, 1024);
            tc_mma(tmem + b * 128 + k * kNComb, ad, bd, idesc_comb, sl > 0 ? 1u : 0u);
          }
          tc_commit(bar(kBarPEmpty + st));
        }
        if (!ok) break;
        tc_commit(bar(kBarDFull + b));
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 10) {
    // --------------------------------------------- A_hat . V MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_av = idesc_bf16_f32(128, 64, false, true);
      const uint32_t abytes = static_cast<uint32_t>(hpc) * 64 * 128;  // A_hat bytes per block
      for (int u = 0; u < 2 && u < n_sub; ++u) mbar_arrive_tx(bar(kBarAFull + u), abytes);
      bool ok = true;
      for (int u = 0; u < n_sub; ++u) {
        const int ab = u & 1;
        const uint32_t aph = (u >> 1) & 1;
        const int vs = (lay.nv == 2) ? (u & 1) : 0;
        const uint32_t vph = (lay.nv == 2) ? ((u >> 1) & 1) : (u & 1);
        if (!mbar_wait_cluster(bar(kBarAFull + ab), aph, p.err) ||
            !mbar_wait(bar(kBarVFull + vs), vph, p.err)) {
          ok = false;
          break;
        }
        // re-arm this buffer for block u+2 before anyone can write it (the
        // peers write block u+2 only after this CTA's A_hat.V(u) completes)
        if (u + 2 < n_sub) mbar_arrive_tx(bar(kBarAFull + ab), abytes);
        fence_async_smem();
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
      if (!ok) *abort_flag = 1;
      tc_commit(bar(kBarO));
    }
  } else if (warp >= 2 && warp <= 9) {
    // ------------------------------------------------- convert + exchange
    const int wq = warp & 3;
    const int sub = (warp - 2) >> 2;               // the two warps of a TMEM quadrant
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
      uint32_t v[2][32];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) tmem_ld32(tq + b * 128 + (2 * kk + sub) * kNComb, v[kk]);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarDEmpty + b));
      if (!warp_wait(bar(kBarAFree + ab), ph ^ 1, p.err, true)) {
        ok = false;
        break;
      }
      const uint32_t afull_local = bar(kBarAFull + ab);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int k = 2 * kk + sub;
        const int r = 2 * k + (wq >> 1);  // combine row within this CTA's 8 rows
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w[j] = pack_bf16x2(__uint_as_float(v[kk][2 * j]), __uint_as_float(v[kk][2 * j + 1]));
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
              st_async_v4(mapa(sb + off, own), e ? hi : lo, mapa(afull_local, own));
            }
          }
        }
      }
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
      __nv_bfloat16* dst = o + (static_cast<size_t>(rbk.seq_start + rloc) * p.H_r + g * hpc + t) * D +
                           sub * (D / 2);
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t x[32];
        if (have) {
          tmem_ld32(tq + 256 + pr * D + sub * (D / 2) + c0, x);
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
