// mf_retrieve_tc.cu — fused Attention Retrieval, bf16, sm_103a.
//
// "Accelerating Cross-Model LLM Inference via Attention Map Reuse", section
// "Practical Implementation Details" and bold header 4: a fused kernel
// reconstructs the receiver's attention from the cached sparse blocks and
// multiplies it by the receiver's values in one pass, so no dense receiver
// map is ever allocated.  The news article "北大MapFlow：注意力图跨模型复用，
// prefill延迟降15%–20%", paragraph "其三": sparse blocks are read, the heads
// are combined linearly on chip, multiplied by the receiver's V and
// accumulated into the output.  Head mapping is linear ("MapFlow System
// Design", item 3): A_hat_i = sum_h W[i,h] * A_h; a block a head did not keep
// counts as zero and nothing is renormalised.
//
// CTA = (64 query rows of one block-row, one receiver KV group g); the group
// CTAs of a block-row are adjacent in the grid so its tiles are read from HBM
// about once and served to the other groups from L2.  It walks
// the ascending union (over sender heads) of the kept block columns of its
// block-row, in 64-column sub-blocks.  For each sub-block:
//   warp 0   TMA: V_g rows of the sub-block (64 x d) and, in chunks of four
//            sender heads, the kept 64 x 64 probability sub-tiles (absent heads
//            are skipped; their chunk mask says so)
//   warps 2-9  combine: A_hat_i = sum_h W[i,h] P_h for the group's receiver
//            heads, fp32 in registers (16 elements x up to 8 heads per
//            thread), rounded once to bf16 into a 128-byte-swizzled K-major
//            operand tile, two receiver heads stacked per 128-row MMA tile
//   warp 1   tcgen05: O_pair += A_hat_pair (128 x 64) . V_g (64 x d), fp32 in
//            TMEM (pairs x d columns), V read as an MN-major operand
// Epilogue: TMEM -> registers -> bf16 O rows (rows beyond the sequence are
// not written; a block-row with no kept tile gets O = 0).
#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kSubRows = 64;
constexpr int kHeadsPerChunk = 4;
constexpr int kSubTileBytes = 64 * 64 * 2;  // 8 KB
constexpr int kPStages = 3;
constexpr int kCombineWarps = 8;
constexpr int kThreads = 64 + 32 * kCombineWarps;
constexpr int kMaxHpg = 8;
constexpr int kMaxHs = 128;

struct RetLayout {
  int p, v, a, w, bar, misc, bytes, abuf_bytes, n_abuf, pairs, vbytes;
  __host__ __device__ RetLayout(int D, int hpg) {
    pairs = (hpg + 1) / 2;
    vbytes = 64 * D * 2;
    abuf_bytes = pairs * 128 * 128;
    n_abuf = (pairs <= 2) ? 2 : 1;
    p = 0;
    v = p + kPStages * kHeadsPerChunk * kSubTileBytes;
    a = v + 2 * vbytes;
    w = a + n_abuf * abuf_bytes;
    bar = w + kMaxHpg * kMaxHs * 4;
    misc = bar + 16 * 8;
    bytes = misc + 64 + 1024;
  }
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try(bar, parity);
  __syncwarp();
  return ok != 0;
}

template <int D, int BLK, int HPGM>
__global__ void __launch_bounds__(kThreads, 1)
    retrieve_bf16_kernel(const __grid_constant__ CUtensorMap tp,
                         const __grid_constant__ CUtensorMap tv, const RetrieveParams p,
                         __nv_bfloat16* __restrict__ o) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hpg = p.H_r / p.H_kv;
  const RetLayout lay(D, hpg);
  // grid x = KV group (fastest), y = slab: the group CTAs of one block-row run
  // side by side and share its sender tiles through L2
  const RowSlab slab = p.slabs[blockIdx.y];
  const int g = blockIdx.x;
  const RowBlock rbk = p.rbs[slab.rb];
  constexpr int kSubPerBlock = BLK / 64;
  const int n_sub = p.union_cnt[slab.rb] * kSubPerBlock;
  const int n_chunks = (p.H_s + kHeadsPerChunk - 1) / kHeadsPerChunk;
  const int row0 = rbk.bi * BLK + slab.half * kSubRows;  // first row, sequence-relative

  auto barPFull = [&](int s) { return sb + lay.bar + 8u * s; };
  auto barPEmpty = [&](int s) { return sb + lay.bar + 8u * (kPStages + s); };
  auto barVFull = [&](int s) { return sb + lay.bar + 8u * (2 * kPStages + s); };
  auto barVEmpty = [&](int s) { return sb + lay.bar + 8u * (2 * kPStages + 2 + s); };
  auto barAFull = [&](int s) { return sb + lay.bar + 8u * (2 * kPStages + 4 + s); };
  auto barAEmpty = [&](int s) { return sb + lay.bar + 8u * (2 * kPStages + 6 + s); };
  const uint32_t barO = sb + lay.bar + 8u * (2 * kPStages + 8);
  volatile int* chunk_mask = reinterpret_cast<volatile int*>(smem + lay.misc);  // [kPStages]
  volatile int* abort_flag = chunk_mask + kPStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + lay.misc + 32);
  float* sW = reinterpret_cast<float*>(smem + lay.w);

  int tcols = lay.pairs * D;
  int talloc = 32;
  while (talloc < tcols) talloc <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(barPFull(s), 1);
      mbar_init(barPEmpty(s), kCombineWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(barVFull(s), 1);
      mbar_init(barVEmpty(s), 1);
      mbar_init(barAFull(s), kCombineWarps);
      mbar_init(barAEmpty(s), 1);
    }
    mbar_init(barO, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // head-map weights of this group: sW[i][h] = W[g*hpg + i][h]
  for (int t = threadIdx.x; t < hpg * p.H_s; t += blockDim.x) {
    const int i = t / p.H_s, hh = t - i * p.H_s;
    sW[i * kMaxHs + hh] = p.W[static_cast<size_t>(g * hpg + i) * p.H_s + hh];
  }
  if (warp == 1) tmem_alloc(smem_u32(tslot), talloc);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tp);
      prefetch_tmap(&tv);
      int k = 0;  // global chunk counter
      bool ok = true;
      int v_issued = 0;
      for (int u = 0; ok && u < n_sub; ++u) {
        const int ue = u / kSubPerBlock, cs = u - ue * kSubPerBlock;
        const int bj = p.union_list[rbk.cand_off + ue];
        const int vs = u & 1;
        if (!mbar_wait(barVEmpty(vs), ((u >> 1) & 1) ^ 1, p.err)) {
          ok = false;
          break;
        }
        mbar_arrive_tx(barVFull(vs), lay.vbytes);
        const int tok0 = rbk.seq_start + bj * BLK + cs * 64;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + lay.v + vs * lay.vbytes + c * 8192, &tv, g * D + c * 64, tok0,
                      barVFull(vs));
        v_issued = u + 1;
        const int* trow = p.tile_of + static_cast<size_t>(rbk.cand_off + bj) * p.H_s;
        for (int hc = 0; hc < n_chunks; ++hc, ++k) {
          const int st = k % kPStages;
          if (!mbar_wait(barPEmpty(st), ((k / kPStages) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          int mask = 0, tix[kHeadsPerChunk];
#pragma unroll
          for (int q = 0; q < kHeadsPerChunk; ++q) {
            const int hh = hc * kHeadsPerChunk + q;
            tix[q] = (hh < p.H_s) ? trow[hh] : -1;
            if (tix[q] >= 0) mask |= 1 << q;
          }
          chunk_mask[st] = mask;
          const int nbytes = __popc(mask) * kSubTileBytes;
          if (nbytes) {
            mbar_arrive_tx(barPFull(st), nbytes);
#pragma unroll
            for (int q = 0; q < kHeadsPerChunk; ++q)
              if (tix[q] >= 0)
                tma_load_2d(sb + lay.p + (st * kHeadsPerChunk + q) * kSubTileBytes, &tp, cs * 64,
                            tix[q] * BLK + slab.half * 64, barPFull(st));
          } else {
            mbar_arrive(barPFull(st));
          }
        }
      }
      if (!ok) *abort_flag = 1;
      // drain copies in flight (bounded)
      for (int kk = (k > kPStages ? k - kPStages : 0); kk < k; ++kk)
        mbar_wait(barPFull(kk % kPStages), (kk / kPStages) & 1, nullptr);
      for (int u = (v_issued > 2 ? v_issued - 2 : 0); u < v_issued; ++u)
        mbar_wait(barVFull(u & 1), (u >> 1) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, true);
      for (int u = 0; u < n_sub; ++u) {
        const int ab = (lay.n_abuf == 2) ? (u & 1) : 0;
        const uint32_t aph = (lay.n_abuf == 2) ? ((u >> 1) & 1) : (u & 1);
        const int vs = u & 1;
        if (!mbar_wait(barAFull(ab), aph, p.err) || !mbar_wait(barVFull(vs), (u >> 1) & 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t abase = sb + lay.a + ab * lay.abuf_bytes;
        const uint32_t vbase = sb + lay.v + vs * lay.vbytes;
        for (int pr = 0; pr < lay.pairs; ++pr) {
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t ad = sdesc_sw128(abase + pr * 16384 + s * 32, 16, 1024);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
              const uint64_t bd = sdesc_sw128(vbase + c * 8192 + s * 2048, 8192, 1024);
              tc_mma(tmem + pr * D + c * 64, ad, bd, idesc, (u > 0 || s > 0) ? 1u : 0u);
            }
          }
        }
        tc_commit(barAEmpty(ab));
        tc_commit(barVEmpty(vs));
      }
      tc_commit(barO);
    }
  } else {
    // ------------------------------------------------------------ combine
    const int t = threadIdx.x - 64;  // 0..255
    const int cw = warp - 2;         // 0..7
    float acc[HPGM][16];
    int k = 0;
    bool ok = true;
    for (int u = 0; ok && u < n_sub; ++u) {
#pragma unroll
      for (int i = 0; i < HPGM; ++i)
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[i][e] = 0.f;
      for (int hc = 0; hc < n_chunks; ++hc, ++k) {
        const int st = k % kPStages;
        if (!warp_wait(barPFull(st), (k / kPStages) & 1, p.err)) {
          ok = false;
          break;
        }
        const int mask = chunk_mask[st];
        for (int q = 0; q < kHeadsPerChunk; ++q) {
          if (!(mask & (1 << q))) continue;
          const int hh = hc * kHeadsPerChunk + q;
          const uint8_t* tileb = smem + lay.p + (st * kHeadsPerChunk + q) * kSubTileBytes;
          float pv[16];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int c = t + 256 * j;  // 16-byte chunk id in the 64x64 sub-tile
            const int r = c >> 3, cg = c & 7;
            const uint4 w4 = *reinterpret_cast<const uint4*>(tileb + sw128_off(r, cg));
            pv[8 * j + 0] = bf16lo(w4.x);
            pv[8 * j + 1] = bf16hi(w4.x);
            pv[8 * j + 2] = bf16lo(w4.y);
            pv[8 * j + 3] = bf16hi(w4.y);
            pv[8 * j + 4] = bf16lo(w4.z);
            pv[8 * j + 5] = bf16hi(w4.z);
            pv[8 * j + 6] = bf16lo(w4.w);
            pv[8 * j + 7] = bf16hi(w4.w);
          }
#pragma unroll
          for (int i = 0; i < HPGM; ++i) {
            if (i < hpg) {
              const float wv = sW[i * kMaxHs + hh];
#pragma unroll
              for (int e = 0; e < 16; ++e) acc[i][e] = fmaf(wv, pv[e], acc[i][e]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(barPEmpty(st));
      }
      if (!ok) break;
      const int ab = (lay.n_abuf == 2) ? (u & 1) : 0;
      const uint32_t aph = (lay.n_abuf == 2) ? ((u >> 1) & 1) : (u & 1);
      if (!warp_wait(barAEmpty(ab), aph ^ 1, p.err)) {
        ok = false;
        break;
      }
      uint8_t* abuf = smem + lay.a + ab * lay.abuf_bytes;
#pragma unroll
      for (int i = 0; i < HPGM; ++i) {
        if (i < hpg) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int c = t + 256 * j;
            const int r = c >> 3, cg = c & 7;
            uint4 w4;
            w4.x = pack_bf16x2(acc[i][8 * j + 0], acc[i][8 * j + 1]);
            w4.y = pack_bf16x2(acc[i][8 * j + 2], acc[i][8 * j + 3]);
            w4.z = pack_bf16x2(acc[i][8 * j + 4], acc[i][8 * j + 5]);
            w4.w = pack_bf16x2(acc[i][8 * j + 6], acc[i][8 * j + 7]);
            *reinterpret_cast<uint4*>(abuf + (i >> 1) * 16384 + sw128_off((i & 1) * 64 + r, cg)) = w4;
          }
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(barAFull(ab));
    }
    if (!ok) *abort_flag = 1;
    // -------------------------------------------------------- epilogue
    const int wq = warp & 3;
    const int colhalf = cw >> 2;  // two warps per TMEM lane quadrant split d
    const int lrow = wq * 32 + lane;  // TMEM lane
    const int i_in_pair = lrow >> 6, r = lrow & 63;
    const int rloc = row0 + r;
    const bool row_ok = rloc < rbk.L;
    const uint32_t tq = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const bool have = n_sub > 0 && ok;
    if (have) warp_wait(barO, 0, p.err);
    tc_fence_after();
    for (int pr = 0; pr < lay.pairs; ++pr) {
      const int i = 2 * pr + i_in_pair;
      const int head = g * hpg + i;
      const bool write = row_ok && i < hpg && *abort_flag == 0;
      __nv_bfloat16* dst = o + (static_cast<size_t>(rbk.seq_start + rloc) * p.H_r + head) * D +
                           colhalf * (D / 2);
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t v[32];
        if (have) {
          tmem_ld32(tq + pr * D + colhalf * (D / 2) + c0, v);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (write) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w4;
            w4.x = pack_bf16x2(__uint_as_float(v[e + 0]), __uint_as_float(v[e + 1]));
            w4.y = pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
            w4.z = pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
            w4.w = pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
            *reinterpret_cast<uint4*>(dst + c0 + e) = w4;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, talloc);
  }
}

template <int D, int BLK, int HPGM>
cudaError_t launch_ret_t(const RetrieveParams& p, const CUtensorMap& tp, const CUtensorMap& tv,
                         void* o, cudaStream_t s) {
  auto kern = retrieve_bf16_kernel<D, BLK, HPGM>;
  const RetLayout lay(D, p.H_r / p.H_kv);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.H_kv, p.n_slabs);
  kern<<<grid, kThreads, lay.bytes, s>>>(tp, tv, p, static_cast<__nv_bfloat16*>(o));
  return cudaGetLastError();
}

}  // namespace

template <int HPGM>
cudaError_t launch_ret_h(const RetrieveParams& p, const CUtensorMap& tp, const CUtensorMap& tv,
                         void* o, cudaStream_t s) {
  if (p.d == 128 && p.B == 64) return launch_ret_t<128, 64, HPGM>(p, tp, tv, o, s);
  if (p.d == 128 && p.B == 128) return launch_ret_t<128, 128, HPGM>(p, tp, tv, o, s);
  if (p.d == 64 && p.B == 64) return launch_ret_t<64, 64, HPGM>(p, tp, tv, o, s);
  if (p.d == 64 && p.B == 128) return launch_ret_t<64, 128, HPGM>(p, tp, tv, o, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_retrieve_bf16(const RetrieveParams& p, const CUtensorMap& tp,
                                 const CUtensorMap& tv, void* o, cudaStream_t s) {
  const int hpg = p.H_r / p.H_kv;
  if (hpg <= 4) return launch_ret_h<4>(p, tp, tv, o, s);
  if (hpg <= kMaxHpg) return launch_ret_h<8>(p, tp, tv, o, s);
  return cudaErrorInvalidValue;
}

}  // namespace mf
