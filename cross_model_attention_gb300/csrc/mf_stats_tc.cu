// mf_stats_tc.cu — Attention State Compressor, step 1 (block statistics) on
// the sm_103a tensor cores, bf16 inputs.
//
// "Accelerating Cross-Model LLM Inference via Attention Map Reuse", section
// "Practical Implementation Details": the compressor filters the sender's map
// before caching it with block-level top-p; the news article
// "北大MapFlow：注意力图跨模型复用，prefill延迟降15%–20%", paragraph "其一",
// adds that it first computes block-level statistics and only then picks
// blocks, never laying out the dense N x N map.  This kernel produces those
// statistics in ONE pass over Q.K^T:
//   row max m_i and row sum l_i of the causal softmax of s_ij = q_i.k_j/sqrt(d),
//   and the probability mass of every candidate B x B block.
//
// CTA = (128 query rows of one sequence, one sender head).  Warp roles:
//   warp 0  TMA producer: Q tile once, K tiles (128 keys) into a 3-4 stage ring
//   warp 1  tcgen05 issuer: S = Q.K^T (M=128, N=128, K=d) into one of two TMEM
//           buffers (fp32, 128 lanes x 128 columns each)
//   statistics warps, one thread per query row (its TMEM lane): running max,
//           lazily re-referenced exp2, per-(row, key-block) partial sums kept
//           in TMEM columns 256..511, running row sum.  A reference value
//           only moves when a 32-column chunk's max exceeds it by more than
//           2^8; the warp's stored partials are then rescaled in TMEM.  Each
//           lane quadrant has two warps: at B = 64 one per 64-column block of
//           every tile, at B = 128 one per S buffer (every second tile, in
//           32-column chunks); each has its own reference and the parts are
//           merged per row at the end.  128 partial columns per warp
//           (sequences up to 16384 tokens at B = 64, 32768 at B = 128).
//   end:    mass[bi][bj] = sum over the block-row's rows of partial/l_ref,
//           reduced across lanes with a 31-shuffle transpose-reduction and
//           across warps in a fixed order (deterministic).
#include <cmath>

#include "mf_internal.cuh"
#include "mf_ptx.cuh"
#include "mf_stats_common.cuh"

namespace mf {
namespace {

constexpr int kRows = 128;
constexpr int kCols = 128;
constexpr uint32_t kPartCol = 256;
constexpr float kTau = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct StatsLayout {
  static constexpr int kChunkBytes = kRows * 128;           // 128 rows x 64 bf16
  static constexpr int kTileBytes = kRows * D * 2;
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kQ = 0;                              // two Q buffers
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kRed = kK + kStages * kTileBytes;    // float [4][256]
  static constexpr int kX = kRed + 4 * 256 * 4;             // float [2][3][128] row-state exchange
  static constexpr int kBar = kX + 2 * 3 * 128 * 4;         // 24 mbarriers
  static constexpr int kSlot = kBar + 24 * 8;
  static constexpr int kFlag = kSlot + 8;
  static constexpr int kBytes = kFlag + 8 + 1024;           // + alignment slack
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try(bar, parity);  // every lane observes the completed phase
  __syncwarp();
  return ok != 0;
}

// Statistics warps per TMEM lane quadrant: at B = 64 two, one per 64-column
// block of every S tile (each loads its 64 columns at once and frees the
// buffer); at B = 128 two, one per S buffer (each takes every second tile in
// 32-column chunks, which keeps its registers in the file).
template <int BLK>
struct StatWarps {
  static constexpr int kHalves = (BLK == 64) ? 2 : 1;  // blocks per tile
  static constexpr int kPar = (BLK == 64) ? 1 : 2;     // buffers split between warps
  static constexpr int kParts = kHalves * kPar;
  static constexpr int kCW = (BLK == 64) ? 64 : 32;    // columns per pass
  static constexpr int kN = 4 * kParts;
  static constexpr int kThreads = 64 + 32 * kN;
};

// Item r of this CTA in a snake order over the heavy-first (tile, head) list:
// round r takes items [r*G, r*G+G), walked forwards on even rounds and
// backwards on odd ones, so every CTA's total work stays within one item of
// the others.  -1 once the list is exhausted.
__device__ __forceinline__ int item_of(int r, int n_items) {
  const int G = gridDim.x;
  const int idx = r * G + ((r & 1) ? (G - 1 - static_cast<int>(blockIdx.x))
                                    : static_cast<int>(blockIdx.x));
  return idx < n_items ? idx : -1;
}

template <int D, int BLK>
__global__ void __launch_bounds__(StatWarps<BLK>::kThreads, 1)
    stats_bf16_kernel(const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk, const CompressParams p) {
  using Lay = StatsLayout<D>;
  constexpr int NS = Lay::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_tiles * p.H_s;

  auto barQFull = [&](int q) { return sb + Lay::kBar + 8u * q; };
  auto barQEmpty = [&](int q) { return sb + Lay::kBar + 8u * (2 + q); };
  auto barFull = [&](int s) { return sb + Lay::kBar + 8u * (4 + s); };
  auto barEmpty = [&](int s) { return sb + Lay::kBar + 8u * (4 + NS + s); };
  auto barSFull = [&](int b) { return sb + Lay::kBar + 8u * (4 + 2 * NS + b); };
  auto barSEmpty = [&](int b) { return sb + Lay::kBar + 8u * (6 + 2 * NS + b); };
  const uint32_t barDone = sb + Lay::kBar + 8u * (8 + 2 * NS);
  volatile int* stat_fail = reinterpret_cast<volatile int*>(smem + Lay::kFlag);

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      mbar_init(barQFull(q), 1);
      mbar_init(barQEmpty(q), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(barFull(s), 1);
      mbar_init(barEmpty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(barSFull(b), 1);
      mbar_init(barSEmpty(b), StatWarps<BLK>::kN / StatWarps<BLK>::kPar);  // the warps of that buffer
    }
    mbar_init(barDone, 1);
    *stat_fail = 0;
    fence_mbar_init();
    if (blockIdx.x == 0 && p.sel_done) *p.sel_done = 0;  // the selection kernel's CTA count
  }
  if (warp == 1) tmem_alloc(sb + Lay::kSlot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + Lay::kSlot);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Q of item r into buffer r&1, K tiles of every item through one ring
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      int kt = 0, nq = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int idx = item_of(r, n_items);
        if (idx < 0) break;
        const RowTile tile = p.tiles[idx / p.H_s];
        const int h = idx % p.H_s;
        const int hk = h / (p.H_s / p.H_ks);
        const int n_ct = p.causal ? tile.tl + 1 : (tile.L + kCols - 1) / kCols;
        const int qb = r & 1;
        if (!mbar_wait(barQEmpty(qb), ((r >> 1) & 1) ^ 1, p.err)) break;
        mbar_arrive_tx(barQFull(qb), Lay::kTileBytes);
        const int qrow = tile.seq_start + tile.tl * kRows;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Lay::kQ + qb * Lay::kTileBytes + c * Lay::kChunkBytes, &tq,
                      h * D + c * 64, qrow, barQFull(qb));
        nq = r + 1;
        for (int n = 0; n < n_ct; ++n, ++kt) {
          const int s = kt % NS;
          if (!mbar_wait(barEmpty(s), ((kt / NS) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_tx(barFull(s), Lay::kTileBytes);
          const uint32_t dst = sb + Lay::kK + s * Lay::kTileBytes;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(dst + c * Lay::kChunkBytes, &tk, hk * D + c * 64,
                        tile.seq_start + n * kCols, barFull(s));
        }
      }
      // drain: copies still in flight complete before the CTA may exit (each
      // wait is on the latest use of its barrier, so its phase is the one of
      // that copy)
      for (int t = (kt > NS ? kt - NS : 0); t < kt; ++t)
        mbar_wait(barFull(t % NS), (t / NS) & 1, nullptr);
      for (int r = (nq > 2 ? nq - 2 : 0); r < nq; ++r)
        mbar_wait(barQFull(r & 1), (r >> 1) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kRows, kCols, false, false);
      int kt = 0, st = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int idx = item_of(r, n_items);
        if (idx < 0) break;
        const RowTile tile = p.tiles[idx / p.H_s];
        const int n_ct = p.causal ? tile.tl + 1 : (tile.L + kCols - 1) / kCols;
        const int qb = r & 1;
        if (!mbar_wait(barQFull(qb), (r >> 1) & 1, p.err)) break;
        const uint32_t qa = sb + Lay::kQ + qb * Lay::kTileBytes;
        for (int n = 0; n < n_ct; ++n, ++kt, ++st) {
          const int s = kt % NS, b = st & 1;
          if (!mbar_wait(barFull(s), (kt / NS) & 1, p.err) ||
              !mbar_wait(barSEmpty(b), ((st >> 1) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = sb + Lay::kK + s * Lay::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Lay::kChunkBytes + (kk & 3) * 32;
            tc_mma(tmem + b * kCols, sdesc_sw128(qa + off, 16, 1024),
                   sdesc_sw128(ka + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
          }
          tc_commit(barEmpty(s));
          tc_commit(barSFull(b));
        }
        tc_commit(barQEmpty(qb));
      }
      tc_commit(barDone);
      mbar_wait(barDone, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------- statistics
    constexpr int kSW = StatWarps<BLK>::kN;
    constexpr int kParts = StatWarps<BLK>::kParts;
    constexpr int kPar = StatWarps<BLK>::kPar;
    constexpr int kCW = StatWarps<BLK>::kCW;
    constexpr int kChunks = BLK / kCW;                // passes over this warp's block
    const int wq = warp & 3;
    const int part = (warp - 2) >> 2;                 // 0 .. kParts-1
    const int half = part % StatWarps<BLK>::kHalves;  // block of the tile
    const int parity = part / StatWarps<BLK>::kHalves;  // S buffer (kPar = 2)
    const int row = wq * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t partcol = kPartCol + part * (256 / kParts);  // this warp's per-block partials
    const float sc = p.scale_log2;
    const float2 sc2 = make_float2(sc, sc);
    float* red = reinterpret_cast<float*>(smem + Lay::kRed);
    float* xs = reinterpret_cast<float*>(smem + Lay::kX);
    int st = 0;
    for (int r = 0;; ++r) {
      const int idx = item_of(r, n_items);
      if (idx < 0) break;
      const RowTile tile = p.tiles[idx / p.H_s];
      const int h = idx % p.H_s;
      const int n_ct = p.causal ? tile.tl + 1 : (tile.L + kCols - 1) / kCols;
      const int row_local = tile.tl * kRows + row;
      const bool row_ok = row_local < tile.L;
      const int n_first = (kPar == 1) ? 0 : ((parity - st) & 1);  // first tile of this warp
      float mtrue = -INFINITY, ref = -INFINITY, lsum = 0.f;
      int nblk = 0;
      bool ok = true;
      for (int n = n_first; n < n_ct; n += kPar) {
        const int sn = st + n;
        const int b = sn & 1;
        if (!warp_wait(barSFull(b), (sn >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float bs = 0.f;  // this block's partial, relative to the current reference
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          float x[kCW];
#pragma unroll
          for (int e = 0; e < kCW; e += 32)
            tmem_ld32(trow + b * kCols + half * 64 + c * kCW + e, reinterpret_cast<uint32_t*>(x) + e);
          tc_wait_ld();
          if (c == kChunks - 1) {  // the whole block is in registers or consumed: free the buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barSEmpty(b));
          }
          const int col0 = n * kCols + half * 64 + c * kCW;
          if (n == n_ct - 1) {  // only the last tile can cross the diagonal or the sequence end
#pragma unroll
            for (int e = 0; e < kCW; ++e) {
              const int j = col0 + e;
              if (!((j < tile.L) && (!p.causal || j <= row_local))) x[e] = -INFINITY;
            }
          }
          // chunk max on the raw scores (scaling by sc > 0 preserves order),
          // four independent chains
          float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
          for (int e = 0; e < kCW; e += 8) {
            m0 = fmax3(m0, x[e], x[e + 1]);
            m1 = fmax3(m1, x[e + 2], x[e + 3]);
            m2 = fmax3(m2, x[e + 4], x[e + 5]);
            m3 = fmax3(m3, x[e + 6], x[e + 7]);
          }
          float bm = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * sc;
          if (!row_ok) bm = -INFINITY;
          mtrue = fmaxf(mtrue, bm);
          float alpha = 1.f;
          if (bm > ref + kTau) {
            alpha = (ref == -INFINITY) ? 0.f : ex2(ref - bm);
            ref = bm;
            lsum *= alpha;
            bs *= alpha;
          }
          if (__any_sync(0xffffffffu, alpha != 1.f) && nblk > 0) {
            tc_wait_st();
            rescale_parts(trow + partcol, nblk, alpha);
          }
          // exp2(x * sc - ref) with one packed FMA per two scores, packed sums
          const float nrs = (ref == -INFINITY) ? 0.f : -ref;
          const float2 nrs2 = make_float2(nrs, nrs);
          // four independent packed accumulators
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          float2 acc2 = make_float2(0.f, 0.f), acc3 = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < kCW; e += 8) {
            float2 t0 = ffma2(make_float2(x[e], x[e + 1]), sc2, nrs2);
            float2 t1 = ffma2(make_float2(x[e + 2], x[e + 3]), sc2, nrs2);
            float2 t2 = ffma2(make_float2(x[e + 4], x[e + 5]), sc2, nrs2);
            float2 t3 = ffma2(make_float2(x[e + 6], x[e + 7]), sc2, nrs2);
            t0.x = ex2(t0.x);
            t0.y = ex2(t0.y);
            t1.x = ex2(t1.x);
            t1.y = ex2(t1.y);
            t2.x = ex2(t2.x);
            t2.y = ex2(t2.y);
            t3.x = ex2(t3.x);
            t3.y = ex2(t3.y);
            acc0 = fadd2(acc0, t0);
            acc1 = fadd2(acc1, t1);
            acc2 = fadd2(acc2, t2);
            acc3 = fadd2(acc3, t3);
          }
          const float2 a01 = fadd2(acc0, acc1), a23 = fadd2(acc2, acc3);
          const float2 a = fadd2(a01, a23);
          bs += a.x + a.y;
        }
        if (!row_ok) bs = 0.f;
        lsum += bs;
        tmem_st1(trow + partcol + nblk, __float_as_uint(bs));
        ++nblk;
      }
      tc_wait_st();
      st += n_ct;
      // ------------------------------------------------------ item epilogue
      // A warp whose wait gave up flags it before the barrier; every warp
      // reads the flag after it, so all take the same exit.
      if (!ok && lane == 0) *stat_fail = 1;
      xs[(part * 3 + 0) * 128 + row] = mtrue;
      xs[(part * 3 + 1) * 128 + row] = ref;
      xs[(part * 3 + 2) * 128 + row] = lsum;
      named_bar(1, 32 * kSW);
      const bool good = (*stat_fail == 0);
      // merge the parts of each row (separate lazy references), in part order
      float M = -INFINITY, Rf = -INFINITY;
#pragma unroll
      for (int q = 0; q < kParts; ++q) {
        M = fmaxf(M, xs[(q * 3 + 0) * 128 + row]);
        Rf = fmaxf(Rf, xs[(q * 3 + 1) * 128 + row]);
      }
      float Lt = 0.f, own_scale = 0.f;
      if (Rf != -INFINITY) {
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
          const float rq = xs[(q * 3 + 1) * 128 + row];
          const float sq = (rq == -INFINITY) ? 0.f : ex2(rq - Rf);
          Lt += xs[(q * 3 + 2) * 128 + row] * sq;
          if (q == part) own_scale = sq;
        }
      }
      const float inv = (row_ok && Lt > 0.f) ? own_scale / Lt : 0.f;
      if (good && row_ok && part == 0) {
        const size_t o = static_cast<size_t>(h) * p.T + tile.seq_start + row_local;
        p.row_max[o] = M * kLn2;
        p.row_sum[o] = Lt * ex2(Rf - M);
      }
      for (int c0 = 0; c0 < nblk; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(trow + partcol + c0, v);
        tc_wait_ld();
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = (c0 + i < nblk) ? __uint_as_float(v[i]) * inv : 0.f;
        const float tot = transpose_reduce32(f);
        const int k = c0 + lane;
        const int n = n_first + kPar * k;  // tile of this warp's k-th partial
        if (k < nblk) red[wq * 256 + (BLK == 64 ? 2 * n + half : n)] = tot;
      }
      tc_fence_before();
      named_bar(1, 32 * kSW);
      if (!good) break;
      const int t0 = threadIdx.x - 64;
      const int nbt = (BLK == 64) ? 2 * n_ct : n_ct;  // block columns covered
      if (BLK == 64) {
        for (int t = t0; t < 2 * nbt; t += 32 * kSW) {
          const int hb = t / nbt, c = t - hb * nbt;
          const int bi = tile.tl * 2 + hb;
          if (bi * 64 >= tile.L) continue;
          const RowBlock rbk = p.rbs[tile.rb0 + hb];
          const int ncand = p.causal ? rbk.bi + 1 : (tile.L + 63) / 64;
          if (c >= ncand) continue;
          const float m = red[(2 * hb) * 256 + c] + red[(2 * hb + 1) * 256 + c];
          p.mass[static_cast<size_t>(h) * p.C + rbk.cand_off + c] = m;
        }
      } else {
        const RowBlock rbk = p.rbs[tile.rb0];
        const int ncand = p.causal ? rbk.bi + 1 : (tile.L + BLK - 1) / BLK;
        for (int c = t0; c < ncand; c += 32 * kSW) {
          const float m = (red[c] + red[256 + c]) + (red[512 + c] + red[768 + c]);
          p.mass[static_cast<size_t>(h) * p.C + rbk.cand_off + c] = m;
        }
      }
      // the next item rewrites xs after this item's second barrier (all xs
      // reads are before it) and red after its own first barrier (all red
      // reads above are before every warp's arrival there)
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int BLK>
cudaError_t launch_stats_t(const CompressParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           cudaStream_t s) {
  auto kern = stats_bf16_kernel<D, BLK>;
  const int smem = StatsLayout<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.n_tiles) * p.H_s;
  if (items <= 0) return cudaSuccess;
  // persistent: one CTA per SM (the 512 TMEM columns and the shared memory
  // allow no second one), each walking its share of the item list
  const int grid = static_cast<int>(items < sms ? items : sms);
  kern<<<grid, StatWarps<BLK>::kThreads, smem, s>>>(tq, tk, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stats_bf16(const CompressParams& p, const CUtensorMap& tq,
                              const CUtensorMap& tk, cudaStream_t s) {
  if (p.d == 128 && p.B == 64) return launch_stats_t<128, 64>(p, tq, tk, s);
  if (p.d == 128 && p.B == 128) return launch_stats_t<128, 128>(p, tq, tk, s);
  if (p.d == 64 && p.B == 64) return launch_stats_t<64, 64>(p, tq, tk, s);
  if (p.d == 64 && p.B == 128) return launch_stats_t<64, 128>(p, tq, tk, s);
  return cudaErrorInvalidValue;
}

}  // namespace mf
