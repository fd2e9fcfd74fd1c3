// mf_stats2_tc.cu — Attention State Compressor, step 1 (block statistics) on
// the sm_103a tensor cores, bf16 inputs: the kernel for rows of at most 128
// candidate blocks, two CTAs per SM.
//
// It computes what stats_bf16_kernel (mf_stats_tc.cu) computes — "Accelerating
// Cross-Model LLM Inference via Attention Map Reuse", section "Practical
// Implementation Details", and the news article
// "北大MapFlow：注意力图跨模型复用，prefill延迟降15%–20%", paragraph "其一":
// in one pass over Q.K^T, the row max m_i and row sum l_i of the causal
// softmax of s_ij = q_i.k_j/sqrt(d), and the probability mass of every
// candidate B x B block — with a smaller footprint per CTA, so that two
// independent CTAs share an SM and one's waits and epilogues overlap the
// other's tiles.
//
// CTA = persistent walker of (128 query rows of one sequence, one sender head)
// items, in the handle's order table when it has one: sequence by sequence,
// heads in chunks whose keys fit in L2, heaviest tiles first within a chunk,
// so that the CTAs running at one time re-read the same keys from L2 (on 16
// packed sequences with 40 KV heads this is 4 % faster than the tile-major
// heavy-first order, which is what a single short sequence gets anyway).
// Warp roles:
//   warp 0  TMA producer: Q of each item (one buffer), K tiles of 64 keys
//           through a 4-6 stage ring that runs on across items
//   warp 1  tcgen05 issuer: S = Q.K^T (M = 128, N = 64, K = d) into one of
//           two TMEM buffers (fp32, columns 0..63 and 64..127)
//   warps 2-5  statistics, one per TMEM lane quadrant, one thread per query
//           row, every tile: tile max, lazily re-referenced exp2 (the
//           reference moves only when a tile's max exceeds it by more than
//           2^8; stored partials are then rescaled), per-(row, block) partial
//           sums in TMEM columns 128..255, running row sum
//   end of item: mass[bi][bj] = sum over the block-row's rows of partial / l,
//           reduced across lanes with a 31-shuffle transpose-reduction and
//           across the quadrants in a fixed order (deterministic).
// TMEM: 256 columns per CTA; shared memory ~100 KB per CTA at d = 128.
#include <cmath>

#include "mf_internal.cuh"
#include "mf_ptx.cuh"
#include "mf_stats_common.cuh"

namespace mf {
namespace {

constexpr int kRows = 128;              // query rows per item
constexpr int kKeys = 64;               // keys per S tile
constexpr uint32_t kPartCol = 128;      // first TMEM column of the partials
constexpr int kMaxBlocks = 128;         // partial columns per row
constexpr float kTau = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kThreads = 192;           // warp 0 TMA, warp 1 MMA, warps 2-5 statistics

template <int D>
struct Stats2Layout {
  static constexpr int kQChunk = kRows * 128;   // 128 rows x 64 bf16
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kKChunk = kKeys * 128;   // 64 keys x 64 bf16
  static constexpr int kKBytes = kKeys * D * 2;
  static constexpr int kStages = (D == 128) ? 4 : 6;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kRed = kK + kStages * kKBytes;  // float [4][kMaxBlocks]
  static constexpr int kBar = kRed + 4 * kMaxBlocks * 4;
  static constexpr int kSlot = kBar + 24 * 8;
  static constexpr int kFlag = kSlot + 8;
  static constexpr int kBytes = kFlag + 8 + 1024;  // + alignment slack
  static_assert(2 * (kBytes + 1024) <= 228 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try(bar, parity);  // every lane observes the completed phase
  __syncwarp();
  return ok != 0;
}

// Item r of this CTA in a snake order over the (tile, head) list:
// round r takes items [r*G, r*G+G), forwards on even rounds and backwards on
// odd ones, so every CTA's total work stays within one item of the others.
// -1 once the list is exhausted.
__device__ __forceinline__ int item_of(int r, int n_items) {
  const int G = gridDim.x;
  const int idx = r * G + ((r & 1) ? (G - 1 - static_cast<int>(blockIdx.x))
                                    : static_cast<int>(blockIdx.x));
  return idx < n_items ? idx : -1;
}

// 64-key tiles of an item: up to the diagonal (causal) or the sequence end.
__device__ __forceinline__ int key_tiles(const RowTile& tile, int causal) {
  return causal ? (tile.tl + 1) * (kRows / kKeys) : (tile.L + kKeys - 1) / kKeys;
}

template <int D, int BLK>
__global__ void __launch_bounds__(kThreads, 2)
    stats2_bf16_kernel(const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap tk, const CompressParams p) {
  using Lay = Stats2Layout<D>;
  constexpr int NS = Lay::kStages;
  constexpr int kTPB = BLK / kKeys;  // S tiles per block: 1 at B = 64, 2 at B = 128
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_tiles * p.H_s;

  const uint32_t barQFull = sb + Lay::kBar;
  const uint32_t barQEmpty = sb + Lay::kBar + 8u;
  auto barFull = [&](int s) { return sb + Lay::kBar + 8u * (2 + s); };
  auto barEmpty = [&](int s) { return sb + Lay::kBar + 8u * (2 + NS + s); };
  auto barSFull = [&](int b) { return sb + Lay::kBar + 8u * (2 + 2 * NS + b); };
  auto barSEmpty = [&](int b) { return sb + Lay::kBar + 8u * (4 + 2 * NS + b); };
  const uint32_t barDone = sb + Lay::kBar + 8u * (6 + 2 * NS);
  volatile int* stat_fail = reinterpret_cast<volatile int*>(smem + Lay::kFlag);

  if (threadIdx.x == 0) {
    mbar_init(barQFull, 1);
    mbar_init(barQEmpty, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(barFull(s), 1);
      mbar_init(barEmpty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(barSFull(b), 1);
      mbar_init(barSEmpty(b), 4);  // the four statistics warps
    }
    mbar_init(barDone, 1);
    *stat_fail = 0;
    fence_mbar_init();
    if (blockIdx.x == 0 && p.sel_done) *p.sel_done = 0;  // the selection kernel's CTA count
  }
  if (warp == 1) tmem_alloc(sb + Lay::kSlot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + Lay::kSlot);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      int kt = 0, nq = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int idx = item_of(r, n_items);
        if (idx < 0) break;
        int ti, h;
        item_tile_head(p, idx, ti, h);
        const RowTile tile = p.tiles[ti];
        const int hk = h / (p.H_s / p.H_ks);
        const int n_ct = key_tiles(tile, p.causal);
        // Q of this item replaces the previous item's once its MMAs are done
        if (!mbar_wait(barQEmpty, (r & 1) ^ 1, p.err)) break;
        mbar_arrive_tx(barQFull, Lay::kQBytes);
        const int qrow = tile.seq_start + tile.tl * kRows;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sb + Lay::kQ + c * Lay::kQChunk, &tq, h * D + c * 64, qrow, barQFull);
        nq = r + 1;
        for (int n = 0; n < n_ct; ++n, ++kt) {
          const int s = kt % NS;
          if (!mbar_wait(barEmpty(s), ((kt / NS) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_tx(barFull(s), Lay::kKBytes);
          const uint32_t dst = sb + Lay::kK + s * Lay::kKBytes;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(dst + c * Lay::kKChunk, &tk, hk * D + c * 64, tile.seq_start + n * kKeys,
                        barFull(s));
        }
      }
      // drain: copies still in flight complete before the CTA may exit (each
      // wait is on the latest use of its barrier)
      for (int t = (kt > NS ? kt - NS : 0); t < kt; ++t) mbar_wait(barFull(t % NS), (t / NS) & 1, nullptr);
      if (nq > 0) mbar_wait(barQFull, (nq - 1) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kRows, kKeys, false, false);
      int kt = 0, st = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int idx = item_of(r, n_items);
        if (idx < 0) break;
        int ti, hi;
        item_tile_head(p, idx, ti, hi);
        const RowTile tile = p.tiles[ti];
        const int n_ct = key_tiles(tile, p.causal);
        if (!mbar_wait(barQFull, r & 1, p.err)) break;
        for (int n = 0; n < n_ct; ++n, ++kt, ++st) {
          const int s = kt % NS, b = st & 1;
          if (!mbar_wait(barFull(s), (kt / NS) & 1, p.err) ||
              !mbar_wait(barSEmpty(b), ((st >> 1) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qa = sb + Lay::kQ, ka = sb + Lay::kK + s * Lay::kKBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            tc_mma(tmem + b * kKeys, sdesc_sw128(qa + (kk >> 2) * Lay::kQChunk + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(ka + (kk >> 2) * Lay::kKChunk + (kk & 3) * 32, 16, 1024), idesc,
                   kk > 0 ? 1u : 0u);
          }
          tc_commit(barEmpty(s));
          tc_commit(barSFull(b));
        }
        if (ok) tc_commit(barQEmpty);  // Q may be replaced once these MMAs finish
      }
      tc_commit(barDone);
      mbar_wait(barDone, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------- statistics
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sc = p.scale_log2;
    const float2 sc2 = make_float2(sc, sc);
    float* red = reinterpret_cast<float*>(smem + Lay::kRed);
    int st = 0;
    for (int r = 0;; ++r) {
      const int idx = item_of(r, n_items);
      if (idx < 0) break;
      int ti, h;
      item_tile_head(p, idx, ti, h);
      const RowTile tile = p.tiles[ti];
      const int n_ct = key_tiles(tile, p.causal);
      const int row_local = tile.tl * kRows + row;
      const bool row_ok = row_local < tile.L;
      float mtrue = -INFINITY, ref = -INFINITY, lsum = 0.f;
      float bs = 0.f;  // this block's partial, relative to the current reference
      int nblk = 0;
      bool ok = true;
      for (int n = 0; n < n_ct; ++n) {
        const int sn = st + n;
        const int b = sn & 1;
        if (!warp_wait(barSFull(b), (sn >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float x[kKeys];
        tmem_ld32(trow + b * kKeys, reinterpret_cast<uint32_t*>(x));
        tmem_ld32(trow + b * kKeys + 32, reinterpret_cast<uint32_t*>(x) + 32);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(barSEmpty(b));  // the tile is in registers
        const int col0 = n * kKeys;
        // only the tiles at the diagonal or the sequence end hold invisible keys
        if (col0 + kKeys > tile.L || (p.causal && col0 + kKeys - 1 > tile.tl * kRows)) {
#pragma unroll
          for (int e = 0; e < kKeys; ++e) {
            const int j = col0 + e;
            if (!((j < tile.L) && (!p.causal || j <= row_local))) x[e] = -INFINITY;
          }
        }
        // tile max on the raw scores (scaling by sc > 0 preserves order),
        // four independent chains
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int e = 0; e < kKeys; e += 8) {
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
          rescale_parts(trow + kPartCol, nblk, alpha);
        }
        // exp2(x * sc - ref) with one packed FMA per two scores, four
        // independent packed accumulators
        const float nrs = (ref == -INFINITY) ? 0.f : -ref;
        const float2 nrs2 = make_float2(nrs, nrs);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        float2 acc2 = make_float2(0.f, 0.f), acc3 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < kKeys; e += 8) {
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
        if (n % kTPB == kTPB - 1 || n == n_ct - 1) {  // the block's last tile
          if (!row_ok) bs = 0.f;
          lsum += bs;
          tmem_st1(trow + kPartCol + nblk, __float_as_uint(bs));
          ++nblk;
          bs = 0.f;
        }
      }
      tc_wait_st();
      st += n_ct;
      // ------------------------------------------------------ item epilogue
      // A warp whose wait gave up flags it before the barrier; every warp
      // reads the flag after it, so all take the same exit.
      if (!ok && lane == 0) *stat_fail = 1;
      named_bar(1, 128);
      const bool good = (*stat_fail == 0);
      const float inv = (row_ok && lsum > 0.f) ? 1.f / lsum : 0.f;
      if (good && row_ok) {
        const size_t o = static_cast<size_t>(h) * p.T + tile.seq_start + row_local;
        p.row_max[o] = mtrue * kLn2;
        p.row_sum[o] = lsum * ex2(ref - mtrue);
      }
      for (int c0 = 0; c0 < nblk; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(trow + kPartCol + c0, v);
        tc_wait_ld();
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = (c0 + i < nblk) ? __uint_as_float(v[i]) * inv : 0.f;
        const float tot = transpose_reduce32(f);
        if (c0 + lane < nblk) red[wq * kMaxBlocks + c0 + lane] = tot;
      }
      tc_fence_before();
      named_bar(1, 128);
      if (!good) break;
      const int t0 = threadIdx.x - 64;
      if (BLK == 64) {
        // block-row hb of the tile = rows of quadrants 2hb and 2hb + 1
        for (int t = t0; t < 2 * nblk; t += 128) {
          const int hb = t / nblk, c = t - hb * nblk;
          const int bi = tile.tl * 2 + hb;
          if (bi * 64 >= tile.L) continue;
          const RowBlock rbk = p.rbs[tile.rb0 + hb];
          const int ncand = p.causal ? rbk.bi + 1 : (tile.L + 63) / 64;
          if (c >= ncand) continue;
          const float m = red[(2 * hb) * kMaxBlocks + c] + red[(2 * hb + 1) * kMaxBlocks + c];
          p.mass[static_cast<size_t>(h) * p.C + rbk.cand_off + c] = m;
        }
      } else {
        const RowBlock rbk = p.rbs[tile.rb0];
        const int ncand = p.causal ? rbk.bi + 1 : (tile.L + BLK - 1) / BLK;
        for (int c = t0; c < ncand; c += 128) {
          const float m = (red[c] + red[kMaxBlocks + c]) + (red[2 * kMaxBlocks + c] + red[3 * kMaxBlocks + c]);
          p.mass[static_cast<size_t>(h) * p.C + rbk.cand_off + c] = m;
        }
      }
      // the next item rewrites red only after its own first barrier, which
      // every warp reaches after the reads above
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int D, int BLK>
cudaError_t launch_stats2_t(const CompressParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            cudaStream_t s) {
  auto kern = stats2_bf16_kernel<D, BLK>;
  const int smem = Stats2Layout<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.n_tiles) * p.H_s;
  if (items <= 0) return cudaSuccess;
  // persistent: two CTAs per SM, each walking its share of the item list
  const long long slots = 2ll * sms;
  const int grid = static_cast<int>(items < slots ? items : slots);
  kern<<<grid, kThreads, smem, s>>>(tq, tk, p);
  return cudaGetLastError();
}

}  // namespace

bool stats2_supported(int max_cand) { return max_cand <= kMaxBlocks; }

cudaError_t launch_stats2_bf16(const CompressParams& p, const CUtensorMap& tq,
                               const CUtensorMap& tk64, cudaStream_t s) {
  if (p.d == 128 && p.B == 64) return launch_stats2_t<128, 64>(p, tq, tk64, s);
  if (p.d == 128 && p.B == 128) return launch_stats2_t<128, 128>(p, tq, tk64, s);
  if (p.d == 64 && p.B == 64) return launch_stats2_t<64, 64>(p, tq, tk64, s);
  if (p.d == 64 && p.B == 128) return launch_stats2_t<64, 128>(p, tq, tk64, s);
  return cudaErrorInvalidValue;
}

}  // namespace mf
