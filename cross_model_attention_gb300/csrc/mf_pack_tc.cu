// mf_pack_tc.cu — Attention State Compressor, step 3: pack the kept
// probability tiles into Block Sparse Row form, bf16 inputs, sm_103a.
//
// "Accelerating Cross-Model LLM Inference via Attention Map Reuse", section
// "Practical Implementation Details": the filtered map is stored in a compact
// Block Sparse Row layout.  Row statistics m_i, l_i come from the statistics
// pass; here only the kept tiles are recomputed (Q.K^T on tcgen05 into TMEM),
// normalised, P_ij = 2^(s_ij*log2(e)/sqrt(d) - m_i*log2(e) - log2(l_i)),
// rounded to bf16 and written with TMA tensor stores from swizzled staging
// buffers (so that every HBM write is a full, coalesced line).
//
// Persistent: two CTAs per SM at B = 64 (one at B = 128) take (128-row tile,
// sender head) items from a global counter, heaviest tiles first, so the
// last items taken are light ones whatever the kept blocks make each item
// cost.  Warp roles: warp 0 TMA loads (Q of
// each item, K blocks through a ring that runs on across items), warp 1
// tcgen05 issue, warps 2-9 normalise and store (two per TMEM lane quadrant,
// one per half of the block's columns; each warp stages its 32 x B/2 slice in
// its own swizzled buffer and issues its own TMA store, so the writer warps
// never wait on one another), warp 10 plans the next item while the
// current one runs: the ascending union of its block-rows' kept columns, the
// rows' statistics, and the col_idx / per-(block, head) tile index entries
// used by the retrieval, with this head's column of the retrieval's
// union-ordered tile table (and, for head 0, the union list).  Plans are
// double-buffered, so item setup is off the critical path.
#include <cmath>

#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kRows = 128;
constexpr int kMaxU = 264;

template <int D, int BLK>
struct PackLayout {
  static constexpr int kQChunk = kRows * 128;
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kKChunk = BLK * 128;            // BLK key rows x 64 bf16
  static constexpr int kKBytes = BLK * D * 2;
  static constexpr int kStages = 3;
  static constexpr int kWarpStage = 32 * BLK;           // one writer warp's 32 rows x BLK/2 bf16
  static constexpr int kStageBytes = 8 * kWarpStage;
  // plan of one item: union columns, their positions in the two kept lists,
  // the rows' exponent offsets, and the item's scalars
  static constexpr int kPlanInts = 3 * kMaxU + kRows + 8;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kStg = kK + kStages * kKBytes;
  static constexpr int kPlan = kStg + kStageBytes;     // two plans
  static constexpr int kFl = kPlan + 2 * kPlanInts * 4; // planner's two flag arrays
  static constexpr int kBar = kFl + 2 * kMaxU * 4;
  static constexpr int kSlot = kBar + 32 * 8;
  static constexpr int kMisc = kSlot + 8;
  static constexpr int kBytes = kMisc + 16 + 1024;
};

// Fields of a plan (int offsets).
constexpr int kPlBj = 0, kPlPos0 = kMaxU, kPlPos1 = 2 * kMaxU, kPlM2 = 3 * kMaxU,
              kPlMeta = 3 * kMaxU + kRows;
// meta: [0] n_u (-1: no more items), [1] head, [2] seq_start, [3] L, [4] tile
// index in the sequence, [5] row_ptr of block-row 0, [6] row_ptr of block-row 1

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try(bar, parity);
  __syncwarp();
  return ok != 0;
}


// Writer warps: two per TMEM lane quadrant, each normalising half of the
// block's columns; one planner warp.
constexpr int kPackThreads = 64 + 256 + 32;

template <int D, int BLK>
__global__ void __launch_bounds__(kPackThreads, (BLK == 64) ? 2 : 1)
    pack_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tvals, const CompressParams p) {
  using Lay = PackLayout<D, BLK>;
  constexpr int NS = Lay::kStages;
  constexpr int kN = BLK;  // MMA N = key block width
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_tiles * p.H_s;
  auto plan = [&](int k) { return reinterpret_cast<int*>(smem + Lay::kPlan) + (k & 1) * Lay::kPlanInts; };
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::kMisc);  // [1] = abort

  const uint32_t barQ = sb + Lay::kBar;
  const uint32_t barQEmpty = sb + Lay::kBar + 8u;
  auto barFull = [&](int s) { return sb + Lay::kBar + 8u * (2 + s); };
  auto barEmpty = [&](int s) { return sb + Lay::kBar + 8u * (2 + NS + s); };
  auto barSFull = [&](int b) { return sb + Lay::kBar + 8u * (2 + 2 * NS + b); };
  auto barSEmpty = [&](int b) { return sb + Lay::kBar + 8u * (4 + 2 * NS + b); };
  auto barReady = [&](int k) { return sb + Lay::kBar + 8u * (6 + 2 * NS + (k & 1)); };
  auto barFree = [&](int k) { return sb + Lay::kBar + 8u * (8 + 2 * NS + (k & 1)); };
  const uint32_t barDone = sb + Lay::kBar + 8u * (10 + 2 * NS);

  if (threadIdx.x == 0) {
    mbar_init(barQ, 1);
    mbar_init(barQEmpty, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(barFull(s), 1);
      mbar_init(barEmpty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(barSFull(b), 1);
      mbar_init(barSEmpty(b), 8);
      mbar_init(barReady(b), 1);
      mbar_init(barFree(b), 10);  // loader, MMA issuer, eight writer warps
    }
    mbar_init(barDone, 1);
    fence_mbar_init();
    misc[1] = 0;
  }
  if (warp == 1) tmem_alloc(sb + Lay::kSlot, 2 * kN < 32 ? 32 : 2 * kN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + Lay::kSlot);

  if (warp == 10) {
    // ------------------------------------------------------------ planner
    int* fl0 = reinterpret_cast<int*>(smem + Lay::kFl);  // position of column bj in kept list 0 (or -1)
    int* fl1 = fl0 + kMaxU;
    // the all-zero tile the retrieval reads for a head's dropped block
    if (blockIdx.x == 0 && p.zero_tile) {
      uint4* z = reinterpret_cast<uint4*>(p.zero_tile);
      for (int i = lane; i < BLK * BLK / 8; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int k = 0;; ++k) {
      if (misc[1]) break;
      if (!warp_wait(barFree(k), ((k >> 1) & 1) ^ 1, p.err)) {
        misc[1] = 1;
        break;
      }
      int* pl = plan(k);
      int idx = 0;
      if (lane == 0) idx = atomicAdd(p.pack_ctr, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (idx >= n_items) {
        // no more items: an empty plan tells the other roles to stop
        if (lane == 0) {
          pl[kPlMeta + 0] = -1;
          mbar_arrive(barReady(k));
        }
        break;
      }
      // item idx: the host's order table, or tile idx / H_s of the
      // heavy-first tile list and head idx % H_s
      int ti, h;
      if (p.items) {
        const int it = p.items[idx];
        ti = it >> 8;
        h = it & 255;
      } else {
        ti = idx / p.H_s;
        h = idx - ti * p.H_s;
      }
      const RowTile tile = p.tiles[ti];
      const int nsub = kRows / BLK;  // 2 for B=64, 1 for B=128
      int rbv[2], kc[2], base[2];
      const int* kl[2];
      for (int t = 0; t < 2; ++t) {
        const bool exists = t < nsub && (tile.tl * kRows + t * BLK) < tile.L;
        rbv[t] = exists ? tile.rb0 + t : -1;
        kc[t] = 0;
        base[t] = 0;
        kl[t] = nullptr;
        if (exists) {
          const int row = h * p.R + rbv[t];
          kc[t] = p.kcount[row];
          base[t] = p.row_ptr[row];
          kl[t] = p.keptcols + static_cast<size_t>(h) * p.C + p.rbs[rbv[t]].cand_off;
        }
      }
      const int nbj = p.causal ? (tile.tl + 1) * (kRows / BLK) : (tile.L + BLK - 1) / BLK;
      for (int i = lane; i < nbj; i += 32) {
        fl0[i] = -1;
        fl1[i] = -1;
      }
      __syncwarp();
      for (int t = 0; t < 2; ++t) {
        if (rbv[t] < 0) continue;
        const int cand_off = p.rbs[rbv[t]].cand_off;
        int* fl = t ? fl1 : fl0;
        for (int i = lane; i < kc[t]; i += 32) {
          const int bj = kl[t][i];
          fl[bj] = i;
          // col_idx and the retrieval's tile index of every kept (block, head)
          p.col_idx[base[t] + i] = bj;
          p.tile_of[static_cast<size_t>(cand_off + bj) * p.H_s + h] = base[t] + i;
        }
      }
      __syncwarp();
      int n = 0;
      for (int c0 = 0; c0 < nbj; c0 += 32) {
        const int bj = c0 + lane;
        const int a = (bj < nbj) ? fl0[bj] : -1, b = (bj < nbj) ? fl1[bj] : -1;
        const bool f = (a >= 0) || (b >= 0);
        const uint32_t m = __ballot_sync(0xffffffffu, f);
        if (f) {
          const int pos = n + __popc(m & ((1u << lane) - 1u));
          pl[kPlBj + pos] = bj;
          pl[kPlPos0 + pos] = a;
          pl[kPlPos1 + pos] = b;
        }
        n += __popc(m);
      }
      // exponent offset of each row: m_i log2(e) + log2(l_i), so that the
      // division by the row sum folds into the exp2
      // the retrieval's tables, from the selection's per-row kept-column
      // masks: this head's tile index at every union column of the block-row
      // (-1 where it dropped the block) and, for head 0, the union list
      if (p.union_in_pack) {
        for (int t = 0; t < 2; ++t) {
          if (rbv[t] < 0) continue;
          const RowBlock rbk = p.rbs[rbv[t]];
          const int ncand = p.causal ? rbk.bi + 1 : (rbk.L + BLK - 1) / BLK;
          // union over the heads of their kept-column masks: lane w + 8j ORs
          // word w of heads j, j + 4, ...; then the four partial ORs combine
          uint32_t mw = 0u;
          for (int hh = lane >> 3; hh < p.H_s; hh += 4)
            mw |= p.kmask[(static_cast<size_t>(hh) * p.R + rbv[t]) * 8 + (lane & 7)];
          mw |= __shfl_xor_sync(0xffffffffu, mw, 8);
          mw |= __shfl_xor_sync(0xffffffffu, mw, 16);
          int pre = (lane < 8) ? __popc(mw) : 0;
#pragma unroll
          for (int off = 1; off < 8; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, pre, off);
            if (lane >= off) pre += y;
          }
          const int ucnt = __shfl_sync(0xffffffffu, pre, 7);
          pre -= (lane < 8) ? __popc(mw) : 0;  // exclusive over the words
          const int* flt = t ? fl1 : fl0;
          for (int c0 = 0; c0 < ncand; c0 += 32) {
            const uint32_t word = __shfl_sync(0xffffffffu, mw, c0 >> 5);
            const int wpre = __shfl_sync(0xffffffffu, pre, c0 >> 5);
            const int bj = c0 + lane;
            if (bj < ncand && ((word >> lane) & 1u)) {
              const int j = wpre + __popc(word & ((1u << lane) - 1u));
              const int pos = flt[bj];
              p.utile[static_cast<size_t>(rbk.cand_off + j) * p.H_s + h] = pos >= 0 ? base[t] + pos : -1;
              if (h == 0) p.union_list[rbk.cand_off + j] = bj;
            }
          }
          if (h == 0 && lane == 0) p.union_cnt[rbv[t]] = ucnt;
        }
      }
      float* m2 = reinterpret_cast<float*>(pl + kPlM2);
      for (int r = lane; r < kRows; r += 32) {
        const int row_local = tile.tl * kRows + r;
        float mm = 0.f;
        if (n > 0 && row_local < tile.L) {
          const size_t o = static_cast<size_t>(h) * p.T + tile.seq_start + row_local;
          mm = p.row_max[o] * 1.4426950408889634f + log2f(p.row_sum[o]);
        }
        m2[r] = mm;
      }
      if (lane == 0) {
        pl[kPlMeta + 0] = n;
        pl[kPlMeta + 1] = h;
        pl[kPlMeta + 2] = tile.seq_start;
        pl[kPlMeta + 3] = tile.L;
        pl[kPlMeta + 4] = tile.tl;
        pl[kPlMeta + 5] = base[0];
        pl[kPlMeta + 6] = base[1];
      }
      // the flags are rewritten for the next item only after every lane has
      // read them; the plan is published by the arrive's release
      __syncwarp();
      if (lane == 0) mbar_arrive(barReady(k));
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------- loader
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tvals);
      int g = 0, nq = 0;
      for (int k = 0;; ++k) {
        if (misc[1]) break;
        if (!mbar_wait(barReady(k), (k >> 1) & 1, p.err)) {
          misc[1] = 1;
          break;
        }
        const int* pl = plan(k);
        const int n_u = pl[kPlMeta + 0], h = pl[kPlMeta + 1];
        if (n_u < 0) break;
        const int y0 = pl[kPlMeta + 2] + pl[kPlMeta + 4] * kRows;
        const int hk = h / (p.H_s / p.H_ks);
        bool ok = true;
        if (n_u > 0) {
          // Q of this item replaces the previous item's once its MMAs are done
          if (!mbar_wait(barQEmpty, (nq & 1) ^ 1, p.err)) {
            ok = false;
          } else {
            mbar_arrive_tx(barQ, Lay::kQBytes);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d(sb + Lay::kQ + c * Lay::kQChunk, &tq, h * D + c * 64, y0, barQ);
            ++nq;
          }
        }
        for (int u = 0; ok && u < n_u; ++u, ++g) {
          const int s = g % NS;
          if (!mbar_wait(barEmpty(s), ((g / NS) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_tx(barFull(s), Lay::kKBytes);
          const uint32_t dst = sb + Lay::kK + s * Lay::kKBytes;
          const int ky = pl[kPlMeta + 2] + pl[kPlBj + u] * BLK;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) tma_load_2d(dst + c * Lay::kKChunk, &tk, hk * D + c * 64, ky, barFull(s));
        }
        mbar_arrive(barFree(k));
        if (!ok) {
          misc[1] = 1;
          break;
        }
      }
      // drain: the last loads of every stage and the last Q
      for (int u = (g > NS ? g - NS : 0); u < g; ++u) mbar_wait(barFull(u % NS), (u / NS) & 1, nullptr);
      if (nq > 0) mbar_wait(barQ, (nq - 1) & 1, nullptr);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kRows, kN, false, false);
      int g = 0, nq = 0;
      for (int k = 0;; ++k) {
        if (misc[1]) break;
        if (!mbar_wait(barReady(k), (k >> 1) & 1, p.err)) {
          misc[1] = 1;
          break;
        }
        const int n_u = plan(k)[kPlMeta + 0];
        if (n_u < 0) break;
        mbar_arrive(barFree(k));
        bool ok = true;
        if (n_u > 0) {
          ok = mbar_wait(barQ, nq & 1, p.err);
          ++nq;
        }
        for (int u = 0; ok && u < n_u; ++u, ++g) {
          const int s = g % NS, b = g & 1;
          if (!mbar_wait(barFull(s), (g / NS) & 1, p.err) ||
              !mbar_wait(barSEmpty(b), ((g >> 1) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qa = sb + Lay::kQ, ka = sb + Lay::kK + s * Lay::kKBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            tc_mma(tmem + b * kN, sdesc_sw128(qa + (kk >> 2) * Lay::kQChunk + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(ka + (kk >> 2) * Lay::kKChunk + (kk & 3) * 32, 16, 1024), idesc,
                   kk > 0 ? 1u : 0u);
          }
          tc_commit(barEmpty(s));
          tc_commit(barSFull(b));
        }
        if (!ok) {
          misc[1] = 1;
          break;
        }
        if (n_u > 0) tc_commit(barQEmpty);  // Q may be replaced once these MMAs finish
      }
      tc_commit(barDone);
      mbar_wait(barDone, 0, nullptr);
    }
  } else {
    // ------------------------------------------------ normalise + store
    constexpr int kHalfCols = BLK / 2;  // columns per writer warp
    const int wq = warp & 3;
    const int ch = (warp - 2) >> 2;     // column half of this warp
    const int row = wq * 32 + lane;
    const int sub = row / BLK;  // which block-row of the tile
    const int rloc0 = wq * 32 - sub * BLK;  // the warp's first row in its block-row
    const uint32_t trow = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sc = p.scale_log2;
    // this warp's staging buffer: 32 rows of BLK/2 bf16 in the layout of the
    // store map's swizzle (64-byte rows at B = 64, 128-byte rows at B = 128)
    const uint32_t wstg = sb + Lay::kStg + (warp - 2) * Lay::kWarpStage;
    uint8_t* wstg_g = smem + Lay::kStg + (warp - 2) * Lay::kWarpStage;
    const float2 sc2 = make_float2(sc, sc);
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (misc[1]) break;
      if (!warp_wait(barReady(k), (k >> 1) & 1, p.err)) break;
      const int* pl = plan(k);
      const int n_u = pl[kPlMeta + 0];
      if (n_u < 0) break;
      const int L = pl[kPlMeta + 3], tl = pl[kPlMeta + 4];
      const int base_sub = pl[kPlMeta + 5 + sub];
      const int* u_pos = pl + (sub == 0 ? kPlPos0 : kPlPos1);
      const int row_local = tl * kRows + row;
      const bool row_ok = row_local < L;
      const float m2 = reinterpret_cast<const float*>(pl + kPlM2)[row];
      const float2 nm2 = make_float2(-m2, -m2);
      for (int u = 0; u < n_u; ++u, ++g) {
        const int b = g & 1;
        if (!warp_wait(barSFull(b), (g >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[kHalfCols];
        {
          uint32_t* r = reinterpret_cast<uint32_t*>(s);
#pragma unroll
          for (int c = 0; c < kHalfCols; c += 32) tmem_ld32(trow + b * kN + ch * kHalfCols + c, r + c);
        }
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(barSEmpty(b));
        const int pos = u_pos[u];
        if (pos < 0) continue;  // this block-row does not keep the block (warp-uniform)
        const int bj = pl[kPlBj + u];
        // the store issued from this warp's buffer one tile ago must have
        // finished reading it
        if (lane == 0) bulk_wait_read_0();
        __syncwarp();
        // only the diagonal block and the sequence's last block need masking
        const bool edge = !row_ok || (bj * BLK + BLK > L) ||
                          (p.causal && bj * BLK + BLK - 1 > tl * kRows + sub * BLK);
        const int c_base = ch * kHalfCols;
#pragma unroll
        for (int c8 = 0; c8 < kHalfCols / 8; ++c8) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float2 t = ffma2(make_float2(s[c8 * 8 + e], s[c8 * 8 + e + 1]), sc2, nm2);
            v[e] = ex2(t.x);
            v[e + 1] = ex2(t.y);
          }
          if (edge) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = bj * BLK + c_base + c8 * 8 + e;
              const bool vis = row_ok && (j < L) && (!p.causal || j <= row_local);
              if (!vis) v[e] = 0.f;
            }
          }
          uint4 w;
          w.x = pack_bf16x2(v[0], v[1]);
          w.y = pack_bf16x2(v[2], v[3]);
          w.z = pack_bf16x2(v[4], v[5]);
          w.w = pack_bf16x2(v[6], v[7]);
          uint32_t off;
          if (BLK == 64) off = lane * 64 + ((c8 ^ ((lane >> 1) & 3)) << 4);  // 64-byte swizzle
          else off = sw128_off(lane, c8);                                     // 128-byte swizzle
          *reinterpret_cast<uint4*>(wstg_g + off) = w;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          // the tiles are read by the retrieval, long after: evict them first
          tma_store_2d_hint(&tvals, wstg, c_base, (base_sub + pos) * BLK + rloc0, policy_evict_first());
          bulk_commit();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(barFree(k));
    }
    if (!ok) misc[1] = 1;
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kN < 32 ? 32 : 2 * kN);
  }
}

template <int D, int BLK>
cudaError_t launch_pack_t(const CompressParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, cudaStream_t s) {
  auto kern = pack_bf16_kernel<D, BLK>;
  const int smem = PackLayout<D, BLK>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.n_tiles) * p.H_s;
  if (items <= 0) return cudaSuccess;
  // persistent: two CTAs per SM at B = 64 (one at B = 128)
  const long long slots = static_cast<long long>(sms) * ((BLK == 64) ? 2 : 1);
  const int grid = static_cast<int>(items < slots ? items : slots);
  kern<<<grid, kPackThreads, smem, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_bf16(const CompressParams& p, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  if (p.d == 128 && p.B == 64) return launch_pack_t<128, 64>(p, tq, tk, tv, s);
  if (p.d == 128 && p.B == 128) return launch_pack_t<128, 128>(p, tq, tk, tv, s);
  if (p.d == 64 && p.B == 64) return launch_pack_t<64, 64>(p, tq, tk, tv, s);
  if (p.d == 64 && p.B == 128) return launch_pack_t<64, 128>(p, tq, tk, tv, s);
  return cudaErrorInvalidValue;
}

}  // namespace mf
