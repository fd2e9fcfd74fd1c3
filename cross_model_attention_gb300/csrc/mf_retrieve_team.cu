// mf_retrieve_team.cu — fused Attention Retrieval, bf16, sm_103a:
// one persistent cooperative kernel in which teams of 8 CTAs (one per
// receiver KV group) pass the combined maps to each other through a small
// L2-resident ring in global memory.
//
// What it computes is the fused retrieval of "Accelerating Cross-Model LLM
// Inference via Attention Map Reuse" (section "Practical Implementation
// Details", bold header 4; head mapping per "MapFlow System Design" item 3) as
// the news article "北大MapFlow：注意力图跨模型复用，prefill延迟降15%–20%"
// describes it in paragraph "其三": read the sparse blocks, combine the sender
// heads on chip, multiply by the receiver's V and accumulate the output:
//   O_i[rows] = sum_bj ( sum_h W[i,h] P_h[rows, bj] ) V_g(i)[bj].
//
// Work split (per 64-row slab of a block-row, one team).  The head combine
// costs H_r multiply-adds per sender-tile element, and one slab's output
// accumulators (H_r heads x 64 rows x d fp32) are four times one SM's tensor
// memory, so the team's 8 CTAs split the slab two ways:
//   * combine: CTA c copies rows 8c..8c+7 of every kept tile of the block
//     (all sender heads; absent heads zero-filled) into a head-interleaved,
//     MN-major operand (each 128-byte source row lands whole in one
//     swizzled line, the layout 16-byte cp.async copies fastest) and
//     computes A_hat[elem, n] with tcgen05 (M = 128 elements = 2 rows x 64
//     keys, N = 32 = 8 KV groups x 4 head slots, K = sender heads, W^T in
//     bf16; slots beyond H_r/8 heads per group have zero weights);
//   * exchange: each thread then holds one element's 32 slots; a warp holds 32
//     consecutive keys of one row, so its 2-byte stores of one slot fill 64
//     contiguous bytes of the team's ring slot in global memory, laid out per
//     group as A_hat [head slot][row][key]; a signalling thread publishes the
//     slot through its ready counter (GPU-scope fence, batched over every
//     block whose stores are complete);
//   * A_hat . V: CTA c owns KV group c: once all 8 slices of a block are in
//     the slot it loads its group's A_hat (one 32 KB TMA box, K-major rows of
//     64 keys) and V_c and accumulates O[(head, row), d] += A_hat . V_c on
//     tcgen05 (two heads x 64 rows per M = 128 tile, N = d) into TMEM over the
//     slab's blocks, then bumps the slot's freed counter.
// The ring (8 slots per team) lives in L2 between its write and its reads
// (the sender tiles are copied with an evict-first L2 policy);
// every sender-tile byte is read from HBM once.  Slabs go to teams heaviest
// first onto the least-loaded team (a host-side table); within a team all
// CTAs walk the same slab list,
// whose records are staged in shared memory at the start.
//
// Warp roles (544 threads): warp 0 TMA loads of V and of the group's A_hat^T,
// warps 11-14 copy sender rows with 16-byte cp.async straight into the
// swizzled operand layout (their tile indices arrive four blocks ahead),
// warp 1 issues the combine MMAs, warps 2-9 convert and store A_hat and
// write each slab's output, warp 10 issues the A_hat.V MMAs, warp 15
// publishes stored blocks, warp 16 mirrors the team's counters into shared
// memory.  Every wait, on a shared-memory barrier, a mirror or a global
// counter, is bounded; the launch is cooperative so a team's CTAs are
// co-resident.
#include "mf_internal.cuh"
#include "mf_ptx.cuh"

namespace mf {
namespace {

constexpr int kTeam = 8;        // CTAs per team = receiver KV groups
constexpr int kThreads = 544;   // warp 0 loads, 1 combine MMA, 2-9 convert, 10 A_hat.V MMA, 11-14 P copies, 15 signals, 16 polls
constexpr int kPThreads = 128;  // P copy threads (warps 11-14)
constexpr int kPBytes = 120 * 1024;  // P ring: whole blocks of head slices (8 rows x 64 columns)
constexpr int kSliceBytes = 8 * 16 * 128;  // a slice of 16 heads; a last slice of <= 8 heads takes half
constexpr int kZeroBytes = 2048;           // two zero atoms: the missing head group of a half slice
constexpr int kPBMax = 3;       // block slots of the P ring at most
constexpr int kNComb = 32;      // combine N: 8 groups x 4 head slots
constexpr int kRing = 8;        // global ring slots per team
constexpr int kASub = 4;        // A_hat slots in shared memory: one head pair (2 x 64 rows x 64 keys) each
constexpr int kPairBytes = 2 * 64 * 64 * 2;
constexpr int kSlotHeads = 4;   // head slots per group
constexpr int kIdxSlots = 8;    // tile-index ring of the copy warps (blocks)
constexpr int kIdxAhead = 4;    // blocks whose tile indices are requested ahead of the copies
constexpr int kMaxSlabs = 32;   // slab records of a team kept in shared memory (later ones from L2)
constexpr int kGroupElems = kSlotHeads * 64 * 64;  // one group's A_hat in a ring slot

// One slab of a team's list (a 64-row half block-row and its kept columns).
struct SlabRec {
  int seq_start, L, bi, cand_off, half, n_sub, rb, pad;
};

// A block slot of the P ring holds the CTA's 8 rows of every sender head in
// slices of 16 heads, [row 8][head group 2][8 heads][128 B] (row stride 2 KB).
// When the last slice has at most 8 heads it is stored as [row 8][8 heads]
// [128 B] (row stride 1 KB), and its MMA descriptor points the missing head
// group at two shared zero atoms after the ring, so no block slot carries
// padding: 40 heads take 40 KB and three block slots fit.
struct TeamLayout {
  int nslice, half_last, slot_bytes, npb, pairs, vbytes, nv;
  int off_p, off_zero, off_a, off_v, off_w, off_s, off_i, off_bar, bytes;
  __host__ __device__ TeamLayout(int D, int Hs, int hpc) {
    nslice = (Hs + 15) / 16;
    half_last = (Hs % 16 != 0 && Hs % 16 <= 8) ? 1 : 0;
    slot_bytes = nslice * kSliceBytes - (half_last ? kSliceBytes / 2 : 0);
    npb = kPBytes / slot_bytes;
    if (npb > kPBMax) npb = kPBMax;
    pairs = (hpc + 1) / 2;
    vbytes = 64 * D * 2;
    const int base = kPBytes + kZeroBytes + kASub * kPairBytes + 4096 + kMaxSlabs * 32 + kIdxSlots * 256;
    nv = (base + 2 * vbytes + 1024 + 448 <= 227 * 1024) ? 2 : 1;
    off_p = 0;
    off_zero = off_p + kPBytes;
    off_a = off_zero + kZeroBytes;
    off_v = off_a + kASub * kPairBytes;
    off_w = off_v + nv * vbytes;
    off_s = off_w + 4096;
    off_i = off_s + kMaxSlabs * 32;
    off_bar = off_i + kIdxSlots * 256;
    bytes = off_bar + 48 * 8 + 64 + 1024;
  }
};

// Offset of slice sl within a block slot, and its row stride.
__device__ __forceinline__ uint32_t slice_off(int sl) { return static_cast<uint32_t>(sl) * kSliceBytes; }
__device__ __forceinline__ uint32_t slice_row_stride(const TeamLayout& lay, int sl) {
  return (lay.half_last && sl == lay.nslice - 1) ? 1024u : 2048u;
}

enum : int {
  kBarVFull = 0, kBarVEmpty = 2, kBarDFull = 4, kBarDEmpty = 6, kBarAFull = 8,
  kBarAEmpty = kBarAFull + kASub, kBarO = kBarAEmpty + kASub, kBarOFree = kBarO + 1,
  kBarStored = kBarOFree + 1, kBarPFull = kBarStored + kRing,
  kBarPEmpty = kBarPFull + kPBMax, kBarIdx = kBarPEmpty + kPBMax, kNumBars = kBarIdx + kIdxSlots
};
static_assert(kNumBars <= 48, "barrier area");

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try(bar, parity);
  __syncwarp();
  return ok != 0;
}

// Shared-memory mirrors of the team's ready / freed counters.  The poller
// warp reads the global counters (one L2 round trip covers all of them) and
// publishes each change here, so the loader's and the convert warps' per-block
// waits are shared-memory reads instead of an L2 round trip per block.  The
// poller's acquire at GPU scope, its release at CTA scope and the waiter's
// acquire at CTA scope chain the other CTAs' stores before the waiter's
// later accesses.
__device__ __forceinline__ uint32_t ld_acquire_cta_shared(const uint32_t* m) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(m)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared(uint32_t* m, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(m)), "r"(v) : "memory");
}
// Bounded wait until the mirror reaches `target`; false on timeout (error
// recorded) or once another role of this CTA has given up.
__device__ __forceinline__ bool wait_mirror(const uint32_t* m, uint32_t target, int* err,
                                            volatile int* abort_flag) {
  if (ld_acquire_cta_shared(m) >= target) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_cta_shared(m) >= target) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        set_error(err, kDevErrTimeout);
        return false;
      }
    }
    if (it > 8) __nanosleep(20);
  }
}
__device__ __forceinline__ bool warp_wait_mirror(const uint32_t* m, uint32_t target, int* err,
                                                 volatile int* abort_flag) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_mirror(m, target, err, abort_flag) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ld_acquire_cta_shared(m);
  __syncwarp();
  return ok != 0;
}

// Slab of round r for a team (the host's longest-first assignment); -1 once
// the team's list is exhausted.
__device__ __forceinline__ int slab_of(int r, int team, const RetrieveParams& p) {
  return r < p.team_stride ? p.team_slabs[team * p.team_stride + r] : -1;
}

template <int kSub>
__device__ __forceinline__ SlabRec load_slab(int r, const RetrieveParams& p, int team) {
  SlabRec x{};
  const int si = slab_of(r, team, p);
  if (si < 0) {
    x.n_sub = -1;
    return x;
  }
  const RowSlab sl = p.slabs[si];
  const RowBlock rb = p.rbs[sl.rb];
  x.seq_start = rb.seq_start;
  x.L = rb.L;
  x.bi = rb.bi;
  x.cand_off = rb.cand_off;
  x.half = sl.half;
  x.rb = sl.rb;
  x.n_sub = p.union_cnt[sl.rb] * kSub;
  return x;
}

// Record r of the team's slab list (n_sub < 0 past the end).
template <int kSub>
__device__ __forceinline__ SlabRec slab_rec(int r, const SlabRec* tab, const RetrieveParams& p,
                                            int team) {
  if (r < kMaxSlabs) return tab[r];
  return load_slab<kSub>(r, p, team);
}

// Walks a team's blocks in order: slab after slab, kept block column after
// kept block column (sub-blocks of 64 columns when B = 128).
struct BlockCursor {
  int r = -1, j = 0;
  bool done = false;
  SlabRec s;
};
template <int kSub>
__device__ __forceinline__ void cursor_settle(BlockCursor& c, const SlabRec* tab,
                                              const RetrieveParams& p, int team) {
  while (c.r < 0 || c.j >= c.s.n_sub) {
    ++c.r;
    c.s = slab_rec<kSub>(c.r, tab, p, team);
    if (c.s.n_sub < 0) {
      c.done = true;
      return;
    }
    c.j = 0;
  }
}

template <int D, int BLK>
__global__ void __launch_bounds__(kThreads, 1)
    retrieve_team_kernel(const __grid_constant__ CUtensorMap ta,
                         const __grid_constant__ CUtensorMap tv, const RetrieveParams p,
                         __nv_bfloat16* __restrict__ o, __nv_bfloat16* __restrict__ ring,
                         uint32_t* __restrict__ flags) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = blockIdx.x / kTeam, g = blockIdx.x % kTeam;
  const int hpc = p.H_r / kTeam;
  const TeamLayout lay(D, p.H_s, hpc);
  constexpr int kSub = BLK / 64;
  uint32_t* const ready = flags + team * (2 * kRing + 1);
  uint32_t* const freed = ready + kRing;
  uint32_t* const done = ready + 2 * kRing;  // CTAs of the team that have finished
  const size_t slot_elems = static_cast<size_t>(kTeam) * kGroupElems;
  __nv_bfloat16* ring_team = ring + static_cast<size_t>(team) * kRing * slot_elems;
  auto bar = [&](int i) { return sb + lay.off_bar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.off_bar + kNumBars * 8);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + lay.off_bar + kNumBars * 8 + 16);
  uint32_t* mirror = reinterpret_cast<uint32_t*>(smem + lay.off_bar + 48 * 8);  // ready[8], freed[8]
  SlabRec* tab = reinterpret_cast<SlabRec*>(smem + lay.off_s);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPBMax; ++s) {
      mbar_init(bar(kBarPFull + s), kPThreads);
      mbar_init(bar(kBarPEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
      mbar_init(bar(kBarDFull + s), 1);
      mbar_init(bar(kBarDEmpty + s), 8);
    }
    for (int s = 0; s < kASub; ++s) {
      mbar_init(bar(kBarAFull + s), 1);
      mbar_init(bar(kBarAEmpty + s), 1);
    }
    mbar_init(bar(kBarO), 1);
    mbar_init(bar(kBarOFree), 8);
    for (int s = 0; s < kRing; ++s) mbar_init(bar(kBarStored + s), 8);
    for (int s = 0; s < kIdxSlots; ++s) mbar_init(bar(kBarIdx + s), kPThreads);
    *abort_flag = 0;
    for (int i = 0; i < 2 * kRing; ++i) mirror[i] = 0u;  // the counters start each launch at 0
    fence_mbar_init();
  }
  // zero the P ring: the lines of padded heads (beyond H_s in the last
  // slice) are never copied and must hold finite values (their weights are 0)
  for (int i = threadIdx.x; i < (kPBytes + kZeroBytes) / 16; i += kThreads)
    *reinterpret_cast<uint4*>(smem + lay.off_p + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  // the team's slab records
  for (int r = threadIdx.x; r < kMaxSlabs; r += kThreads) tab[r] = load_slab<kSub>(r, p, team);
  // W^T as the combine's B operand: row n = 4 * group + head slot (32 rows;
  // receiver head group * H_r/8 + slot), 64 bf16 sender-head entries per row,
  // 128-byte swizzle; zero for unused slots and beyond H_s.
  for (int t = threadIdx.x; t < kNComb * 64; t += kThreads) {
    const int n = t >> 6, k = t & 63;
    const int gs = n >> 2, ts = n & 3;
    const int i = gs * hpc + ts;
    const float wv = (ts < hpc && k < p.H_s) ? p.W[static_cast<size_t>(i) * p.H_s + k] : 0.f;
    *reinterpret_cast<__nv_bfloat16*>(smem + lay.off_w + sw128_off(n, k >> 3) + (k & 7) * 2) =
        __float2bfloat16_rn(wv);
  }
  fence_async_smem();
  if (warp == 1) tmem_alloc(smem_u32(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);

  if (warp == 0) {
    // --------------------------------------------- V and A_hat tile loader
    if (lane == 0) {
      prefetch_tmap(&ta);
      prefetch_tmap(&tv);
      bool ok = true;
      int u = 0;
      for (int r = 0; ok; ++r) {
        const SlabRec sr = slab_rec<kSub>(r, tab, p, team);
        if (sr.n_sub < 0) break;
        int bj_next = sr.n_sub > 0 ? p.union_list[sr.cand_off] : 0;
        for (int j = 0; j < sr.n_sub; ++j, ++u) {
          const int bj = bj_next;  // read one block ahead
          if (j + 1 < sr.n_sub) bj_next = p.union_list[sr.cand_off + (j + 1) / kSub];
          const int cs = j % kSub;
          const int vs = (lay.nv == 2) ? (u & 1) : 0;
          const uint32_t vph = (lay.nv == 2) ? ((u >> 1) & 1) : (u & 1);
          if (!mbar_wait(bar(kBarVEmpty + vs), vph ^ 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_tx(bar(kBarVFull + vs), lay.vbytes);
          const int tok0 = sr.seq_start + bj * BLK + cs * 64;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sb + lay.off_v + vs * lay.vbytes + c * 8192, &tv, g * D + c * 64, tok0,
                        bar(kBarVFull + vs));
          // this group's A_hat of block u, once all 8 slices are in the ring
          // slot, one head pair per shared-memory slot (a pair's slot frees
          // as soon as its own MMAs are done)
          const int s = u % kRing;
          if (!wait_mirror(mirror + s, static_cast<uint32_t>(kTeam * (u / kRing + 1)), p.err,
                           abort_flag)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          const int y = ((team * kRing + s) * kTeam + g) * (kGroupElems / 64);
          for (int pr = 0; pr < lay.pairs; ++pr) {
            const int q = u * lay.pairs + pr, as = q % kASub;
            if (!mbar_wait(bar(kBarAEmpty + as), ((q / kASub) & 1) ^ 1, p.err)) {
              ok = false;
              break;
            }
            mbar_arrive_tx(bar(kBarAFull + as), static_cast<uint32_t>(kPairBytes));
            tma_load_2d(sb + lay.off_a + as * kPairBytes, &ta, 0, y + pr * 128, bar(kBarAFull + as));
          }
          if (!ok) break;
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp >= 11 && warp <= 14) {
    // ------------------------------------------------------ P row producer
    // Thread t copies, for slice-local head h = t/8 and 16-byte chunk
    // cg = t%8, rows 8g..8g+7 of that head's kept tile (64 columns of this
    // sub-block) into the slice layout [row 8][head group 2][8 heads][128 B]
    // with the 128-byte swizzle; a dropped or padded head is zero-filled.
    const int t = threadIdx.x - 11 * 32;
    const int hl = t >> 3, cg = t & 7;
    // (a half slice holds heads hl < 8 only, so its head group is always 0)
    const uint32_t dst0 = sb + lay.off_p + (hl >> 3) * 1024 + sw128_off(hl & 7, cg);
    const size_t row_bytes = static_cast<size_t>(BLK) * 2;
    const char* vbase = reinterpret_cast<const char*>(p.values);
    // Tile indices come through a shared-memory ring filled by cp.async
    // kIdxAhead blocks ahead (thread t < H_s copies head t's entry of the
    // union-ordered table), so no copy waits on a global load.  A slot is
    // rewritten kIdxSlots - kIdxAhead blocks after its use; the copy warps
    // cannot drift that far apart (a block's copies need every warp's
    // arrivals on the previous blocks' slices).
    const int* idx_ring = reinterpret_cast<const int*>(smem + lay.off_i);
    BlockCursor ic;
    cursor_settle<kSub>(ic, tab, p, team);
    int n_req = 0;
    auto request_next = [&]() {
      if (ic.done) return;
      const int slot = n_req % kIdxSlots;
      if (t < p.H_s)
        cp_async4(sb + lay.off_i + slot * 256 + t * 4,
                  p.utile + static_cast<size_t>(ic.s.cand_off + ic.j / kSub) * p.H_s + t);
      cp_async_arrive(bar(kBarIdx + slot));
      ++n_req;
      ++ic.j;
      cursor_settle<kSub>(ic, tab, p, team);
    };
    for (int i = 0; i < kIdxAhead; ++i) request_next();
    bool ok = true;
    int u = 0;
    for (int r = 0; ok; ++r) {
      const SlabRec sr = slab_rec<kSub>(r, tab, p, team);
      if (sr.n_sub < 0) break;
      for (int j = 0; ok && j < sr.n_sub; ++j, ++u) {
        const int cs = j % kSub;
        request_next();
        if (!warp_wait(bar(kBarIdx + u % kIdxSlots), (u / kIdxSlots) & 1, p.err)) {
          ok = false;
          break;
        }
        const int* irow = idx_ring + (u % kIdxSlots) * 64;
        // sender tiles are read once: evicted from L2 before the exchange ring
        const uint64_t pol = policy_evict_first();
        int tix[4];
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          const int h = sl * 16 + hl;
          tix[sl] = (sl < lay.nslice && h < p.H_s) ? irow[h] : -1;
        }
        // the block slot of block u - npb has been consumed
        const int pb = u % lay.npb;
        int good = 1;
        if (lane == 0) good = mbar_wait(bar(kBarPEmpty + pb), ((u / lay.npb) & 1) ^ 1, p.err) ? 1 : 0;
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          if (sl >= lay.nslice || sl * 16 + hl >= p.H_s) continue;  // padded heads stay zero
          const int tt = tix[sl];
          const char* src = vbase +
                            (static_cast<size_t>(tt >= 0 ? tt : 0) * BLK + sr.half * 64 + 8 * g) *
                                row_bytes +
                            cs * 128 + cg * 16;
          const uint32_t nbytes = tt >= 0 ? 16u : 0u;  // a dropped head is zero-filled
          const uint32_t dst = dst0 + pb * lay.slot_bytes + slice_off(sl);
          const uint32_t rstride = slice_row_stride(lay, sl);
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) cp_async16_hint(dst + rr * rstride, src + rr * row_bytes, nbytes, pol);
        }
        cp_async_arrive(bar(kBarPFull + pb));
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (warp == 1) {
    // ------------------------------------------------- combine MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_comb = idesc_bf16_f32(128, kNComb, true, false);
      bool ok = true;
      int u = 0;
      for (int r = 0; ok; ++r) {
        const SlabRec sr = slab_rec<kSub>(r, tab, p, team);
        if (sr.n_sub < 0) break;
        for (int j = 0; ok && j < sr.n_sub; ++j, ++u) {
          const int b = u & 1, pb = u % lay.npb;
          if (!mbar_wait(bar(kBarDEmpty + b), ((u >> 1) & 1) ^ 1, p.err) ||
              !mbar_wait(bar(kBarPFull + pb), (u / lay.npb) & 1, p.err)) {
            ok = false;
            break;
          }
          fence_async_smem();  // rows were written by cp.async (generic proxy)
          tc_fence_after();
          const uint32_t wbase = sb + lay.off_w;
          for (int sl = 0; sl < lay.nslice; ++sl) {
            const uint32_t pbase = sb + lay.off_p + pb * lay.slot_bytes + slice_off(sl);
            const uint32_t rstride = slice_row_stride(lay, sl);
            const uint64_t bd = sdesc_sw128(wbase + sl * 32, 16, 1024);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // rows 2k, 2k+1 of the slice: LBO = row stride, SBO = the second
              // head group (the next atom, or for a half slice the zero atoms)
              const uint32_t a0 = pbase + 2 * k * rstride;
              const uint32_t sbo = (rstride == 2048u) ? 1024u : (sb + lay.off_zero) - a0;
              const uint64_t ad = sdesc_sw128(a0, rstride, sbo);
              tc_mma(tmem + b * 128 + k * kNComb, ad, bd, idesc_comb, sl > 0 ? 1u : 0u);
            }
          }
          tc_commit(bar(kBarPEmpty + pb));
          tc_commit(bar(kBarDFull + b));
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 10) {
    // --------------------------------------------- A_hat . V MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_av = idesc_bf16_f32(128, D, false, true);
      bool ok = true;
      int u = 0;
      for (int r = 0; ok; ++r) {
        const SlabRec sr = slab_rec<kSub>(r, tab, p, team);
        if (sr.n_sub < 0) break;
        // the previous slab's output has been read out of TMEM
        if (r > 0 && !mbar_wait(bar(kBarOFree), (r - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        for (int j = 0; j < sr.n_sub; ++j, ++u) {
          const int vs = (lay.nv == 2) ? (u & 1) : 0;
          const uint32_t vph = (lay.nv == 2) ? ((u >> 1) & 1) : (u & 1);
          if (!mbar_wait(bar(kBarVFull + vs), vph, p.err)) {
            ok = false;
            break;
          }
          const uint32_t vbase = sb + lay.off_v + vs * lay.vbytes;
          // O[(head, row), d] += A_hat[(head, row), key] V[key, d], two heads
          // (128 rows of A_hat, K-major) per MMA, 16 keys per step; V is
          // MN-major with d chunks of 64 at 8 KB
          for (int pr = 0; pr < lay.pairs; ++pr) {
            const int q = u * lay.pairs + pr, as = q % kASub;
            if (!mbar_wait(bar(kBarAFull + as), (q / kASub) & 1, p.err)) {
              ok = false;
              break;
            }
            // every pair of block u is in: this CTA has its copy of the ring
            // slot (the copies are complete, so no ordering beyond the count
            // itself is needed)
            if (pr == lay.pairs - 1) red_relaxed_gpu_add(freed + u % kRing, 1u);
            tc_fence_after();
            const uint32_t abase = sb + lay.off_a + as * kPairBytes;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint64_t ad = sdesc_sw128(abase + s * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(vbase + s * 2048, 8192, 1024);
              tc_mma(tmem + 256 + pr * D, ad, bd, idesc_av, (j > 0 || s > 0) ? 1u : 0u);
            }
            tc_commit(bar(kBarAEmpty + as));
          }
          if (!ok) break;
          tc_commit(bar(kBarVEmpty + vs));
        }
        if (!ok) break;
        tc_commit(bar(kBarO));  // this slab's accumulation is complete
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 16) {
    // --------------------------------------------------------------- poller
    // Lane i < 8 follows ready[i], lane 8 + i freed[i]: one acquire load per
    // lane per round (all in one L2 round trip), each change published to
    // the shared-memory mirror.  A lane stops once its counter reaches the
    // value the team's last block gives it, or when the CTA gives up.
    if (lane < 2 * kRing) {
      const int sl = lane & (kRing - 1);
      const uint32_t* src = (lane < kRing ? ready : freed) + sl;
      int total = 0;
      for (int r = 0;; ++r) {
        const SlabRec sr = slab_rec<kSub>(r, tab, p, team);
        if (sr.n_sub < 0) break;
        total += sr.n_sub;
      }
      const uint32_t final_v =
          static_cast<uint32_t>(kTeam * (total > sl ? (total - sl + kRing - 1) / kRing : 0));
      uint32_t last = 0;
      unsigned long long t0 = globaltimer();
      while (last < final_v) {
        const uint32_t v = ld_acquire_gpu(src);
        if (v != last) {
          st_release_cta_shared(mirror + lane, v);
          last = v;
          t0 = globaltimer();
          continue;
        }
        if (*abort_flag) break;
        if (globaltimer() - t0 > kWaitLimitNs) {
          set_error(p.err, kDevErrTimeout);
          *abort_flag = 1;
          break;
        }
        __nanosleep(32);
      }
    }
  } else if (warp == 15) {
    // ------------------------------------------------------------ signaller
    // Publishes blocks whose A_hat slices this CTA's convert warps have
    // stored: waits for the CTA-local barrier of the oldest unpublished
    // block, takes every later block that is also complete, then one GPU-scope
    // fence covers them all before the ready counters move.  The fence waits
    // for the stores to reach L2; keeping it here keeps the convert warps
    // streaming.
    if (lane == 0) {
      int total = 0;
      for (int r = 0;; ++r) {
        const SlabRec sr = slab_rec<kSub>(r, tab, p, team);
        if (sr.n_sub < 0) break;
        total += sr.n_sub;
      }
      bool ok = true;
      for (int u = 0; ok && u < total;) {
        if (!mbar_wait(bar(kBarStored + u % kRing), (u / kRing) & 1, p.err)) {
          ok = false;
          break;
        }
        int v = u + 1;
        while (v < total && v < u + kRing && mbar_try(bar(kBarStored + v % kRing), (v / kRing) & 1))
          ++v;
        fence_acq_rel_gpu();
        for (int w = u; w < v; ++w) red_relaxed_gpu_add(ready + w % kRing, 1u);
        u = v;
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------ convert + store + epilogue
    // Combine chunk k (TMEM columns k*32..k*32+31 of buffer b) holds rows 2k,
    // 2k+1 of this CTA's 8; TMEM lane L is row 2k + L/64, key L%64.  The two
    // warps of a lane quadrant take alternate chunks.
    const int wq = warp & 3;
    const int sub = (warp - 2) >> 2;               // the two warps of a TMEM quadrant
    const uint32_t tq = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const int key = (wq & 1) * 32 + lane;
    bool ok = true;
    int u = 0;
    for (int r = 0; ok; ++r) {
      const SlabRec sr = slab_rec<kSub>(r, tab, p, team);
      if (sr.n_sub < 0) break;
      const int row0 = sr.bi * BLK + sr.half * 64;
      for (int j = 0; ok && j < sr.n_sub; ++j, ++u) {
        const int b = u & 1;
        if (!warp_wait(bar(kBarDFull + b), (u >> 1) & 1, p.err)) {
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
        // every owner has its copy of the slot's previous contents
        const int s = u % kRing;
        if (u >= kRing && !warp_wait_mirror(mirror + kRing + s,
                                            static_cast<uint32_t>(kTeam * (u / kRing)), p.err,
                                            abort_flag)) {
          ok = false;
          break;
        }
        __nv_bfloat16* slot_base = ring_team + static_cast<size_t>(s) * slot_elems;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int rr = 2 * (2 * kk + sub) + (wq >> 1);  // row within this CTA's 8
          // [group][head slot][row 8g + rr][key]; column n = 4 * group + slot
          __nv_bfloat16* dst = slot_base + (8 * g + rr) * 64 + key;
#pragma unroll
          for (int n = 0; n < kNComb; ++n) {
            if ((n & 3) < hpc)
              dst[static_cast<size_t>(n) * 64 * 64] = __float2bfloat16_rn(__uint_as_float(v[kk][n]));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarStored + s));  // release.cta: the signaller publishes
      }
      if (!ok) break;
      // ------------------------------------------------------ slab epilogue
      const int L = wq * 32 + lane;  // TMEM lane: head 2pr + L/64, row L%64
      const int rl = L & 63;
      const int rloc = row0 + rl;
      const bool row_ok = rloc < sr.L;
      const bool have = sr.n_sub > 0;
      if (!warp_wait(bar(kBarO), r & 1, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int pr = 0; pr < lay.pairs; ++pr) {
        const int t = 2 * pr + (L >> 6);
        const bool write = row_ok && t < hpc;
        __nv_bfloat16* dst =
            o + (static_cast<size_t>(sr.seq_start + rloc) * p.H_r + g * hpc + t) * D + sub * (D / 2);
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarOFree));
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // The team's last CTA to finish (every wait above is bounded, so all get
  // here) leaves the team's counters at zero for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(done, 1u) == static_cast<uint32_t>(kTeam - 1)) {
      for (int i = 0; i < 2 * kRing; ++i) ready[i] = 0u;  // ready, then freed
      *done = 0u;
      __threadfence();
    }
  }
}

template <int D, int BLK>
cudaError_t launch_team_t(const RetrieveParams& p, const CUtensorMap& ta, const CUtensorMap& tv,
                          void* o, void* ring, uint32_t* flags, int n_teams, cudaStream_t s) {
  auto kern = retrieve_team_kernel<D, BLK>;
  const TeamLayout lay(D, p.H_s, p.H_r / kTeam);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_teams * kTeam, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = lay.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tv, p, static_cast<__nv_bfloat16*>(o),
                            static_cast<__nv_bfloat16*>(ring), flags);
}

}  // namespace

bool retrieve_team_supported(int H_s, int H_r, int H_kv, int d, int B) {
  return H_kv == kTeam && H_r % kTeam == 0 && H_r / kTeam <= kSlotHeads && H_s <= 64 &&
         (d == 64 || d == 128) && (B == 64 || B == 128);
}

int retrieve_team_count(int n_slabs, int sms) {
  int t = sms / kTeam;
  if (t > n_slabs) t = n_slabs;
  return t < 1 ? 1 : t;
}

size_t retrieve_team_ring_bytes(int n_teams) {
  return static_cast<size_t>(n_teams) * kRing * kTeam * kGroupElems * 2;
}

size_t retrieve_team_flag_bytes(int n_teams) {
  return static_cast<size_t>(n_teams) * (2 * kRing + 1) * sizeof(uint32_t);
}

int retrieve_team_ring_box_rows(int) { return kPairBytes / 128; }

int retrieve_team_ring_rows(int n_teams) { return n_teams * kRing * kTeam * (kGroupElems / 64); }

cudaError_t launch_retrieve_team(const RetrieveParams& p, const CUtensorMap& ta,
                                 const CUtensorMap& tv, void* o, void* ring, uint32_t* flags,
                                 int n_teams, cudaStream_t s) {
  if (p.d == 128 && p.B == 64) return launch_team_t<128, 64>(p, ta, tv, o, ring, flags, n_teams, s);
  if (p.d == 128 && p.B == 128) return launch_team_t<128, 128>(p, ta, tv, o, ring, flags, n_teams, s);
  if (p.d == 64 && p.B == 64) return launch_team_t<64, 64>(p, ta, tv, o, ring, flags, n_teams, s);
  if (p.d == 64 && p.B == 128) return launch_team_t<64, 128>(p, ta, tv, o, ring, flags, n_teams, s);
  return cudaErrorInvalidValue;
}

}  // namespace mf
