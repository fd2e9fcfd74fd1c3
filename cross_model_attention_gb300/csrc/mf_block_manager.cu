// mf_block_manager.cu — the block manager: compressed block-row states cached
// under prefix hashes, and BSR views assembled from them.
//
// [Summary] "Accelerating Cross-Model LLM Inference via Attention Map Reuse",
// "Practical Implementation Details", and [Article] "北大MapFlow：注意力图跨模型
// 复用，prefill延迟降15%–20%", part "其二": compressed states are indexed by hashes that
// carry the preceding context, so a request sharing a prefix finds the states
// of its shared positions, and one sender state serves every receiver mapped
// to it.  Reading: under a causal mask, block-row bi of a sequence (its
// selection and kept tiles for every head) depends only on the tokens of
// blocks 0..bi, so the chained hash of those blocks names it.  An entry holds
// one block-row of one sender layer: the kept tiles of all heads, in slots of
// one device tile pool, and their (candidate column, head) positions.  A view
// is an ordinary BSR layer whose tile table points into the pool; the
// retrieval kernels read it as they read a compressed layer.
//
// Host side: an index keyed by (layer key, hash), an LRU order over entries no
// view pins, and a free list of pool slots.  Device side: one gather kernel
// that copies newly cached tiles from a compressed layer into their slots.
#include <cstdint>
#include <cstring>
#include <memory>
#include <set>
#include <unordered_map>

#include "mf_handle.h"

namespace mf {

struct BmEntry {
  int key_layer = 0;
  uint64_t hash = 0;
  int bi = 0, rows = 0;     // block-row index within its sequence, valid rows
  std::vector<int> where;   // per kept tile: candidate column * H_s + head
  std::vector<int> slots;   // pool slot of each kept tile
  int pins = 0;             // views that reference this entry
  uint64_t tick = 0;        // last insert or lookup (LRU)
};

}  // namespace mf

using namespace mf;

struct mf_bm_s {
  int H_s = 0, B = 0, d = 0;
  long long cap = 0;            // tile slots; slot `cap` is the all-zero tile
  uint16_t* pool = nullptr;     // [(cap + 1)][B][B] bf16
  mf_alloc_fn alloc = nullptr;
  mf_free_fn dealloc = nullptr;
  void* ctx = nullptr;
  struct Key {
    int layer;
    uint64_t hash;
    bool operator==(const Key& o) const { return layer == o.layer && hash == o.hash; }
  };
  struct KeyHash {
    size_t operator()(const Key& k) const { return (size_t)(k.hash ^ (0x9E3779B97F4A7C15ull * (uint64_t)(k.layer + 1))); }
  };
  std::unordered_map<Key, std::unique_ptr<BmEntry>, KeyHash> index;
  std::set<std::pair<uint64_t, BmEntry*>> lru;  // unpinned entries, oldest first
  std::vector<int> free_slots;
  uint64_t tick = 0;
  long long hits = 0, misses = 0, evictions = 0, pinned_entries = 0;
};

namespace {

// splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", 2014): a bijective 64-bit mix.
inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

void* pool_alloc(mf_bm_t bm, size_t bytes, cudaStream_t s) {
  if (bm->alloc) return bm->alloc(bytes, bm->ctx, s);
  void* p = nullptr;
  if (cudaMallocAsync(&p, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

void pool_free(mf_bm_t bm, void* p, cudaStream_t s) {
  if (!p) return;
  if (bm->dealloc) bm->dealloc(p, bm->ctx, s);
  else cudaFreeAsync(p, s);
}

void touch(mf_bm_t bm, BmEntry* e) {
  if (e->pins == 0) bm->lru.erase({e->tick, e});
  e->tick = ++bm->tick;
  if (e->pins == 0) bm->lru.insert({e->tick, e});
}

void pin(mf_bm_t bm, BmEntry* e) {
  if (e->pins++ == 0) {
    bm->lru.erase({e->tick, e});
    ++bm->pinned_entries;
  }
}

// The least recently used unpinned entries whose slots, with the free ones,
// give `need` slots (nothing is changed yet); false if the pinned entries,
// or those the current call touched, leave too few.
bool plan_room(mf_bm_t bm, size_t need, uint64_t protect_from, std::vector<BmEntry*>* victims) {
  size_t have = bm->free_slots.size();
  for (auto it = bm->lru.begin(); have < need; ++it) {
    if (it == bm->lru.end()) return false;
    BmEntry* e = it->second;
    if (e->tick >= protect_from) return false;  // touched by the current call
    victims->push_back(e);
    have += e->slots.size();
  }
  return true;
}

// Evicts the planned victims: their slots join the free list.
void evict(mf_bm_t bm, const std::vector<BmEntry*>& victims, int64_t* evicted) {
  for (BmEntry* e : victims) {
    bm->lru.erase({e->tick, e});
    for (int sl : e->slots) bm->free_slots.push_back(sl);
    bm->index.erase(mf_bm_s::Key{e->key_layer, e->hash});  // frees e
    ++bm->evictions;
    if (evicted) ++*evicted;
  }
}

// Copies tile pairs[i].x of `src` into slot pairs[i].y of `dst`, one CTA per
// tile at a time, 16-byte vectors.
__global__ void __launch_bounds__(256) bm_gather_tiles_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                              const int2* __restrict__ pairs, int n, int tile_u4) {
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int2 pr = pairs[i];
    const uint4* s = src + static_cast<size_t>(pr.x) * tile_u4;
    uint4* t = dst + static_cast<size_t>(pr.y) * tile_u4;
    for (int j = threadIdx.x; j < tile_u4; j += blockDim.x) t[j] = s[j];
  }
}

}  // namespace

namespace mf {

void bm_unpin(LayerState& L) {
  mf_bm_t bm = L.view_bm;
  for (BmEntry* e : L.view_pins) {
    if (--e->pins == 0) {
      --bm->pinned_entries;
      bm->lru.insert({e->tick, e});
    }
  }
  L.view_pins.clear();
  L.view_bm = nullptr;
}

}  // namespace mf

extern "C" {

int mf_prefix_hashes(const int32_t* tokens, const int32_t* cu_seqlens, const int32_t* q_begin, int n_seqs, int B,
                     uint64_t seed, uint64_t* hashes_out, int64_t capacity, int64_t* n_out) {
  if (!tokens || !cu_seqlens || !n_out) return fail(MF_ERR_ARG, "NULL pointer argument");
  if (n_seqs < 1 || B < 1) return fail(MF_ERR_ARG, "n_seqs and B must be >= 1");
  if (cu_seqlens[0] != 0) return fail(MF_ERR_ARG, "cu_seqlens[0] must be 0");
  int64_t R = 0;
  for (int s = 0; s < n_seqs; ++s) {
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    if (L < 0) return fail(MF_ERR_ARG, "cu_seqlens must be non-decreasing");
    const int qb = q_begin ? q_begin[s] : 0;
    if (qb < 0 || qb > L || (qb % B != 0 && qb != L))
      return fail(MF_ERR_ARG, "q_begin[%d] = %d is neither a block start nor the sequence's end", s, qb);
    if (qb < L) R += (L + B - 1) / B - qb / B;
  }
  *n_out = R;
  if (!hashes_out) return MF_OK;  // size query
  if (capacity < R) return fail(MF_ERR_ARG, "hashes_out holds %lld, %lld needed", (long long)capacity, (long long)R);
  int64_t r = 0;
  for (int s = 0; s < n_seqs; ++s) {
    const int a = cu_seqlens[s], L = cu_seqlens[s + 1] - a;
    uint64_t h = mix64(seed ^ 0x6A09E667F3BCC909ull);
    const int qb = q_begin ? q_begin[s] : 0;
    for (int b0 = 0; b0 < L; b0 += B) {
      const int n = std::min(B, L - b0);
      h = mix64(h ^ (0x9E3779B97F4A7C15ull * (uint64_t)n));  // the block's length
      for (int i = 0; i < n; ++i) h = mix64(h ^ (uint64_t)(uint32_t)tokens[a + b0 + i]);
      if (b0 >= qb) hashes_out[r++] = h;  // the chain runs over the prefix too
    }
  }
  return MF_OK;
}

int mf_bm_create(mf_bm_t* out, int H_s, int B, int64_t tile_capacity, mf_alloc_fn alloc_fn, mf_free_fn free_fn,
                 void* alloc_ctx, void* stream) {
  if (!out) return fail(MF_ERR_ARG, "out is NULL");
  *out = nullptr;
  if (H_s < 1) return fail(MF_ERR_ARG, "H_s must be >= 1");
  if ((alloc_fn == nullptr) != (free_fn == nullptr))
    return fail(MF_ERR_ARG, "alloc_fn and free_fn must both be set or both be NULL");
  if (B != 64 && B != 128) return fail(MF_ERR_UNSUPPORTED, "block size %d (supported: 64, 128)", B);
  if (tile_capacity < 1 || tile_capacity >= (1ll << 31) - 1) return fail(MF_ERR_ARG, "tile_capacity out of range");
  auto bm = std::make_unique<mf_bm_s>();
  bm->H_s = H_s;
  bm->B = B;
  bm->cap = tile_capacity;
  bm->alloc = alloc_fn;
  bm->dealloc = free_fn;
  bm->ctx = alloc_ctx;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tile = (size_t)B * B * 2;
  bm->pool = (uint16_t*)pool_alloc(bm.get(), (size_t)(tile_capacity + 1) * tile, s);
  if (!bm->pool) return fail(MF_ERR_OOM, "tile pool of %lld tiles", (long long)tile_capacity);
  // the all-zero tile the retrieval reads for a head's dropped block
  cudaError_t e = cudaMemsetAsync(reinterpret_cast<char*>(bm->pool) + (size_t)tile_capacity * tile, 0, tile, s);
  if (e != cudaSuccess) {
    pool_free(bm.get(), bm->pool, s);
    return cuda_fail(e, "zero tile");
  }
  bm->free_slots.reserve((size_t)tile_capacity);
  for (long long i = tile_capacity - 1; i >= 0; --i) bm->free_slots.push_back((int)i);
  *out = bm.release();
  return MF_OK;
}

int mf_bm_destroy(mf_bm_t bm) {
  if (!bm) return MF_OK;
  if (bm->pinned_entries > 0)
    return fail(MF_ERR_STATE, "%lld cached block-rows are still used by views", bm->pinned_entries);
  pool_free(bm, bm->pool, nullptr);
  delete bm;
  return MF_OK;
}

int mf_bm_insert(mf_bm_t bm, int key_layer, mf_bsr_t h, int layer, const uint64_t* hashes, int64_t* counts,
                 void* stream) {
  if (!bm || !h || !hashes) return fail(MF_ERR_ARG, "NULL handle or hashes");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  if (h->H_s != bm->H_s || h->B != bm->B) return fail(MF_ERR_ARG, "the handle's H_s or B differs from the manager's");
  if (!h->causal) return fail(MF_ERR_UNSUPPORTED, "non-causal block-rows depend on the whole sequence");
  LayerState& L = h->layers[layer];
  if (!L.valid) return fail(MF_ERR_STATE, "layer %d has not been compressed", layer);
  if (L.offloaded) return fail(MF_ERR_STATE, "layer %d is offloaded", layer);
  if (bm->d && L.d != bm->d) return fail(MF_ERR_ARG, "d = %d differs from the cached layers' %d", L.d, bm->d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.ready) MF_CUDA(cudaStreamWaitEvent(s, L.ready, 0), "wait for the layer's prefetch");
  const int H = h->H_s;
  // the layer's tile table: which tile holds (candidate, head), -1 if dropped
  std::vector<int> tile_of((size_t)H * h->C);
  MF_CUDA(cudaMemcpyAsync(tile_of.data(), L.tile_of, tile_of.size() * 4, cudaMemcpyDeviceToHost, s), "tile table copy");
  MF_CUDA(cudaStreamSynchronize(s), "tile table copy");
  const uint64_t call_tick = bm->tick + 1;
  int64_t inserted = 0, present = 0, evicted = 0;
  struct NewRow {
    int rb;
    std::vector<int> where, src;
  };
  std::vector<NewRow> fresh;
  std::unordered_map<uint64_t, int> fresh_of;  // hashes repeated within this call
  size_t need = 0;
  for (int rb = 0; rb < h->R; ++rb) {
    const RowBlock& rbk = h->rbs[rb];
    auto it = bm->index.find(mf_bm_s::Key{key_layer, hashes[rb]});
    if (it != bm->index.end()) {
      BmEntry* e = it->second.get();
      if (e->bi != rbk.bi || e->rows != std::min(h->B, rbk.L - rbk.bi * h->B))
        return fail(MF_ERR_ARG, "hash of block-row %d names a cached block-row of another shape", rb);
      touch(bm, e);
      ++present;
      continue;
    }
    auto fr = fresh_of.find(hashes[rb]);
    if (fr != fresh_of.end()) {
      const RowBlock& first = h->rbs[fresh[fr->second].rb];
      if (first.bi != rbk.bi || std::min(h->B, first.L - first.bi * h->B) != std::min(h->B, rbk.L - rbk.bi * h->B))
        return fail(MF_ERR_ARG, "block-rows %d and %d share a hash but not a shape", fresh[fr->second].rb, rb);
      ++present;
      continue;
    }
    NewRow nr;
    nr.rb = rb;
    for (int bj = 0; bj <= rbk.bi; ++bj)
      for (int hh = 0; hh < H; ++hh) {
        const int t = tile_of[(size_t)(rbk.cand_off + bj) * H + hh];
        if (t >= 0) {
          nr.where.push_back(bj * H + hh);
          nr.src.push_back(t);
        }
      }
    need += nr.where.size();
    fresh_of[hashes[rb]] = (int)fresh.size();
    fresh.push_back(std::move(nr));
  }
  if (need > (size_t)bm->cap) return fail(MF_ERR_OOM, "%zu new tiles exceed the pool's %lld", need, bm->cap);
  int sms = 0;
  MF_CUDA(sm_count(&sms), "device query");
  // the device copy list first: nothing below changes the cache until every
  // step that can fail has succeeded (all or nothing)
  int2* pairs_d = nullptr;
  if (need > 0) {
    pairs_d = (int2*)pool_alloc(bm, need * sizeof(int2), s);
    if (!pairs_d) return fail(MF_ERR_OOM, "copy list allocation failed");
  }
  std::vector<BmEntry*> victims;
  if (!plan_room(bm, need, call_tick, &victims)) {
    pool_free(bm, pairs_d, s);
    return fail(MF_ERR_OOM, "the pool has %zu free tiles for %zu new ones; the rest are pinned or in use by this call",
                bm->free_slots.size(), need);
  }
  // the slots the new tiles take: the victims' first, then free ones from the
  // back of the free list; the victims stay cached until the copy is queued
  std::vector<int> take;
  take.reserve(need);
  for (BmEntry* v : victims)
    for (int sl : v->slots)
      if (take.size() < need) take.push_back(sl);
  const size_t from_free = need - take.size();
  for (size_t i = 0; i < from_free; ++i) take.push_back(bm->free_slots[bm->free_slots.size() - 1 - i]);
  std::vector<int2> pairs;
  pairs.reserve(need);
  std::vector<std::unique_ptr<BmEntry>> made;
  made.reserve(fresh.size());
  for (NewRow& nr : fresh) {
    const RowBlock& rbk = h->rbs[nr.rb];
    auto e = std::make_unique<BmEntry>();
    e->key_layer = key_layer;
    e->hash = hashes[nr.rb];
    e->bi = rbk.bi;
    e->rows = std::min(h->B, rbk.L - rbk.bi * h->B);
    e->where = std::move(nr.where);
    e->slots.resize(e->where.size());
    for (size_t i = 0; i < e->slots.size(); ++i) {
      e->slots[i] = take[pairs.size()];
      pairs.push_back(make_int2(nr.src[i], e->slots[i]));
    }
    made.push_back(std::move(e));
  }
  if (!pairs.empty()) {
    cudaError_t e = cudaMemcpyAsync(pairs_d, pairs.data(), pairs.size() * sizeof(int2), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) {
      const int grid = (int)std::min<size_t>(pairs.size(), (size_t)sms * 8);
      const int tile_u4 = bm->B * bm->B * 2 / 16;
      bm_gather_tiles_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(L.values),
                                                  reinterpret_cast<uint4*>(bm->pool), pairs_d, (int)pairs.size(),
                                                  tile_u4);
      e = cudaGetLastError();
    }
    // the host list was pageable: the copy has consumed it on return
    pool_free(bm, pairs_d, s);
    if (e != cudaSuccess) return cuda_fail(e, "tile gather");
  }
  // commit: the victims leave the cache (their slots not taken return to the
  // free list), the taken free slots leave it, the new entries enter the index
  bm->free_slots.resize(bm->free_slots.size() - from_free);
  {
    const size_t before = bm->free_slots.size();
    evict(bm, victims, &evicted);
    // evict() appended every victim slot; keep only those not taken
    std::vector<int> rest;
    size_t skipped = 0;
    for (size_t i = before; i < bm->free_slots.size(); ++i)
      if (skipped < need - from_free) ++skipped; else rest.push_back(bm->free_slots[i]);
    bm->free_slots.resize(before);
    bm->free_slots.insert(bm->free_slots.end(), rest.begin(), rest.end());
  }
  for (auto& e : made) {
    e->tick = ++bm->tick;
    bm->lru.insert({e->tick, e.get()});
    const uint64_t hsh = e->hash;
    bm->index.emplace(mf_bm_s::Key{key_layer, hsh}, std::move(e));
    ++inserted;
  }
  bm->d = L.d;
  if (counts) {
    counts[0] = inserted;
    counts[1] = present;
    counts[2] = evicted;
  }
  return MF_OK;
}

int mf_bm_match(mf_bm_t bm, int key_layer, const uint64_t* hashes, int n, int* n_hit) {
  if (!bm || !hashes || !n_hit) return fail(MF_ERR_ARG, "NULL argument");
  int k = 0;
  while (k < n) {
    auto it = bm->index.find(mf_bm_s::Key{key_layer, hashes[k]});
    if (it == bm->index.end()) break;
    touch(bm, it->second.get());
    ++k;
  }
  bm->hits += k;
  bm->misses += (k < n) ? 1 : 0;
  *n_hit = k;
  return MF_OK;
}

int mf_bm_assemble(mf_bm_t bm, int key_layer, const uint64_t* hashes, mf_bsr_t h, int layer, void* stream) {
  if (!bm || !h || !hashes) return fail(MF_ERR_ARG, "NULL handle or hashes");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  if (h->H_s != bm->H_s || h->B != bm->B) return fail(MF_ERR_ARG, "the handle's H_s or B differs from the manager's");
  if (!h->causal) return fail(MF_ERR_UNSUPPORTED, "non-causal block-rows are not cached");
  const int H = h->H_s;
  std::vector<BmEntry*> rows((size_t)h->R);
  for (int rb = 0; rb < h->R; ++rb) {
    auto it = bm->index.find(mf_bm_s::Key{key_layer, hashes[rb]});
    if (it == bm->index.end()) return fail(MF_ERR_ARG, "block-row %d is not cached", rb);
    const RowBlock& rbk = h->rbs[rb];
    BmEntry* e = it->second.get();
    if (e->bi != rbk.bi || e->rows != std::min(h->B, rbk.L - rbk.bi * h->B))
      return fail(MF_ERR_ARG, "hash of block-row %d names a cached block-row of another shape", rb);
    rows[rb] = e;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerState& L = h->layers[layer];
  release_layer(h, L, s);
  const MetaLayout ml = meta_layout(h);
  L.meta = dev_alloc(h, ml.bytes, s);
  L.meta_bytes = ml.bytes;
  if (!L.meta) return fail(MF_ERR_OOM, "allocation of %zu bytes failed", ml.bytes);
  carve_meta(L, ml);
  std::vector<int> tile_of((size_t)H * h->C, -1);
  long long ntiles = 0;
  for (int rb = 0; rb < h->R; ++rb) {
    const BmEntry* e = rows[rb];
    const int off = h->rbs[rb].cand_off;
    for (size_t i = 0; i < e->where.size(); ++i) {
      const int bj = e->where[i] / H, hh = e->where[i] % H;
      tile_of[(size_t)(off + bj) * H + hh] = e->slots[i];
    }
    ntiles += (long long)e->where.size();
  }
  MF_CUDA(cudaMemcpyAsync(L.tile_of, tile_of.data(), tile_of.size() * 4, cudaMemcpyHostToDevice, s),
          "tile table upload");
  CompressParams cp{};
  cp.rbs = h->rbs_d;
  cp.H_s = H;
  cp.B = h->B;
  cp.causal = 1;
  cp.R = h->R;
  cp.C = h->C;
  cp.tile_of = L.tile_of;
  cp.union_cnt = L.union_cnt;
  cp.union_list = L.union_list;
  cp.utile = L.utile;
  h->launches[MF_K_UNION] += 1;
  MF_CUDA(launch_union(cp, s), "union kernel");
  L.values = bm->pool;
  L.capacity = bm->cap;  // the pool's zero tile
  L.nnz = ntiles;
  L.nnz_known = true;
  L.stream = s;
  int rc = make_map(&L.pmap, L.values, h->B, (uint64_t)(bm->cap + 1) * h->B, (uint64_t)h->B * 2, 64, 64);
  if (rc != MF_OK) {
    release_layer(h, L, s);
    return rc;
  }
  L.view_bm = bm;
  for (BmEntry* e : rows) {
    pin(bm, e);
    L.view_pins.push_back(e);
  }
  L.valid = true;
  L.dtype = MF_DTYPE_BF16;
  L.d = bm->d;
  L.p = 0.f;
  return MF_OK;
}

int mf_bm_stats(mf_bm_t bm, int64_t* out) {
  if (!bm || !out) return fail(MF_ERR_ARG, "NULL argument");
  out[0] = (int64_t)bm->index.size();
  out[1] = bm->cap - (int64_t)bm->free_slots.size();
  out[2] = bm->cap;
  out[3] = bm->hits;
  out[4] = bm->misses;
  out[5] = bm->evictions;
  out[6] = bm->pinned_entries;
  return MF_OK;
}

}  // extern "C"
