// mf_api.cu — the C ABI of libmapflow (declared in include/mapflow.h):
// argument validation, the per-handle block grid, device buffers, TMA
// tensor maps, and the launch sequence of the compressor and the retrieval.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <map>
#include <vector>

#include "../../include/mapflow.h"
#include "mf_handle.h"
#include "mf_internal.cuh"

using namespace mf;

namespace mf {

static thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------ tensor maps --
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 map: `inner` elements per row, `rows` rows, `stride` bytes between
// rows; box = box_inner x box_rows; 128-byte swizzle; out-of-range reads give 0.
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t stride,
             uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return fail(MF_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (driver too old?)");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {stride};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MF_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MF_OK;
}

}  // namespace mf

namespace mf {

void* dev_alloc(mf_bsr_t h, size_t bytes, cudaStream_t s) {
  if (bytes == 0) bytes = 256;
  if (h->alloc) return h->alloc(bytes, h->ctx, s);
  void* p = nullptr;
  if (cudaMallocAsync(&p, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

void dev_free(mf_bsr_t h, void* p, cudaStream_t s) {
  if (!p) return;
  if (h->dealloc) h->dealloc(p, h->ctx, s);
  else cudaFreeAsync(p, s);
}

void release_layer(mf_bsr_t h, LayerState& L, cudaStream_t s) {
  dev_free(h, L.meta, s);
  if (!L.view_bm) dev_free(h, L.values, s);  // a view's tiles belong to the block manager
  dev_free(h, L.col_idx, s);
  if (L.view_bm) bm_unpin(L);
  if (L.ready) {
    cudaEventSynchronize(L.ready);  // no copy may still use the host buffers
    cudaEventDestroy(L.ready);
  }
  if (L.h_meta) cudaFreeHost(L.h_meta);
  if (L.h_values) cudaFreeHost(L.h_values);
  if (L.h_colidx) cudaFreeHost(L.h_colidx);
  L = LayerState();
}

static size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

MetaLayout meta_layout(const mf_bsr_s* h) {
  const size_t HC = (size_t)h->H_s * h->C, HT = (size_t)h->H_s * h->T, HR = (size_t)h->H_s * h->R;
  MetaLayout m{};
  size_t off = 0;
  m.mass = off; off += align_up(HC * 4);
  m.max = off; off += align_up(HT * 4);
  m.sum = off; off += align_up(HT * 4);
  m.kc = off; off += align_up(HR * 4);
  m.kept = off; off += align_up(HC * 4);
  m.rp = off; off += align_up((HR + 1) * 4);
  m.tile = off; off += align_up(HC * 4);
  m.uc = off; off += align_up((size_t)h->R * 4);
  m.ul = off; off += align_up((size_t)h->C * 4);
  m.ut = off; off += align_up(HC * 4);
  m.km = off; off += align_up(HR * 8 * 4);
  m.nnz = off; off += 256;
  m.bytes = off;
  return m;
}

void carve_meta(LayerState& L, const MetaLayout& m) {
  if (!L.meta) {
    L.mass = L.row_max = L.row_sum = nullptr;
    L.kcount = L.keptcols = L.row_ptr = L.tile_of = L.union_cnt = L.union_list = L.utile = nullptr;
    L.kmask = nullptr;
    L.nnz_dev = nullptr;
    return;
  }
  char* mb = static_cast<char*>(L.meta);
  L.mass = (float*)(mb + m.mass);
  L.row_max = (float*)(mb + m.max);
  L.row_sum = (float*)(mb + m.sum);
  L.kcount = (int*)(mb + m.kc);
  L.keptcols = (int*)(mb + m.kept);
  L.row_ptr = (int*)(mb + m.rp);
  L.tile_of = (int*)(mb + m.tile);
  L.union_cnt = (int*)(mb + m.uc);
  L.union_list = (int*)(mb + m.ul);
  L.utile = (int*)(mb + m.ut);
  L.kmask = (uint32_t*)(mb + m.km);
  L.nnz_dev = (long long*)(mb + m.nnz);
}
}  // namespace mf

namespace {

cudaEvent_t take_event(mf_bsr_t h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Runs one kernel launch, counting it and (when profiling) bracketing it with
// events on its stream.
template <typename F>
cudaError_t timed(mf_bsr_t h, int kind, cudaStream_t s, F&& launch) {
  h->launches[kind] += 1;
  if (!((h->prof_mask >> kind) & 1u)) return launch();
  cudaEvent_t a = take_event(h), b = take_event(h);
  if (a) cudaEventRecord(a, s);
  cudaError_t e = launch();
  if (b) cudaEventRecord(b, s);
  if (a && b) h->prof.push_back(ProfRec{kind, a, b});
  return e;
}

int check_shapes(int dtype, int d, int B) {
  if (B != 64 && B != 128) return 0;
  if (d != 64 && d != 128) return 0;
  if (dtype == MF_DTYPE_BF16) return 1;
  if (dtype == MF_DTYPE_F32) return !(d == 128 && B == 128);
  return 0;
}

}  // namespace

extern "C" {

int mf_version(void) { return 100; }

const char* mf_last_error(void) { return g_last_error.c_str(); }

int mf_supported(int dtype, int d, int B) { return check_shapes(dtype, d, B); }

int mf_bsr_create(mf_bsr_t* out, int n_layers, int T, int H_s, int B, int causal,
                  const int32_t* cu_seqlens_host, int n_seqs, mf_alloc_fn alloc_fn,
                  mf_free_fn free_fn, void* alloc_ctx) {
  return mf_bsr_create_chunked(out, n_layers, T, H_s, B, causal, cu_seqlens_host, nullptr, n_seqs,
                               alloc_fn, free_fn, alloc_ctx);
}

int mf_bsr_create_chunked(mf_bsr_t* out, int n_layers, int T, int H_s, int B, int causal,
                          const int32_t* cu_seqlens_host, const int32_t* q_begin_host, int n_seqs,
                          mf_alloc_fn alloc_fn, mf_free_fn free_fn, void* alloc_ctx) {
  if (!out) return fail(MF_ERR_ARG, "out is NULL");
  *out = nullptr;
  if (n_layers < 1 || T < 1 || H_s < 1 || n_seqs < 1 || !cu_seqlens_host)
    return fail(MF_ERR_ARG, "n_layers, T, H_s, n_seqs must be >= 1 and cu_seqlens non-NULL");
  if ((alloc_fn == nullptr) != (free_fn == nullptr))
    return fail(MF_ERR_ARG, "alloc_fn and free_fn must both be set or both be NULL");
  if (B != 64 && B != 128) return fail(MF_ERR_UNSUPPORTED, "block size %d (supported: 64, 128)", B);
  if (H_s > 128) return fail(MF_ERR_UNSUPPORTED, "H_s = %d > 128", H_s);
  if (causal != 0 && causal != 1) return fail(MF_ERR_ARG, "causal must be 0 or 1");
  if (cu_seqlens_host[0] != 0) return fail(MF_ERR_ARG, "cu_seqlens[0] must be 0");
  for (int s = 0; s < n_seqs; ++s) {
    const int L = cu_seqlens_host[s + 1] - cu_seqlens_host[s];
    if (L < 0) return fail(MF_ERR_ARG, "cu_seqlens must be non-decreasing (sequence %d)", s);
    if (L > 256 * B)
      return fail(MF_ERR_UNSUPPORTED, "sequence %d has length %d > 256*B = %d", s, L, 256 * B);
  }
  if (cu_seqlens_host[n_seqs] != T)
    return fail(MF_ERR_ARG, "cu_seqlens[n_seqs] = %d != T = %d", cu_seqlens_host[n_seqs], T);
  if (q_begin_host) {
    if (!causal) return fail(MF_ERR_UNSUPPORTED, "query chunks need a causal mask");
    long long rows = 0;
    for (int s = 0; s < n_seqs; ++s) {
      const int L = cu_seqlens_host[s + 1] - cu_seqlens_host[s], qb = q_begin_host[s];
      if (qb < 0 || qb > L || (qb % 128 != 0 && qb != L))
        return fail(MF_ERR_ARG, "q_begin[%d] = %d must be a multiple of 128 in [0, %d], or %d", s, qb, L, L);
      rows += L - qb;
    }
    if (rows == 0) return fail(MF_ERR_ARG, "the chunks hold no query rows");
  }

  mf_bsr_t h = new mf_bsr_s();
  h->n_layers = n_layers;
  h->T = T;
  h->H_s = H_s;
  h->B = B;
  h->causal = causal;
  h->n_seqs = n_seqs;
  h->alloc = alloc_fn;
  h->dealloc = free_fn;
  h->ctx = alloc_ctx;
  h->cu.assign(cu_seqlens_host, cu_seqlens_host + n_seqs + 1);
  h->q_begin.assign(n_seqs, 0);
  if (q_begin_host) h->q_begin.assign(q_begin_host, q_begin_host + n_seqs);
  long long cand = 0;
  for (int s = 0; s < n_seqs; ++s) {
    const int start = h->cu[s], L = h->cu[s + 1] - h->cu[s];
    if (h->q_begin[s] == L) continue;  // an empty chunk
    const int nb = (L + B - 1) / B;
    // query block-rows from q_begin on (a chunk over a prefix); keys from 0
    const int b0 = h->q_begin[s] / B;
    const int rb_first = (int)h->rbs.size();  // the handle's index of block-row b0
    for (int bi = b0; bi < nb; ++bi) {
      h->rbs.push_back(RowBlock{start, L, bi, (int)cand});
      cand += causal ? bi + 1 : nb;
      h->max_cand = std::max(h->max_cand, causal ? bi + 1 : nb);
      for (int half = 0; half < B / 64; ++half)
        if (bi * B + half * 64 < L) h->slabs.push_back(RowSlab{rb_first + bi - b0, half});
    }
    const int nt = (L + 127) / 128;
    for (int tl = h->q_begin[s] / 128; tl < nt; ++tl)
      h->tiles.push_back(RowTile{start, L, tl, rb_first + tl * (128 / B) - b0});
  }
  if (cand > (1ll << 30)) {
    delete h;
    return fail(MF_ERR_UNSUPPORTED, "too many candidate blocks");
  }
  // heaviest tiles first: causal work grows with the tile index
  std::stable_sort(h->tiles.begin(), h->tiles.end(),
                   [&](const RowTile& a, const RowTile& b) {
                     const int wa = causal ? a.tl : 0, wb = causal ? b.tl : 0;
                     return wa > wb;
                   });
  // Sequences longest first.  Work that reads a sequence's keys or values
  // again for every item (the pack's K, the retrieval's V) runs sequence by
  // sequence, so the items in flight at one time share what they read in L2;
  // the last items are then the light ones of the shortest sequence.
  std::vector<int> seq_rank(n_seqs);
  {
    std::vector<int> order(n_seqs);
    for (int s = 0; s < n_seqs; ++s) order[s] = s;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
      return h->cu[a + 1] - h->cu[a] > h->cu[b + 1] - h->cu[b];
    });
    for (int r = 0; r < n_seqs; ++r) seq_rank[order[r]] = r;
  }
  std::map<int, int> rank_of_start;  // sequence start token -> rank
  for (int s = 0; s < n_seqs; ++s) rank_of_start[h->cu[s]] = seq_rank[s];
  // heaviest slabs first within each sequence (causal: work grows with the
  // block-row index) so the tail of the retrieval grid is short
  std::stable_sort(h->slabs.begin(), h->slabs.end(), [&](const RowSlab& a, const RowSlab& b) {
    const RowBlock& ra = h->rbs[a.rb];
    const RowBlock& rb = h->rbs[b.rb];
    const int sa = rank_of_start[ra.seq_start], sb = rank_of_start[rb.seq_start];
    if (sa != sb) return sa < sb;
    const int wa = causal ? ra.bi : 0, wb = causal ? rb.bi : 0;
    return wa > wb;
  });
  // The pack's and the two-CTA statistics kernel's items (tile, head):
  // sequence by sequence, and within a sequence in chunks of heads whose keys
  // (at most d = 128) fit in a share of L2, heaviest tiles first within a
  // chunk.  A sequence whose keys fit in 48 MB is one chunk, and then the
  // order is the tile-major heavy-first order; longer ones are chunked, with
  // 12 MB of keys per chunk for the pack (its tile stores stream through L2)
  // and 96 MB for the statistics (measured on 16 packed sequences).
  if (H_s < 256) {
    std::vector<std::vector<int>> by_rank(n_seqs);
    for (int t = 0; t < (int)h->tiles.size(); ++t)
      by_rank[rank_of_start[h->tiles[t].seq_start]].push_back(t);  // tl descending when causal
    auto build_order = [&](long long chunk_bytes, std::vector<int>& out) {
      for (int r = 0; r < n_seqs; ++r) {
        if (by_rank[r].empty()) continue;
        const long long L = h->tiles[by_rank[r][0]].L;
        const long long per_head = L * 128 * 2;
        // a sequence whose keys fit in 48 MB stays one chunk; chunks hold a
        // multiple of 8 query heads when H_s allows, so that no chunk splits
        // a GQA group of 1, 2, 4 or 8 heads (the handle does not know H_ks;
        // the byte budget counts every query head's keys, an upper bound)
        int hc = per_head * H_s <= (48ll << 20)
                     ? H_s
                     : (int)std::max(1ll, std::min<long long>(H_s, chunk_bytes / per_head));
        if (hc < H_s && H_s % 8 == 0) hc = std::min(H_s, (hc + 7) / 8 * 8);
        for (int c0 = 0; c0 < H_s; c0 += hc)
          for (int t : by_rank[r])
            for (int hh = c0; hh < std::min(H_s, c0 + hc); ++hh) out.push_back(t << 8 | hh);
      }
    };
    build_order(12ll << 20, h->pack_items);
    build_order(96ll << 20, h->stats_items);
  }
  h->R = (int)h->rbs.size();
  h->C = (int)cand;
  h->n_tiles = (int)h->tiles.size();
  h->n_slabs = (int)h->slabs.size();
  h->layers.resize(n_layers);

  auto put = [&](void** dst, const void* src, size_t bytes) -> int {
    void* p = dev_alloc(h, bytes, nullptr);
    if (!p) return fail(MF_ERR_OOM, "allocation of %zu bytes failed", bytes);
    *dst = p;
    if (src) {
      cudaError_t e = cudaMemcpy(p, src, bytes, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(tables)");
    }
    return MF_OK;
  };
  int rc = put((void**)&h->rbs_d, h->rbs.data(), sizeof(RowBlock) * h->rbs.size());
  if (rc == MF_OK) rc = put((void**)&h->tiles_d, h->tiles.data(), sizeof(RowTile) * h->tiles.size());
  if (rc == MF_OK) rc = put((void**)&h->slabs_d, h->slabs.data(), sizeof(RowSlab) * h->slabs.size());
  if (rc == MF_OK && !h->pack_items.empty())
    rc = put((void**)&h->pack_items_d, h->pack_items.data(), sizeof(int) * h->pack_items.size());
  if (rc == MF_OK && !h->stats_items.empty())
    rc = put((void**)&h->stats_items_d, h->stats_items.data(), sizeof(int) * h->stats_items.size());
  if (rc == MF_OK) rc = put((void**)&h->err_d, nullptr, sizeof(int));
  if (rc == MF_OK) {
    cudaError_t e = cudaMemset(h->err_d, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMallocHost((void**)&h->host_pinned, 2 * sizeof(long long));
    if (e != cudaSuccess) rc = cuda_fail(e, "handle setup");
  }
  if (rc == MF_OK) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = cuda_fail(e, "handle setup sync");
  }
  if (rc != MF_OK) {
    std::string msg = g_last_error;
    mf_bsr_destroy(h);
    g_last_error = msg;
    return rc;
  }
  *out = h;
  return MF_OK;
}

void mf_bsr_destroy(mf_bsr_t h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (auto& r : h->prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : h->event_pool) cudaEventDestroy(e);
  for (auto& L : h->layers) release_layer(h, L, nullptr);
  dev_free(h, h->rbs_d, nullptr);
  dev_free(h, h->tiles_d, nullptr);
  dev_free(h, h->pack_items_d, nullptr);
  dev_free(h, h->stats_items_d, nullptr);
  dev_free(h, h->slabs_d, nullptr);
  dev_free(h, h->err_d, nullptr);
  dev_free(h, h->ring, nullptr);
  dev_free(h, h->ring_flags, nullptr);
  dev_free(h, h->team_slabs_d, nullptr);
  cudaDeviceSynchronize();
  if (h->host_pinned) cudaFreeHost(h->host_pinned);
  delete h;
}

int mf_compress(mf_bsr_t h, int layer, const void* q, const void* k, int dtype, int T, int H_s,
                int H_ks, int d, int B, float p, int causal, void* stream) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer %d out of range", layer);
  if (!q || !k) return fail(MF_ERR_ARG, "q and k must be non-NULL");
  if (T != h->T || H_s != h->H_s || B != h->B || causal != h->causal)
    return fail(MF_ERR_ARG, "T/H_s/B/causal differ from the handle's");
  if (H_ks < 1 || H_s % H_ks != 0) return fail(MF_ERR_ARG, "H_s %% H_ks != 0");
  if (!(p > 0.f && p <= 1.f)) return fail(MF_ERR_ARG, "p must be in (0, 1]");
  if (dtype != MF_DTYPE_BF16 && dtype != MF_DTYPE_F32) return fail(MF_ERR_ARG, "unknown dtype");
  if (!check_shapes(dtype, d, B))
    return fail(MF_ERR_UNSUPPORTED, "dtype %d with d = %d, B = %d is not built", dtype, d, B);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerState& L = h->layers[layer];
  if (L.meta || L.values || L.col_idx || L.offloaded || L.ready) release_layer(h, L, s);

  const size_t HC = (size_t)h->H_s * h->C;
  const MetaLayout ml = meta_layout(h);
  L.meta = dev_alloc(h, ml.bytes, s);
  if (!L.meta) return fail(MF_ERR_OOM, "allocation of %zu bytes failed", ml.bytes);
  L.meta_bytes = ml.bytes;
  carve_meta(L, ml);

  CompressParams cp{};
  cp.rbs = h->rbs_d;
  cp.tiles = h->tiles_d;
  cp.n_tiles = h->n_tiles;
  cp.items = h->pack_items_d;
  cp.stats_items = h->stats_items_d;
  cp.T = T;
  cp.H_s = H_s;
  cp.H_ks = H_ks;
  cp.d = d;
  cp.B = B;
  cp.causal = causal;
  cp.R = h->R;
  cp.C = h->C;
  cp.max_cand = h->max_cand;
  cp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  cp.p = p;
  cp.mass = L.mass;
  cp.row_max = L.row_max;
  cp.row_sum = L.row_sum;
  cp.kcount = L.kcount;
  cp.keptcols = L.keptcols;
  cp.row_ptr = L.row_ptr;
  cp.tile_of = L.tile_of;
  cp.union_cnt = L.union_cnt;
  cp.union_list = L.union_list;
  cp.utile = L.utile;
  cp.kmask = (dtype == MF_DTYPE_BF16) ? L.kmask : nullptr;
  cp.nnz_out = L.nnz_dev;
  cp.pack_ctr = reinterpret_cast<int*>(L.nnz_dev + 1);  // in the 256-byte scalar slot
  cp.sel_done = reinterpret_cast<int*>(L.nnz_dev + 1) + 1;
  cp.err = h->err_d;

  CUtensorMap tq{}, tk{}, tk_pack{};
  int rc;
  if (dtype == MF_DTYPE_BF16) {
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(k) & 15))
      return fail(MF_ERR_ARG, "q and k must be 16-byte aligned");
    if ((rc = make_map(&tq, q, (uint64_t)H_s * d, T, (uint64_t)H_s * d * 2, 64, 128)) != MF_OK) return rc;
    if ((rc = make_map(&tk_pack, k, (uint64_t)H_ks * d, T, (uint64_t)H_ks * d * 2, 64, B)) != MF_OK) return rc;
    if (stats2_supported(h->max_cand)) {
      // two CTAs per SM on 64-key tiles (rows of at most 128 candidate blocks)
      CUtensorMap tk64 = tk_pack;
      if (B != 64 &&
          (rc = make_map(&tk64, k, (uint64_t)H_ks * d, T, (uint64_t)H_ks * d * 2, 64, 64)) != MF_OK)
        return rc;
      MF_CUDA(timed(h, MF_K_STATS, s, [&] { return launch_stats2_bf16(cp, tq, tk64, s); }),
              "statistics kernel");
    } else {
      if ((rc = make_map(&tk, k, (uint64_t)H_ks * d, T, (uint64_t)H_ks * d * 2, 64, 128)) != MF_OK) return rc;
      MF_CUDA(timed(h, MF_K_STATS, s, [&] { return launch_stats_bf16(cp, tq, tk, s); }),
              "statistics kernel");
    }
  } else {
    MF_CUDA(timed(h, MF_K_STATS, s,
                  [&] { return launch_stats_f32(cp, (const float*)q, (const float*)k, s); }),
            "statistics kernel (fp32)");
  }
  MF_CUDA(timed(h, MF_K_SELECT, s, [&] { return launch_select(cp, s); }), "selection kernel");
  long long cap;
  if (h->exact_alloc) {
    // exact size: learn nnz first (the one host round trip of this mode)
    MF_CUDA(cudaMemcpyAsync(&h->host_pinned[0], L.nnz_dev, sizeof(long long), cudaMemcpyDeviceToHost, s),
            "nnz copy");
    MF_CUDA(cudaMemcpyAsync(&h->host_pinned[1], h->err_d, sizeof(int), cudaMemcpyDeviceToHost, s),
            "error word copy");
    MF_CUDA(cudaStreamSynchronize(s), "compress sync");
    const int dev_err = static_cast<int>(h->host_pinned[1] & 0xffffffff);
    if (dev_err) {
      cudaMemsetAsync(h->err_d, 0, sizeof(int), s);
      release_layer(h, L, s);
      return fail(MF_ERR_TIMEOUT, "a device-side wait timed out in the compressor");
    }
    cap = h->host_pinned[0];
    L.nnz = cap;
    L.nnz_known = true;
  } else {
    // upper bound (every candidate kept): no host round trip; nnz stays on
    // the device until someone asks for it
    cap = (long long)HC;
    L.nnz_known = false;
  }
  L.capacity = cap;
  L.stream = s;
  L.values_bytes = (size_t)cap * B * B * 2;
  L.colidx_bytes = (size_t)cap * 4;
  // one extra all-zero tile after the kept ones: the retrieval reads it in
  // place of a head's dropped block
  L.values = (uint16_t*)dev_alloc(h, L.values_bytes + (size_t)B * B * 2, s);
  L.col_idx = (int*)dev_alloc(h, L.colidx_bytes, s);
  if (!L.values || !L.col_idx) {
    release_layer(h, L, s);
    return fail(MF_ERR_OOM, "allocation of %zu bytes for the BSR values failed", L.values_bytes);
  }
  cp.col_idx = L.col_idx;
  // the bf16 pack kernel writes the zero tile itself; the selection kernel
  // has reset every candidate's tile index
  if (dtype != MF_DTYPE_BF16 || cap == 0)
    MF_CUDA(cudaMemsetAsync(reinterpret_cast<char*>(L.values) + L.values_bytes, 0, (size_t)B * B * 2, s),
            "zero tile");
  else
    cp.zero_tile = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(L.values) + L.values_bytes);
  // the bf16 pack kernel writes the retrieval's union tables from the
  // selection's masks
  cp.union_in_pack = (dtype == MF_DTYPE_BF16 && cap > 0) ? 1 : 0;
  if (cap > 0) {
    if (dtype == MF_DTYPE_BF16) {
      CUtensorMap tvals{};
      // the pack kernel's writer warps each store 32 rows x B/2 columns
      if ((rc = make_map(&tvals, L.values, B, (uint64_t)cap * B, (uint64_t)B * 2, B / 2, 32,
                         B == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B)) != MF_OK)
        return rc;
      MF_CUDA(timed(h, MF_K_PACK, s, [&] { return launch_pack_bf16(cp, tq, tk_pack, tvals, s); }),
              "pack kernel");
    } else {
      MF_CUDA(timed(h, MF_K_PACK, s,
                    [&] { return launch_pack_f32(cp, (const float*)q, (const float*)k, L.values, s); }),
              "pack kernel (fp32)");
    }
  }
  if (!cp.union_in_pack)
    MF_CUDA(timed(h, MF_K_UNION, s, [&] { return launch_union(cp, s); }), "union kernel");
  if ((rc = make_map(&L.pmap, L.values, B, (uint64_t)(cap + 1) * B, (uint64_t)B * 2, 64, 64)) != MF_OK)
    return rc;
  L.valid = true;
  L.dtype = dtype;
  L.d = d;
  L.p = p;
  return MF_OK;
}

int mf_retrieve(mf_bsr_t h, const float* W, const void* v, void* o, int dtype, int H_r, int H_kv,
                int d, const int32_t* layer_map_host, int n, void* stream) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (!W || !v || !o || !layer_map_host) return fail(MF_ERR_ARG, "NULL pointer argument");
  if (n < 1) return fail(MF_ERR_ARG, "n must be >= 1");
  if (H_r < 1 || H_kv < 1 || H_r % H_kv != 0) return fail(MF_ERR_ARG, "H_r %% H_kv != 0");
  if (dtype != MF_DTYPE_BF16 && dtype != MF_DTYPE_F32) return fail(MF_ERR_ARG, "unknown dtype");
  if (!check_shapes(dtype, d, h->B))
    return fail(MF_ERR_UNSUPPORTED, "dtype %d with d = %d, B = %d is not built", dtype, d, h->B);
  const int hpg = H_r / H_kv;
  if (dtype == MF_DTYPE_BF16 && hpg > 8)
    return fail(MF_ERR_UNSUPPORTED, "H_r / H_kv = %d > 8", hpg);
  if (dtype == MF_DTYPE_BF16 && ((reinterpret_cast<uintptr_t>(v) & 15) || (reinterpret_cast<uintptr_t>(o) & 15)))
    return fail(MF_ERR_ARG, "v and o must be 16-byte aligned");
  for (int x = 0; x < n; ++x) {
    const int sl = layer_map_host[x];
    if (sl < 0 || sl >= h->n_layers) return fail(MF_ERR_ARG, "layer_map[%d] = %d out of range", x, sl);
    const LayerState& L = h->layers[sl];
    if (!L.valid) return fail(MF_ERR_STATE, "sender layer %d has not been compressed", sl);
    if (L.offloaded) return fail(MF_ERR_STATE, "sender layer %d is offloaded (mf_bsr_prefetch it)", sl);
    if (L.d != d) return fail(MF_ERR_ARG, "d = %d differs from the compressed layer's %d", d, L.d);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // a prefetch may still be copying a layer in on another stream
  for (int x = 0; x < n; ++x) {
    const LayerState& L = h->layers[layer_map_host[x]];
    if (L.ready) MF_CUDA(cudaStreamWaitEvent(s, L.ready, 0), "wait for the layer's prefetch");
  }
  const size_t esz = (dtype == MF_DTYPE_BF16) ? 2 : 4;
  const size_t v_layer = (size_t)h->T * H_kv * d * esz;
  const size_t o_layer = (size_t)h->T * H_r * d * esz;
  for (int x = 0; x < n; ++x) {
    const LayerState& L = h->layers[layer_map_host[x]];
    RetrieveParams rp{};
    rp.rbs = h->rbs_d;
    rp.slabs = h->slabs_d;
    rp.n_slabs = h->n_slabs;
    rp.T = h->T;
    rp.H_s = h->H_s;
    rp.H_r = H_r;
    rp.H_kv = H_kv;
    rp.d = d;
    rp.B = h->B;
    rp.R = h->R;
    rp.C = h->C;
    rp.tile_of = L.tile_of;
    rp.union_cnt = L.union_cnt;
    rp.union_list = L.union_list;
    rp.utile = L.utile;
    rp.W = W + (size_t)x * H_r * h->H_s;
    rp.zero_tile = (int)L.capacity;
    rp.values = L.values;
    rp.err = h->err_d;
    const char* vx = static_cast<const char*>(v) + x * v_layer;
    char* ox = static_cast<char*>(o) + x * o_layer;
    if (dtype == MF_DTYPE_BF16) {
      CUtensorMap tv{};
      int rc = make_map(&tv, vx, (uint64_t)H_kv * d, h->T, (uint64_t)H_kv * d * 2, 64, 64);
      if (rc != MF_OK) return rc;
      if (retrieve_team_supported(h->H_s, H_r, H_kv, d, h->B)) {
        int sms = 0;
        MF_CUDA(sm_count(&sms), "device query");
        const int teams = retrieve_team_count(h->n_slabs, sms);
        if (!h->ring) {
          const int cap = retrieve_team_count(1 << 30, sms);
          h->ring = dev_alloc(h, retrieve_team_ring_bytes(cap), s);
          h->ring_flags = (uint32_t*)dev_alloc(h, retrieve_team_flag_bytes(cap), s);
          if (!h->ring || !h->ring_flags) return fail(MF_ERR_OOM, "exchange ring allocation failed");
          // zero once: each launch leaves the counters at zero when it ends
          MF_CUDA(cudaMemsetAsync(h->ring_flags, 0, retrieve_team_flag_bytes(cap), s), "ring reset");
          h->ring_teams = cap;
        }
        if (h->team_slab_teams != teams) {
          // Work of a slab ~ its candidate blocks (causal: bi + 1); slabs come
          // heaviest first, each goes to the team with the least work so far.
          std::vector<std::vector<int>> lists(teams);
          std::vector<long long> load(teams, 0);
          for (int i = 0; i < h->n_slabs; ++i) {
            const RowBlock& rb = h->rbs[h->slabs[i].rb];
            const long long wgt = h->causal ? rb.bi + 1 : (rb.L + h->B - 1) / h->B;
            int best = 0;
            for (int t = 1; t < teams; ++t)
              if (load[t] < load[best]) best = t;
            lists[best].push_back(i);
            load[best] += wgt;
          }
          int stride = 1;
          for (auto& l : lists) stride = std::max(stride, (int)l.size());
          h->team_slabs.assign((size_t)teams * stride, -1);
          for (int t = 0; t < teams; ++t)
            for (size_t j = 0; j < lists[t].size(); ++j) h->team_slabs[(size_t)t * stride + j] = lists[t][j];
          dev_free(h, h->team_slabs_d, s);
          h->team_slabs_d = (int*)dev_alloc(h, h->team_slabs.size() * sizeof(int), s);
          if (!h->team_slabs_d) return fail(MF_ERR_OOM, "slab table allocation failed");
          MF_CUDA(cudaMemcpyAsync(h->team_slabs_d, h->team_slabs.data(), h->team_slabs.size() * sizeof(int),
                                  cudaMemcpyHostToDevice, s),
                  "slab table copy");
          h->team_slab_teams = teams;
          h->team_stride = stride;
        }
        rp.team_slabs = h->team_slabs_d;
        rp.team_stride = h->team_stride;
        CUtensorMap ta{};
        rc = make_map(&ta, h->ring, 64, (uint64_t)retrieve_team_ring_rows(h->ring_teams), 128, 64,
                      (uint32_t)retrieve_team_ring_box_rows(H_r));
        if (rc != MF_OK) return rc;
        MF_CUDA(timed(h, MF_K_RETRIEVE, s,
                      [&] {
                        return launch_retrieve_team(rp, ta, tv, ox, h->ring, h->ring_flags, teams, s);
                      }),
                "retrieval kernel (team)");
      } else {
        MF_CUDA(timed(h, MF_K_RETRIEVE, s,
                      [&] { return launch_retrieve_bf16(rp, L.pmap, tv, ox, s); }),
                "retrieval kernel");
      }
    } else {
      MF_CUDA(timed(h, MF_K_RETRIEVE, s,
                    [&] {
                      return launch_retrieve_f32(rp, L.values, (const float*)vx, (float*)ox, s);
                    }),
              "retrieval kernel (fp32)");
    }
  }
  return MF_OK;
}

}  // extern "C"

namespace {
// Reads a layer's kept-tile count from the device (waits for its compress).
int ensure_nnz(mf_bsr_t h, LayerState& L) {
  if (L.nnz_known) return MF_OK;
  MF_CUDA(cudaMemcpyAsync(&h->host_pinned[0], L.nnz_dev, sizeof(long long), cudaMemcpyDeviceToHost,
                          L.stream),
          "nnz copy");
  MF_CUDA(cudaStreamSynchronize(L.stream), "nnz sync");
  L.nnz = h->host_pinned[0];
  L.nnz_known = true;
  return MF_OK;
}
}  // namespace

extern "C" {

int mf_bsr_set_exact(mf_bsr_t h, int exact) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  h->exact_alloc = exact != 0;
  return MF_OK;
}

int mf_bsr_info(mf_bsr_t h, int layer, int64_t* nnz, int64_t* n_rows, int64_t* n_cand) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  LayerState& L = h->layers[layer];
  if (!L.valid) return fail(MF_ERR_STATE, "layer %d has not been compressed", layer);
  if (nnz) {
    const int rc = ensure_nnz(h, L);
    if (rc != MF_OK) return rc;
  }
  if (nnz) *nnz = L.nnz;
  if (n_rows) *n_rows = (int64_t)h->H_s * h->R;
  if (n_cand) *n_cand = (int64_t)h->H_s * h->C;
  return MF_OK;
}

int mf_bsr_export(mf_bsr_t h, int layer, const int32_t** row_ptr, const int32_t** col_idx,
                  const uint16_t** values, const float** mass, const float** row_max,
                  const float** row_sum) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  const LayerState& L = h->layers[layer];
  if (!L.valid) return fail(MF_ERR_STATE, "layer %d has not been compressed", layer);
  if (L.view_bm) return fail(MF_ERR_STATE, "layer %d is a block-manager view (its tiles are the manager's)", layer);
  if (L.offloaded) return fail(MF_ERR_STATE, "layer %d is offloaded", layer);
  if (row_ptr) *row_ptr = L.row_ptr;
  if (col_idx) *col_idx = L.col_idx;
  if (values) *values = L.values;
  if (mass) *mass = L.mass;
  if (row_max) *row_max = L.row_max;
  if (row_sum) *row_sum = L.row_sum;
  return MF_OK;
}

int mf_bsr_copy(mf_bsr_t h, int layer, int32_t* row_ptr, int32_t* col_idx, uint16_t* values,
                float* mass, float* row_max, float* row_sum, void* stream) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  LayerState& L = h->layers[layer];
  if (!L.valid) return fail(MF_ERR_STATE, "layer %d has not been compressed", layer);
  if (L.view_bm) return fail(MF_ERR_STATE, "layer %d is a block-manager view (its tiles are the manager's)", layer);
  if (L.offloaded) return fail(MF_ERR_STATE, "layer %d is offloaded", layer);
  if (col_idx || values) {
    const int rc = ensure_nnz(h, L);
    if (rc != MF_OK) return rc;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.ready) MF_CUDA(cudaStreamWaitEvent(s, L.ready, 0), "wait for the layer's prefetch");
  const size_t HR = (size_t)h->H_s * h->R, HC = (size_t)h->H_s * h->C, HT = (size_t)h->H_s * h->T;
  auto cp = [&](void* dst, const void* src, size_t bytes) {
    return (dst && bytes) ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s) : cudaSuccess;
  };
  MF_CUDA(cp(row_ptr, L.row_ptr, (HR + 1) * 4), "row_ptr copy");
  MF_CUDA(cp(col_idx, L.col_idx, (size_t)L.nnz * 4), "col_idx copy");
  MF_CUDA(cp(values, L.values, (size_t)L.nnz * h->B * h->B * 2), "values copy");
  MF_CUDA(cp(mass, L.mass, HC * 4), "mass copy");
  MF_CUDA(cp(row_max, L.row_max, HT * 4), "row_max copy");
  MF_CUDA(cp(row_sum, L.row_sum, HT * 4), "row_sum copy");
  return MF_OK;
}

int mf_bsr_release_layer(mf_bsr_t h, int layer) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  release_layer(h, h->layers[layer], nullptr);
  return MF_OK;
}

int mf_bsr_offload(mf_bsr_t h, int layer, void* stream) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  LayerState& L = h->layers[layer];
  if (!L.valid) return fail(MF_ERR_STATE, "layer %d has not been compressed", layer);
  if (L.view_bm) return fail(MF_ERR_STATE, "layer %d is a block-manager view (its tiles are the manager's)", layer);
  if (L.offloaded) return MF_OK;
  int rc = ensure_nnz(h, L);  // only the kept tiles travel
  if (rc != MF_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.ready) MF_CUDA(cudaStreamWaitEvent(s, L.ready, 0), "wait for the layer's prefetch");
  const size_t vbytes = (size_t)L.nnz * h->B * h->B * 2, cbytes = (size_t)L.nnz * 4;
  if (!L.h_meta) MF_CUDA(cudaMallocHost(&L.h_meta, L.meta_bytes), "pinned host allocation");
  if (L.h_values_cap < vbytes) {
    if (L.h_values) cudaFreeHost(L.h_values);
    L.h_values = nullptr;
    L.h_values_cap = 0;
    MF_CUDA(cudaMallocHost(&L.h_values, vbytes), "pinned host allocation");
    L.h_values_cap = vbytes;
  }
  if (L.h_colidx_cap < cbytes) {
    if (L.h_colidx) cudaFreeHost(L.h_colidx);
    L.h_colidx = nullptr;
    L.h_colidx_cap = 0;
    MF_CUDA(cudaMallocHost(&L.h_colidx, cbytes), "pinned host allocation");
    L.h_colidx_cap = cbytes;
  }
  MF_CUDA(cudaMemcpyAsync(L.h_meta, L.meta, L.meta_bytes, cudaMemcpyDeviceToHost, s), "offload copy");
  if (vbytes) MF_CUDA(cudaMemcpyAsync(L.h_values, L.values, vbytes, cudaMemcpyDeviceToHost, s), "offload copy");
  if (cbytes) MF_CUDA(cudaMemcpyAsync(L.h_colidx, L.col_idx, cbytes, cudaMemcpyDeviceToHost, s), "offload copy");
  // the device buffers go back to the allocator behind the copies
  dev_free(h, L.meta, s);
  dev_free(h, L.values, s);
  dev_free(h, L.col_idx, s);
  L.meta = nullptr;
  L.values = nullptr;
  L.col_idx = nullptr;
  carve_meta(L, meta_layout(h));  // null until the prefetch
  if (!L.ready) MF_CUDA(cudaEventCreateWithFlags(&L.ready, cudaEventDisableTiming), "event");
  MF_CUDA(cudaEventRecord(L.ready, s), "event record");
  L.offloaded = true;
  return MF_OK;
}

int mf_bsr_prefetch(mf_bsr_t h, int layer, void* stream) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (layer < 0 || layer >= h->n_layers) return fail(MF_ERR_ARG, "layer out of range");
  LayerState& L = h->layers[layer];
  if (!L.valid) return fail(MF_ERR_STATE, "layer %d has not been compressed", layer);
  if (!L.offloaded) return MF_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MF_CUDA(cudaStreamWaitEvent(s, L.ready, 0), "wait for the layer's offload");
  const int B = h->B;
  const long long nnz = L.nnz;
  const size_t vbytes = (size_t)nnz * B * B * 2, cbytes = (size_t)nnz * 4;
  const MetaLayout ml = meta_layout(h);
  L.meta = dev_alloc(h, ml.bytes, s);
  L.values = (uint16_t*)dev_alloc(h, vbytes + (size_t)B * B * 2, s);
  L.col_idx = (int*)dev_alloc(h, cbytes ? cbytes : 4, s);
  if (!L.meta || !L.values || !L.col_idx) {
    dev_free(h, L.meta, s);
    dev_free(h, L.values, s);
    dev_free(h, L.col_idx, s);
    L.meta = nullptr;
    L.values = nullptr;
    L.col_idx = nullptr;
    return fail(MF_ERR_OOM, "device allocation for the prefetch failed");
  }
  carve_meta(L, ml);
  MF_CUDA(cudaMemcpyAsync(L.meta, L.h_meta, ml.bytes, cudaMemcpyHostToDevice, s), "prefetch copy");
  if (vbytes) MF_CUDA(cudaMemcpyAsync(L.values, L.h_values, vbytes, cudaMemcpyHostToDevice, s), "prefetch copy");
  if (cbytes) MF_CUDA(cudaMemcpyAsync(L.col_idx, L.h_colidx, cbytes, cudaMemcpyHostToDevice, s), "prefetch copy");
  // the retrieval's all-zero tile, right after the kept ones
  MF_CUDA(cudaMemsetAsync(reinterpret_cast<char*>(L.values) + vbytes, 0, (size_t)B * B * 2, s), "zero tile");
  L.capacity = nnz;
  L.values_bytes = vbytes;
  L.colidx_bytes = cbytes;
  const int rc = make_map(&L.pmap, L.values, B, (uint64_t)(nnz + 1) * B, (uint64_t)B * 2, 64, 64);
  if (rc != MF_OK) return rc;
  L.stream = s;
  MF_CUDA(cudaEventRecord(L.ready, s), "event record");
  L.offloaded = false;
  return MF_OK;
}

int mf_calibrate_head_map(mf_bsr_t sender, int sender_layer, mf_bsr_t receiver, int receiver_layer,
                          float ridge, float* W_out, void* stream) {
  if (!sender || !receiver || !W_out) return fail(MF_ERR_ARG, "NULL handle or W_out");
  if (sender_layer < 0 || sender_layer >= sender->n_layers || receiver_layer < 0 ||
      receiver_layer >= receiver->n_layers)
    return fail(MF_ERR_ARG, "layer out of range");
  if (!(ridge >= 0.f)) return fail(MF_ERR_ARG, "ridge must be >= 0");
  if (sender->T != receiver->T || sender->B != receiver->B || sender->causal != receiver->causal ||
      sender->cu != receiver->cu || sender->q_begin != receiver->q_begin)
    return fail(MF_ERR_ARG, "the two handles must share sequences, block size and causality");
  const int H_s = sender->H_s, H_r = receiver->H_s;
  if (H_s + H_r > kCalibRows)
    return fail(MF_ERR_UNSUPPORTED, "H_s + H_r = %d > %d", H_s + H_r, kCalibRows);
  LayerState& SL = sender->layers[sender_layer];
  LayerState& RL = receiver->layers[receiver_layer];
  if (!SL.valid || !RL.valid) return fail(MF_ERR_STATE, "both layers must be compressed");
  if (SL.offloaded || RL.offloaded) return fail(MF_ERR_STATE, "both layers must be on the device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (SL.ready) MF_CUDA(cudaStreamWaitEvent(s, SL.ready, 0), "wait for the layer's prefetch");
  if (RL.ready) MF_CUDA(cudaStreamWaitEvent(s, RL.ready, 0), "wait for the layer's prefetch");
  const int n = H_s + H_r;
  const int grid = calib_grid(sender->C);
  const size_t gbytes = (size_t)n * n * sizeof(double);
  const size_t pbytes = (size_t)grid * kCalibRows * kCalibRows * sizeof(float);
  char* scratch = (char*)dev_alloc(sender, gbytes + pbytes, s);
  if (!scratch) return fail(MF_ERR_OOM, "allocation of %zu bytes failed", gbytes + pbytes);
  double* G_d = reinterpret_cast<double*>(scratch);
  CalibParams cp{SL.tile_of, SL.values, RL.tile_of, RL.values, sender->C, H_s, H_r, sender->B,
                 reinterpret_cast<float*>(scratch + gbytes), sender->err_d};
  // the Gram matrix of [sender heads; receiver heads] over every stored entry
  std::vector<double> G((size_t)n * n);
  cudaError_t e = launch_calib_gram(cp, grid, G_d, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(G.data(), G_d, gbytes, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&sender->host_pinned[1], sender->err_d, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  dev_free(sender, scratch, s);
  if (e != cudaSuccess) return cuda_fail(e, "calibration kernel");
  if (static_cast<int>(sender->host_pinned[1] & 0xffffffff)) {
    cudaMemsetAsync(sender->err_d, 0, sizeof(int), s);
    return fail(MF_ERR_TIMEOUT, "a device-side wait timed out in the calibration kernel");
  }
  // Cholesky factor of the sender block plus ridge: L L^T = G_ss + ridge I
  std::vector<double> L((size_t)H_s * H_s, 0.0);
  for (int i = 0; i < H_s; ++i) {
    for (int j = 0; j <= i; ++j) {
      double acc = G[(size_t)i * n + j] + (i == j ? (double)ridge : 0.0);
      for (int k = 0; k < j; ++k) acc -= L[(size_t)i * H_s + k] * L[(size_t)j * H_s + k];
      if (i == j) {
        if (!(acc > 0.0))
          return fail(MF_ERR_ARG, "the sender heads' Gram matrix is singular (pass ridge > 0)");
        L[(size_t)i * H_s + i] = std::sqrt(acc);
      } else {
        L[(size_t)i * H_s + j] = acc / L[(size_t)j * H_s + j];
      }
    }
  }
  // each receiver head: solve L L^T w = C_i with C_i[h] = G[H_s + i][h]
  std::vector<double> y(H_s), w(H_s);
  for (int i = 0; i < H_r; ++i) {
    for (int a = 0; a < H_s; ++a) {
      double acc = G[(size_t)(H_s + i) * n + a];
      for (int k = 0; k < a; ++k) acc -= L[(size_t)a * H_s + k] * y[k];
      y[a] = acc / L[(size_t)a * H_s + a];
    }
    for (int a = H_s - 1; a >= 0; --a) {
      double acc = y[a];
      for (int k = a + 1; k < H_s; ++k) acc -= L[(size_t)k * H_s + a] * w[k];
      w[a] = acc / L[(size_t)a * H_s + a];
    }
    for (int a = 0; a < H_s; ++a) W_out[(size_t)i * H_s + a] = (float)w[a];
  }
  return MF_OK;
}

int mf_device_status(mf_bsr_t h, void* stream) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MF_CUDA(cudaMemcpyAsync(&h->host_pinned[1], h->err_d, sizeof(int), cudaMemcpyDeviceToHost, s),
          "error word copy");
  MF_CUDA(cudaStreamSynchronize(s), "status sync");
  const int e = static_cast<int>(h->host_pinned[1] & 0xffffffff);
  if (e) {
    cudaMemsetAsync(h->err_d, 0, sizeof(int), s);
    cudaStreamSynchronize(s);
    return fail(MF_ERR_TIMEOUT, "a device-side wait timed out");
  }
  return MF_OK;
}

int mf_profile_kinds(mf_bsr_t h, int mask) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  const unsigned m = static_cast<unsigned>(mask) & ((1u << MF_K_COUNT) - 1u);
  if (m) {
    for (auto& r : h->prof) {
      h->event_pool.push_back(r.a);
      h->event_pool.push_back(r.b);
    }
    h->prof.clear();
    for (auto& c : h->launches) c = 0;
  }
  h->prof_mask = m;
  return MF_OK;
}

int mf_profile(mf_bsr_t h, int enable) {
  return mf_profile_kinds(h, enable ? static_cast<int>((1u << MF_K_COUNT) - 1u) : 0);
}

int mf_profile_read(mf_bsr_t h, int kernel, int64_t* launches, double* total_ms) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (kernel < 0 || kernel >= MF_K_COUNT) return fail(MF_ERR_ARG, "unknown kernel kind");
  double tot = 0.0;
  for (auto& r : h->prof) {
    if (r.kind != kernel) continue;
    MF_CUDA(cudaEventSynchronize(r.b), "event sync");
    float ms = 0.f;
    MF_CUDA(cudaEventElapsedTime(&ms, r.a, r.b), "event elapsed");
    tot += ms;
  }
  if (launches) *launches = h->launches[kernel];
  if (total_ms) *total_ms = tot;
  return MF_OK;
}

int mf_select_noalloc(const float* mass, const int32_t* cu_seqlens_host, int n_seqs, int H_s,
                      int B, int causal, float p, int32_t* row_ptr, int32_t* col_idx,
                      int64_t col_capacity, int64_t* nnz, void* stream) {
  if (!mass || !cu_seqlens_host || !row_ptr || !col_idx || !nnz)
    return fail(MF_ERR_ARG, "NULL pointer argument");
  if (n_seqs < 1 || H_s < 1) return fail(MF_ERR_ARG, "n_seqs and H_s must be >= 1");
  if (B != 64 && B != 128) return fail(MF_ERR_UNSUPPORTED, "block size %d (supported: 64, 128)", B);
  if (causal != 0 && causal != 1) return fail(MF_ERR_ARG, "causal must be 0 or 1");
  if (!(p > 0.f && p <= 1.f)) return fail(MF_ERR_ARG, "p must be in (0, 1]");
  if (cu_seqlens_host[0] != 0) return fail(MF_ERR_ARG, "cu_seqlens[0] must be 0");
  std::vector<RowBlock> rbs;
  long long cand = 0;
  for (int s = 0; s < n_seqs; ++s) {
    const int start = cu_seqlens_host[s], L = cu_seqlens_host[s + 1] - cu_seqlens_host[s];
    if (L < 0) return fail(MF_ERR_ARG, "cu_seqlens must be non-decreasing (sequence %d)", s);
    if (L > 256 * B)
      return fail(MF_ERR_UNSUPPORTED, "sequence %d has length %d > 256*B = %d", s, L, 256 * B);
    const int nb = (L + B - 1) / B;
    for (int bi = 0; bi < nb; ++bi) {
      rbs.push_back(RowBlock{start, L, bi, (int)cand});
      cand += causal ? bi + 1 : nb;
    }
  }
  const long long R = (long long)rbs.size();
  if (R == 0) return fail(MF_ERR_ARG, "no tokens");
  if (col_capacity < (long long)H_s * cand)
    return fail(MF_ERR_ARG, "col_capacity %lld < H_s * candidates = %lld",
                (long long)col_capacity, (long long)H_s * cand);
  const size_t need = noalloc_needed_bytes(R, H_s, cand);
  if (need > noalloc_scratch_bytes())
    return fail(MF_ERR_UNSUPPORTED,
                "this selection needs %zu bytes of scratch; the no-allocation entry point "
                "reserves %zu bytes per device",
                need, noalloc_scratch_bytes());
  MF_CUDA(launch_select_noalloc(rbs.data(), (int)R, (int)cand, H_s, B, causal, p, mass, row_ptr,
                                col_idx, reinterpret_cast<long long*>(nnz),
                                static_cast<cudaStream_t>(stream)),
          "no-allocation selection");
  return MF_OK;
}

int mf_selftest_wait(mf_bsr_t h, int limit_ms, void* stream) {
  if (!h) return fail(MF_ERR_ARG, "handle is NULL");
  if (limit_ms < 1 || limit_ms > 10000) return fail(MF_ERR_ARG, "limit_ms must be in [1, 10000]");
  MF_CUDA(launch_selftest_wait(h->err_d, (unsigned long long)limit_ms * 1000000ull,
                               static_cast<cudaStream_t>(stream)),
          "self-test kernel");
  return MF_OK;
}

}  // extern "C"
