// mf_handle.h — host-side internals shared by the ABI's translation units:
// the BSR handle and its per-layer state, error reporting, device allocation
// through the handle's allocator, and TMA tensor-map encoding.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <string>
#include <vector>

#include "../../include/mapflow.h"
#include "mf_internal.cuh"

namespace mf {
struct BmEntry;  // a block-row state cached by a block manager
}

// --------------------------------------------------------------- handle --
struct LayerState {
  bool valid = false;
  int dtype = -1;
  int d = 0;
  float p = 0.f;
  long long nnz = 0;       // valid when nnz_known
  bool nnz_known = false;
  long long capacity = 0;  // tiles allocated for kept blocks (zero tile at this index)
  cudaStream_t stream = nullptr;
  void* meta = nullptr;    // one allocation carved into the arrays below
  size_t meta_bytes = 0;
  float* mass = nullptr;
  float* row_max = nullptr;
  float* row_sum = nullptr;
  int* kcount = nullptr;
  int* keptcols = nullptr;
  int* row_ptr = nullptr;
  int* tile_of = nullptr;
  int* union_cnt = nullptr;
  int* union_list = nullptr;
  int* utile = nullptr;
  uint32_t* kmask = nullptr;
  long long* nnz_dev = nullptr;
  int* col_idx = nullptr;
  uint16_t* values = nullptr;
  size_t values_bytes = 0, colidx_bytes = 0;
  CUtensorMap pmap;  // values as [(nnz+1)*B rows][B cols], 64x64 boxes (per-group retrieval)
  // while offloaded: the layer's arrays in pinned host memory owned by the
  // handle (meta whole, the nnz kept tiles, col_idx); device pointers null
  bool offloaded = false;
  void* h_meta = nullptr;
  void* h_values = nullptr;
  void* h_colidx = nullptr;
  size_t h_values_cap = 0, h_colidx_cap = 0;  // allocated host bytes
  cudaEvent_t ready = nullptr;  // end of the last offload's or prefetch's copies
  // a view assembled by a block manager: `values` is the manager's tile pool
  // (not owned), the pinned entries stay cached until the view is released
  mf_bm_t view_bm = nullptr;
  std::vector<mf::BmEntry*> view_pins;
};

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};

struct mf_bsr_s {
  bool exact_alloc = false;  // size the BSR exactly (one stream sync per layer)
  unsigned prof_mask = 0;  // kernel kinds timed with events
  long long launches[MF_K_COUNT] = {0};
  std::vector<ProfRec> prof;
  std::vector<cudaEvent_t> event_pool;
  int n_layers = 0, T = 0, H_s = 0, B = 0, causal = 1, n_seqs = 0;
  int R = 0, C = 0, max_cand = 0, n_tiles = 0, n_slabs = 0;
  std::vector<int> cu;
  std::vector<int> q_begin;  // per sequence: first query row (0, or a chunk's start)
  std::vector<mf::RowBlock> rbs;
  std::vector<mf::RowTile> tiles;
  std::vector<mf::RowSlab> slabs;
  mf::RowBlock* rbs_d = nullptr;
  mf::RowTile* tiles_d = nullptr;
  // the pack kernel's item order: tile index << 8 | head (sequence-major)
  std::vector<int> pack_items;
  int* pack_items_d = nullptr;
  // the two-CTA statistics kernel's item order (same form, larger key chunks)
  std::vector<int> stats_items;
  int* stats_items_d = nullptr;
  mf::RowSlab* slabs_d = nullptr;
  int* err_d = nullptr;
  long long* host_pinned = nullptr;  // [0] nnz, [1] error word
  mf_alloc_fn alloc = nullptr;
  mf_free_fn dealloc = nullptr;
  void* ctx = nullptr;
  std::vector<LayerState> layers;
  // team retrieval's exchange ring (allocated on first use, sized for the
  // device's team count)
  void* ring = nullptr;
  uint32_t* ring_flags = nullptr;
  int ring_teams = 0;
  // team retrieval's slab lists (longest-first onto the least-loaded team)
  std::vector<int> team_slabs;
  int* team_slabs_d = nullptr;
  int team_slab_teams = 0, team_stride = 0;
};

namespace mf {

// Records the message for mf_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);

#define MF_CUDA(call, what)                     \
  do {                                          \
    cudaError_t e_ = (call);                    \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// 2-D bf16 map: `inner` elements per row, `rows` rows, `stride` bytes between
// rows; box = box_inner x box_rows; out-of-range reads give 0.
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t stride,
             uint32_t box_inner, uint32_t box_rows,
             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// Device memory through the handle's allocator (stream-ordered).
void* dev_alloc(mf_bsr_t h, size_t bytes, cudaStream_t s);
void dev_free(mf_bsr_t h, void* p, cudaStream_t s);
// Frees a layer's buffers (and a view's pins) and resets its state.
void release_layer(mf_bsr_t h, LayerState& L, cudaStream_t s);

// Byte offsets of a layer's arrays in its one scratch allocation ("meta").
struct MetaLayout {
  size_t mass, max, sum, kc, kept, rp, tile, uc, ul, ut, km, nnz, bytes;
};
MetaLayout meta_layout(const mf_bsr_s* h);
// Points the layer's array pointers into its scratch allocation (all null
// when the layer has none on the device).
void carve_meta(LayerState& L, const MetaLayout& m);

// Drops the pins a block-manager view holds on its cached entries.
void bm_unpin(LayerState& L);

}  // namespace mf
