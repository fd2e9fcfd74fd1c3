// mf_internal.cuh — shared host/device structures and kernel launchers of
// libmapflow (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

namespace mf {

// One global block-row (a B-row block of one packed sequence).
struct RowBlock {
  int seq_start;  // first token of the sequence in the packed batch
  int L;          // sequence length
  int bi;         // block-row index within the sequence
  int cand_off;   // offset of this block-row's candidates in a head's mass row
};

// One 128-query-row tile of a sequence (the compressor's CTA unit).
struct RowTile {
  int seq_start;
  int L;
  int tl;   // tile index within the sequence (rows 128*tl .. 128*tl+127)
  int rb0;  // global block-row of the tile's first block-row
};

// One 64-row slab of a block-row (the retrieval's CTA unit).
struct RowSlab {
  int rb;    // global block-row
  int half;  // 0 for B = 64; 0/1 for B = 128
};

struct CompressParams {
  const RowBlock* rbs;
  const RowTile* tiles;
  int n_tiles;
  const int* items;  // pack order: [n_tiles * H_s] tile index << 8 | head, or null (tile-major)
  const int* stats_items;  // the two-CTA statistics kernel's order, same form, or null
  int T, H_s, H_ks, d, B, causal;
  int R;            // block-rows
  int C;            // candidates per head
  int max_cand;     // most candidates of one block-row
  float scale_log2; // log2(e) / sqrt(d)
  float p;
  // outputs / intermediates
  float* mass;      // [H_s][C]
  float* row_max;   // [H_s][T]  natural-log units
  float* row_sum;   // [H_s][T]
  int* kcount;      // [H_s*R]
  int* keptcols;    // [H_s][C]  per row: kept block columns, ascending
  int* row_ptr;     // [H_s*R + 1]
  int* col_idx;     // [nnz]
  int* tile_of;     // [C][H_s]  tile index of (block-row cand, head) or -1
  int* union_cnt;   // [R]
  int* union_list;  // [C]
  int* utile;       // [C][H_s]  tile_of in union order: row cand_off + j is union column j
  long long* nnz_out;  // device scalar
  int* pack_ctr;    // device scalar: the pack kernel's next item (reset by the selection kernel)
  int* sel_done;    // device scalar: selection CTAs finished (reset by the statistics kernel)
  uint16_t* zero_tile;  // the all-zero tile after the kept ones (bf16 pack writes it), or null
  uint32_t* kmask;  // [H_s*R][8] kept columns of each BSR row as bit masks (bf16 path), or null
  int union_in_pack;  // 1: the bf16 pack kernel writes union_cnt / union_list / utile
  int* err;
};

struct RetrieveParams {
  const RowBlock* rbs;
  const RowSlab* slabs;
  int n_slabs;
  int T, H_s, H_r, H_kv, d, B;
  int R, C;
  const int* tile_of;     // [C][H_s]
  const int* union_cnt;   // [R]
  const int* union_list;  // [C]
  const int* utile;       // [C][H_s] tile_of in union order
  const int* team_slabs;  // team retrieval: [n_teams][team_stride] slab indices, -1 padded
  int team_stride;
  const float* W;         // [H_r][H_s] of this receiver layer
  int zero_tile;          // index of an all-zero tile (= nnz)
  const uint16_t* values; // [nnz+1][B][B] bf16 tiles
  int* err;
};

// SM count of the current device, queried once per device.
inline cudaError_t sm_count(int* out) {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  *out = v;
  return cudaSuccess;
}

// -------------------------------------------------------------- launchers --
// All return cudaError_t of the launch (cudaSuccess when enqueued).
// Head-map calibration: Gram matrix of the stacked head maps of two BSR
// layers over one block grid (rows 0..H_s-1 sender heads, then receiver heads).
constexpr int kCalibRows = 96;
struct CalibParams {
  const int* s_tile_of;      // sender [C][H_s] kept tile index or -1
  const uint16_t* s_values;  // sender tiles [.][B][B] bf16
  const int* r_tile_of;      // receiver [C][H_r]
  const uint16_t* r_values;
  int C, H_s, H_r, B;
  float* partial;            // [grid][kCalibRows][kCalibRows] per-CTA sums
  int* err;                  // device error word (bounded waits)
};
// CTAs for C candidate blocks (two per SM at most, none idle).
int calib_grid(int C);
// The Gram kernel, then the fixed-order fp64 sum of its partials into
// G [n][n], n = H_s + H_r.
cudaError_t launch_calib_gram(const CalibParams& p, int grid, double* G, cudaStream_t s);

// Statistics with two CTAs per SM (64-key S tiles) for rows of at most 128
// candidate blocks; tk64 boxes are 64 keys high.
bool stats2_supported(int max_cand);
cudaError_t launch_stats2_bf16(const CompressParams& p, const CUtensorMap& tq,
                               const CUtensorMap& tk64, cudaStream_t s);
cudaError_t launch_stats_bf16(const CompressParams& p, const CUtensorMap& tq,
                              const CUtensorMap& tk, cudaStream_t s);
cudaError_t launch_stats_f32(const CompressParams& p, const float* q, const float* k,
                             cudaStream_t s);
// Selection and, in its last CTA, the row_ptr scan.
cudaError_t launch_select(const CompressParams& p, cudaStream_t s);
cudaError_t launch_pack_bf16(const CompressParams& p, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tvals,
                             cudaStream_t s);
cudaError_t launch_pack_f32(const CompressParams& p, const float* q, const float* k,
                            uint16_t* values, cudaStream_t s);
cudaError_t launch_union(const CompressParams& p, cudaStream_t s);
cudaError_t launch_retrieve_bf16(const RetrieveParams& p, const CUtensorMap& tp,
                                 const CUtensorMap& tv, void* o, cudaStream_t s);
// Team retrieval: persistent cooperative kernel, teams of 8 CTAs exchanging
// the combined maps through a ring in global memory (`ring` of
// retrieve_team_ring_bytes, `flags` of retrieve_team_flag_bytes, zeroed
// once: every launch leaves them at zero; `ta` maps the ring as
// retrieve_team_ring_rows x 64 bf16
// with boxes of 64 x retrieve_team_ring_box_rows).
bool retrieve_team_supported(int H_s, int H_r, int H_kv, int d, int B);
int retrieve_team_count(int n_slabs, int sms);
size_t retrieve_team_ring_bytes(int n_teams);
size_t retrieve_team_flag_bytes(int n_teams);
int retrieve_team_ring_box_rows(int H_r);
int retrieve_team_ring_rows(int n_teams);
cudaError_t launch_retrieve_team(const RetrieveParams& p, const CUtensorMap& ta,
                                 const CUtensorMap& tv, void* o, void* ring, uint32_t* flags,
                                 int n_teams, cudaStream_t s);
cudaError_t launch_retrieve_f32(const RetrieveParams& p, const uint16_t* values, const float* v,
                                float* o, cudaStream_t s);

// No-allocation selection (scratch in a static device array; mf_noalloc.cu).
size_t noalloc_scratch_bytes();
size_t noalloc_needed_bytes(long long R, long long H_s, long long C);
cudaError_t launch_select_noalloc(const RowBlock* rbs_host, int R, int C, int H_s, int B,
                                  int causal, float p, const float* mass, int* row_ptr,
                                  int* col_idx, long long* nnz, cudaStream_t s);

cudaError_t launch_selftest_wait(int* err, unsigned long long limit_ns, cudaStream_t s);

}  // namespace mf
