/*
 * mapflow.h — C ABI of the GB300 (sm_103a) hot path of cross-model
 * attention-map reuse.
 *
 * The method is described on two pages:
 *   [Summary] "Accelerating Cross-Model LLM Inference via Attention Map Reuse"
 *             (paper summary page), sections "MapFlow System Design",
 *             "Practical Implementation Details" and bold headers 2-4;
 *   [Article] "北大MapFlow：注意力图跨模型复用，prefill延迟降15%–20%" (news
 *             article), the paragraphs "其一" (compressor: block statistics,
 *             then block selection, no dense map) and "其三" (retrieval: heads
 *             combined on chip, multiplied by the receiver's V, accumulated).
 *
 * Two calls carry the method:
 *   mf_compress  — the Attention State Compressor: causal-softmax row
 *                  statistics of a sender layer's Q.K^T/sqrt(d), B x B block
 *                  masses, block-level top-p per (head, block-row), and the
 *                  kept probability tiles packed as Block Sparse Row (BSR).
 *   mf_retrieve  — the fused Attention Retrieval: for receiver layer j, reads
 *                  the BSR of sender layer m(j), combines the sender heads as
 *                  A_hat_i = sum_h W_j[i,h] * A_h on chip (missing blocks are
 *                  zero, no renormalisation) and multiplies by the receiver's
 *                  V of head i's KV group, accumulating O_i; no dense A_hat is
 *                  ever written to memory.
 *
 * Conventions (all calls):
 *   - Every pointer argument is a DEVICE pointer unless its name ends in
 *     "_host".  The caller owns every buffer it passes; the handle owns the
 *     BSR buffers it allocates (through the caller's allocator when one is
 *     given, else cudaMallocAsync on the call's stream).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Work is enqueued on it; calls return before the GPU finishes, except
 *     where a call states that it synchronises.
 *   - Every call returns an mf_status (MF_OK = 0).  Nothing throws across the
 *     ABI.  On failure mf_last_error() returns a message (thread-local).
 *   - Sequences are packed: token t of sequence s lives at row
 *     cu_seqlens[s] + t of every [T, H, d] tensor.  Block grids start at each
 *     sequence's first token; tiles never straddle sequences.
 *   - Layouts are dense row-major: Q [T][H_s][d], K [T][H_ks][d],
 *     V [T][H_kv][d], O [T][H_r][d], W [H_r][H_s].
 *   - GQA grouping is contiguous: query head h uses KV head h / (H_q/H_kv).
 *   - There is no CPU fallback: without a usable sm_103a GPU every compute
 *     call fails with MF_ERR_CUDA.
 */
#ifndef MAPFLOW_H_
#define MAPFLOW_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MF_API __attribute__((visibility("default")))
#else
#define MF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MF_OK              0
#define MF_ERR_ARG         1  /* invalid argument (NULL, negative, inconsistent) */
#define MF_ERR_UNSUPPORTED 2  /* valid but outside the compiled shapes        */
#define MF_ERR_CUDA        3  /* CUDA runtime / launch error                  */
#define MF_ERR_OOM         4  /* allocator returned NULL                      */
#define MF_ERR_TIMEOUT     5  /* a device-side wait hit its limit             */
#define MF_ERR_STATE       6  /* call order (e.g. retrieve before compress)   */

/* ---- element types ------------------------------------------------------ */
#define MF_DTYPE_F32  0   /* IEEE fp32                                      */
#define MF_DTYPE_BF16 1   /* bfloat16 (stored as uint16)                    */

typedef struct mf_bsr_s* mf_bsr_t;   /* opaque; owns BSR state of n layers */
typedef struct mf_bm_s* mf_bm_t;     /* opaque; block manager (prefix-hash cache) */

/* Optional caller allocator (e.g. a framework's caching allocator).  Must
 * return a device pointer aligned to >= 256 bytes usable on `stream`, or
 * NULL on failure.  `free_fn` releases a pointer returned by `alloc_fn`. */
typedef void* (*mf_alloc_fn)(size_t bytes, void* ctx, void* stream);
typedef void  (*mf_free_fn)(void* ptr, void* ctx, void* stream);

/* Library version: major*10000 + minor*100 + patch. */
MF_API int mf_version(void);

/* Message of the last failed call on this thread ("" if none). */
MF_API const char* mf_last_error(void);

/* Shapes the library supports (for callers that want to check first). */
MF_API int mf_supported(int dtype, int d, int B);

/*
 * mf_bsr_create — create a handle that will hold the compressed attention
 * state of `n_layers` sender layers over one packed batch.
 *
 *   n_layers          number of sender layers the handle can hold (>= 1)
 *   T                 total packed tokens (= cu_seqlens_host[n_seqs])
 *   H_s               sender query heads
 *   B                 block size (64 or 128)
 *   causal            1 = causal attention (candidates bj <= bi), 0 = full
 *   cu_seqlens_host   HOST int32 [n_seqs+1], cu[0] = 0, non-decreasing,
 *                     cu[n_seqs] = T; every sequence length <= 256*B
 *   n_seqs            number of packed sequences (>= 1)
 *   alloc_fn/free_fn  optional allocator pair (both NULL or both set)
 *   alloc_ctx         passed back to the allocator
 *
 * Errors: MF_ERR_ARG on inconsistent arguments, MF_ERR_UNSUPPORTED on B or
 * sequence lengths outside the build, MF_ERR_CUDA / MF_ERR_OOM when the small
 * per-handle tables cannot be placed on the device.  Synchronous.
 */
MF_API int mf_bsr_create(mf_bsr_t* out, int n_layers, int T, int H_s, int B, int causal,
                  const int32_t* cu_seqlens_host, int n_seqs,
                  mf_alloc_fn alloc_fn, mf_free_fn free_fn, void* alloc_ctx);

/*
 * mf_bsr_create_chunked — a handle whose query rows start at q_begin[s] in
 * each sequence while its keys start at 0: a prefill chunk over a prefix
 * ([Article], the paragraph after "其三": the system runs inside a serving
 * engine with chunked prefill; reading: a chunk's block-rows are the full
 * sequence's block-rows from q_begin on, computed against every earlier
 * key).  mf_compress then
 * computes, and mf_retrieve writes, only the chunk's rows: q and o keep the
 * full packed layout [T, ...] (rows before q_begin are neither read nor
 * written), k and v cover the whole prefix.  Block-row order, R and C count
 * only the chunk's block-rows.  With a block manager this is how a request
 * whose prefix is cached compresses only its new block-rows
 * (mf_prefix_hashes with the same q_begin names them).
 *   q_begin_host  HOST int32 [n_seqs], each a multiple of 128 in [0, L_s],
 *                 or L_s (an empty chunk); NULL: mf_bsr_create.  The chunks
 *                 must hold >= 1 row
 * Causal only (MF_ERR_UNSUPPORTED otherwise).  Other arguments and errors as
 * mf_bsr_create.
 */
MF_API int mf_bsr_create_chunked(mf_bsr_t* out, int n_layers, int T, int H_s, int B, int causal,
                                 const int32_t* cu_seqlens_host, const int32_t* q_begin_host,
                                 int n_seqs, mf_alloc_fn alloc_fn, mf_free_fn free_fn,
                                 void* alloc_ctx);

/* Release every buffer of the handle (waits for the device first). */
MF_API void mf_bsr_destroy(mf_bsr_t h);

/*
 * mf_compress — Attention State Compressor for one sender layer
 * ([Summary] "Practical Implementation Details"; [Article] "其一").
 *
 *   layer    0-based slot in the handle (< n_layers); an existing state in
 *            that slot is released first
 *   q        [T][H_s][d]  sender queries of the layer (dtype)
 *   k        [T][H_ks][d] sender keys of the layer (dtype)
 *   dtype    MF_DTYPE_BF16 (tensor-core path) or MF_DTYPE_F32
 *   T,H_s,B,causal  must equal the handle's
 *   H_ks     sender KV heads, H_s % H_ks == 0
 *   d        head dimension, 64 or 128
 *   p        top-p threshold, 0 < p <= 1
 *
 * Computes, per head h and row i, m_i = max_j s_ij and
 * l_i = sum_j exp(s_ij - m_i) with s_ij = q_i.k_j/sqrt(d) over the keys the
 * row may see; the probability mass of every candidate B x B block; the
 * block-level top-p of every (head, block-row): sort by mass descending,
 * ties to the lower block column, keep the shortest prefix whose cumulative
 * mass reaches p of the row's total, evaluated exactly in fixed point
 * (q_b = rint(mass_b * 2^32), P_q = rint(p * 2^20), keep the smallest k with
 * 2^20 * sum_{t<k} q_(t) >= P_q * sum_b q_b); and the BSR of the kept tiles:
 *   row_ptr int32 [H_s*R + 1]   rows ordered head-major, then global
 *                               block-row (R = sum_s ceil(L_s/B))
 *   col_idx int32 [nnz]         block column relative to the sequence's first
 *                               block, ascending within a row
 *   values  bf16  [nnz][B][B]   P_ij = exp(s_ij - m_i)/l_i, zero above the
 *                               diagonal and outside the sequence
 * By default the call is fully asynchronous: the values buffer is sized for
 * the upper bound (every candidate kept, plus one all-zero tile used by the
 * retrieval) and nnz stays on the device until mf_bsr_info/_copy asks for it;
 * a device-side timeout is then reported by mf_device_status.  After
 * mf_bsr_set_exact(h, 1) the call instead synchronises `stream` once to size
 * the buffer exactly and reports MF_ERR_TIMEOUT itself.
 * Errors: MF_ERR_ARG, MF_ERR_UNSUPPORTED, MF_ERR_OOM, MF_ERR_CUDA,
 * MF_ERR_TIMEOUT (exact mode: a device wait gave up; the layer is left empty).
 */
MF_API int mf_compress(mf_bsr_t h, int layer, const void* q, const void* k, int dtype,
                int T, int H_s, int H_ks, int d, int B, float p, int causal,
                void* stream);

/*
 * mf_retrieve — fused Attention Retrieval for n receiver layers
 * ([Summary] "Practical Implementation Details" and bold header 4;
 * [Article] "其三"; head mapping per [Summary] "MapFlow System Design" 3).
 *
 *   W               fp32 [n][H_r][H_s]  head-mapping weights of each layer
 *   v               [n][T][H_kv][d]     receiver values (dtype)
 *   o               [n][T][H_r][d]      output (dtype), fully overwritten
 *   dtype           MF_DTYPE_BF16 or MF_DTYPE_F32 (must match the layer's
 *                   compress dtype family: bf16 retrieval needs d in {64,128})
 *   H_r, H_kv       receiver query / KV heads, H_r % H_kv == 0,
 *                   H_r/H_kv <= 8 (d = 128) or <= 16 (d = 64)
 *   d               head dimension (= the compressed layers' d)
 *   layer_map_host  HOST int32 [n]: handle slot (sender layer) used by call
 *                   layer x; each slot must hold a compressed state
 *   n               number of receiver layers in this call (>= 1)
 *
 * O_i[t] = sum over the kept blocks (h, bi, bj) of block-row bi of t:
 *          W[i,h] * P_h[t, bj cols] @ V_g(i)[bj rows], fp32 accumulation.
 * Rows of blocks with no kept tile get O = 0.  Asynchronous.
 * With 8 KV heads and H_r <= 32 (bf16) the kernel is a cooperative launch
 * whose CTAs pass partial results through a small exchange ring owned by the
 * handle (about 40 MB, allocated with the handle's allocator on the first such
 * call, on `stream`): calls of one handle must therefore not run concurrently
 * on different streams.
 * Errors: MF_ERR_ARG, MF_ERR_UNSUPPORTED, MF_ERR_STATE, MF_ERR_CUDA, MF_ERR_OOM.
 */
MF_API int mf_retrieve(mf_bsr_t h, const float* W, const void* v, void* o, int dtype,
                int H_r, int H_kv, int d, const int32_t* layer_map_host, int n,
                void* stream);

/*
 * mf_bsr_set_exact — 1: size each layer's BSR exactly (mf_compress then
 * synchronises its stream once); 0 (default): allocate the upper bound and
 * never synchronise.
 */
MF_API int mf_bsr_set_exact(mf_bsr_t h, int exact);

/*
 * mf_bsr_info — sizes of a compressed layer: nnz (kept tiles), rows
 * (H_s*R), candidates (H_s * sum of candidate blocks per block-row).  Asking
 * for nnz of an asynchronously compressed layer waits for that compress.
 */
MF_API int mf_bsr_info(mf_bsr_t h, int layer, int64_t* nnz, int64_t* n_rows, int64_t* n_cand);

/*
 * mf_bsr_export — device pointers (owned by the handle, valid until the
 * layer is released or recompressed) to a compressed layer:
 *   row_ptr  int32 [H_s*R+1], col_idx int32 [nnz], values bf16 [nnz][B][B],
 *   mass     fp32 [H_s][C] candidate masses (per head: block-rows in global
 *            order, each with its candidates bj = 0.. in order),
 *   row_max  fp32 [H_s][T] (m_i), row_sum fp32 [H_s][T] (l_i).
 * Any output pointer may be NULL.
 */
MF_API int mf_bsr_export(mf_bsr_t h, int layer, const int32_t** row_ptr, const int32_t** col_idx,
                  const uint16_t** values, const float** mass, const float** row_max,
                  const float** row_sum);

/*
 * mf_bsr_copy — copy a compressed layer into caller-owned DEVICE buffers
 * (sizes as for mf_bsr_export; any destination may be NULL).  Asynchronous on
 * `stream`.
 */
MF_API int mf_bsr_copy(mf_bsr_t h, int layer, int32_t* row_ptr, int32_t* col_idx, uint16_t* values,
                float* mass, float* row_max, float* row_sum, void* stream);

/* mf_bsr_release_layer — free one layer's state (per-layer streaming). */
MF_API int mf_bsr_release_layer(mf_bsr_t h, int layer);

/*
 * mf_bsr_offload — move a compressed layer to pinned host memory owned by the
 * handle and give its device buffers back to the allocator, asynchronously on
 * `stream` (learns nnz first: one sync of the layer's stream if not known).
 * Only the kept tiles travel.  The layer stays valid; mf_retrieve,
 * mf_bsr_export and mf_bsr_copy reject it (MF_ERR_STATE) until
 * mf_bsr_prefetch brings it back.  Work that reads the layer on other streams
 * must be ordered before `stream` by the caller.
 *
 * mf_bsr_prefetch — bring an offloaded layer back to the device,
 * asynchronously on `stream` (typically a copy stream, so that the transfer
 * overlaps other work); mf_retrieve and mf_bsr_copy on any stream wait for its
 * copies by themselves (an event recorded here).
 *
 * Together they let a caller keep on the device only the sender layers the
 * next receiver layers read, and fetch the next ones while the receiver
 * recomputes its first layers ([Article] "其二": the cached state is fetched
 * while the receiver's first layers are recomputed).  No-ops on a layer that
 * is already where asked.  Errors: MF_ERR_ARG, MF_ERR_STATE, MF_ERR_OOM,
 * MF_ERR_CUDA.
 */
MF_API int mf_bsr_offload(mf_bsr_t h, int layer, void* stream);
MF_API int mf_bsr_prefetch(mf_bsr_t h, int layer, void* stream);

/* ---------------------------------------------------------------------------
 * Block manager: compressed block-rows cached under prefix hashes
 *
 * [Summary] "Practical Implementation Details" (a block manager indexes the
 * cache by prefix hash) and [Article] "其二" (states are indexed by hashes
 * that carry the preceding context; a request finds the cached blocks of its
 * shared prefix; one sender state serves several receivers).  Reading: under
 * a causal mask block-row bi of a sequence (selection and kept tiles of every
 * head) depends only on the tokens of blocks 0..bi, so it is keyed by the
 * chained hash of those blocks and shared by every sequence that has the same
 * prefix.  An entry is one block-row of one layer (the caller's layer key):
 * its kept tiles of every head, stored once in a device tile pool, and their
 * positions.  A view is an ordinary layer of a BSR handle whose tile table
 * points into the pool; mf_retrieve reads it like a compressed layer, and
 * mf_calibrate_head_map accepts it; export, copy and offload refuse it
 * (MF_ERR_STATE).  Non-causal handles are refused (MF_ERR_UNSUPPORTED): their
 * block-rows depend on the whole sequence.  A manager is not thread-safe.
 * ------------------------------------------------------------------------- */

/*
 * mf_prefix_hashes — chained 64-bit hashes of the B-token blocks of each
 * packed sequence: each block's hash mixes the previous block's hash (or
 * `seed` for block 0), the block's length and its tokens (splitmix64
 * finaliser), so a ragged last block never matches a full one.
 *   tokens      HOST int32 [cu_seqlens[n_seqs]]
 *   cu_seqlens  HOST int32 [n_seqs + 1]
 *   q_begin     HOST int32 [n_seqs] or NULL: hashes only of the block-rows
 *               from q_begin[s] on (a multiple of B, or L_s), as a chunked handle
 *               (mf_bsr_create_chunked) orders them; the chain still runs
 *               over the tokens before
 *   hashes_out  HOST uint64 [capacity], filled in the block-row order of a
 *               handle made with the same cu_seqlens, q_begin and B; NULL:
 *               only *n_out
 *   n_out       the number of block-rows R
 * Errors: MF_ERR_ARG.
 */
MF_API int mf_prefix_hashes(const int32_t* tokens, const int32_t* cu_seqlens, const int32_t* q_begin,
                            int n_seqs, int B, uint64_t seed, uint64_t* hashes_out, int64_t capacity,
                            int64_t* n_out);

/*
 * mf_bm_create / mf_bm_destroy — a manager for block-rows of H_s heads and
 * block size B with a device pool of `tile_capacity` bf16 B x B tiles (plus
 * one all-zero tile), allocated through alloc_fn (cudaMallocAsync if NULL)
 * on `stream`.  Destroy fails with MF_ERR_STATE while a view pins entries.
 * Errors: MF_ERR_ARG, MF_ERR_UNSUPPORTED (B), MF_ERR_OOM, MF_ERR_CUDA.
 */
MF_API int mf_bm_create(mf_bm_t* out, int H_s, int B, int64_t tile_capacity, mf_alloc_fn alloc_fn,
                        mf_free_fn free_fn, void* alloc_ctx, void* stream);
MF_API int mf_bm_destroy(mf_bm_t bm);

/*
 * mf_bm_insert — cache the block-rows of compressed `layer` of handle `h`
 * under (key_layer, hashes[rb]), hashes HOST uint64 [R] as mf_prefix_hashes
 * gives them.  Block-rows already cached are only marked used; new ones get
 * pool slots (least recently used unpinned entries are evicted to make room)
 * and their kept tiles are copied into the pool by a gather kernel on
 * `stream`.  Reads the layer's tile table to the host (synchronises
 * `stream`).  counts (optional, HOST int64 [3]): block-rows inserted, found
 * cached, entries evicted.  A hash that names a cached block-row of another
 * position or length is MF_ERR_ARG; more new tiles than the unpinned pool
 * holds is MF_ERR_OOM.  A failed insert inserts and evicts nothing (the
 * entries it would evict leave the cache only once the copy is queued);
 * cached block-rows it found are still marked used.
 */
MF_API int mf_bm_insert(mf_bm_t bm, int key_layer, mf_bsr_t h, int layer, const uint64_t* hashes,
                        int64_t* counts, void* stream);

/*
 * mf_bm_match — the length of the longest run hashes[0..k) cached under
 * key_layer (the shared prefix, in block-rows), through *n_hit.
 */
MF_API int mf_bm_match(mf_bm_t bm, int key_layer, const uint64_t* hashes, int n, int* n_hit);

/*
 * mf_bm_assemble — make `layer` of handle `h` a view of the cached block-rows
 * hashes[0..R) (HOST uint64 [R] in h's block-row order): the tile table and
 * the retrieval's union tables are built on `stream` (one small kernel), the
 * tiles stay in the pool.  The entries stay pinned (not evicted) until the
 * layer is released, recompressed or re-assembled.  A hash that is not cached,
 * or that names a block-row of another position or length, is MF_ERR_ARG.
 */
MF_API int mf_bm_assemble(mf_bm_t bm, int key_layer, const uint64_t* hashes, mf_bsr_t h, int layer,
                          void* stream);

/*
 * mf_bm_stats — HOST int64 [7]: entries, pool tiles in use, pool capacity,
 * block-rows found by mf_bm_match, mf_bm_match calls that stopped short,
 * entries evicted, entries pinned by views.
 */
MF_API int mf_bm_stats(mf_bm_t bm, int64_t* out);

/*
 * mf_calibrate_head_map — fit the head map W offline from two compressed
 * layers over the same packed sequences ([Summary] "MapFlow System Design"
 * item 3: the receiver's map of a reused layer is a linear transformation of
 * the mapped sender layer's head maps, learned offline).  Reading: least
 * squares over every map entry, each map as its BSR stores it (dropped blocks
 * zero):  W = argmin sum_i |A_i - sum_h W[i,h] P_h|^2 + ridge |W|^2, where
 * P_h are the `sender` layer's heads and A_i the `receiver` layer's (a handle
 * made for the receiver's heads, typically compressed at p = 1).
 *   W_out  HOST fp32 [H_r][H_s]
 *   ridge  >= 0, added to the sender heads' Gram matrix
 * The Gram matrices are accumulated on the GPU from the bf16 tiles (fp32
 * partials, summed in fp64 on the host) and the H_s x H_s system is solved
 * on the host (Cholesky, fp64).  Synchronises `stream`.  Both handles must
 * share sequences, block size and causality; H_s + H_r <= 96.
 * Errors: MF_ERR_ARG (incl. a singular Gram matrix: pass ridge > 0),
 * MF_ERR_UNSUPPORTED, MF_ERR_STATE, MF_ERR_OOM, MF_ERR_CUDA.
 */
MF_API int mf_calibrate_head_map(mf_bsr_t sender, int sender_layer, mf_bsr_t receiver,
                                 int receiver_layer, float ridge, float* W_out, void* stream);

/*
 * mf_device_status — synchronise `stream` and read the handle's device
 * error word (set by bounded device-side waits).  Returns MF_OK,
 * MF_ERR_TIMEOUT (and clears the word), or MF_ERR_CUDA.
 */
MF_API int mf_device_status(mf_bsr_t h, void* stream);

/* ---- per-kernel timing (CUDA events on the launching stream) ------------ */
#define MF_K_STATS    0   /* compressor statistics (Q.K^T, row stats, masses) */
#define MF_K_SELECT   1   /* block-level top-p                                */
#define MF_K_SCAN     2   /* row_ptr scan (done by the selection kernel's last
                             CTA: no launches of its own)                     */
#define MF_K_PACK     3   /* BSR pack (kept-tile recompute + store)           */
#define MF_K_UNION    4   /* retrieval plan (union of kept columns); on the
                             bf16 path the pack kernel writes it: no launches */
#define MF_K_RETRIEVE 5   /* fused retrieval                                  */
#define MF_K_COUNT    6

/*
 * mf_profile — enable (1) or disable (0) event timing of every kernel the
 * handle launches; enabling clears earlier records.  Launch counts are kept
 * whether timing is on or not (reset by enabling).
 */
MF_API int mf_profile(mf_bsr_t h, int enable);

/*
 * mf_profile_kinds — like mf_profile, but times only the kernel kinds whose
 * bit (1 << MF_K_*) is set in `mask` (0 disables timing).  Fewer event pairs
 * in the stream: launch counts stay complete for every kind.
 */
MF_API int mf_profile_kinds(mf_bsr_t h, int mask);

/*
 * mf_profile_read — launches and summed device time (ms) of one kernel kind
 * since profiling was enabled.  Waits for the recorded events.
 */
MF_API int mf_profile_read(mf_bsr_t h, int kernel, int64_t* launches, double* total_ms);

/*
 * mf_select_noalloc — block-level top-p selection and BSR structure from a
 * caller's block masses, allocating NO device memory.  The pages have no
 * counterpart of this call: it exists for callers that cannot allocate when
 * they select — engines that reserve almost all device memory up front and
 * forbid further cudaMalloc, and latency-critical loops that cannot pay
 * cudaFree's implicit device synchronisation.
 *
 *   mass             fp32 [H_s][C] candidate masses in mf_bsr_export's layout
 *                    (input; e.g. exported from mf_compress)
 *   cu_seqlens_host  HOST int32 [n_seqs+1] (as for mf_bsr_create)
 *   H_s, B, causal, p  as for mf_compress
 *   row_ptr          int32 [H_s*R + 1] output
 *   col_idx          int32 output with room for col_capacity entries;
 *                    col_capacity must be >= H_s*C (every candidate kept)
 *   nnz              DEVICE int64 output: number of kept tiles
 *
 * The selection rule and the output are exactly mf_compress's row_ptr and
 * col_idx for the same masses.  Intermediates live in one file-scope static
 * device array of 16 MiB per device (held by every GPU that loads the
 * library until the process exits); a call needing more is rejected with
 * MF_ERR_UNSUPPORTED.  The first call on each device looks up that array's
 * device address (cudaGetSymbolAddress) — make that first call before any
 * stream capture.  All calls on a device share the array: calls that overlap
 * on the GPU (different streams without ordering) race; calls ordered on one
 * stream are safe.  Nothing needs clearing between calls.  The host table of
 * block-rows is copied to the device from a pageable host buffer that the
 * call owns; such a copy has read the host buffer before cudaMemcpyAsync
 * returns, so the call frees it on return; the kernels run asynchronously on
 * `stream`.
 */
MF_API int mf_select_noalloc(const float* mass, const int32_t* cu_seqlens_host, int n_seqs,
                             int H_s, int B, int causal, float p, int32_t* row_ptr,
                             int32_t* col_idx, int64_t col_capacity, int64_t* nnz, void* stream);

/*
 * mf_selftest_wait — failure-detection self-test (no counterpart on the
 * pages).  Launches one thread that waits on a device barrier nothing will
 * complete, bounded by `limit_ms` milliseconds (1..10000); the wait gives up,
 * records a timeout in the handle's device error word and returns, leaving
 * the context usable.  A following mf_device_status returns MF_ERR_TIMEOUT.
 */
MF_API int mf_selftest_wait(mf_bsr_t h, int limit_ms, void* stream);

#ifdef __cplusplus
}
#endif

#endif  /* MAPFLOW_H_ */
