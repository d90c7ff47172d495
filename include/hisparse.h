/*
 * hisparse.h -- C ABI of libhisparse: the HiSparse decode-time KV-row swap-in
 * and the indexed KV-row movers, as hand-written CUDA kernels for GB300
 * (sm_103a).
 *
 * Conventions shared by every entry point
 *  - All calls are asynchronous and stream-ordered on `stream` (a CUDA runtime
 *    stream handle; NULL is the legacy default stream).  The library owns no
 *    memory, allocates nothing, and keeps no state between calls beyond a
 *    once-per-process kernel attribute set-up.
 *  - "device" pointers must be readable/writable by the GPU: device memory
 *    (or managed memory).  Pool pointers may also be pinned host memory
 *    (cudaHostAlloc / cudaHostRegister), read over the host link.
 *  - The synchronous return value covers argument errors and launch errors
 *    (hs_err).  Problems found in the data while the kernel runs are reported
 *    through optional per-row or per-call status words (HS_ST_* bits).
 *  - On any non-HS_OK return, hs_last_error() holds a message for the calling
 *    thread.  Empty work (batch == 0, top_k == 0, n == 0) returns HS_OK and
 *    launches nothing.
 *  - No floating point is involved: rows are opaque bytes.
 */
#ifndef HISPARSE_H
#define HISPARSE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA runtime stream (cudaStream_t has this exact type). */
typedef struct CUstream_st* hs_stream_t;

typedef enum hs_err {
  HS_OK = 0,
  HS_ERR_ARG = 1,         /* a pointer, size, stride or memory type is unusable */
  HS_ERR_UNSUPPORTED = 2, /* valid, but outside what this build supports */
  HS_ERR_CUDA = 3         /* a CUDA runtime call or the launch failed */
} hs_err;

/* Status bits written by the kernels (0 = clean). */
#define HS_ST_DUP_ID 1        /* a valid id repeated within a row: later copies got -1 */
#define HS_ST_BAD_POOL_ROW 2  /* a miss's pool row was outside [0, pool_num_rows): -1, not a miss */
#define HS_ST_BAD_LRU_SLOT 4  /* an LRU entry was outside [0, hot_size) or repeated a slot */
#define HS_ST_BAD_HOT_ROW 8   /* a miss's hot row was outside [0, hot_num_rows): -1, no copy */
#define HS_ST_TIMEOUT 16      /* a bounded wait inside a kernel gave up (see hs_swap_in) */
#define HS_ST_BAD_STATE 32    /* req_state[b] >= num_states: row emitted -1 */
#define HS_ST_BAD_INDEX 64    /* a mover index was out of range: that row was skipped */

/* hs_swap_in_args.flags */
#define HS_SEQ_LENS_I64 1  /* seq_lens is int64 (else int32) */
#define HS_REQ_STATE_I64 2 /* req_state is int64 (else int32) */
/* The call may start while the kernel before it in the stream is still
 * running (programmatic dependent launch): until that kernel has completed it
 * reads only seq_lens, req_state, num_real, slot_tokens, slot_rows and lru,
 * and writes nothing.  Set it only when no kernel still in flight in the
 * stream writes those six buffers; topk_ids and every other buffer may be
 * written by the preceding kernel.  One more condition when that kernel lets
 * its dependents start before its last writes (griddepcontrol.launch_dependents
 * early, as hs_swap_in and hs_gather_misses do): it must not write pool_k,
 * pool_v or the resident block table, which are read through the read-only
 * data path (valid only for data unchanged while the reading grid exists). */
#define HS_OVERLAP_PREV 4

/*
 * hs_swap_in -- resolve each batch row's top-k token ids against the row's
 * device hot buffer, assign LRU slots to misses, copy the missing KV rows from
 * the pool into the hot buffer, and emit each entry's hot-buffer row.
 *
 * Defined by: SGLang jit_kernel/csrc/hisparse.cuh, load_cache_to_device_buffer
 * and load_cache_to_device_buffer_kernel (one row per batch entry: padding
 * exit, short-sequence fast path, newest-token slot, LRU walk with hits kept
 * and evictables compacted, misses in top-k order taking least recently used
 * slots, LRU writeback, per-miss row copy); vLLM
 * csrc/libtorch_stable/hisparse_kernels.cu, hisparse_resolve_residency_kernel
 * (invalid ids resolve to -1, padding rows publish -1, corruption tripwires,
 * hit/miss statistics).
 *
 * Per batch row b (rows are independent):
 *  - padding: b >= *num_real, or req_state[b] < 0 -> out[b][*] = -1,
 *    miss_count 0, status 0, state untouched.  req_state[b] >= num_states ->
 *    the same with status HS_ST_BAD_STATE.
 *  - r = req_state[b], L = seq_lens[b].  If L <= hot_size (fast path):
 *    out[b][i] = slot_rows[r][t] for i < min(L, top_k) and 0 <= t < L, else -1
 *    (t = topk_ids[b][i]); state untouched.
 *  - otherwise an id t is valid iff 0 <= t < L.  Invalid ids and repeats of an
 *    earlier valid id (HS_ST_DUP_ID) emit -1.  t == L-1 (the newest token)
 *    emits slot_rows[r][hot_size]; slot hot_size is never read or written
 *    otherwise.  Every other valid id is a hit if some LRU slot s holds it
 *    (slot_tokens[r][s] == t; out = slot_rows[r][s]), else a miss candidate.
 *    A candidate with pool_rows[r][t] outside [0, pool_num_rows) (or
 *    t >= pool_rows_cols) emits -1 (HS_ST_BAD_POOL_ROW).  The m-th remaining
 *    miss in top-k order takes the m-th evictable slot in LRU order, emits
 *    slot_rows[r][s], records slot_tokens[r][s] = t and copies row_bytes bytes
 *    of pool_k row pool_rows[r][t] to hot_k row slot_rows[r][s] (and pool_v to
 *    hot_v).  The LRU row becomes [untouched evictables][misses][hits], each
 *    group in its previous order (misses in top-k order).
 *  - tripwires: an LRU entry outside [0, hot_size), or a slot already listed
 *    earlier in the same LRU row, is never a hit and stays evictable
 *    (HS_ST_BAD_LRU_SLOT); a miss given such an entry, or a slot whose hot row
 *    is outside [0, hot_num_rows) (HS_ST_BAD_HOT_ROW), emits -1 and writes no
 *    token and no bytes but still counts as a miss.
 *  - time-out: the kernel's waits for its own staging copies are bounded.  If
 *    one runs out in any CTA of a row, the whole row is left alone: status[b]
 *    is exactly HS_ST_TIMEOUT, miss_count[b] is 0, and out_rows, the plan,
 *    the LRU row, the slot tokens, the stats and the hot buffer are not
 *    written.  It means the GPU did not complete a copy within about a
 *    second; treat the context as suspect.
 *
 * Layouts (all row-major with the given element strides; device memory unless
 * noted):
 *  topk_ids    int32 [batch, >=top_k]           stride topk_stride
 *  seq_lens    int32/int64 [batch]              (flags & HS_SEQ_LENS_I64)
 *  req_state   int32/int64 [batch]              (flags & HS_REQ_STATE_I64)
 *  num_real    int32 [1] or NULL (all rows real)
 *  slot_tokens int32 [num_states, >=hot_size+1] in/out, -1 = empty slot
 *  slot_rows   int32 [num_states, >=hot_size+1] hot-buffer row of each slot
 *  lru         int16 [num_states, >=hot_size]   in/out, least recent first
 *  pool_rows   int64 [num_states, pool_rows_cols] pool row of each token
 *  pool_k/_v   bytes [pool_num_rows, row_bytes] device or pinned host; pool_v NULL = K only
 *  hot_k/_v    bytes [hot_num_rows, row_bytes]  device; hot_v NULL iff pool_v NULL
 *  out_rows    int32 [batch, >=top_k]           stride out_stride
 *  miss_count  int32 [batch] or NULL; stats uint64 [2] (+= hits, misses) or NULL;
 *  status      int32 [batch] or NULL (per-row HS_ST_* bits, overwritten)
 *  miss_src    int64 [batch, >=top_k] or NULL  stride plan_stride  } the miss plan,
 *  miss_dst    int32 [batch, >=top_k] or NULL  stride plan_stride  } for replay by
 *  miss_mask   int32 [batch, >=top_k] or NULL  stride mask_stride  } hs_gather_misses
 *  max_seq_len 0 (unknown) or a bound on the sequence lengths: a row with
 *              seq_lens[b] > max_seq_len emits -1 with HS_ST_BAD_STATE and
 *              changes no state.  A bound lets the library use a more compact
 *              request hash (faster); results are the same.
 *  src_bt      int32 [num_states, >=src_bt_blocks] or NULL   source block table
 *  res_bt      int32 [num_states, >=res_bt_blocks] or NULL   resident block table
 *
 * Block tables (optional; vLLM csrc/libtorch_stable/hisparse_kernels.cu,
 * hisparse_resolve_residency_kernel, Phase 1), both indexed by the row's
 * state row r, for a valid id t that is the first copy of its value:
 *  - resident: when e = res_bt[r][t / res_block_size] (block index below
 *    res_bt_blocks) is >= 0 and != res_null_block, the entry emits
 *    e * res_block_size + t % res_block_size and is not looked up, not a hit
 *    and not a miss (also on the short-sequence path).  This precedes the
 *    newest-token rule;
 *  - source (replaces pool_rows, which may then be NULL): the pool row of t is
 *    g = src_bt[r][t / src_block_size] * src_block_size + t % src_block_size;
 *    when the block index is not below src_bt_blocks, the entry is <= 0 or
 *    g >= pool_num_rows, the entry behaves as an invalid id (-1, no status
 *    bit).  The newest token needs no source row.
 *
 * Miss plan (optional; vLLM csrc/libtorch_stable/hisparse_kernels.cu,
 * hisparse_gather_plan_kernel and hisparse_gather_compact_kernel): for the
 * row's m-th miss (m < miss_count[b], top-k order) miss_src[b][m] is the pool
 * row it was copied from and miss_dst[b][m] the hot row it was given (-1 when
 * it was given none); entries past the miss count are not written.
 * miss_mask[b][i] is 1 when top-k entry i was one of the row's misses, else 0
 * (all 0 for padding rows and short sequences).  miss_src and miss_dst go
 * together and need miss_count.
 *
 * Limits: 1 <= top_k <= hot_size <= 32767 (slots are int16).  Up to
 * hot_size 8192 each row runs on a cluster of up to 8 CTAs; every CTA holds the
 * row's ids, LRU order, slot tokens, slot rows and a hash of 2*top_k..8*top_k
 * slots (the most that fits), plus its share of the per-position state.  Above
 * 8192 each row runs on one CTA (the hs_swap_in_layers kernel), which keeps
 * the slot tokens and rows in global memory when they do not fit.  Either way
 * the row's state must fit one CTA's shared memory (hs_swap_in_smem_bytes),
 * else HS_ERR_UNSUPPORTED.  hot_num_rows <= INT32_MAX.
 * Preconditions (not checked): distinct req_state values within one call;
 * slot_rows values distinct across the slots the call can touch; pool and hot
 * buffers do not overlap; no other work writes these buffers concurrently.
 * Ownership: the caller owns every buffer; nothing is retained after return.
 */
typedef struct hs_swap_in_args {
  int32_t batch;    /* B */
  int32_t top_k;    /* K */
  int32_t hot_size; /* H */
  int32_t flags;    /* HS_SEQ_LENS_I64 | HS_REQ_STATE_I64 | HS_OVERLAP_PREV */
  const int32_t* num_real;
  const int32_t* topk_ids; int64_t topk_stride;
  const void* seq_lens;
  const void* req_state;
  int64_t num_states;
  int32_t* slot_tokens; int64_t slot_tokens_stride;
  const int32_t* slot_rows; int64_t slot_rows_stride;
  int16_t* lru; int64_t lru_stride;
  const int64_t* pool_rows; int64_t pool_rows_stride; int64_t pool_rows_cols;
  const void* pool_k; const void* pool_v; int64_t pool_num_rows;
  void* hot_k; void* hot_v; int64_t hot_num_rows;
  int64_t row_bytes;
  int32_t* out_rows; int64_t out_stride;
  int32_t* miss_count;
  unsigned long long* stats;
  int32_t* status;
  int64_t* miss_src; int32_t* miss_dst; int64_t plan_stride;
  int32_t* miss_mask; int64_t mask_stride;
  const int32_t* src_bt; int64_t src_bt_stride; int32_t src_bt_blocks; int32_t src_block_size;
  const int32_t* res_bt; int64_t res_bt_stride; int32_t res_bt_blocks; int32_t res_block_size;
  int32_t res_null_block;
  int64_t max_seq_len; /* 0, or a bound on every seq_lens[b] (lets the library pack its hash) */
} hs_swap_in_args;

hs_err hs_swap_in(const hs_swap_in_args* args, hs_stream_t stream);

/*
 * hs_swap_in_timeout_selftest -- hs_swap_in with one CTA of every full-path
 * row made to give up one of its bounded waits at once (zero polls), so that
 * the time-out path runs without any GPU fault or hang: the copy it gave up
 * on is still waited out before the CTA exits.  rank >= 0 picks that CTA of
 * each row's cluster (mod the cluster size), rank < 0 the last one; which = 0
 * gives up the wait for the row's staged state, 1 the wait for its top-k row.
 * Every full-path row must then report exactly HS_ST_TIMEOUT with miss_count
 * 0 and no other write (see hs_swap_in); padding and short-sequence rows do
 * not wait and run as usual.  Defined by this library (the pages bound no
 * waits).  Errors: those of hs_swap_in, and HS_ERR_ARG for which not 0 or 1.
 */
hs_err hs_swap_in_timeout_selftest(const hs_swap_in_args* args, int32_t rank, int32_t which,
                                   hs_stream_t stream);

/*
 * hs_swap_in_layers -- hs_swap_in for several layers at once, when the caller
 * has every layer's top-k rows: layers[l] is layer l's complete argument
 * block, and the result for each layer is exactly what hs_swap_in(&layers[l])
 * would give, layer by layer.  All batch rows of all layers are resolved by
 * one grid (one CTA per row and layer), so a decode step's layers share the
 * GPU instead of running one small launch after another.  This is a variant
 * of the pages' per-layer call (SGLang jit_kernel/csrc/hisparse.cuh,
 * load_cache_to_device_buffer, runs once per layer); its rules, status bits
 * and time-out behaviour are those of hs_swap_in.
 *
 *  layers      host array of num_layers argument blocks (read during the call
 *              only).  Every block must agree with layers[0] in batch, top_k,
 *              hot_size, flags, row_bytes, max_seq_len, every stride, every
 *              row count (num_states, pool_rows_cols, pool_num_rows,
 *              hot_num_rows), the block-table geometry, and in which optional
 *              pointers are NULL; only the pointers themselves may differ.
 *              Otherwise HS_ERR_ARG.
 *  num_layers  >= 0 (0 launches nothing); any number (launched 64 layers at a
 *              time, in order)
 * Preconditions (not checked): no two layers write the same buffer (state
 * rows, hot buffers, outputs, plans, status words; a shared stats counter is
 * fine, it is added to atomically).  Read-only buffers (pools, slot_rows,
 * pool_rows, tables, top-k rows, request metadata) may be shared.
 * Limits: those of hs_swap_in; per CTA the row's state must fit shared memory
 * (top_k up to a few thousand with any hot_size <= 32767), else
 * HS_ERR_UNSUPPORTED.
 */
hs_err hs_swap_in_layers(const hs_swap_in_args* layers, int32_t num_layers,
                         hs_stream_t stream);

/*
 * hs_swap_in_layers_timeout_selftest -- hs_swap_in_layers with every
 * full-path row made to give up one bounded wait at once (which = 0: the
 * staged state; 1: the top-k row), as hs_swap_in_timeout_selftest does for
 * the per-layer call: those rows report exactly HS_ST_TIMEOUT with
 * miss_count 0 and write nothing else.  Defined by this library.
 */
hs_err hs_swap_in_layers_timeout_selftest(const hs_swap_in_args* layers, int32_t num_layers,
                                          int32_t which, hs_stream_t stream);

/* Shared memory (bytes) per CTA that a swap-in row needs for (top_k, hot_size):
 * split over the largest cluster (8 CTAs) up to hot_size 8192, the one-CTA
 * kernel's least above it; 0 if the pair is outside [1, 32767] or
 * top_k > hot_size.  The call returns HS_ERR_UNSUPPORTED when this exceeds the
 * device's per-CTA shared memory. */
int64_t hs_swap_in_smem_bytes(int32_t top_k, int32_t hot_size);

/*
 * hs_store_kv -- scatter n_tokens rows: k_dst row loc[t] = k_src row t, and
 * likewise V.  Defined by: tokenspeed tokenspeed_kernel/ops/kvcache/triton.py,
 * store_kv_cache and _store_kv_cache_kernel (per-token K/V scatter; source
 * leading axis of any stride, rows contiguous).
 *
 *  k_src, v_src  device bytes; row t at k_src + t*src_k_stride (bytes); v_src
 *                NULL = K only (then v_dst must be NULL)
 *  k_dst, v_dst  device bytes [dst_rows] rows of dst_stride bytes
 *  loc           device int64 [n_tokens]
 *  row_bytes     bytes per row (any >= 1; strides >= row_bytes)
 *  status        device int32 [1] or NULL: HS_ST_BAD_INDEX is OR-ed in when a
 *                loc is outside [0, dst_rows) (that token is skipped)
 * Precondition (not checked): loc values are distinct; src and dst do not overlap.
 */
hs_err hs_store_kv(const void* k_src, const void* v_src, int64_t src_k_stride,
                   int64_t src_v_stride, void* k_dst, void* v_dst, int64_t dst_stride,
                   int64_t dst_rows, const int64_t* loc, int64_t n_tokens, int64_t row_bytes,
                   int32_t* status, hs_stream_t stream);

/* hs_transfer_kv's has_v word: bit 0 says the V pointers follow the K
 * pointers; HS_XFER_DEVICE_SOURCES asserts that every source pointer is
 * device memory, which lets the library move 16-byte-aligned rows with bulk
 * (TMA) copies. */
#define HS_XFER_HAS_V 1
#define HS_XFER_DEVICE_SOURCES 2

/*
 * hs_transfer_kv -- indexed row gather/scatter over layers: for every pair n
 * and every pointer pair p in [0, num_layers * (1 + has_v)),
 * dst_ptrs[p] row dst_idx[n] = src_ptrs[p] row src_idx[n].  With has_v the
 * arrays hold num_layers K pointers followed by num_layers V pointers.
 * num_layers == 1 is the per-layer transfer.  Defined by: tokenspeed
 * tokenspeed_kernel/ops/kvcache/triton.py, transfer_kv_per_layer(_mla) and
 * transfer_kv_all_layer(_mla) (per-layer base pointers in uint64 arrays, one
 * index pair copied across all layers); SGLang jit_kernel/csrc/hisparse.cuh,
 * transfer_cache_dsv4_mla_kernel (the same all-layer form).
 *
 *  src_ptrs, dst_ptrs  device uint64 arrays of base addresses (device or pinned
 *                      host for sources; device for destinations)
 *  src_idx, dst_idx    device int64 [n]
 *  src_stride/dst_stride  row pitch in bytes (>= row_bytes); src_rows/dst_rows
 *                      bound the indices
 *  status              device int32 [1] or NULL: HS_ST_BAD_INDEX when a pair is
 *                      out of range (the pair is skipped for every layer);
 *                      HS_ST_TIMEOUT if a bulk copy's bounded wait gave up
 *  has_v               HS_XFER_HAS_V | HS_XFER_DEVICE_SOURCES (other bits:
 *                      HS_ERR_ARG)
 * Precondition (not checked): dst_idx values are distinct; sources and
 * destinations do not overlap; with HS_XFER_DEVICE_SOURCES every source is
 * device memory.
 */
hs_err hs_transfer_kv(const uint64_t* src_ptrs, const uint64_t* dst_ptrs, int32_t num_layers,
                      int32_t has_v, const int64_t* src_idx, const int64_t* dst_idx, int64_t n,
                      int64_t src_stride, int64_t dst_stride, int64_t src_rows,
                      int64_t dst_rows, int64_t row_bytes, int32_t* status,
                      hs_stream_t stream);

/* Input element types of hs_fp8_store_kv. */
#define HS_DT_F32 0
#define HS_DT_F16 1
#define HS_DT_BF16 2

/*
 * hs_fp8_store_kv -- quantise K/V to FP8 E4M3 and scatter them into a paged
 * KV cache.  Defined by: tokenspeed tokenspeed_kernel/ops/kvcache/triton.py,
 * fused_fp8_set_kv_buffer and _fused_fp8_set_kv_buffer_kernel.  For token t
 * with slot L = cache_loc[t] (skipped, with HS_ST_BAD_INDEX OR-ed into
 * *status, when L is outside [0, num_slots)), page = L / page_size and
 * offset = L % page_size; for every head h < num_kv_heads and d < head_dim:
 *   y = x                               (k_scale / v_scale NULL), or
 *   y = fp32(x * fp32(1 / scale))       (the inverse divided in fp32)
 *   cache[page*cache_stride_page + offset*cache_stride_offset + h*cache_stride_head + d]
 *     = e4m3(y)
 * where e4m3 rounds to nearest, ties to even, saturates finite overflow and
 * infinities to +-448 and keeps NaN a NaN (OCP E4M3 "FN": bias 7, no
 * infinities, S.1111.111 = NaN).
 *
 *  k, v          device [n_tokens, num_kv_heads, head_dim] of in_dtype
 *                (HS_DT_F32 / F16 / BF16), token and head strides in elements,
 *                dims contiguous; v NULL = K only (then v_cache NULL)
 *  k_cache/v_cache  device bytes; strides in bytes (dims contiguous); a flat
 *                cache [slots, heads, dim] is page_size-row pages with
 *                cache_stride_page = page_size * cache_stride_offset
 *  cache_loc     device int64 [n_tokens]
 *  k_scale/v_scale  device fp32 [1] or NULL
 *  status        device int32 [1] or NULL
 * Limits: num_slots < 2^32 (else HS_ERR_UNSUPPORTED).
 * Precondition (not checked): cache_loc values are distinct; inputs and caches
 * do not overlap.
 */
hs_err hs_fp8_store_kv(const void* k, const void* v, int32_t in_dtype, int64_t k_stride_token,
                       int64_t k_stride_head, int64_t v_stride_token, int64_t v_stride_head,
                       void* k_cache, void* v_cache, int64_t cache_stride_page,
                       int64_t cache_stride_offset, int64_t cache_stride_head,
                       int32_t page_size, int64_t num_slots, const int64_t* cache_loc,
                       int64_t n_tokens, int32_t num_kv_heads, int32_t head_dim,
                       const float* k_scale, const float* v_scale, int32_t* status,
                       hs_stream_t stream);

/*
 * hs_invalidate_tokens -- drop resident copies of rewritten tokens: for each
 * n < n_tokens, with r = state_rows[n] and t = tokens[n], every slot
 * s < hot_size of state row r with slot_tokens[r][s] == t becomes -1, so the
 * next swap-in fetches the new row.  r < 0 or t < 0 is skipped; r >=
 * num_states is skipped with HS_ST_BAD_INDEX OR-ed into *status.  Slot
 * hot_size (the newest token's) is not touched.  Defined by: vLLM
 * csrc/libtorch_stable/hisparse_kernels.cu, hisparse_invalidate_written_slots
 * (restated for request-relative slot tokens).
 *
 *  slot_tokens  device int32 [num_states, >= hot_size + 1], stride in elements
 *  state_rows   device int64 [n_tokens]; tokens device int32 [n_tokens]
 *  status       device int32 [1] or NULL
 * Limits: n_tokens * ceil(hot_size / 1024) < 2^31 (else HS_ERR_UNSUPPORTED).
 */
hs_err hs_invalidate_tokens(int32_t* slot_tokens, int64_t slot_tokens_stride, int32_t hot_size,
                            int64_t num_states, const int64_t* state_rows,
                            const int32_t* tokens, int64_t n_tokens, int32_t* status,
                            hs_stream_t stream);

/*
 * hs_gather_misses -- replay a swap-in's miss plan onto the layers that share
 * the resolving layer's indices (same slot assignment, other bytes): for
 * b < batch, m < min(max(miss_count[b], 0), top_k) and every pointer pair p in
 * [0, num_layers * (1 + has_v)), with s = miss_src[b][m], d = miss_dst[b][m]:
 * d < 0 is skipped; s outside [0, pool_num_rows) or d >= hot_num_rows skips
 * the miss (for every layer) and ORs HS_ST_BAD_INDEX into *status; otherwise
 * row d of hot_ptrs[p] = row s of pool_ptrs[p].  With has_v the arrays hold
 * num_layers K pointers followed by num_layers V pointers, as in
 * hs_transfer_kv.  No LRU state is read or written.  Defined by: vLLM
 * csrc/libtorch_stable/hisparse_kernels.cu, hisparse_gather_plan_kernel and
 * hisparse_gather_compact_kernel (shared-layer plan replay; per-row miss lists
 * bounded by per-row counts, fixed shape for graph capture).
 *
 *  pool_ptrs   device uint64 [num_layers * (1 + has_v)]: pools of
 *              [pool_num_rows, row_bytes] contiguous rows, device or pinned host
 *  hot_ptrs    device uint64, same length: device hot buffers [hot_num_rows, row_bytes]
 *  miss_src    device int64 [batch, >=top_k], miss_dst device int32, both stride plan_stride
 *  miss_count  device int32 [batch]
 *  status      device int32 [1] or NULL
 *  flags       HS_GATHER_HAS_V (the V pointers follow the K pointers; written
 *              has_v above) | HS_OVERLAP_PREV (the launch may start while the
 *              preceding kernel in the stream still runs; it reads the plan, the
 *              counts and the pointer arrays, and writes, only after that kernel
 *              has finished, so the plan may come from the swap-in right before
 *              it; the plan and counts are read through L2.  If that kernel
 *              starts its dependents early, it must not write the pools or the
 *              pointer arrays, read through the read-only data path).  Other
 *              bits: HS_ERR_ARG.
 * Precondition (not checked): the miss_dst values a call copies to are distinct.
 */
#define HS_GATHER_HAS_V 1
hs_err hs_gather_misses(const uint64_t* pool_ptrs, const uint64_t* hot_ptrs, int32_t num_layers,
                        int32_t flags, int64_t pool_num_rows, int64_t hot_num_rows,
                        int64_t row_bytes, const int64_t* miss_src, const int32_t* miss_dst,
                        int64_t plan_stride, const int32_t* miss_count, int32_t batch,
                        int32_t top_k, int32_t* status, hs_stream_t stream);

/*
 * hs_probe_read -- measurement utility, not part of the method: stream-read
 * `bytes` bytes (16-byte aligned pointer, bytes % 16 == 0) from device or
 * pinned host memory with every SM, folding them into *sink (device uint64
 * [1]).  Used to measure the host-link read bandwidth that bounds swap-ins
 * from a pinned-host pool.
 */
hs_err hs_probe_read(const void* src, int64_t bytes, unsigned long long* sink,
                     hs_stream_t stream);

/* Text for an hs_err code. */
const char* hs_err_string(int32_t err);

/* Name of one HS_ST_* status bit ("" for a value that is not a single known bit). */
const char* hs_status_string(int32_t bit);

/* Message for the calling thread's last non-HS_OK return ("" if none). */
const char* hs_last_error(void);

/* ABI version of this header. */
/*
 * hs_wait_selftest -- checks that a bounded wait that runs out hands control
 * back: one block initialises an mbarrier that nothing arms and waits on it
 * with the swap-in's bounded mbarrier wait (the one behind HS_ST_TIMEOUT, see
 * hs_swap_in), at most max_polls polls, then ORs HS_ST_TIMEOUT into *status.
 * No copy is in flight on that barrier, so giving up is safe; the context
 * stays usable for the calls that follow.  Defined by this library (the
 * pages bound no waits).
 *
 *  max_polls  >= 0 (each poll may suspend the thread briefly; ~1e3 is quick)
 *  status     device int32 [1], required
 * Errors: HS_ERR_ARG for max_polls < 0 or a NULL status.
 */
hs_err hs_wait_selftest(int32_t max_polls, int32_t* status, hs_stream_t stream);

#define HS_ABI_VERSION 8
int32_t hs_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HISPARSE_H */
