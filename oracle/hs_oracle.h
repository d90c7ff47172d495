/*
 * hs_oracle.h -- plain single-threaded CPU oracle for the HiSparse KV-row
 * swap-in and the indexed KV-row movers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this library: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant generator with
 * the CUDA path; the status-bit values below restate the public interface.
 *
 * Every pointer here is a HOST pointer.  Floating point never occurs: the
 * method moves bytes and does integer bookkeeping ("The kernels only move
 * bytes; they are dtype agnostic", vLLM csrc/libtorch_stable/hisparse_kernels.cu,
 * file header).
 */
#ifndef HS_ORACLE_H
#define HS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Per-row status bits (restated from the public interface). */
#define HSO_ST_DUP_ID 1
#define HSO_ST_BAD_POOL_ROW 2
#define HSO_ST_BAD_LRU_SLOT 4
#define HSO_ST_BAD_HOT_ROW 8
#define HSO_ST_TIMEOUT 16
#define HSO_ST_BAD_STATE 32
#define HSO_ST_BAD_INDEX 64

typedef struct hso_swap_in_args {
  int32_t batch;    /* B */
  int32_t top_k;    /* K */
  int32_t hot_size; /* H: LRU-managed slots [0,H); slot H holds the newest token */
  int32_t num_real; /* rows b >= num_real are padding; -1 means all rows are real */
  const int32_t* topk_ids; int64_t topk_stride;        /* [B, K] */
  const int64_t* seq_lens;                              /* [B] */
  const int64_t* req_state;                             /* [B] state row per batch row */
  int64_t num_states;                                   /* R */
  int32_t* slot_tokens; int64_t slot_tokens_stride;     /* [R, >=H+1] in/out */
  const int32_t* slot_rows; int64_t slot_rows_stride;   /* [R, >=H+1] */
  int16_t* lru; int64_t lru_stride;                     /* [R, >=H] in/out */
  const int64_t* pool_rows; int64_t pool_rows_stride; int64_t pool_rows_cols; /* [R, cols] */
  const uint8_t* pool_k; const uint8_t* pool_v; int64_t pool_num_rows;       /* pool_v may be NULL */
  uint8_t* hot_k; uint8_t* hot_v; int64_t hot_num_rows;                      /* hot_v NULL iff pool_v NULL */
  int64_t row_bytes;                                    /* S */
  int32_t* out_rows; int64_t out_stride;                /* [B, K] */
  int32_t* miss_count;                                  /* [B] or NULL */
  uint64_t* stats;                                      /* [2] accumulated, or NULL */
  int32_t* status;                                      /* [B] or NULL */
  /* Optional plan outputs (NULL = not written), for replay onto layers that
   * share this call's indices: the row's m-th miss (m < miss_count[b]) came
   * from pool row miss_src[b][m] and was given hot row miss_dst[b][m] (-1 when
   * it got none); entries past the miss count are left as they were.
   * miss_mask[b][i] = 1 when top-k entry i was one of the row's misses. */
  int64_t* miss_src; int32_t* miss_dst; int64_t plan_stride;   /* [B, >=K] */
  int32_t* miss_mask; int64_t mask_stride;                      /* [B, >=K] */
  /* Optional block tables, both indexed by the row's state row r (vLLM
   * hisparse_resolve_residency_kernel, Phase 1).
   * Source table (replaces pool_rows when not NULL): the pool row of token t is
   * g = src_bt[r][t / src_block_size] * src_block_size + t % src_block_size when
   * the block index is below src_bt_blocks, the entry is > 0 and g <
   * pool_num_rows; otherwise the entry is invalid (-1, no state change).
   * Resident table: when e = res_bt[r][t / res_block_size] (block index below
   * res_bt_blocks) is >= 0 and != res_null_block, token t is served from the
   * device: out = e * res_block_size + t % res_block_size, and the entry is not
   * looked up, not a hit and not a miss. */
  const int32_t* src_bt; int64_t src_bt_stride; int32_t src_bt_blocks; int32_t src_block_size;
  const int32_t* res_bt; int64_t res_bt_stride; int32_t res_bt_blocks; int32_t res_block_size;
  int32_t res_null_block;
  /* 0, or a bound on the sequence lengths: a row with seq_len > max_seq_len is
   * a bad-state row (-1, miss_count 0, HSO_ST_BAD_STATE, no state change). */
  int64_t max_seq_len;
} hso_swap_in_args;

/* Returns 0, or -1 when an argument is unusable (the oracle does not try to
 * mirror every synchronous check of the CUDA library). */
int hso_swap_in(const hso_swap_in_args* a);

/* Invalidates resident copies of rewritten tokens (vLLM
 * hisparse_invalidate_written_slots_kernel, restated for request-relative slot
 * tokens): for each n, with r = state_rows[n] and t = tokens[n]: every slot
 * s < hot_size of state row r with slot_tokens[r][s] == t becomes -1.  r < 0
 * or t < 0 is skipped; r >= num_states is skipped with HSO_ST_BAD_INDEX. */
int hso_invalidate_tokens(int32_t* slot_tokens, int64_t slot_tokens_stride, int32_t hot_size,
                          int64_t num_states, const int64_t* state_rows, const int32_t* tokens,
                          int64_t n, int32_t* status);

/* Replays a swap-in's miss plan onto another layer's pool and hot buffer:
 * for b < batch, m < min(max(miss_count[b], 0), top_k): d = miss_dst[b][m],
 * s = miss_src[b][m]; d < 0 is skipped silently; s outside [0,pool_num_rows)
 * or d >= hot_num_rows is skipped with HSO_ST_BAD_INDEX OR-ed into *status;
 * otherwise hot row d = pool row s (K, and V when pool_v is not NULL). */
int hso_gather_misses(const uint8_t* pool_k, const uint8_t* pool_v, int64_t pool_num_rows,
                      uint8_t* hot_k, uint8_t* hot_v, int64_t hot_num_rows, int64_t row_bytes,
                      const int64_t* miss_src, const int32_t* miss_dst, int64_t plan_stride,
                      const int32_t* miss_count, int32_t batch, int32_t top_k, int32_t* status);

/* dst_k[loc[t]] = k_src[t] (and V), tokens in order; loc out of [0,dst_rows)
 * is skipped with HSO_ST_BAD_INDEX OR-ed into *status. */
int hso_store_kv(const uint8_t* k_src, const uint8_t* v_src, int64_t src_k_stride,
                 int64_t src_v_stride, uint8_t* k_dst, uint8_t* v_dst, int64_t dst_stride,
                 int64_t dst_rows, const int64_t* loc, int64_t n_tokens, int64_t row_bytes,
                 int32_t* status);

/* For n in order, for each of the num_layers*(1+has_v) pointer pairs p:
 * dst_ptrs[p] row dst_idx[n] = src_ptrs[p] row src_idx[n].  Out-of-range
 * indices skip the pair with HSO_ST_BAD_INDEX. */
int hso_transfer_kv(const uint64_t* src_ptrs, const uint64_t* dst_ptrs, int32_t num_layers,
                    int32_t has_v, const int64_t* src_idx, const int64_t* dst_idx, int64_t n,
                    int64_t src_stride, int64_t dst_stride, int64_t src_rows, int64_t dst_rows,
                    int64_t row_bytes, int32_t* status);

/* FP8 (E4M3, OCP "FN" variant: bias 7, no infinities, max finite 448, NaN =
 * S.1111.111) encoding of a float: round to nearest, ties to even; finite
 * overflow and infinities saturate to +-448; NaN gives 0x7F | sign << 7. */
uint8_t hso_e4m3_from_float(float x);
/* out[i] = hso_e4m3_from_float(x[i]) for i < n. */
void hso_e4m3_encode_array(const float* x, uint8_t* out, int64_t n);

/* Input element types of hso_fp8_store_kv. */
#define HSO_IN_F32 0
#define HSO_IN_F16 1
#define HSO_IN_BF16 2

/* Quantise K/V rows to FP8 E4M3 and scatter them into a paged cache (tokenspeed
 * tokenspeed_kernel/ops/kvcache/triton.py, fused_fp8_set_kv_buffer):
 * for token t with slot L = loc[t] (skipped with HSO_ST_BAD_INDEX when outside
 * [0, num_slots)), page = L / page_size and offset = L % page_size; for every
 * head h and dim d, y = x (no scale) or y = fp32(x * inv_scale) and
 * cache[page*c_page + offset*c_off + h*c_head + d] = e4m3(y), where
 * inv_scale = fp32(1 / scale) as the pages' host code computes it.  Input
 * strides are in elements (dim stride 1), cache strides in bytes (dim stride
 * 1).  v / v_cache may be NULL (K only); k_scale / v_scale NULL: no scaling. */
int hso_fp8_store_kv(const void* k, const void* v, int32_t in_dtype, int64_t k_stride_token,
                     int64_t k_stride_head, int64_t v_stride_token, int64_t v_stride_head,
                     uint8_t* k_cache, uint8_t* v_cache, int64_t c_page, int64_t c_off,
                     int64_t c_head, int32_t page_size, int64_t num_slots, const int64_t* loc,
                     int64_t n_tokens, int32_t num_heads, int32_t head_dim, const float* k_scale,
                     const float* v_scale, int32_t* status);

#ifdef __cplusplus
}
#endif
#endif /* HS_ORACLE_H */
