/*
 * hs_oracle.cpp -- plain, slow, single-threaded CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  It shares no code
 * with the CUDA library.  Membership uses std::unordered_map / std::vector,
 * bytes move with memcpy, and every step is taken in the order the pages
 * state it, one batch row after another, with no blocking or fusion.
 *
 * Sources (page title, section):
 *  - SGLang jit_kernel/csrc/hisparse.cuh, load_cache_to_device_buffer_kernel:
 *    padding exit, short-sequence fast path, newest-token binding, LRU walk
 *    (hits forward / evictables backward), miss compaction in top-k order,
 *    LRU writeback, per-miss row copy.
 *  - vLLM csrc/libtorch_stable/hisparse_kernels.cu,
 *    hisparse_resolve_residency_kernel: invalid entries resolved to -1,
 *    padding rows publish -1, corruption tripwires (LRU slot out of range,
 *    eviction slot out of range), hit/miss statistics, the same writeback
 *    stated a second way.
 *  - vLLM csrc/libtorch_stable/hisparse_kernels.cu, hisparse_gather_plan_kernel
 *    and hisparse_gather_compact_kernel: a resolving layer's miss plan (which
 *    entries missed, which pool row went to which hot row) replayed onto a
 *    layer that shares its indices, with no LRU resolution.
 *  - tokenspeed tokenspeed_kernel/ops/kvcache/triton.py, fused_fp8_set_kv_buffer:
 *    K/V rows optionally multiplied by an inverse scale in fp32, converted to
 *    FP8 E4M3 and scattered into a paged cache (the encoding is written here
 *    from the format's definition: sign, 4 exponent bits with bias 7, 3
 *    mantissa bits, subnormals at exponent 0, S.1111.111 = NaN).
 *  - tokenspeed tokenspeed_kernel/ops/kvcache/triton.py, store_kv_cache and
 *    transfer_kv_per_layer / transfer_kv_all_layer(_mla): indexed row scatter
 *    and gather over per-layer pointer arrays.
 *
 * Readings where the pages are silent or disagree (all restated in the design
 * notes):
 *  - an id is valid iff 0 <= id < seq_len; invalid ids emit -1 and change no state;
 *  - among repeated valid ids in one row the first occurrence wins; later
 *    copies emit -1 and raise DUP_ID;
 *  - the newest token (id == seq_len-1) emits slot_rows[r][H]; the swap-in never
 *    reads or writes slot H's token or bytes;
 *  - padding rows (b >= num_real, or a negative state row) emit -1, miss_count 0;
 *  - an LRU entry outside [0,H), or a slot already seen earlier in the same
 *    LRU row, is a corrupt entry: it is never a hit and is kept as evictable;
 *  - a miss candidate whose pool row is out of [0,P) emits -1 and is not a miss;
 *  - a miss whose eviction slot is corrupt, or whose hot row is out of
 *    [0,hot_num_rows), emits -1 and changes no token and no bytes, but still
 *    counts as a miss and is still moved in the LRU order;
 *  - exactly row_bytes bytes are copied for any row size and alignment.
 *
 * HSO_MUTANT (compile-time, default 0) plants one deliberate mistake so a
 * test can show that the oracle's pins catch it.  Product builds never set it.
 */
#include "hs_oracle.h"

#include <cmath>
#include <cstring>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#ifndef HSO_MUTANT
#define HSO_MUTANT 0
#endif

namespace {

void pad_row(const hso_swap_in_args* a, int32_t b) {
  int32_t* out = a->out_rows + (int64_t)b * a->out_stride;
  for (int32_t i = 0; i < a->top_k; ++i) out[i] = -1;
  if (a->miss_count) a->miss_count[b] = 0;
  if (a->status) a->status[b] = 0;
}

// Block-table lookups (see hso_swap_in_args): -1 when the token has no row.
int64_t resident_row(const hso_swap_in_args* a, int64_t r, int32_t t) {
  if (!a->res_bt) return -1;
  const int64_t blk = t / a->res_block_size;
  if (blk >= a->res_bt_blocks) return -1;
  const int32_t e = a->res_bt[r * a->res_bt_stride + blk];
  if (e < 0 || e == a->res_null_block) return -1;
  return (int64_t)e * a->res_block_size + t % a->res_block_size;
}
int64_t source_row(const hso_swap_in_args* a, int64_t r, int32_t t) {
  const int64_t blk = t / a->src_block_size;
  if (blk >= a->src_bt_blocks) return -1;
  const int32_t e = a->src_bt[r * a->src_bt_stride + blk];
#if HSO_MUTANT == 15
  if (e < 0) return -1;  // planted: block 0 taken as mapped
#else
  if (e <= 0) return -1;
#endif
  const int64_t g = (int64_t)e * a->src_block_size + t % a->src_block_size;
  return g < a->pool_num_rows ? g : -1;
}

void swap_in_row(const hso_swap_in_args* a, int32_t b) {
  const int32_t K = a->top_k;
  const int32_t H = a->hot_size;
  int32_t* out = a->out_rows + (int64_t)b * a->out_stride;
  const int32_t* ids = a->topk_ids + (int64_t)b * a->topk_stride;
  if (a->miss_mask)
    for (int32_t i = 0; i < K; ++i) a->miss_mask[(int64_t)b * a->mask_stride + i] = 0;

  // Step 1: CUDA-graph padding rows.
  if (a->num_real >= 0 && b >= a->num_real) { pad_row(a, b); return; }
  const int64_t r = a->req_state[b];
  if (r < 0) { pad_row(a, b); return; }
  if (r >= a->num_states) {
    pad_row(a, b);
    if (a->status) a->status[b] = HSO_ST_BAD_STATE;
    return;
  }
  const int64_t Lb = a->seq_lens[b];
  if (a->max_seq_len > 0 && Lb > a->max_seq_len) {  // outside the caller's bound
    pad_row(a, b);
    if (a->status) a->status[b] = HSO_ST_BAD_STATE;
    return;
  }
  int32_t* tokens = a->slot_tokens + r * a->slot_tokens_stride;
  const int32_t* rows = a->slot_rows + r * a->slot_rows_stride;
  int16_t* lru = a->lru + r * a->lru_stride;
  const int64_t* pool_rows = a->pool_rows ? a->pool_rows + r * a->pool_rows_stride : nullptr;
  int32_t st = 0;

  // Step 3: fast path -- the whole sequence fits the hot buffer in order.
#if HSO_MUTANT == 5
  if (Lb < H) {
#else
  if (Lb <= H) {
#endif
    const int64_t count = Lb < K ? Lb : K;
    for (int32_t i = 0; i < K; ++i) {
      const int32_t t = ids[i];
#if HSO_MUTANT == 10
      out[i] = (t >= 0 && t < Lb) ? rows[t] : -1;
#else
      out[i] = (i < count && t >= 0 && t < Lb) ? rows[t] : -1;
#endif
      if (i < count && t >= 0 && t < Lb) {  // a resident block serves the token
        const int64_t rr = resident_row(a, r, t);
        if (rr >= 0) out[i] = (int32_t)rr;
      }
    }
    if (a->miss_count) a->miss_count[b] = 0;
    if (a->status) a->status[b] = 0;
    return;
  }

  // Step 4: classify the entries in top-k order.
  for (int32_t i = 0; i < K; ++i) out[i] = -1;
  std::unordered_map<int32_t, int32_t> want;  // token id -> top-k entry
  std::unordered_set<int32_t> seen;
#if HSO_MUTANT == 3
  std::unordered_map<int32_t, int32_t> last_of;
  for (int32_t i = 0; i < K; ++i) last_of[ids[i]] = i;
#endif
  for (int32_t i = 0; i < K; ++i) {
    const int32_t t = ids[i];
    if (t < 0 || (int64_t)t >= Lb) continue;  // invalid: -1, no state change
#if HSO_MUTANT == 3
    if (last_of[t] != i) { st |= HSO_ST_DUP_ID; continue; }
#else
    if (seen.count(t)) { st |= HSO_ST_DUP_ID; continue; }
    seen.insert(t);
#endif
    const int64_t rr = resident_row(a, r, t);
    if (rr >= 0) { out[i] = (int32_t)rr; continue; }  // served from a resident block
#if HSO_MUTANT != 4
    if ((int64_t)t == Lb - 1) { out[i] = rows[H]; continue; }  // newest slot
#endif
    if (a->src_bt && source_row(a, r, t) < 0) continue;  // no source row: invalid
    want[t] = i;
  }

  // Step 5: walk the LRU order from least to most recently used.
  std::vector<int32_t> hits, evict;
  std::vector<char> evict_bad;  // parallel to evict: corrupt LRU entry
  std::vector<char> resolved(K, 0);
  std::unordered_set<int32_t> slot_seen;
  for (int32_t p = 0; p < H; ++p) {
    const int32_t s = lru[p];
    if (s < 0 || s >= H || slot_seen.count(s)) {  // corruption tripwire
      st |= HSO_ST_BAD_LRU_SLOT;
      evict.push_back(s);
      evict_bad.push_back(1);
      continue;
    }
    slot_seen.insert(s);
    const int32_t tok = tokens[s];
    auto it = want.find(tok);
    if (it != want.end() && !resolved[it->second]) {
      resolved[it->second] = 1;
      out[it->second] = rows[s];
      hits.push_back(s);
    } else {
      evict.push_back(s);
      evict_bad.push_back(0);
    }
  }

  // Step 6: miss candidates in top-k order; a bad pool row is not a miss.
  struct Miss { int32_t i; int32_t id; int64_t pool_row; };
  std::vector<Miss> misses;
  for (int32_t i = 0; i < K; ++i) {
    const int32_t t = ids[i];
    auto it = want.find(t);
    if (it == want.end() || it->second != i || resolved[i]) continue;
    const int64_t pr = a->src_bt ? source_row(a, r, t)
                                 : (((int64_t)t < a->pool_rows_cols) ? pool_rows[t] : -1);
#if HSO_MUTANT == 8
    if (pr < 0 || pr > a->pool_num_rows) {
#else
    if (pr < 0 || pr >= a->pool_num_rows) {
#endif
      st |= HSO_ST_BAD_POOL_ROW;
      continue;
    }
    misses.push_back({i, t, pr});
  }
  const int32_t M = (int32_t)misses.size();

  // Step 7: the m-th miss takes the m-th least recently used evictable slot.
#if HSO_MUTANT == 2
  std::vector<int32_t> order(evict.rbegin(), evict.rend());
  std::vector<char> order_bad(evict_bad.rbegin(), evict_bad.rend());
#else
  const std::vector<int32_t>& order = evict;
  const std::vector<char>& order_bad = evict_bad;
#endif
  int32_t applied = 0;
  for (int32_t m = 0; m < M; ++m) {
    const Miss& ms = misses[m];
    if (a->miss_mask) a->miss_mask[(int64_t)b * a->mask_stride + ms.i] = 1;
    if (a->miss_src) {
      a->miss_src[(int64_t)b * a->plan_stride + m] = ms.pool_row;
      a->miss_dst[(int64_t)b * a->plan_stride + m] = -1;  // set below once a row is given
    }
    const int32_t s = order[m];
    if (order_bad[m]) { st |= HSO_ST_BAD_LRU_SLOT; continue; }
    const int32_t hr = rows[s];
    if (hr < 0 || (int64_t)hr >= a->hot_num_rows) { st |= HSO_ST_BAD_HOT_ROW; continue; }
    // Corrupt entries (out of range, or a repeat of an earlier slot) were
    // marked in the walk, so every slot written here is distinct.
    out[ms.i] = hr;
#if HSO_MUTANT == 12
    if (a->miss_src) a->miss_dst[(int64_t)b * a->plan_stride + m] = s;
#else
    if (a->miss_src) a->miss_dst[(int64_t)b * a->plan_stride + m] = hr;
#endif
    tokens[s] = ms.id;
#if HSO_MUTANT == 6
    const int64_t src_row = ms.id;
#else
    const int64_t src_row = ms.pool_row;
#endif
    std::memcpy(a->hot_k + (int64_t)hr * a->row_bytes, a->pool_k + src_row * a->row_bytes,
                (size_t)a->row_bytes);
    if (a->pool_v)
      std::memcpy(a->hot_v + (int64_t)hr * a->row_bytes, a->pool_v + src_row * a->row_bytes,
                  (size_t)a->row_bytes);
    ++applied;
  }

  // Step 8: LRU writeback -- stale evictables, then this step's misses in
  // top-k order, then the hits in their previous relative order (MRU end).
  std::vector<int32_t> next;
  next.reserve(H);
  const int32_t E = (int32_t)evict.size();
#if HSO_MUTANT == 1
  for (int32_t q = M; q < E; ++q) next.push_back(evict[q]);
  for (int32_t s : hits) next.push_back(s);
  for (int32_t q = 0; q < M; ++q) next.push_back(evict[q]);
#elif HSO_MUTANT == 7
  for (int32_t q = M; q < E; ++q) next.push_back(evict[q]);
  for (int32_t q = 0; q < M; ++q) next.push_back(evict[q]);
  for (auto it = hits.rbegin(); it != hits.rend(); ++it) next.push_back(*it);
#else
  for (int32_t q = M; q < E; ++q) next.push_back(order[q]);
  for (int32_t q = 0; q < M; ++q) next.push_back(order[q]);
  for (int32_t s : hits) next.push_back(s);
#endif
  for (int32_t p = 0; p < H; ++p) lru[p] = (int16_t)next[p];

#if HSO_MUTANT == 9
  const int32_t reported = applied;
#else
  const int32_t reported = M;
  (void)applied;
#endif
  if (a->miss_count) a->miss_count[b] = reported;
  if (a->stats) {
    a->stats[0] += (uint64_t)hits.size();
    a->stats[1] += (uint64_t)reported;
  }
  if (a->status) a->status[b] = st;
}

}  // namespace

extern "C" int hso_swap_in(const hso_swap_in_args* a) {
  if (!a || a->top_k < 0 || a->hot_size < 1 || a->top_k > a->hot_size || a->row_bytes < 1)
    return -1;
  if (a->batch <= 0 || a->top_k == 0) return 0;
  for (int32_t b = 0; b < a->batch; ++b) swap_in_row(a, b);
  return 0;
}

extern "C" int hso_invalidate_tokens(int32_t* slot_tokens, int64_t slot_tokens_stride,
                                     int32_t hot_size, int64_t num_states,
                                     const int64_t* state_rows, const int32_t* tokens, int64_t n,
                                     int32_t* status) {
  if (hot_size < 0 || n < 0 || num_states < 0) return -1;
  for (int64_t q = 0; q < n; ++q) {
    const int64_t r = state_rows[q];
    const int32_t t = tokens[q];
    if (r < 0 || t < 0) continue;
    if (r >= num_states) {
      if (status) *status |= HSO_ST_BAD_INDEX;
      continue;
    }
    int32_t* row = slot_tokens + r * slot_tokens_stride;
#if HSO_MUTANT == 16
    for (int32_t s = 0; s <= hot_size; ++s)  // planted: slot H included
#else
    for (int32_t s = 0; s < hot_size; ++s)
#endif
      if (row[s] == t) row[s] = -1;
  }
  return 0;
}

extern "C" int hso_gather_misses(const uint8_t* pool_k, const uint8_t* pool_v,
                                 int64_t pool_num_rows, uint8_t* hot_k, uint8_t* hot_v,
                                 int64_t hot_num_rows, int64_t row_bytes, const int64_t* miss_src,
                                 const int32_t* miss_dst, int64_t plan_stride,
                                 const int32_t* miss_count, int32_t batch, int32_t top_k,
                                 int32_t* status) {
  if (row_bytes < 1 || batch < 0 || top_k < 0) return -1;
  for (int32_t b = 0; b < batch; ++b) {
    int32_t n = miss_count[b];
    if (n < 0) n = 0;
#if HSO_MUTANT == 11
    if (n > top_k + 1) n = top_k + 1;
    for (int32_t m = 0; m <= n && m < top_k; ++m) {
#else
    if (n > top_k) n = top_k;
    for (int32_t m = 0; m < n; ++m) {
#endif
      const int64_t s = miss_src[(int64_t)b * plan_stride + m];
      const int32_t d = miss_dst[(int64_t)b * plan_stride + m];
      if (d < 0) continue;  // this miss was given no hot row
      if (s < 0 || s >= pool_num_rows || (int64_t)d >= hot_num_rows) {
        if (status) *status |= HSO_ST_BAD_INDEX;
        continue;
      }
      std::memcpy(hot_k + (int64_t)d * row_bytes, pool_k + s * row_bytes, (size_t)row_bytes);
      if (pool_v)
        std::memcpy(hot_v + (int64_t)d * row_bytes, pool_v + s * row_bytes, (size_t)row_bytes);
    }
  }
  return 0;
}

extern "C" int hso_store_kv(const uint8_t* k_src, const uint8_t* v_src, int64_t src_k_stride,
                            int64_t src_v_stride, uint8_t* k_dst, uint8_t* v_dst,
                            int64_t dst_stride, int64_t dst_rows, const int64_t* loc,
                            int64_t n_tokens, int64_t row_bytes, int32_t* status) {
  if (row_bytes < 1 || n_tokens < 0) return -1;
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t d = loc[t];
    if (d < 0 || d >= dst_rows) {
      if (status) *status |= HSO_ST_BAD_INDEX;
      continue;
    }
    std::memcpy(k_dst + d * dst_stride, k_src + t * src_k_stride, (size_t)row_bytes);
    if (v_src) std::memcpy(v_dst + d * dst_stride, v_src + t * src_v_stride, (size_t)row_bytes);
  }
  return 0;
}

extern "C" int hso_transfer_kv(const uint64_t* src_ptrs, const uint64_t* dst_ptrs,
                               int32_t num_layers, int32_t has_v, const int64_t* src_idx,
                               const int64_t* dst_idx, int64_t n, int64_t src_stride,
                               int64_t dst_stride, int64_t src_rows, int64_t dst_rows,
                               int64_t row_bytes, int32_t* status) {
  if (row_bytes < 1 || n < 0 || num_layers < 0) return -1;
  const int32_t pairs = num_layers * (has_v ? 2 : 1);
  for (int64_t i = 0; i < n; ++i) {
    const int64_t s = src_idx[i], d = dst_idx[i];
    if (s < 0 || s >= src_rows || d < 0 || d >= dst_rows) {
      if (status) *status |= HSO_ST_BAD_INDEX;
      continue;
    }
    for (int32_t p = 0; p < pairs; ++p) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(src_ptrs[p]);
      uint8_t* dst = reinterpret_cast<uint8_t*>(dst_ptrs[p]);
      std::memcpy(dst + d * dst_stride, src + s * src_stride, (size_t)row_bytes);
    }
  }
  return 0;
}

namespace {

// Round half to even of a non-negative double.
double round_half_even(double q) {
  const double fl = std::floor(q);
  const double r = q - fl;
  if (r > 0.5) return fl + 1.0;
  if (r < 0.5) return fl;
#if HSO_MUTANT == 13
  return fl + 1.0;  // planted: ties away from zero
#else
  return std::fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
#endif
}

float decode_input(const void* base, int64_t idx, int32_t dtype) {
  if (dtype == HSO_IN_F32) {
    return static_cast<const float*>(base)[idx];
  }
  const uint16_t h = static_cast<const uint16_t*>(base)[idx];
  if (dtype == HSO_IN_BF16) {  // the upper half of an IEEE binary32
    const uint32_t bits = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return f;
  }
  // IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits
  const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = std::ldexp(static_cast<double>(m), -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = std::ldexp(1.0 + m / 1024.0, e - 15);
  return static_cast<float>(sign ? -v : v);
}

}  // namespace

extern "C" uint8_t hso_e4m3_from_float(float x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  if (std::isnan(x)) return sign | 0x7F;
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 448.0) return sign | 0x7E;  // saturate (finite overflow and infinities)
  if (a < std::ldexp(1.0, -6)) {
    // subnormal range: value = m * 2^-9, m in [0, 8]; m == 8 is the first normal
    const double m = round_half_even(a * 512.0);
    return sign | static_cast<uint8_t>(m);
  }
  int e2;
  const double fr = std::frexp(a, &e2);  // a = fr * 2^e2, fr in [0.5, 1)
  int e = e2 - 1;                        // a = (2 fr) * 2^e, 2 fr in [1, 2)
  double m = round_half_even((2.0 * fr - 1.0) * 8.0);
  if (m == 8.0) {
    m = 0.0;
    ++e;
  }
  return sign | static_cast<uint8_t>(((e + 7) << 3) | static_cast<int>(m));
}

extern "C" void hso_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = hso_e4m3_from_float(x[i]);
}

extern "C" int hso_fp8_store_kv(const void* k, const void* v, int32_t in_dtype,
                                int64_t k_stride_token, int64_t k_stride_head,
                                int64_t v_stride_token, int64_t v_stride_head, uint8_t* k_cache,
                                uint8_t* v_cache, int64_t c_page, int64_t c_off, int64_t c_head,
                                int32_t page_size, int64_t num_slots, const int64_t* loc,
                                int64_t n_tokens, int32_t num_heads, int32_t head_dim,
                                const float* k_scale, const float* v_scale, int32_t* status) {
  // the inverse scales, divided in fp32 like the pages' host code
  const float inv_k_val = k_scale ? 1.0f / *k_scale : 1.0f;
  const float inv_v_val = v_scale ? 1.0f / *v_scale : 1.0f;
  const float* inv_k = k_scale ? &inv_k_val : nullptr;
  const float* inv_v = v_scale ? &inv_v_val : nullptr;
  if (in_dtype < HSO_IN_F32 || in_dtype > HSO_IN_BF16 || page_size < 1 || n_tokens < 0 ||
      num_heads < 0 || head_dim < 0 || (v == nullptr) != (v_cache == nullptr))
    return -1;
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t L = loc[t];
    if (L < 0 || L >= num_slots) {
      if (status) *status |= HSO_ST_BAD_INDEX;
      continue;
    }
#if HSO_MUTANT == 14
    const int64_t page = L % page_size, off = L / page_size;  // planted: swapped
#else
    const int64_t page = L / page_size, off = L % page_size;
#endif
    for (int kv = 0; kv < (v ? 2 : 1); ++kv) {
      const void* in = kv ? v : k;
      const int64_t st = kv ? v_stride_token : k_stride_token;
      const int64_t sh = kv ? v_stride_head : k_stride_head;
      uint8_t* cache = kv ? v_cache : k_cache;
      const float* inv = kv ? inv_v : inv_k;
      for (int32_t h = 0; h < num_heads; ++h)
        for (int32_t d = 0; d < head_dim; ++d) {
          const float x = decode_input(in, t * st + h * sh + d, in_dtype);
          const float y = inv ? x * *inv : x;  // one fp32 multiply, rounded to fp32
          cache[page * c_page + off * c_off + h * c_head + d] = hso_e4m3_from_float(y);
        }
    }
  }
  return 0;
}
