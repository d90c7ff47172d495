// hs_swap_in_rows.cu -- the HiSparse decode-time swap-in with one CTA per
// (batch row, layer) problem, for sm_103a.
//
// The same method as hs_swap_in.cu (SGLang jit_kernel/csrc/hisparse.cuh,
// load_cache_to_device_buffer, with the invalid-entry rules, padding rows and
// tripwires of vLLM csrc/libtorch_stable/hisparse_kernels.cu,
// hisparse_resolve_residency_kernel), laid out for many independent problems
// per launch: hs_swap_in_layers resolves every row of several layers in one
// grid, and hs_swap_in sends rows longer than the cluster kernel's register
// tiles here.  One CTA of 512 threads owns a problem and does its whole
// bookkeeping once -- no work is repeated across CTAs -- and two such CTAs
// share an SM, so one's memory waits overlap the other's bookkeeping.
//
// No per-position state stays in registers across phases, so any hot size up
// to 32767 works; what a phase needs from an earlier one is in shared memory:
//   P0 stage    the LRU row, and where they fit the slot tokens and slot rows,
//               by TMA bulk copies on an mbarrier (thread 0 polls, bounded);
//   P1 request  valid ids into the request map: direct (a bitmap over token
//               ids, word prefixes, rank -> entry) when the caller bounds the
//               sequence length, else the hash (Knuth multiplicative, linear
//               probing, a thread's first CASes issued together) and a 4 KB
//               filter; a second pass only if an id repeats;
//   P2 walk     every position probes its slot's token; the lowest position
//               holding a wanted token claims the entry (atomicMin).  The same
//               pass checks the LRU row: entries outside [0, H) are corrupt;
//               a slot listed twice keeps its lowest position (only when the
//               atomicOr bitmap saw a repeat does one warp mark the later
//               positions, and the walk runs again without them);
//      hits     claimed entries set their position's bit in a hit bitmap;
//               candidates fetch their pool rows with LDGSTS;
//   P3 ranks    popc of the bitmap words and one warp scan give each position
//               its hits-before count;
//   P4 misses   ballot/popc over entries in top-k order gives each miss its
//               rank m; miss m takes the m-th non-hit position in LRU order
//               (found by a binary search over the word prefixes), emits its
//               hot row and records the slot's new token;
//   P5 LRU      the new order [stale evictables][misses][hits] is built in
//               shared memory and stored coalesced;
//   P6 copy     (miss, chunk) items over all threads, loads before stores.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "hs_device.cuh"
#include "hs_host.h"
#include "hs_swap_in_common.cuh"

namespace hs {
namespace {

constexpr int kRowThreads = 512;
constexpr int kRowCopyUnroll = 6;
constexpr int kRowFilterBits = 15;  // request filter: 2^15 bits = 4 KB
constexpr int kRowMaxLayers = 64;   // layers per launch (kernel-parameter space)

// Shared-memory layout of one CTA, computed on the host.  Regions whose
// contents are dead by a later phase are reused: the hash region holds the
// misses' source and destination byte offsets for the copy (it is >= 16K
// bytes), the token region the candidates' pool rows (without block tables)
// and then the new LRU order.
struct RowLayout {
  int hash_bits;
  int map;                    // kMapWide / kMapPacked / kMapDirect
  int direct_words;           // bitmap words of the direct map (max_seq_len / 32, rounded up)
  int o_dpre, o_dent;         // direct map: word prefixes (uint16), dense rank -> entry (int32)
  int stage_tok, stage_rows;  // slot tokens / slot rows staged (else read from global memory)
  int o_hash, o_filter, o_ids, o_lru, o_tok, o_prs, o_rows, o_claim, o_code;
  int o_sbits, o_dup, o_hit, o_cntp, o_cnte, o_misc, o_wsum, o_bar;
  int total;
};

inline int take_(int* o, int64_t bytes) {
  const int r = *o;
  *o += static_cast<int>((bytes + 15) & ~int64_t{15});
  return r;
}

// map: kMapDirect takes max_len (the caller's sequence bound) and ignores
// bits; the hash forms take bits.
RowLayout make_row_layout(int K, int H, int map, int bits, int64_t max_len, bool stage_tok,
                          bool stage_rows, bool tables) {
  RowLayout L{};
  L.map = map;
  L.hash_bits = bits;
  L.stage_tok = stage_tok;
  L.stage_rows = stage_rows;
  const int64_t k = K, h = H, nw = (H + 31) / 32;
  int o = 0;
  if (map == kMapDirect) {  // bitmap | word prefixes | rank -> entry, then the copy offsets
    const int64_t dw = (max_len + 31) / 32;
    L.direct_words = static_cast<int>(dw);
    const int64_t pre = (4 * dw + 15) & ~int64_t{15};
    const int64_t ent = pre + ((2 * dw + 15) & ~int64_t{15});
    L.o_hash = take_(&o, std::max<int64_t>(ent + 4 * k, 16 * k));
    L.o_dpre = L.o_hash + static_cast<int>(pre);
    L.o_dent = L.o_hash + static_cast<int>(ent);
    L.o_filter = take_(&o, 0);
  } else {
    L.o_hash = take_(&o, std::max<int64_t>(int64_t{4} << bits, 16 * k));
    L.o_filter = take_(&o, 4 << (kRowFilterBits - 5));
  }
  L.o_ids = take_(&o, 4 * k + 16);
  L.o_lru = take_(&o, 2 * h + 16);
  int64_t tok_bytes = 2 * h + 16;  // the new LRU order
  if (stage_tok) tok_bytes = std::max(tok_bytes, 4 * h + 16);
  if (!tables) tok_bytes = std::max(tok_bytes, 8 * k);
  L.o_tok = take_(&o, tok_bytes);
  L.o_prs = tables ? take_(&o, 8 * k) : L.o_tok;
  L.o_rows = stage_rows ? take_(&o, 4 * (h + 1) + 16) : 0;
  L.o_claim = take_(&o, 4 * k);
  L.o_code = take_(&o, k);
  L.o_sbits = take_(&o, 4 * nw);
  L.o_dup = take_(&o, 4 * nw);
  L.o_hit = take_(&o, 4 * nw);
  L.o_cntp = take_(&o, 4 * nw);
  L.o_cnte = take_(&o, 4 * ((k + 31) / 32));
  L.o_misc = take_(&o, 64);
  L.o_wsum = take_(&o, 4 * 33);
  L.o_bar = take_(&o, 16);
  L.total = o;
  return L;
}

// Pointers of one layer's call (every other argument is the same for all
// layers of a launch).
struct RowLayerPtrs {
  const int32_t* num_real;
  const int32_t* topk_ids;
  const void* seq_lens;
  const void* req_state;
  int32_t* slot_tokens;
  const int32_t* slot_rows;
  int16_t* lru;
  const int64_t* pool_rows;
  const unsigned char* pool_k;
  const unsigned char* pool_v;
  unsigned char* hot_k;
  unsigned char* hot_v;
  int32_t* out_rows;
  int32_t* miss_count;
  unsigned long long* stats;
  int32_t* status;
  int64_t* miss_src;
  int32_t* miss_dst;
  int32_t* miss_mask;
  const int32_t* src_bt;
  const int32_t* res_bt;
};

struct RowCommon {
  int32_t batch, top_k, hot_size, flags;
  int64_t topk_stride, num_states, slot_tokens_stride, slot_rows_stride, lru_stride;
  int64_t pool_rows_stride, pool_rows_cols, pool_num_rows, hot_num_rows, row_bytes;
  int64_t out_stride, plan_stride, mask_stride, max_seq_len;
  int64_t src_bt_stride, res_bt_stride;
  int32_t src_bt_blocks, src_bs, res_bt_blocks, res_bs, res_null;
  int32_t entry_bits, copy_width, fail_wait;
  int32_t prefetch_rows;  // device pools, 16-byte rows: a miss's row is prefetched into L2
  uint32_t chunks_per_row;
  FastDiv div_src_bs, div_res_bs, div_chunks, div_batch;
  RowLayout lay;
};

template <int NL>
struct RowParams {
  RowCommon c;
  RowLayerPtrs ly[NL];
};

enum { kRmFlags = 0, kRmRepeat = 1, kRmSlotRepeat = 2, kRmHits = 3, kRmMisses = 4 };

__device__ __forceinline__ bool bit_of(const uint32_t* bits, int x) {
  return (bits[x >> 5] >> (x & 31)) & 1u;
}

// The exit of a CTA whose bounded wait ran out (block-uniform): the row is
// left alone -- status exactly HS_ST_TIMEOUT, miss count 0, nothing else
// written -- and the CTA waits, with a much larger bound, for its own bulk
// copies still in flight before its shared memory is released.
__device__ __noinline__ void rows_timeout_exit(int32_t* status, int32_t* miss_count, int b,
                                               uint64_t* bar, bool ids_issued) {
  if (threadIdx.x == 0) {
    if (status) status[b] = HS_ST_TIMEOUT;
    if (miss_count) miss_count[b] = 0;
    mbar_wait(bar + 1, 0, kDrainPolls, kDrainNs);
    if (ids_issued) mbar_wait(bar, 0, kDrainPolls, kDrainNs);
  }
  __syncthreads();
}

// P6: copy misses [0, n): the row at byte offset src[m] of the pool goes to
// byte offset dst[m] of the hot buffer (skipped when dst[m] < 0).  Work items
// are (miss, chunk) over all threads, kRowCopyUnroll loads before the stores.
// One round of copy items, w0 + u * kRowThreads for u < kRowCopyUnroll:
// loads only (the caller stores them with copy_store_round).
template <int G, int U = kRowCopyUnroll>
__device__ __forceinline__ void copy_load_round(const RowCommon& p, const unsigned char* pool,
                                                unsigned char* hot, uint32_t total, uint32_t w0,
                                                const int64_t* src, const int64_t* dst,
                                                typename Chunk<G>::T* v, unsigned char** to) {
  const uint32_t cpr = p.chunks_per_row;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint32_t w = w0 + u * kRowThreads;
    to[u] = nullptr;
    if (w < total) {
      const uint32_t m = cpr == 1 ? w : fast_div(w, p.div_chunks);
      const uint32_t off = (w - m * cpr) * G;
      const int64_t d = dst[m];
      if (d >= 0) {
        v[u] = Chunk<G>::ld(pool + src[m] + off);
        to[u] = hot + d + off;
      }
    }
  }
}
template <int G, int U = kRowCopyUnroll>
__device__ __forceinline__ void copy_store_round(const typename Chunk<G>::T* v,
                                                 unsigned char* const* to) {
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (to[u] != nullptr) Chunk<G>::st(to[u], v[u]);
}
// Items from `first` on (first is a multiple of kRowThreads).
template <int G>
__device__ __forceinline__ void copy_misses(const RowCommon& p, const unsigned char* pool,
                                            unsigned char* hot, int n, const int64_t* src,
                                            const int64_t* dst, uint32_t first = 0) {
  const uint32_t total = static_cast<uint32_t>(n) * p.chunks_per_row;
  for (uint32_t w0 = first + threadIdx.x; w0 < total; w0 += kRowThreads * kRowCopyUnroll) {
    typename Chunk<G>::T v[kRowCopyUnroll];
    unsigned char* to[kRowCopyUnroll];
    copy_load_round<G>(p, pool, hot, total, w0, src, dst, v, to);
    copy_store_round<G>(v, to);
  }
}

template <int NL, bool kTables, int kMap>
__global__ void __launch_bounds__(kRowThreads, 2)
    swap_in_rows_kernel(const __grid_constant__ RowParams<NL> P) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RowCommon& p = P.c;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const unsigned lanes_before = (1u << lane) - 1u;
  const uint32_t layer = p.batch == 1 ? blockIdx.x : fast_div(blockIdx.x, p.div_batch);
  const int b = static_cast<int>(blockIdx.x - layer * static_cast<uint32_t>(p.batch));
  const RowLayerPtrs& q = P.ly[layer];
  const int K = p.top_k;
  const int H = p.hot_size;
  const RowLayout& L = p.lay;

  // ---- P0: request metadata; the short-sequence and padding exits issue no
  // copy.  With HS_OVERLAP_PREV nothing is written and the top-k row is not
  // read before grid_dep_wait().
  grid_dep_launch_dependents();
  const bool overlap = (p.flags & HS_OVERLAP_PREV) != 0;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.o_bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    fence_mbar_init();
  }
  const int32_t* ids_g = q.topk_ids + static_cast<int64_t>(b) * p.topk_stride;
  int32_t* out_g = q.out_rows + static_cast<int64_t>(b) * p.out_stride;
  int32_t* mask_g = q.miss_mask ? q.miss_mask + static_cast<int64_t>(b) * p.mask_stride : nullptr;
  const bool pad_nr = q.num_real != nullptr && b >= __ldg(q.num_real);
  const int64_t r = (p.flags & HS_REQ_STATE_I64)
                        ? __ldg(static_cast<const int64_t*>(q.req_state) + b)
                        : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(q.req_state) + b));
  const int64_t Lb = (p.flags & HS_SEQ_LENS_I64)
                         ? __ldg(static_cast<const int64_t*>(q.seq_lens) + b)
                         : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(q.seq_lens) + b));
  const bool too_long = p.max_seq_len > 0 && Lb > p.max_seq_len;
  if (pad_nr || r < 0 || r >= p.num_states || too_long) {  // padding / bad state row
    grid_dep_wait();
    for (int i = tid; i < K; i += kRowThreads) {
      out_g[i] = -1;
      if (mask_g) mask_g[i] = 0;
    }
    if (tid == 0) {
      if (q.miss_count) q.miss_count[b] = 0;
      if (q.status) q.status[b] = (pad_nr || r < 0) ? 0 : HS_ST_BAD_STATE;
    }
    return;
  }
  const int32_t* rows_g = q.slot_rows + r * p.slot_rows_stride;
  if (Lb <= H) {  // short sequence: every token sits in its own slot
    grid_dep_wait();
    const int64_t count = Lb < K ? Lb : K;
    for (int i = tid; i < K; i += kRowThreads) {
      const int32_t t = __ldcg(ids_g + i);
      int32_t o = -1;
      if (i < count && t >= 0 && t < Lb) {
        o = __ldg(rows_g + t);
        const uint32_t rb = q.res_bt != nullptr ? div_any(t, p.div_res_bs) : 0u;
        if (q.res_bt != nullptr && rb < static_cast<uint32_t>(p.res_bt_blocks)) {
          const int32_t e = __ldg(q.res_bt + r * p.res_bt_stride + rb);
          if (e >= 0 && e != p.res_null) o = e * p.res_bs + (t - static_cast<int32_t>(rb) * p.res_bs);
        }
      }
      out_g[i] = o;
      if (mask_g) mask_g[i] = 0;
    }
    if (tid == 0) {
      if (q.miss_count) q.miss_count[b] = 0;
      if (q.status) q.status[b] = 0;
    }
    return;
  }

  const uint32_t lim = Lb < (1ll << 31) ? static_cast<uint32_t>(Lb) : 0x80000000u;
  const int32_t newest = Lb - 1 <= INT32_MAX ? static_cast<int32_t>(Lb - 1) : -1;
  int32_t* tokens_g = q.slot_tokens + r * p.slot_tokens_stride;
  int16_t* lru_g = q.lru + r * p.lru_stride;
  int16_t* lru = reinterpret_cast<int16_t*>(smem + L.o_lru +
                                            (reinterpret_cast<uintptr_t>(lru_g) & 15u));
  int32_t* tok_s = reinterpret_cast<int32_t*>(smem + L.o_tok +
                                              (reinterpret_cast<uintptr_t>(tokens_g) & 15u));
  int32_t* rows_s = reinterpret_cast<int32_t*>(smem + L.o_rows +
                                               (reinterpret_cast<uintptr_t>(rows_g) & 15u));
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L.o_ids +
                                            (reinterpret_cast<uintptr_t>(ids_g) & 15u));
  const StageSplit sp_lru = stage_split(lru_g, 2LL * H);
  const StageSplit sp_tok = stage_split(tokens_g, L.stage_tok ? 4LL * H : 0);
  const StageSplit sp_rows = stage_split(rows_g, L.stage_rows ? 4LL * (H + 1) : 0);
  const StageSplit sp_ids = stage_split(ids_g, 4LL * K);
  if (tid == 0) {
    mbar_arrive_expect_tx(bar + 1, sp_lru.body + sp_tok.body + sp_rows.body);
    stage_body(lru, lru_g, sp_lru, bar + 1);
    if (L.stage_tok) stage_body(tok_s, tokens_g, sp_tok, bar + 1);
    if (L.stage_rows) stage_body(rows_s, rows_g, sp_rows, bar + 1);
    if (!overlap) {  // the top-k row is final already
      mbar_arrive_expect_tx(bar, sp_ids.body);
      stage_body(ids, ids_g, sp_ids, bar);
    }
  }
  bool ids_issued = !overlap;
  StagePending pend_ids{-1, 0u};
  if (!overlap) pend_ids = stage_edges(ids_g, 4LL * K, sp_ids, tid);
  const StagePending pend_lru = stage_edges(lru_g, 2LL * H, sp_lru, tid);
  const StagePending pend_tok =
      L.stage_tok ? stage_edges(tokens_g, 4LL * H, sp_tok, tid) : StagePending{-1, 0u};
  const StagePending pend_rows =
      L.stage_rows ? stage_edges(rows_g, 4LL * (H + 1), sp_rows, tid) : StagePending{-1, 0u};
  // Slot tokens and slot rows: the staged copies, or global memory when they
  // did not fit (plain loads: this kernel writes the tokens later).
  const int32_t* tokp = L.stage_tok ? tok_s : tokens_g;
  const int32_t* rowp = L.stage_rows ? rows_s : rows_g;

  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + L.o_hash);
  uint32_t* filter = reinterpret_cast<uint32_t*>(smem + L.o_filter);
  int64_t* prs = reinterpret_cast<int64_t*>(smem + L.o_prs);
  int32_t* claim = reinterpret_cast<int32_t*>(smem + L.o_claim);
  int8_t* code = reinterpret_cast<int8_t*>(smem + L.o_code);
  uint32_t* sbits = reinterpret_cast<uint32_t*>(smem + L.o_sbits);
  uint32_t* dup = reinterpret_cast<uint32_t*>(smem + L.o_dup);
  uint32_t* hit = reinterpret_cast<uint32_t*>(smem + L.o_hit);
  int32_t* cntp = reinterpret_cast<int32_t*>(smem + L.o_cntp);
  int32_t* cnte = reinterpret_cast<int32_t*>(smem + L.o_cnte);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.o_misc);
  int32_t* wsum = reinterpret_cast<int32_t*>(smem + L.o_wsum);
  const DirectMap dm{tab, reinterpret_cast<uint16_t*>(smem + L.o_dpre),
                     reinterpret_cast<int32_t*>(smem + L.o_dent)};
  const int nwq = static_cast<int>((Lb + 31) >> 5);  // direct map: bitmap words of this row
  const int nw = (H + 31) / 32;
  {  // whole 16-byte words: every region is padded to 16 bytes
    int4* c4 = reinterpret_cast<int4*>(claim);
    for (int i = tid; i < (K + 3) / 4; i += kRowThreads)
      c4[i] = make_int4(kUnclaimed, kUnclaimed, kUnclaimed, kUnclaimed);
    if constexpr (kMap == kMapDirect) {
      int4* b4 = reinterpret_cast<int4*>(dm.bm);
      for (int i = tid; i < (nwq + 3) / 4; i += kRowThreads) b4[i] = make_int4(0, 0, 0, 0);
      int4* e4 = reinterpret_cast<int4*>(dm.ent);
      for (int i = tid; i < (K + 3) / 4; i += kRowThreads)
        e4[i] = make_int4(kUnclaimed, kUnclaimed, kUnclaimed, kUnclaimed);
    } else {
      int4* t4 = reinterpret_cast<int4*>(tab);
      for (int i = tid; i < (1 << L.hash_bits) / 4; i += kRowThreads)
        t4[i] = make_int4(-1, -1, -1, -1);
      int4* f4 = reinterpret_cast<int4*>(filter);
      for (int i = tid; i < (1 << (kRowFilterBits - 7)); i += kRowThreads)
        f4[i] = make_int4(0, 0, 0, 0);
    }
    for (int i = tid; i < nw; i += kRowThreads) {
      sbits[i] = 0u;
      dup[i] = 0u;
      hit[i] = 0u;
    }
    if (tid < 16) misc[tid] = 0;
  }
  __syncthreads();  // the barriers' initialisation is visible
  stage_finish(lru, pend_lru);
  stage_finish(tok_s, pend_tok);
  stage_finish(rows_s, pend_rows);

  int32_t my_flags = 0;

  // ---- P1 (request): the top-k row, written by the preceding kernel.
  grid_dep_wait();
  if (overlap) {
    pend_ids = stage_edges(ids_g, 4LL * K, sp_ids, tid);
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, sp_ids.body);
      stage_body(ids, ids_g, sp_ids, bar);
    }
    ids_issued = true;
  }
  stage_finish(ids, pend_ids);
  if (!block_wait(bar, 0, p.fail_wait == 1 ? 0u : kMaxPolls)) {
    rows_timeout_exit(q.status, q.miss_count, b, bar, ids_issued);
    return;
  }
  // Block tables: each valid id's entries are loaded with LDGSTS into prs and
  // read back after the hash insert by the thread that loaded them.
  int2* tbl = reinterpret_cast<int2*>(prs);  // {resident entry, source entry}
  if (kTables) {
    for (int i = tid; i < K; i += kRowThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) >= lim) continue;
      const uint32_t rb = q.res_bt != nullptr ? div_any(t, p.div_res_bs) : 0u;
      if (q.res_bt != nullptr && rb < static_cast<uint32_t>(p.res_bt_blocks))
        cp_async_4(&tbl[i].x, q.res_bt + r * p.res_bt_stride + rb);
      else
        tbl[i].x = -1;
      const uint32_t sb = q.src_bt != nullptr ? div_any(t, p.div_src_bs) : 0u;
      if (q.src_bt != nullptr && sb < static_cast<uint32_t>(p.src_bt_blocks))
        cp_async_4(&tbl[i].y, q.src_bt + r * p.src_bt_stride + sb);
      else
        tbl[i].y = 0;
    }
    cp_async_commit();
  }
  constexpr bool kPacked = kMap == kMapPacked;
  const ReqHash<kPacked> hsh{tab, L.hash_bits, p.entry_bits};
  if constexpr (kMap == kMapDirect) {
    // Mark the requested ids (a bit already set is a repeated id), then the
    // words' prefixes (each thread a run of words), then rank -> entry.
    bool rep = false;
    for (int i = tid; i < K; i += kRowThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) >= lim) continue;
      const uint32_t bit = 1u << (t & 31);
      rep |= (atomicOr(&dm.bm[t >> 5], bit) & bit) != 0u;
    }
    if (rep) misc[kRmRepeat] = 1;
    __syncthreads();
    const int per = (nwq + kRowThreads - 1) / kRowThreads;
    const int w0 = tid * per, w1 = min(nwq, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(dm.bm[w]);
    int total;
    int run = block_exclusive_sum(cnt, wsum, &total);
    for (int w = w0; w < w1; ++w) {
      dm.pre[w] = static_cast<uint16_t>(run);
      run += __popc(dm.bm[w]);
    }
    __syncthreads();
    const bool any_rep = misc[kRmRepeat] != 0;
    for (int i = tid; i < K; i += kRowThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) >= lim) continue;
      const int d = dm.rank(t, dm.bm[t >> 5]);
      if (any_rep)
        atomicMin(&dm.ent[d], i);
      else
        dm.ent[d] = i;
    }
  } else {
    bool rep = false;
    for (int g0 = 0; g0 < K; g0 += 4 * kRowThreads) {
      int32_t tv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = g0 + u * kRowThreads + tid;
        tv[u] = i < K ? ids[i] : -1;
      }
      if constexpr (kPacked) {  // first probes issued together, collisions after
        uint32_t h0[4], old[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          old[u] = ReqHash<true>::kEmpty;
          h0[u] = 0u;
          if (static_cast<uint32_t>(tv[u]) >= lim) continue;
          const uint32_t fb = filter_bit(tv[u], kRowFilterBits);
          atomicOr(&filter[fb >> 5], 1u << (fb & 31));
          h0[u] = hsh.first(tv[u]);
          old[u] = atomicCAS(&tab[h0[u]], ReqHash<true>::kEmpty,
                             (static_cast<uint32_t>(tv[u]) << hsh.eb) |
                                 static_cast<uint32_t>(g0 + u * kRowThreads + tid));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (old[u] == ReqHash<true>::kEmpty) continue;  // inserted (or not valid)
          if ((old[u] >> hsh.eb) == static_cast<uint32_t>(tv[u]))
            rep = true;
          else
            rep |= hsh.insert_from(tv[u], g0 + u * kRowThreads + tid, (h0[u] + 1u) & hsh.mask());
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (static_cast<uint32_t>(tv[u]) >= lim) continue;
          const uint32_t fb = filter_bit(tv[u], kRowFilterBits);
          atomicOr(&filter[fb >> 5], 1u << (fb & 31));
          rep |= hsh.insert(tv[u], g0 + u * kRowThreads + tid);
        }
      }
    }
    if (rep) misc[kRmRepeat] = 1;  // a repeated id: resolved below
  }
  if (kTables) {  // resident ids and ids without a source row are not wanted
    cp_async_wait_all();
    for (int i = tid; i < K; i += kRowThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) >= lim) continue;
      const int2 e = tbl[i];
      int8_t c = 0;
      int64_t row = -1;
      if (q.res_bt != nullptr && e.x >= 0 && e.x != p.res_null) {
        c = kResident;
        const int32_t off = t - static_cast<int32_t>(div_any(t, p.div_res_bs)) * p.res_bs;
        row = static_cast<int64_t>(e.x) * p.res_bs + off;
      } else if (q.src_bt != nullptr && t != newest) {
        const int32_t off = t - static_cast<int32_t>(div_any(t, p.div_src_bs)) * p.src_bs;
        const int64_t g = static_cast<int64_t>(e.y) * p.src_bs + off;
        if (e.y <= 0 || g >= p.pool_num_rows)
          c = kUnmapped;
        else
          row = g;  // the candidate's pool row, if it misses
      }
      code[i] = c;
      prs[i] = row;
    }
  }
  __syncthreads();
  const bool id_repeat = misc[kRmRepeat] != 0;
  if (kMap != kMapDirect && id_repeat) {  // rare: each repeated id's smallest entry becomes canonical
    for (int i = tid; i < K; i += kRowThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) < lim) hsh.make_min(t, i);
    }
    __syncthreads();
  }
  // The canonical entry of a valid id, -1 when it is not requested.
  auto map_find = [&](int32_t t) -> int32_t {
    if constexpr (kMap == kMapDirect)
      return dm.find(t);
    else
      return hsh.find(t);
  };

  // The request map needed only the top-k row: the state's copies had until
  // now to arrive.
  if (!block_wait(bar + 1, 0, p.fail_wait == 0 ? 0u : kMaxPolls)) {
    rows_timeout_exit(q.status, q.miss_count, b, bar, ids_issued);
    return;
  }

  // ---- P2: walk the LRU order; the lowest position holding a wanted token
  // claims it.  The first walk also checks the LRU row: a slot outside [0, H)
  // is a corrupt entry, and a slot already seen (atomicOr bitmap) means a slot
  // repeats -- rare: then one warp marks every position whose slot appeared at
  // a lower position, the claims are cleared and the walk runs again without
  // those positions.
  auto walk = [&](bool first_walk, bool skip_dups) {
  for (int x0 = 0; x0 < H; x0 += 4 * kRowThreads) {
    int32_t tk[4];
    bool ok[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + u * kRowThreads + tid;
      const int s = x < H ? lru[x] : -1;
      const bool in_range = x < H && s >= 0 && s < H;
      if (first_walk && x < H) {
        if (in_range) {
          const uint32_t bit = 1u << (s & 31);
          if (atomicOr(&sbits[s >> 5], bit) & bit) misc[kRmSlotRepeat] = 1;
        } else {
          my_flags |= HS_ST_BAD_LRU_SLOT;
        }
      }
      ok[u] = in_range && !(skip_dups && bit_of(dup, x));
      tk[u] = ok[u] ? tokp[s] : -1;
      ok[u] = ok[u] && static_cast<uint32_t>(tk[u]) < lim && tk[u] != newest;
    }
    int f[4];
    if constexpr (kMap == kMapDirect) {  // exact: no filter, no probe chains
      uint32_t bw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) bw[u] = ok[u] ? dm.bm[tk[u] >> 5] : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        f[u] = ((bw[u] >> (tk[u] & 31)) & 1u) ? dm.ent[dm.rank(tk[u], bw[u])] : -1;
    } else {
    uint32_t fw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      fw[u] = ok[u] ? filter[filter_bit(tk[u], kRowFilterBits) >> 5] : 0u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ok[u] = ok[u] && ((fw[u] >> (filter_bit(tk[u], kRowFilterBits) & 31)) & 1u);
      f[u] = -1;
    }
    if constexpr (kPacked) {  // first probes together, the rare longer chains after
      uint32_t kv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) kv[u] = ok[u] ? tab[hsh.first(tk[u])] : ReqHash<true>::kEmpty;
      const uint32_t emask = (1u << hsh.eb) - 1u;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!ok[u] || kv[u] == ReqHash<true>::kEmpty) continue;
        if ((kv[u] >> hsh.eb) == static_cast<uint32_t>(tk[u]))
          f[u] = static_cast<int32_t>(kv[u] & emask);
        else
          f[u] = hsh.find_from(tk[u], (hsh.first(tk[u]) + 1u) & hsh.mask());
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (ok[u]) f[u] = hsh.find(tk[u]);
    }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (kTables && f[u] >= 0 && code[f[u]] != 0) f[u] = -1;  // resident or unmapped: not wanted
      if (f[u] >= 0) atomicMin(&claim[f[u]], x0 + u * kRowThreads + tid);
    }
  }
  };
  walk(true, false);
  __syncthreads();
  const bool slot_repeat = misc[kRmSlotRepeat] != 0;
  if (slot_repeat) {  // rare: `hit` serves as the seen-set of the in-order pass
    if (warp == 0) {
      for (int base = 0; base < H; base += 32) {
        const int x = base + lane;
        const int s = x < H ? lru[x] : -1;
        const bool valid = x < H && s >= 0 && s < H;
        const unsigned same = __match_any_sync(kFullMask, valid ? s : -1 - lane);
        const bool first = valid && (__ffs(same) - 1) == lane;
        const bool seen = valid && bit_of(hit, s);
        __syncwarp();
        if (first && !seen) atomicOr(&hit[s >> 5], 1u << (s & 31));
        const unsigned dmask = __ballot_sync(kFullMask, valid && (!first || seen));
        if (lane == 0) dup[base >> 5] = dmask;
        __syncwarp();
      }
    }
    for (int i = tid; i < K; i += kRowThreads) claim[i] = kUnclaimed;
    __syncthreads();
    for (int i = tid; i < nw; i += kRowThreads) hit[i] = 0u;
    my_flags |= HS_ST_BAD_LRU_SLOT;  // a repeated slot's later positions are corrupt entries
    walk(false, true);
    __syncthreads();
  }
  // Claimed entries mark their position as a hit; the pool rows of the miss
  // candidates (valid, not newest, unclaimed, canonical) are fetched with
  // LDGSTS so the loads overlap P3.
  const int64_t* pool_rows_g = q.pool_rows ? q.pool_rows + r * p.pool_rows_stride : nullptr;
  for (int i = tid; i < K; i += kRowThreads) {
    const int32_t c = claim[i];
    if (c != kUnclaimed) atomicOr(&hit[c >> 5], 1u << (c & 31));
    const int32_t t = ids[i];
    const bool valid = static_cast<uint32_t>(t) < lim;
    const int8_t pre = (kTables && valid) ? code[i] : 0;
    if (pre == kResident) continue;
    const bool cand = valid && t != newest && pre == 0 && c == kUnclaimed &&
                      (!id_repeat || map_find(t) == i);
    if (q.src_bt != nullptr) {
      if (!cand) prs[i] = -1;
    } else if (cand && t < p.pool_rows_cols) {
      cp_async_8(&prs[i], pool_rows_g + t);
    } else {
      prs[i] = -1;
    }
  }
  cp_async_commit();
  __syncthreads();

  // ---- P3: hits before each bitmap word (one warp scan).
  for (int w = tid; w < nw; w += kRowThreads) cntp[w] = __popc(hit[w]);
  __syncthreads();
  if (warp == 0) {
    const int nh = warp_scan_array(cntp, nw, lane);
    if (lane == 0) misc[kRmHits] = nh;
  }
  // The m-th evictable in LRU order is the m-th position that is not a hit:
  // the last word with at most m non-hits before it (binary search on the
  // prefixes), then the right bit of that word.  Only the misses look theirs up.
  auto evictable = [&](int m) -> int {
    int lo = 0, hi = nw - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (32 * mid - cntp[mid] <= m) lo = mid;
      else hi = mid - 1;
    }
    uint32_t free_bits = ~hit[lo];
    if (lo == nw - 1 && (H & 31)) free_bits &= (1u << (H & 31)) - 1u;
    return 32 * lo + static_cast<int>(__fns(free_bits, 0, m - (32 * lo - cntp[lo]) + 1));
  };

  // ---- P4: entries in top-k order.
  cp_async_wait_all();
  __syncthreads();
  for (int base = 0; base < K; base += kRowThreads) {
    const int i = base + tid;
    bool miss = false;
    if (i < K) {
      const int32_t t = ids[i];
      int8_t c;
      if (static_cast<uint32_t>(t) >= lim) {
        c = kInvalid;
      } else if (id_repeat && map_find(t) != i) {
        c = kRepeat;
        my_flags |= HS_ST_DUP_ID;
      } else if (kTables && code[i] == kResident) {
        c = kResident;
      } else if (t == newest) {
        c = kNewest;
      } else if (kTables && code[i] == kUnmapped) {
        c = kInvalid;  // no source row: like an invalid id
      } else if (claim[i] != kUnclaimed) {
        c = kHit;
      } else {
        const int64_t pr = prs[i];
        if (pr >= 0 && pr < p.pool_num_rows) {
          c = kMiss;
          miss = true;
          if (p.prefetch_rows) {  // in L2 by the time P6 copies it
            bulk_prefetch_l2(q.pool_k + pr * p.row_bytes, static_cast<uint32_t>(p.row_bytes));
            if (q.pool_v != nullptr)
              bulk_prefetch_l2(q.pool_v + pr * p.row_bytes, static_cast<uint32_t>(p.row_bytes));
          }
        } else {
          c = kBadPool;
          my_flags |= HS_ST_BAD_POOL_ROW;
        }
      }
      code[i] = c;
    }
    const unsigned m = __ballot_sync(kFullMask, miss);
    if (lane == 0 && base + warp * 32 < K) cnte[(base >> 5) + warp] = __popc(m);
  }
  __syncthreads();
  if (warp == 0) {
    const int nm = warp_scan_array(cnte, (K + 31) / 32, lane);
    if (lane == 0) misc[kRmMisses] = nm;
  }
  __syncthreads();
  const int NH = misc[kRmHits];
  const int M = misc[kRmMisses];
  const int E = H - NH;
  // The hash is dead: it now holds each miss's source and destination byte
  // offsets (the destination -1 when the miss got no hot row).
  int64_t* jsrc = reinterpret_cast<int64_t*>(smem + L.o_hash);
  int64_t* jdst = jsrc + K;
  for (int base = 0; base < K; base += kRowThreads) {
    const int i = base + tid;
    const bool mine = i < K;
    const int8_t c = mine ? code[i] : kInvalid;
    const unsigned m = __ballot_sync(kFullMask, c == kMiss);
    if (mine && mask_g) mask_g[i] = c == kMiss;
    if (c == kMiss) {
      const int mm = cnte[i >> 5] + __popc(m & lanes_before);  // the row's mm-th miss
      const int x = evictable(mm);                             // takes the mm-th evictable
      const int s = lru[x];
      int32_t d = -1;
      if (s >= 0 && s < H && !(slot_repeat && bit_of(dup, x))) {  // not a corrupt entry
        const int32_t hr = rowp[s];
        if (hr >= 0 && hr < p.hot_num_rows) {
          d = hr;
          tokens_g[s] = ids[i];
        } else {
          my_flags |= HS_ST_BAD_HOT_ROW;
        }
      }
      const int64_t pr = prs[i];
      out_g[i] = d;
      jsrc[mm] = pr * p.row_bytes;
      jdst[mm] = d >= 0 ? static_cast<int64_t>(d) * p.row_bytes : -1;
      if (q.miss_src) {
        q.miss_src[b * p.plan_stride + mm] = pr;
        q.miss_dst[b * p.plan_stride + mm] = d;
      }
    } else if (mine) {
      int32_t o = -1;
      if (c == kNewest) o = rowp[H];  // the newest token lives in slot H
      if (kTables && c == kResident) o = static_cast<int32_t>(prs[i]);
      if (c == kHit) o = rowp[lru[claim[i]]];
      out_g[i] = o;
    }
  }
  __syncthreads();  // prs is dead; the token region takes the new LRU order

  // ---- P5: the new LRU order [stale evictables][misses][hits].
  int16_t* nlru = reinterpret_cast<int16_t*>(smem + L.o_tok);
  for (int x = tid; x < H; x += kRowThreads) {
    const uint32_t hw = hit[x >> 5];
    const uint32_t bit = 1u << (x & 31);
    const int hb = cntp[x >> 5] + __popc(hw & (bit - 1u));
    int pos;
    if (hw & bit) {
      pos = E + hb;
    } else {
      const int e = x - hb;
      pos = e >= M ? e - M : E - M + e;
    }
    nlru[pos] = lru[x];
  }
  if (my_flags) atomicOr(&misc[kRmFlags], my_flags);
  __syncthreads();
  if ((reinterpret_cast<uintptr_t>(lru_g) & 15u) == 0) {  // 16-byte stores, then the tail
    const int n16 = H / 8;
    const uint4* s4 = reinterpret_cast<const uint4*>(nlru);
    uint4* g4 = reinterpret_cast<uint4*>(lru_g);
    for (int i = tid; i < n16; i += kRowThreads) g4[i] = s4[i];
    for (int x = n16 * 8 + tid; x < H; x += kRowThreads) lru_g[x] = nlru[x];
  } else {
    for (int x = tid; x < H; x += kRowThreads) lru_g[x] = nlru[x];
  }
  if (tid == 0) {
    if (q.miss_count) q.miss_count[b] = M;
    if (q.status) q.status[b] = misc[kRmFlags];
    if (q.stats) {
      atomicAdd(q.stats, static_cast<unsigned long long>(NH));
      atomicAdd(q.stats + 1, static_cast<unsigned long long>(M));
    }
  }

  // ---- P6: copy the misses' rows.
  if (p.copy_width == 16) {
    copy_misses<16>(p, q.pool_k, q.hot_k, M, jsrc, jdst);
    if (q.pool_v != nullptr) copy_misses<16>(p, q.pool_v, q.hot_v, M, jsrc, jdst);
  } else if (p.copy_width == 4) {
    copy_misses<4>(p, q.pool_k, q.hot_k, M, jsrc, jdst);
    if (q.pool_v != nullptr) copy_misses<4>(p, q.pool_v, q.hot_v, M, jsrc, jdst);
  } else {
    copy_misses<1>(p, q.pool_k, q.hot_k, M, jsrc, jdst);
    if (q.pool_v != nullptr) copy_misses<1>(p, q.pool_v, q.hot_v, M, jsrc, jdst);
  }
}

template <int NL>
using RowKernelFn = void (*)(const RowParams<NL>);

template <int NL, bool kTables>
RowKernelFn<NL> pick_rows_map(int map) {
  if (map == kMapDirect) return swap_in_rows_kernel<NL, kTables, kMapDirect>;
  if (map == kMapPacked) return swap_in_rows_kernel<NL, kTables, kMapPacked>;
  return swap_in_rows_kernel<NL, kTables, kMapWide>;
}
template <int NL>
RowKernelFn<NL> pick_rows_kernel(bool tables, int map) {
  return tables ? pick_rows_map<NL, true>(map) : pick_rows_map<NL, false>(map);
}

// Layer geometry that must agree across the layers of one launch.
bool same_geometry(const hs_swap_in_args& a, const hs_swap_in_args& z) {
  return a.batch == z.batch && a.top_k == z.top_k && a.hot_size == z.hot_size &&
         a.flags == z.flags && a.topk_stride == z.topk_stride && a.num_states == z.num_states &&
         a.slot_tokens_stride == z.slot_tokens_stride &&
         a.slot_rows_stride == z.slot_rows_stride && a.lru_stride == z.lru_stride &&
         a.pool_rows_stride == z.pool_rows_stride && a.pool_rows_cols == z.pool_rows_cols &&
         a.pool_num_rows == z.pool_num_rows && a.hot_num_rows == z.hot_num_rows &&
         a.row_bytes == z.row_bytes && a.out_stride == z.out_stride &&
         a.plan_stride == z.plan_stride && a.mask_stride == z.mask_stride &&
         a.max_seq_len == z.max_seq_len && a.src_bt_stride == z.src_bt_stride &&
         a.src_bt_blocks == z.src_bt_blocks && a.src_block_size == z.src_block_size &&
         a.res_bt_stride == z.res_bt_stride && a.res_bt_blocks == z.res_bt_blocks &&
         a.res_block_size == z.res_block_size && a.res_null_block == z.res_null_block &&
         (a.num_real == nullptr) == (z.num_real == nullptr) &&
         (a.pool_v == nullptr) == (z.pool_v == nullptr) &&
         (a.pool_rows == nullptr) == (z.pool_rows == nullptr) &&
         (a.miss_count == nullptr) == (z.miss_count == nullptr) &&
         (a.stats == nullptr) == (z.stats == nullptr) &&
         (a.status == nullptr) == (z.status == nullptr) &&
         (a.miss_src == nullptr) == (z.miss_src == nullptr) &&
         (a.miss_mask == nullptr) == (z.miss_mask == nullptr) &&
         (a.src_bt == nullptr) == (z.src_bt == nullptr) &&
         (a.res_bt == nullptr) == (z.res_bt == nullptr);
}

RowLayerPtrs layer_ptrs(const hs_swap_in_args& a) {
  RowLayerPtrs y;
  y.num_real = a.num_real;
  y.topk_ids = a.topk_ids;
  y.seq_lens = a.seq_lens;
  y.req_state = a.req_state;
  y.slot_tokens = a.slot_tokens;
  y.slot_rows = a.slot_rows;
  y.lru = a.lru;
  y.pool_rows = a.pool_rows;
  y.pool_k = static_cast<const unsigned char*>(a.pool_k);
  y.pool_v = static_cast<const unsigned char*>(a.pool_v);
  y.hot_k = static_cast<unsigned char*>(a.hot_k);
  y.hot_v = static_cast<unsigned char*>(a.hot_v);
  y.out_rows = a.out_rows;
  y.miss_count = a.miss_count;
  y.stats = a.stats;
  y.status = a.status;
  y.miss_src = a.miss_src;
  y.miss_dst = a.miss_dst;
  y.miss_mask = a.miss_mask;
  y.src_bt = a.src_bt;
  y.res_bt = a.res_bt;
  return y;
}

template <int NL>
hs_err launch_rows(const RowCommon& c, const hs_swap_in_args* layers, int n, bool tables,
                   int device, hs_stream_t stream, const char* who) {
  RowParams<NL> prm;
  prm.c = c;
  for (int l = 0; l < n; ++l) prm.ly[l] = layer_ptrs(layers[l]);
  for (int l = n; l < NL; ++l) prm.ly[l] = prm.ly[0];
  const RowKernelFn<NL> fn = pick_rows_kernel<NL>(tables, c.lay.map);
  hs_err err = ensure_smem(reinterpret_cast<const void*>(fn), device, c.lay.total);
  if (err != HS_OK) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c.batch) * static_cast<unsigned>(n), 1, 1);
  cfg.blockDim = dim3(kRowThreads, 1, 1);
  cfg.dynamicSmemBytes = c.lay.total;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (c.flags & HS_OVERLAP_PREV) ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, prm);
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "%s launch: %s", who, cudaGetErrorString(e));
  return HS_OK;
}

// Shared-memory plan: two CTAs per SM when it fits (slot tokens and rows
// staged, a request hash of four then two slots per id), else one.
// The request map is direct when the caller bounds the sequence length
// (max_len > 0) and it fits, else the packed hash when `packed`, else the wide.
hs_err pick_row_layout(int K, int H, bool tables, bool packed, int64_t max_len,
                       const DeviceInfo& dev, const char* who, RowLayout* out) {
  const int two = dev.max_smem_per_sm / 2 - 1024;
  const int budgets[2] = {two < dev.max_smem_optin ? two : dev.max_smem_optin,
                          dev.max_smem_optin};
  const bool stage[3][2] = {{true, true}, {true, false}, {false, false}};
  const int hash_map = packed ? kMapPacked : kMapWide;
  for (int budget : budgets)
    for (const auto& st : stage) {
      if (max_len > 0 && max_len <= (int64_t{1} << 24)) {
        const RowLayout L =
            make_row_layout(K, H, kMapDirect, 0, max_len, st[0], st[1], tables);
        if (L.total <= budget) {
          *out = L;
          return HS_OK;
        }
      }
      for (int mult = 4; mult >= 2; mult /= 2) {
        const RowLayout L =
            make_row_layout(K, H, hash_map, hash_bits_for(K, mult), 0, st[0], st[1], tables);
        if (L.total <= budget) {
          *out = L;
          return HS_OK;
        }
      }
    }
  return fail(HS_ERR_UNSUPPORTED,
              "%s: top_k %d / hot_size %d need more shared memory per CTA than the device's %d B",
              who, K, H, dev.max_smem_optin);
}

}  // namespace

int64_t swap_in_rows_min_smem(int K, int H, bool tables) {
  return make_row_layout(K, H, kMapPacked, hash_bits_for(K, 2), 0, false, false, tables).total;
}

hs_err swap_in_rows_launch(const hs_swap_in_args* layers, int num_layers, hs_stream_t stream,
                           const char* who, int fail_wait) {
  const hs_swap_in_args& a = layers[0];
  for (int l = 1; l < num_layers; ++l)
    if (!same_geometry(a, layers[l]))
      return fail(HS_ERR_ARG,
                  "%s: layer %d differs from layer 0 in a size, stride, flag or in which "
                  "optional buffers it gives (only pointers may differ)",
                  who, l);
  // The copy width is the narrowest any layer's buffers allow.
  SwapInDerived dv{};
  int width = 16;
  bool pools_device = true;
  for (int l = 0; l < num_layers; ++l) {
    hs_err err = derive_swap_in(&layers[l], who, &dv);
    if (err != HS_OK) return err;
    width = dv.copy_width < width ? dv.copy_width : width;
    pools_device = pools_device && dv.pools_device;
  }
  DeviceInfo dev;
  hs_err err = current_device(&dev);
  if (err != HS_OK) return err;
  RowLayout lay;
  err = pick_row_layout(a.top_k, a.hot_size, dv.tables, dv.packed, a.max_seq_len, dev, who,
                        &lay);
  if (err != HS_OK) return err;
  if (static_cast<int64_t>(a.batch) * kRowMaxLayers > INT32_MAX)
    return fail(HS_ERR_UNSUPPORTED, "%s: batch too large", who);

  RowCommon c{};
  c.batch = a.batch;
  c.top_k = a.top_k;
  c.hot_size = a.hot_size;
  c.flags = a.flags;
  c.topk_stride = a.topk_stride;
  c.num_states = a.num_states;
  c.slot_tokens_stride = a.slot_tokens_stride;
  c.slot_rows_stride = a.slot_rows_stride;
  c.lru_stride = a.lru_stride;
  c.pool_rows_stride = a.pool_rows_stride;
  c.pool_rows_cols = a.pool_rows_cols;
  c.pool_num_rows = a.pool_num_rows;
  c.hot_num_rows = a.hot_num_rows;
  c.row_bytes = a.row_bytes;
  c.out_stride = a.out_stride;
  c.plan_stride = a.plan_stride;
  c.mask_stride = a.mask_stride;
  c.max_seq_len = a.max_seq_len;
  c.src_bt_stride = a.src_bt_stride;
  c.res_bt_stride = a.res_bt_stride;
  c.src_bt_blocks = a.src_bt_blocks;
  c.src_bs = a.src_block_size;
  c.res_bt_blocks = a.res_bt_blocks;
  c.res_bs = a.res_block_size;
  c.res_null = a.res_null_block;
  c.entry_bits = dv.entry_bits;
  c.copy_width = width;
  c.prefetch_rows = width == 16 && pools_device;
  c.fail_wait = fail_wait;
  c.chunks_per_row = static_cast<uint32_t>(a.row_bytes / width);
  c.div_src_bs = dv.div_src_bs;
  c.div_res_bs = dv.div_res_bs;
  c.div_chunks = FastDiv{fastdiv_magic(c.chunks_per_row), c.chunks_per_row};
  c.div_batch = FastDiv{fastdiv_magic(static_cast<uint32_t>(a.batch)),
                        static_cast<uint32_t>(a.batch)};
  c.lay = lay;
  if (static_cast<uint64_t>(c.chunks_per_row) * static_cast<uint64_t>(a.top_k) >= (1ull << 32))
    return fail(HS_ERR_UNSUPPORTED, "%s: top_k * row chunks must be < 2^32", who);
  for (int l0 = 0; l0 < num_layers; l0 += kRowMaxLayers) {
    const int n = num_layers - l0 < kRowMaxLayers ? num_layers - l0 : kRowMaxLayers;
    err = n == 1 ? launch_rows<1>(c, layers + l0, n, dv.tables, dev.device, stream, who)
                 : launch_rows<kRowMaxLayers>(c, layers + l0, n, dv.tables, dev.device, stream,
                                              who);
    if (err != HS_OK) return err;
  }
  return HS_OK;
}

}  // namespace hs

extern "C" hs_err hs_swap_in_layers(const hs_swap_in_args* layers, int32_t num_layers,
                                    hs_stream_t stream) {
  hs::CallRange range("hs_swap_in_layers");
  using namespace hs;
  clear_error();
  if (num_layers < 0) return fail(HS_ERR_ARG, "hs_swap_in_layers: num_layers must be >= 0");
  if (num_layers == 0) return HS_OK;
  if (layers == nullptr) return fail(HS_ERR_ARG, "hs_swap_in_layers: layers is NULL");
  bool any_empty = false;
  for (int l = 0; l < num_layers; ++l) {
    bool empty = false;
    hs_err err = check_swap_in_args(&layers[l], "hs_swap_in_layers", 32767, &empty);
    if (err != HS_OK) return err;
    any_empty |= empty;
  }
  if (any_empty) {  // batch or top_k is 0: nothing to launch if every layer agrees
    for (int l = 1; l < num_layers; ++l)
      if (layers[l].batch != layers[0].batch || layers[l].top_k != layers[0].top_k)
        return fail(HS_ERR_ARG, "hs_swap_in_layers: layer %d differs from layer 0 in batch or top_k", l);
    return HS_OK;
  }
  return swap_in_rows_launch(layers, num_layers, stream, "hs_swap_in_layers", -1);
}

extern "C" hs_err hs_swap_in_layers_timeout_selftest(const hs_swap_in_args* layers,
                                                     int32_t num_layers, int32_t which,
                                                     hs_stream_t stream) {
  using namespace hs;
  clear_error();
  if (which != 0 && which != 1)
    return fail(HS_ERR_ARG, "hs_swap_in_layers_timeout_selftest: which must be 0 or 1");
  if (num_layers < 1 || layers == nullptr)
    return fail(HS_ERR_ARG, "hs_swap_in_layers_timeout_selftest: need layers");
  bool empty = false;
  for (int l = 0; l < num_layers; ++l) {
    hs_err err = check_swap_in_args(&layers[l], "hs_swap_in_layers_timeout_selftest", 32767,
                                    &empty);
    if (err != HS_OK || empty) return err;
  }
  return swap_in_rows_launch(layers, num_layers, stream, "hs_swap_in_layers_timeout_selftest",
                             which);
}
