// hs_swap_in.cu -- the HiSparse decode-time swap-in for sm_103a.
//
// Defined by SGLang jit_kernel/csrc/hisparse.cuh (load_cache_to_device_buffer
// and its kernel) with the invalid-entry rules, padding rows and corruption
// tripwires of vLLM csrc/libtorch_stable/hisparse_kernels.cu
// (hisparse_resolve_residency_kernel).
//
// Each batch row runs on a cluster of C CTAs (C = 1..8, chosen so that
// batch * C covers the SMs).  Every CTA of the cluster computes the row's
// whole bookkeeping in its own shared memory -- it is cheap, local and
// identical in every CTA -- and then applies only its share of the writes:
// CTA j owns top-k entries [j*E, (j+1)*E) (their outputs, their misses'
// token records and row copies) and LRU positions [j*P, (j+1)*P) (their place
// in the new LRU order).  Exchanging per-position results through
// distributed shared memory instead was measured slower than recomputing
// them.  The only cross-CTA step is one split cluster barrier: no CTA writes
// the row's LRU order or slot tokens before every CTA has staged them.
//
//   P0 stage    the row's LRU order, slot tokens and slot rows into shared
//               memory by TMA bulk copies completed on an mbarrier (head and
//               tail bytes through registers); thread 0 alone polls it;
//   P1 state    check the LRU row is a permutation of the slots (one atomicOr
//               bitmap pass; a lowest-position pass only if a slot repeats)
//               and gather each position's slot token into registers;
//      request  then the top-k row: all valid ids into an open-addressing
//               table (Knuth multiplicative hash, linear probing, a thread's
//               first CASes issued together) and a 16 KB bitmap filter; only
//               when an id repeats does a second pass make its smallest entry
//               index canonical;
//   P2 walk     every position probes its slot's token; the lowest position
//               holding a wanted token claims the entry (atomicMin); the
//               candidates then look up their pool rows (LDGSTS);
//   P3/P4 count position-ordered ballot/popc gives hits per chunk; entries
//               in top-k order are classified (a miss's pool row is then
//               prefetched into L2 by the CTA owning it) and ballot/popc gives
//               misses per chunk; two warps scan both at once: hit ranks, the
//               evictables in LRU order, and each miss's rank m;
//   P4 assign   the m-th miss takes the m-th evictable; the CTA owning the
//               entry emits its output, records the slot's new token and
//               queues the row copy;
//   P5 LRU      each CTA writes its positions' places in the new order
//               [stale evictables][misses][hits];
//   P6 copy     (miss, 16-byte chunk) work items over all threads: read-only
//               no-L1 loads from the pool (HBM or pinned host memory), L2-only
//               stores into the hot buffer.
//
// With HS_OVERLAP_PREV the launch may begin while the preceding kernel in the
// stream is still running: before the grid-dependency wait (right after the
// state's copies are issued) it reads only request metadata and state rows;
// the top-k row is read after the wait, and nothing is written to global
// memory before it.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "hs_device.cuh"
#include "hs_host.h"
#include "hs_swap_in_common.cuh"

namespace hs {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxItems = 8;  // LRU positions per thread: hot_size <= 8192
constexpr int kCopyUnroll = 4;
constexpr int kMaxCluster = 8;

constexpr int kBloomBits = 17;  // request filter: 2^17 bits = 16 KB

struct Layout {
  int hash_bits, hash_size, slice_p, slice_e;
  int o_hash, o_bloom, o_prs, o_ids, o_lru, o_tok, o_rows, o_mark, o_sbits, o_claim, o_evl, o_cntp, o_cnte, o_code, o_misc, o_bar, o_jsrc, o_jdst;
  int total;
};

__host__ __device__ inline int take(int* o, int bytes) {
  const int r = *o;
  *o += (bytes + 15) & ~15;
  return r;
}

// Shared-memory layout of one CTA.  Slices are whole 32-element chunks so a
// warp's ballot covers one chunk of the row.
__host__ __device__ inline Layout make_layout(int K, int H, int C, int bits) {
  Layout L;
  L.hash_bits = bits;
  L.hash_size = 1 << bits;
  L.slice_p = ((H + C - 1) / C + 31) & ~31;
  L.slice_e = ((K + C - 1) / C + 31) & ~31;
  const int chunks_p = (H + 31) / 32, chunks_e = (K + 31) / 32;
  int o = 0;
  L.o_hash = take(&o, 4 * L.hash_size);   // the request hash (ReqHash)
  L.o_bloom = take(&o, 4 << (kBloomBits - 5));  // one bit per hashed requested id
  L.o_prs = take(&o, 8 * K);              // pool row of each miss candidate (LDGSTS)
  L.o_ids = take(&o, 4 * K + 16);         // staged top-k row
  L.o_lru = take(&o, 2 * H + 16);         // staged LRU order
  L.o_tok = take(&o, 4 * H + 16);         // staged slot tokens [0, H)
  L.o_rows = take(&o, 4 * (H + 1) + 16);  // staged slot rows [0, H]
  L.o_mark = take(&o, 4 * H);             // slot -> lowest LRU position (repeated slots only)
  L.o_sbits = take(&o, 4 * ((H + 31) / 32));  // slots seen in the LRU row
  L.o_claim = take(&o, 4 * K);            // entry -> lowest position holding its token
  L.o_evl = take(&o, 4 * H);              // evictables in LRU order: slot | corrupt << 16
  L.o_cntp = take(&o, 4 * chunks_p);      // per-chunk hit counts -> exclusive prefixes
  L.o_cnte = take(&o, 4 * chunks_e);      // per-chunk miss counts -> exclusive prefixes
  L.o_code = take(&o, K);                 // per-entry classification
  L.o_misc = take(&o, 4 * 8);
  L.o_bar = take(&o, 16);                 // mbarriers: [0] top-k row, [1] state row
  L.o_jsrc = take(&o, 8 * L.slice_e);     // my misses: pool row
  L.o_jdst = take(&o, 4 * L.slice_e);     // my misses: hot row or -1
  L.total = o;
  return L;
}

struct SwapInParams {
  int32_t top_k, hot_size, cluster, hash_bits, flags;
  const int32_t* num_real;
  const int32_t* topk_ids;
  int64_t topk_stride;
  const void* seq_lens;
  const void* req_state;
  int64_t num_states;
  int32_t* slot_tokens;
  int64_t slot_tokens_stride;
  const int32_t* slot_rows;
  int64_t slot_rows_stride;
  int16_t* lru;
  int64_t lru_stride;
  const int64_t* pool_rows;
  int64_t pool_rows_stride, pool_rows_cols;
  const unsigned char* pool_k;
  const unsigned char* pool_v;
  int64_t pool_num_rows;
  unsigned char* hot_k;
  unsigned char* hot_v;
  int64_t hot_num_rows;
  int64_t row_bytes;
  int32_t* out_rows;
  int64_t out_stride;
  int32_t* miss_count;
  unsigned long long* stats;
  int32_t* status;
  int64_t* miss_src;  // optional miss plan
  int32_t* miss_dst;
  int64_t plan_stride;
  int32_t* miss_mask;
  int64_t mask_stride;
  const int32_t* src_bt;  // optional block tables, indexed by state row
  int64_t src_bt_stride;
  int32_t src_bt_blocks, src_bs;
  const int32_t* res_bt;
  int64_t res_bt_stride;
  int32_t res_bt_blocks, res_bs, res_null;
  FastDiv div_src_bs, div_res_bs;  // dividers by the two block sizes
  uint32_t chunks_per_row;  // row_bytes / copy width
  FastDiv div_chunks;
  Layout lay;               // shared-memory layout, computed once on the host
  int32_t entry_bits;       // bits of a top-k entry index in the packed hash
  int64_t max_seq_len;      // 0, or a bound on every row's sequence length
  int32_t copy_width;       // 16, 4 or 1 bytes per copy chunk
  int32_t prefetch_rows;    // device pools, 16-byte rows: a miss's row is prefetched into L2
  int32_t fail_rank;        // self-test: this cluster rank's wait gives up at once (-1: none)
  int32_t fail_wait;        // self-test: 0 = the state-row wait, 1 = the top-k-row wait
};

enum {
  kMiscFlags = 0, kMiscRepeat = 1, kMiscSlotRepeat = 2, kMiscHits = 3, kMiscMisses = 4,
  kMiscTimeout = 5,    // this CTA's bounded wait ran out
  kMiscRowTimeout = 6  // some CTA of the row's cluster ran out
};

__device__ __forceinline__ uint32_t bloom_bit(int32_t key) { return filter_bit(key, kBloomBits); }

// The exit of a CTA whose bounded wait ran out (block-uniform; the CTA has
// arrived at the row's first cluster barrier).  It completes both cluster
// barriers so that its peers' waits complete, reports the time-out (with no
// other write: its peers see the time-out too and leave the row alone), and
// waits, with a much larger bound, for its own bulk copies still in flight
// before its shared memory is released.  If even that bound runs out the CTA
// returns with the copy outstanding; HS_ST_TIMEOUT then says the context is
// suspect.
__device__ __noinline__ void timeout_tail(const SwapInParams& p, int b, int j, int C,
                                          uint64_t* bar) {
  cluster_wait();
  if (C > 1) cluster_arrive_relaxed();
  if (threadIdx.x == 0) {
    if (p.status) {
      if (j == 0)
        p.status[b] = HS_ST_TIMEOUT;
      else
        atomicOr(p.status + b, HS_ST_TIMEOUT);
    }
    if (j == 0 && p.miss_count) p.miss_count[b] = 0;
    mbar_wait(bar + 1, 0, kDrainPolls, kDrainNs);
    mbar_wait(bar, 0, kDrainPolls, kDrainNs);
  }
  __syncthreads();
  if (C > 1) cluster_wait();
}

// P6: copy this CTA's misses, work item = (miss, chunk).
template <int G>
__device__ __forceinline__ void copy_rows(const SwapInParams& p, const unsigned char* pool,
                                          unsigned char* hot, int n, const int64_t* jsrc,
                                          const int32_t* jdst) {
  using Ch = Chunk<G>;
  const uint32_t cpr = p.chunks_per_row;
  const uint32_t total = static_cast<uint32_t>(n) * cpr;
  for (uint32_t w0 = threadIdx.x; w0 < total; w0 += kThreads * kCopyUnroll) {
    typename Ch::T v[kCopyUnroll];
    unsigned char* dst[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const uint32_t w = w0 + u * kThreads;
      dst[u] = nullptr;
      if (w < total) {
        const uint32_t m = cpr == 1 ? w : fast_div(w, p.div_chunks);
        const uint32_t c = w - m * cpr;
        const int32_t d = jdst[m];
        if (d >= 0) {
          const int64_t off = static_cast<int64_t>(c) * G;
          v[u] = Ch::ld(pool + jsrc[m] * p.row_bytes + off);
          dst[u] = hot + static_cast<int64_t>(d) * p.row_bytes + off;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (dst[u] != nullptr) Ch::st(dst[u], v[u]);
  }
}

// IT = LRU positions per thread (position k * 1024 + tid for k < IT); their
// slot, claimed entry and hit flag stay in registers from P1 to P5, and each
// phase handles them as batched, independent loads.
// kTables: the call passes block tables (compiled out of the common case).
// kPacked: the packed request hash (the caller bounds the sequence lengths).
template <int IT, bool kTables, bool kPacked>
__global__ void __launch_bounds__(kThreads, 1) swap_in_kernel(const SwapInParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const unsigned lanes_before = (1u << lane) - 1u;
  const int C = p.cluster;
  const int j = static_cast<int>(cluster_rank());
  const int b = blockIdx.x / C;
  const int K = p.top_k;
  const int H = p.hot_size;
  const Layout& L = p.lay;
  const int p0 = min(H, j * L.slice_p), p1 = min(H, p0 + L.slice_p);  // my LRU positions
  const int e0 = min(K, j * L.slice_e), e1 = min(K, e0 + L.slice_e);  // my entries

  // ---- P0: request metadata and the state row.  With HS_OVERLAP_PREV this
  // grid may start while the preceding kernel in the stream still runs: until
  // grid_dep_wait() it reads only the request's metadata and state row and
  // writes nothing to global memory; the top-k row is read after the wait.
  // Rows are staged by bulk copies (their 16-byte-aligned bodies) completed
  // on two mbarriers, one per row kind, each used for one phase; the
  // unaligned head and tail bytes go through registers.  Copies are issued
  // only on the full path, so the padding and short-sequence exits leave
  // nothing in flight.
  grid_dep_launch_dependents();
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.o_bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    fence_mbar_init();
  }
  const int32_t* ids_g = p.topk_ids + static_cast<int64_t>(b) * p.topk_stride;
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L.o_ids +
                                            (reinterpret_cast<uintptr_t>(ids_g) & 15u));
  const StageSplit sp_ids = stage_split(ids_g, 4LL * K);
  StagePending pend_ids{-1, 0u};
  auto stage_ids = [&]() {
    pend_ids = stage_edges(ids_g, 4LL * K, sp_ids, tid);
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, sp_ids.body);
      stage_body(ids, ids_g, sp_ids, bar);
    }
  };

  int32_t* out_g = p.out_rows + static_cast<int64_t>(b) * p.out_stride;
  const bool pad_nr = p.num_real != nullptr && b >= __ldg(p.num_real);
  const int64_t r = (p.flags & HS_REQ_STATE_I64)
                        ? __ldg(static_cast<const int64_t*>(p.req_state) + b)
                        : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(p.req_state) + b));
  const int64_t Lb = (p.flags & HS_SEQ_LENS_I64)
                         ? __ldg(static_cast<const int64_t*>(p.seq_lens) + b)
                         : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(p.seq_lens) + b));

  const bool too_long = p.max_seq_len > 0 && Lb > p.max_seq_len;  // outside the caller's bound
  if (pad_nr || r < 0 || r >= p.num_states || too_long) {  // padding / bad state row
    grid_dep_wait();
    for (int i = e0 + tid; i < e1; i += kThreads) {
      out_g[i] = -1;
      if (p.miss_mask) p.miss_mask[b * p.mask_stride + i] = 0;
    }
    if (j == 0 && tid == 0) {
      if (p.miss_count) p.miss_count[b] = 0;
      if (p.status) p.status[b] = (pad_nr || r < 0) ? 0 : HS_ST_BAD_STATE;
    }
    return;
  }

  const int32_t* rows_g = p.slot_rows + r * p.slot_rows_stride;
  if (Lb <= H) {  // fast path: the whole sequence sits in the hot buffer in order
    grid_dep_wait();
    // Each CTA reads only its own entries' ids, straight from global memory
    // through L2 (the preceding kernel may have written them).
    const int64_t count = Lb < K ? Lb : K;
    for (int i = e0 + tid; i < e1; i += kThreads) {
      const int32_t t = __ldcg(ids_g + i);
      int32_t o = -1;
      if (i < count && t >= 0 && t < Lb) {
        o = __ldg(rows_g + t);
        const uint32_t rb = p.res_bt != nullptr ? div_any(t, p.div_res_bs) : 0u;
        if (p.res_bt != nullptr && rb < static_cast<uint32_t>(p.res_bt_blocks)) {  // a resident block
          const int32_t e = __ldg(p.res_bt + r * p.res_bt_stride + rb);
          if (e >= 0 && e != p.res_null) o = e * p.res_bs + (t - static_cast<int32_t>(rb) * p.res_bs);
        }
      }
      out_g[i] = o;
      if (p.miss_mask) p.miss_mask[b * p.mask_stride + i] = 0;
    }
    if (j == 0 && tid == 0) {
      if (p.miss_count) p.miss_count[b] = 0;
      if (p.status) p.status[b] = 0;
    }
    return;
  }

  // A top-k id t is valid iff 0 <= t < Lb: as one unsigned compare against
  // min(Lb, 2^31); the newest token is Lb - 1 (no int32 id matches -1 here).
  const uint32_t lim = Lb < (1ll << 31) ? static_cast<uint32_t>(Lb) : 0x80000000u;
  const int32_t newest = Lb - 1 <= INT32_MAX ? static_cast<int32_t>(Lb - 1) : -1;
  int32_t* tokens_g = p.slot_tokens + r * p.slot_tokens_stride;
  int16_t* lru_g = p.lru + r * p.lru_stride;
  int16_t* lru = reinterpret_cast<int16_t*>(smem + L.o_lru +
                                            (reinterpret_cast<uintptr_t>(lru_g) & 15u));
  int32_t* tok = reinterpret_cast<int32_t*>(smem + L.o_tok +
                                            (reinterpret_cast<uintptr_t>(tokens_g) & 15u));
  int32_t* rows = reinterpret_cast<int32_t*>(smem + L.o_rows +
                                             (reinterpret_cast<uintptr_t>(rows_g) & 15u));
  const StageSplit sp_lru = stage_split(lru_g, 2LL * H);
  const StageSplit sp_tok = stage_split(tokens_g, 4LL * H);
  const StageSplit sp_rows = stage_split(rows_g, 4LL * (H + 1));
  if (tid == 0) {
    mbar_arrive_expect_tx(bar + 1, sp_lru.body + sp_tok.body + sp_rows.body);
    stage_body(lru, lru_g, sp_lru, bar + 1);
    stage_body(tok, tokens_g, sp_tok, bar + 1);
    stage_body(rows, rows_g, sp_rows, bar + 1);
  }
  // The grid-dependency wait comes right after the state's copies are
  // issued, and the top-k row's copy right after it (without early start the
  // wait returns at once).  The CTAs that set a launch's length are the last
  // to get an SM, after the preceding kernel has ended: for them the wait is
  // free, and the row's fetch overlaps the fills and the state half below.
  // A CTA that started early does those after the wait, with time to spare.
  grid_dep_wait();
  stage_ids();
  const StagePending pend_lru = stage_edges(lru_g, 2LL * H, sp_lru, tid);
  const StagePending pend_tok = stage_edges(tokens_g, 4LL * H, sp_tok, tid);
  const StagePending pend_rows = stage_edges(rows_g, 4LL * (H + 1), sp_rows, tid);

  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + L.o_hash);
  uint32_t* bloom = reinterpret_cast<uint32_t*>(smem + L.o_bloom);
  int64_t* prs = reinterpret_cast<int64_t*>(smem + L.o_prs);
  int32_t* mark = reinterpret_cast<int32_t*>(smem + L.o_mark);
  uint32_t* sbits = reinterpret_cast<uint32_t*>(smem + L.o_sbits);
  int32_t* claim = reinterpret_cast<int32_t*>(smem + L.o_claim);
  int32_t* evl = reinterpret_cast<int32_t*>(smem + L.o_evl);
  int32_t* cntp = reinterpret_cast<int32_t*>(smem + L.o_cntp);
  int32_t* cnte = reinterpret_cast<int32_t*>(smem + L.o_cnte);
  int8_t* code = reinterpret_cast<int8_t*>(smem + L.o_code);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.o_misc);
  int64_t* jsrc = reinterpret_cast<int64_t*>(smem + L.o_jsrc);
  int32_t* jdst = reinterpret_cast<int32_t*>(smem + L.o_jdst);
  {
    int4* t4 = reinterpret_cast<int4*>(tab);
    for (int i = tid; i < L.hash_size / 4; i += kThreads) t4[i] = make_int4(-1, -1, -1, -1);
  }
  {  // whole 16-byte words: every region is padded to 16 bytes
    int4* c4 = reinterpret_cast<int4*>(claim);
    for (int i = tid; i < (K + 3) / 4; i += kThreads)
      c4[i] = make_int4(kUnclaimed, kUnclaimed, kUnclaimed, kUnclaimed);
    int4* b4 = reinterpret_cast<int4*>(bloom);
    for (int i = tid; i < (1 << (kBloomBits - 7)); i += kThreads) b4[i] = make_int4(0, 0, 0, 0);
    int4* s4 = reinterpret_cast<int4*>(sbits);
    for (int i = tid; i < ((H + 31) / 32 + 3) / 4; i += kThreads) s4[i] = make_int4(0, 0, 0, 0);
  }
  if (tid < 8) misc[tid] = 0;
  __syncthreads();  // the barriers' initialisation is visible
  stage_finish(lru, pend_lru);
  stage_finish(tok, pend_tok);
  stage_finish(rows, pend_rows);
  // A wait that runs out in any CTA of the row leaves the whole row alone:
  // each CTA records its outcome in misc[kMiscTimeout] before the cluster
  // barrier, and after it every CTA reads all of them (below, before the
  // row's first write).
  const uint32_t polls_state = (p.fail_rank == j && p.fail_wait == 0) ? 0u : kMaxPolls;
  if (!block_wait(bar + 1, 0, polls_state)) {
    if (tid == 0) {
      misc[kMiscTimeout] = 1;
      fence_acq_rel_cluster();
    }
    cluster_arrive_relaxed();
    timeout_tail(p, b, j, C, bar);
    return;
  }
  // ---- P1 (state half): check the LRU row is a permutation of the slots.
  int32_t my_flags = 0;
  int sl[IT];  // the slot at each of my LRU positions
#pragma unroll
  for (int k = 0; k < IT; ++k) {
    const int q = k * kThreads + tid;
    sl[k] = q < H ? lru[q] : 0;
  }
#pragma unroll
  for (int k = 0; k < IT; ++k) {
    if (k * kThreads + tid >= H) continue;
    if (sl[k] >= 0 && sl[k] < H) {
      const uint32_t bit = 1u << (sl[k] & 31);
      if (atomicOr(&sbits[sl[k] >> 5], bit) & bit) misc[kMiscSlotRepeat] = 1;
    } else {
      my_flags |= HS_ST_BAD_LRU_SLOT;
    }
  }
  __syncthreads();
  const bool slot_repeat = misc[kMiscSlotRepeat] != 0;
  if (slot_repeat) {  // rare: a slot listed twice keeps its lowest position
#pragma unroll
    for (int k = 0; k < IT; ++k)
      if (k * kThreads + tid < H && sl[k] >= 0 && sl[k] < H) mark[sl[k]] = kUnclaimed;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < IT; ++k)
      if (k * kThreads + tid < H && sl[k] >= 0 && sl[k] < H) atomicMin(&mark[sl[k]], k * kThreads + tid);
    __syncthreads();
  }
  // The token each of my positions holds, if it could be wanted.
  int f[IT];  // per position: the wanted entry it holds, -1 none, -2 corrupt entry
  int32_t tk[IT];
  bool ok[IT];
  {
#pragma unroll
    for (int k = 0; k < IT; ++k) {
      const int q = k * kThreads + tid;
      ok[k] = q < H && sl[k] >= 0 && sl[k] < H;
    }
    if (slot_repeat) {
#pragma unroll
      for (int k = 0; k < IT; ++k)
        if (ok[k]) ok[k] = mark[sl[k]] == k * kThreads + tid;
    }
#pragma unroll
    for (int k = 0; k < IT; ++k) {
      f[k] = ok[k] ? -1 : -2;
      tk[k] = ok[k] ? tok[sl[k]] : -1;
    }
#pragma unroll
    for (int k = 0; k < IT; ++k)
      ok[k] = ok[k] && static_cast<uint32_t>(tk[k]) < lim && tk[k] != newest;
  }

  // ---- P1 (request half): the top-k row, written by the preceding kernel.
  stage_finish(ids, pend_ids);
  const uint32_t polls_ids = (p.fail_rank == j && p.fail_wait == 1) ? 0u : kMaxPolls;
  const bool ids_ok = block_wait(bar, 0, polls_ids);
  // Every CTA of the row has staged the state (and recorded whether its waits
  // ran out) once all have arrived here; the matching wait comes before the
  // walk, well before the row's first write.  Thread 0, which saw the copies
  // complete and wrote the outcome, releases; the others arrive relaxed.
  if (tid == 0) {
    if (!ids_ok) misc[kMiscTimeout] = 1;
    fence_acq_rel_cluster();
  }
  cluster_arrive_relaxed();
  if (!ids_ok) {
    timeout_tail(p, b, j, C, bar);
    return;
  }
  // Block tables: each valid id's entries are loaded with LDGSTS into prs
  // (free until P2's candidate prefetch), read back after the hash insert by
  // the thread that loaded them.
  constexpr bool tables = kTables;
  int2* tbl = reinterpret_cast<int2*>(prs);  // {resident entry, source entry}
  if (tables) {
    for (int i = tid; i < K; i += kThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) >= lim) continue;
      const uint32_t rb = p.res_bt != nullptr ? div_any(t, p.div_res_bs) : 0u;
      if (p.res_bt != nullptr && rb < static_cast<uint32_t>(p.res_bt_blocks))
        cp_async_4(&tbl[i].x, p.res_bt + r * p.res_bt_stride + rb);
      else
        tbl[i].x = -1;
      const uint32_t sb = p.src_bt != nullptr ? div_any(t, p.div_src_bs) : 0u;
      if (p.src_bt != nullptr && sb < static_cast<uint32_t>(p.src_bt_blocks))
        cp_async_4(&tbl[i].y, p.src_bt + r * p.src_bt_stride + sb);
      else
        tbl[i].y = 0;
    }
    cp_async_commit();
  }
  // Hash the valid ids; only when an id repeats does a second pass make its
  // smallest entry index canonical.
  const ReqHash<kPacked> hsh{tab, L.hash_bits, p.entry_bits};
  if constexpr (kPacked && IT <= 4) {  // my entries' first probes batched, collisions after
    int32_t tv[IT];
    uint32_t h0[IT], old[IT];
#pragma unroll
    for (int k = 0; k < IT; ++k) tv[k] = k * kThreads + tid < K ? ids[k * kThreads + tid] : -1;
#pragma unroll
    for (int k = 0; k < IT; ++k) {
      old[k] = ReqHash<true>::kEmpty;
      if (static_cast<uint32_t>(tv[k]) >= lim) continue;
      const uint32_t bb = bloom_bit(tv[k]);
      atomicOr(&bloom[bb >> 5], 1u << (bb & 31));
      h0[k] = hsh.first(tv[k]);
      old[k] = atomicCAS(&tab[h0[k]], ReqHash<true>::kEmpty,
                         (static_cast<uint32_t>(tv[k]) << hsh.eb) | (k * kThreads + tid));
    }
    bool rep = false;
#pragma unroll
    for (int k = 0; k < IT; ++k) {
      if (old[k] == ReqHash<true>::kEmpty) continue;  // inserted (or not valid)
      if ((old[k] >> hsh.eb) == static_cast<uint32_t>(tv[k]))
        rep = true;
      else
        rep |= hsh.insert_from(tv[k], k * kThreads + tid, (h0[k] + 1u) & hsh.mask());
    }
    if (rep) misc[kMiscRepeat] = 1;  // a repeated id: resolved below
  } else {
    for (int i = tid; i < K; i += kThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) < lim) {
        const uint32_t bb = bloom_bit(t);
        atomicOr(&bloom[bb >> 5], 1u << (bb & 31));
        if (hsh.insert(t, i)) misc[kMiscRepeat] = 1;  // a repeated id: resolved below
      }
    }
  }
  if (tables) {  // resident ids and ids without a source row are not wanted
    cp_async_wait_all();
    for (int i = tid; i < K; i += kThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) >= lim) continue;
      const int2 e = tbl[i];
      int8_t c = 0;
      int64_t row = -1;
      if (p.res_bt != nullptr && e.x >= 0 && e.x != p.res_null) {
        c = kResident;
        const int32_t off = t - static_cast<int32_t>(div_any(t, p.div_res_bs)) * p.res_bs;
        row = static_cast<int64_t>(e.x) * p.res_bs + off;
      } else if (p.src_bt != nullptr && t != newest) {
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
  if (misc[kMiscRepeat]) {  // rare
    for (int i = tid; i < K; i += kThreads) {
      const int32_t t = ids[i];
      if (static_cast<uint32_t>(t) < lim) hsh.make_min(t, i);
    }
    __syncthreads();
  }

  // Every CTA of the row has staged its state and recorded whether a wait ran
  // out.  Warp 0 reads the peers' outcomes from their shared memory now; the
  // loads complete during the walk.
  cluster_wait();
  int peer_timeout = 0;
  if (C > 1 && warp == 0 && lane < C) peer_timeout = peer_ld(peer_addr(&misc[kMiscTimeout], lane));

  // ---- P2: walk the LRU order; the lowest position holding a wanted token claims it.
  {
    uint32_t bw[IT];
#pragma unroll
    for (int k = 0; k < IT; ++k) bw[k] = ok[k] ? bloom[bloom_bit(tk[k]) >> 5] : 0u;
#pragma unroll
    for (int k = 0; k < IT; ++k) ok[k] = ok[k] && ((bw[k] >> (bloom_bit(tk[k]) & 31)) & 1u);
    if constexpr (kPacked) {  // first probes batched, the rare longer chains after
      uint32_t kv[IT];
#pragma unroll
      for (int k = 0; k < IT; ++k) kv[k] = ok[k] ? tab[hsh.first(tk[k])] : ReqHash<true>::kEmpty;
      const uint32_t emask = (1u << hsh.eb) - 1u;
#pragma unroll
      for (int k = 0; k < IT; ++k) {
        if (!ok[k] || kv[k] == ReqHash<true>::kEmpty) continue;
        if ((kv[k] >> hsh.eb) == static_cast<uint32_t>(tk[k]))
          f[k] = static_cast<int32_t>(kv[k] & emask);
        else
          f[k] = hsh.find_from(tk[k], (hsh.first(tk[k]) + 1u) & hsh.mask());
      }
    } else {
#pragma unroll
      for (int k = 0; k < IT; ++k)
        if (ok[k]) f[k] = hsh.find(tk[k]);
    }
    if (tables) {  // a resident id or one without a source row is not wanted
#pragma unroll
      for (int k = 0; k < IT; ++k)
        if (f[k] >= 0 && code[f[k]] != 0) f[k] = -1;
    }
#pragma unroll
    for (int k = 0; k < IT; ++k)
      if (f[k] >= 0) atomicMin(&claim[f[k]], k * kThreads + tid);
  }
  if (C > 1 && warp == 0) {
    const unsigned any = __ballot_sync(kFullMask, peer_timeout != 0);
    if (lane == 0 && any) misc[kMiscRowTimeout] = 1;
  }
  __syncthreads();
  if (C > 1) {
    // This CTA no longer reads its peers' shared memory: the second cluster
    // barrier, waited on at exit, keeps every CTA alive until all have read.
    cluster_arrive_relaxed();
    if (misc[kMiscRowTimeout]) {  // a wait ran out in another CTA: leave the row alone
      if (j == 0 && tid == 0) {
        if (p.status) p.status[b] = HS_ST_TIMEOUT;
        if (p.miss_count) p.miss_count[b] = 0;
      }
      cluster_wait();
      return;
    }
  }
  // Pool rows of the miss candidates (wanted, not newest, not claimed), loaded
  // with LDGSTS now so the load overlaps P3.
  const bool id_repeat = misc[kMiscRepeat] != 0;
  // (With a source block table prs already holds the translated rows; for a
  // resident entry it holds the resident row.)
  const int64_t* pool_rows_g = p.pool_rows ? p.pool_rows + r * p.pool_rows_stride : nullptr;
  for (int i = tid; i < K; i += kThreads) {
    const int32_t t = ids[i];
    const bool valid = static_cast<uint32_t>(t) < lim;
    const int8_t pre = (tables && valid) ? code[i] : 0;
    if (pre == kResident) continue;
    const bool cand = valid && t != newest && pre == 0 && claim[i] == kUnclaimed &&
                      (!id_repeat || hsh.find(t) == i);
    if (p.src_bt != nullptr) {
      if (!cand) prs[i] = -1;
    } else if (cand && t < p.pool_rows_cols) {
      cp_async_8(&prs[i], pool_rows_g + t);
    } else {
      prs[i] = -1;
    }
  }
  cp_async_commit();

  // ---- P3/P4 counts: hits per chunk of LRU positions, then (once this
  // thread's own pool-row loads have landed) each entry's class and the
  // misses per chunk of entries.  One barrier, then one warp scans each.
  const int chunks_p = (H + 31) / 32;
  bool hit[IT];
  unsigned hm[IT];
  {
    int cl[IT];
#pragma unroll
    for (int k = 0; k < IT; ++k) cl[k] = f[k] >= 0 ? claim[f[k]] : -1;
#pragma unroll
    for (int k = 0; k < IT; ++k) {
      hit[k] = f[k] >= 0 && cl[k] == k * kThreads + tid;
      hm[k] = __ballot_sync(kFullMask, hit[k]);
      if (lane == 0 && k * kThreads + warp * 32 < H) cntp[k * 32 + warp] = __popc(hm[k]);
    }
  }
  // ---- P4: entries in top-k order (a thread reads back only the pool rows
  // its own loads fetched).
  cp_async_wait_all();
  const int chunks_e = (K + 31) / 32;
  for (int base = 0; base < K; base += kThreads) {
    const int i = base + tid;
    bool miss = false;
    if (i < K) {
      const int32_t t = ids[i];
      int8_t c;
      if (static_cast<uint32_t>(t) >= lim) {
        c = kInvalid;
      } else if (id_repeat && hsh.find(t) != i) {
        c = kRepeat;
        my_flags |= HS_ST_DUP_ID;
      } else if (tables && code[i] == kResident) {
        c = kResident;
      } else if (t == newest) {
        c = kNewest;
      } else if (tables && code[i] == kUnmapped) {
        c = kInvalid;  // no source row: like an invalid id
      } else if (claim[i] != kUnclaimed) {
        c = kHit;
      } else {
        const int64_t pr = prs[i];
        if (pr >= 0 && pr < p.pool_num_rows) {
          c = kMiss;
          miss = true;
          if (p.prefetch_rows && i >= e0 && i < e1) {  // in L2 by the time P6 copies it
            bulk_prefetch_l2(p.pool_k + pr * p.row_bytes, static_cast<uint32_t>(p.row_bytes));
            if (p.pool_v != nullptr)
              bulk_prefetch_l2(p.pool_v + pr * p.row_bytes, static_cast<uint32_t>(p.row_bytes));
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
    const int nh = warp_scan_array(cntp, chunks_p, lane);
    if (lane == 0) misc[kMiscHits] = nh;
  } else if (warp == 1) {
    const int nm = warp_scan_array(cnte, chunks_e, lane);
    if (lane == 0) misc[kMiscMisses] = nm;
  }
  __syncthreads();
  // ---- P3: hit ranks in LRU order; evictables compacted in LRU order.
  int hb[IT];  // hits before each of my positions
#pragma unroll
  for (int k = 0; k < IT; ++k) {
    const int q = k * kThreads + tid;
    hb[k] = 0;
    if (q >= H) continue;
    hb[k] = cntp[k * 32 + warp] + __popc(hm[k] & lanes_before);
    if (!hit[k]) {
      const bool corrupt = f[k] == -2;
      if (corrupt) my_flags |= HS_ST_BAD_LRU_SLOT;
      evl[q - hb[k]] = (corrupt ? 0x10000 : 0) | (sl[k] & 0xFFFF);
    }
  }

  __syncthreads();  // the evictables are listed before the misses take them
  const int NH = misc[kMiscHits];
  const int M = misc[kMiscMisses];
  const int E = H - NH;
  const int my_first_miss = e0 < K ? cnte[e0 >> 5] : M;
  // Only my own entries: their chunks are whole and 32-aligned, so a warp's
  // ballot covers one chunk.  A miss's pool row is still in prs.
  for (int base = e0; base < e1; base += kThreads) {
    const int i = base + tid;
    const bool mine = i < e1;
    const int8_t c = mine ? code[i] : kInvalid;
    const unsigned m = __ballot_sync(kFullMask, c == kMiss);
    if (mine && p.miss_mask) p.miss_mask[b * p.mask_stride + i] = c == kMiss;
    if (c == kMiss) {
      const int64_t my_pr = prs[i];
      const int mm = cnte[i >> 5] + __popc(m & lanes_before);  // the row's mm-th miss
      const int32_t e = evl[mm];                               // takes the mm-th evictable
      int32_t d = -1;
      if (!(e >> 16)) {
        const int s = static_cast<int16_t>(e & 0xFFFF);
        const int32_t hr = rows[s];
        if (hr >= 0 && hr < p.hot_num_rows) {
          d = hr;
          tokens_g[s] = ids[i];
        }
      }
      out_g[i] = d;
      jsrc[mm - my_first_miss] = my_pr;
      jdst[mm - my_first_miss] = d;
      if (p.miss_src) {
        p.miss_src[b * p.plan_stride + mm] = my_pr;
        p.miss_dst[b * p.plan_stride + mm] = d;
      }
    } else if (mine) {
      int32_t o = -1;
      if (c == kNewest) o = rows[H];  // the newest token lives in slot H
      if (c == kResident) o = static_cast<int32_t>(prs[i]);
      if (c == kHit) o = rows[lru[claim[i]]];
      out_g[i] = o;
    }
  }
  if (j == 0) {  // the row's status covers every miss's hot row
    for (int mm = tid; mm < M; mm += kThreads) {
      const int32_t e = evl[mm];
      if (e >> 16) continue;
      const int32_t hr = rows[static_cast<int16_t>(e & 0xFFFF)];
      if (hr < 0 || hr >= p.hot_num_rows) my_flags |= HS_ST_BAD_HOT_ROW;
    }
  }

  // ---- P5: my positions' places in the new LRU order.
#pragma unroll
  for (int k = 0; k < IT; ++k) {
    const int q = k * kThreads + tid;
    if (q < p0 || q >= p1) continue;
    int pos;
    if (hit[k]) {
      pos = E + hb[k];
    } else {
      const int e = q - hb[k];
      pos = e >= M ? e - M : E - M + e;
    }
    lru_g[pos] = static_cast<int16_t>(sl[k]);
  }
  if (my_flags) atomicOr(&misc[kMiscFlags], my_flags);
  __syncthreads();
  if (j == 0 && tid == 0) {
    if (p.miss_count) p.miss_count[b] = M;
    if (p.status) p.status[b] = misc[kMiscFlags];
    if (p.stats) {
      atomicAdd(p.stats, static_cast<unsigned long long>(NH));
      atomicAdd(p.stats + 1, static_cast<unsigned long long>(M));
    }
  }

  // ---- P6: copy my misses' rows.
  const int my_m = (e1 < K ? cnte[e1 >> 5] : M) - my_first_miss;
  if (p.copy_width == 16) {
    copy_rows<16>(p, p.pool_k, p.hot_k, my_m, jsrc, jdst);
    if (p.pool_v != nullptr) copy_rows<16>(p, p.pool_v, p.hot_v, my_m, jsrc, jdst);
  } else if (p.copy_width == 4) {
    copy_rows<4>(p, p.pool_k, p.hot_k, my_m, jsrc, jdst);
    if (p.pool_v != nullptr) copy_rows<4>(p, p.pool_v, p.hot_v, my_m, jsrc, jdst);
  } else {
    copy_rows<1>(p, p.pool_k, p.hot_k, my_m, jsrc, jdst);
    if (p.pool_v != nullptr) copy_rows<1>(p, p.pool_v, p.hot_v, my_m, jsrc, jdst);
  }
  if (C > 1) cluster_wait();  // no peer still reads this CTA's shared memory
}

using KernelFn = void (*)(const SwapInParams);

template <bool kTables, bool kPacked>
KernelFn pick_items(int items) {
  switch (items) {
    case 1: return swap_in_kernel<1, kTables, kPacked>;
    case 2: return swap_in_kernel<2, kTables, kPacked>;
    case 4: return swap_in_kernel<4, kTables, kPacked>;
    default: return swap_in_kernel<8, kTables, kPacked>;
  }
}

// Cluster size for a batch: the largest power of two <= 8 with batch * C <=
// SMs (at least 1), raised while the per-CTA state does not fit shared memory.
int pick_cluster(int batch, int K, int H, int bits, const DeviceInfo& dev) {
  int C = 1;
  while (C < kMaxCluster && static_cast<int64_t>(batch) * C * 2 <= dev.sm_count) C *= 2;
  while (C < kMaxCluster && make_layout(K, H, C, bits).total > dev.max_smem_optin) C *= 2;
  return C;
}

}  // namespace
}  // namespace hs

extern "C" int64_t hs_swap_in_smem_bytes(int32_t top_k, int32_t hot_size) {
  if (top_k < 1 || hot_size < 1 || hot_size > 32767 || top_k > hot_size) return 0;
  if (hot_size > hs::kMaxItems * hs::kThreads)  // one CTA per row
    return hs::swap_in_rows_min_smem(top_k, hot_size, false);
  return hs::make_layout(top_k, hot_size, hs::kMaxCluster, hs::hash_bits_for(top_k, 2)).total;
}

namespace hs {
namespace {

// hs_swap_in, with the self-test's forced time-out: fail_rank -1 = none, -2 =
// the last CTA of each row's cluster, else that rank (mod the cluster size).
hs_err swap_in_launch(const hs_swap_in_args* a, hs_stream_t stream, int fail_rank,
                      int fail_wait) {
  bool empty = false;
  hs_err err = check_swap_in_args(a, "hs_swap_in", 32767, &empty);
  if (err != HS_OK || empty) return err;
  if (a->hot_size > kMaxItems * kThreads)  // the one-CTA-per-row kernel takes larger rows
    return swap_in_rows_launch(a, 1, stream, "hs_swap_in", fail_rank == -1 ? -1 : fail_wait);
  SwapInDerived dv;
  err = derive_swap_in(a, "hs_swap_in", &dv);
  if (err != HS_OK) return err;

  DeviceInfo dev;
  err = current_device(&dev);
  if (err != HS_OK) return err;
  // A request hash of >= 8 slots per id in its packed form (load <= 1/8)
  // keeps probe chains short; smaller where shared memory is tight.
  int bits = hash_bits_for(a->top_k, 8);
  int C = pick_cluster(a->batch, a->top_k, a->hot_size, bits, dev);
  for (int mult = 4; mult >= 2 && make_layout(a->top_k, a->hot_size, C, bits).total >
                                       dev.max_smem_optin;
       mult /= 2) {
    bits = hash_bits_for(a->top_k, mult);
    C = pick_cluster(a->batch, a->top_k, a->hot_size, bits, dev);
  }
  const Layout L = make_layout(a->top_k, a->hot_size, C, bits);
  if (L.total > dev.max_smem_optin)
    return fail(HS_ERR_UNSUPPORTED,
                "hs_swap_in: top_k %d / hot_size %d need %d B of shared memory per CTA even "
                "split over %d CTAs, the device allows %d B",
                a->top_k, a->hot_size, L.total, C, dev.max_smem_optin);
  if (static_cast<int64_t>(a->batch) * C > INT32_MAX)
    return fail(HS_ERR_UNSUPPORTED, "hs_swap_in: batch too large");

  SwapInParams p;
  p.top_k = a->top_k;
  p.hot_size = a->hot_size;
  p.cluster = C;
  p.hash_bits = bits;
  p.flags = a->flags;
  p.num_real = a->num_real;
  p.topk_ids = a->topk_ids;
  p.topk_stride = a->topk_stride;
  p.seq_lens = a->seq_lens;
  p.req_state = a->req_state;
  p.num_states = a->num_states;
  p.slot_tokens = a->slot_tokens;
  p.slot_tokens_stride = a->slot_tokens_stride;
  p.slot_rows = a->slot_rows;
  p.slot_rows_stride = a->slot_rows_stride;
  p.lru = a->lru;
  p.lru_stride = a->lru_stride;
  p.pool_rows = a->pool_rows;
  p.pool_rows_stride = a->pool_rows_stride;
  p.pool_rows_cols = a->pool_rows_cols;
  p.pool_k = static_cast<const unsigned char*>(a->pool_k);
  p.pool_v = static_cast<const unsigned char*>(a->pool_v);
  p.pool_num_rows = a->pool_num_rows;
  p.hot_k = static_cast<unsigned char*>(a->hot_k);
  p.hot_v = static_cast<unsigned char*>(a->hot_v);
  p.hot_num_rows = a->hot_num_rows;
  p.row_bytes = a->row_bytes;
  p.out_rows = a->out_rows;
  p.out_stride = a->out_stride;
  p.miss_count = a->miss_count;
  p.stats = a->stats;
  p.status = a->status;
  p.miss_src = a->miss_src;
  p.miss_dst = a->miss_dst;
  p.plan_stride = a->plan_stride;
  p.miss_mask = a->miss_mask;
  p.src_bt = a->src_bt;
  p.src_bt_stride = a->src_bt_stride;
  p.src_bt_blocks = a->src_bt_blocks;
  p.src_bs = a->src_block_size;
  p.res_bt = a->res_bt;
  p.res_bt_stride = a->res_bt_stride;
  p.res_bt_blocks = a->res_bt_blocks;
  p.res_bs = a->res_block_size;
  p.res_null = a->res_null_block;
  p.div_src_bs = dv.div_src_bs;
  p.div_res_bs = dv.div_res_bs;
  p.mask_stride = a->mask_stride;
  p.chunks_per_row = dv.chunks_per_row;
  p.div_chunks = FastDiv{fastdiv_magic(dv.chunks_per_row), dv.chunks_per_row};
  p.lay = L;
  p.entry_bits = dv.entry_bits;
  p.max_seq_len = a->max_seq_len;
  p.copy_width = dv.copy_width;
  p.prefetch_rows = dv.copy_width == 16 && dv.pools_device;
  p.fail_rank = fail_rank == -1 ? -1 : (fail_rank < 0 ? C - 1 : fail_rank % C);
  p.fail_wait = fail_wait;

  int items = 1;
  while (items * kThreads < a->hot_size) items *= 2;
  KernelFn fn = dv.tables ? (dv.packed ? pick_items<true, true>(items) : pick_items<true, false>(items))
                          : (dv.packed ? pick_items<false, true>(items) : pick_items<false, false>(items));
  err = ensure_smem(reinterpret_cast<const void*>(fn), dev.device, L.total);
  if (err != HS_OK) return err;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a->batch) * C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (a->flags & HS_OVERLAP_PREV) ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p);
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "hs_swap_in launch: %s", cudaGetErrorString(e));
  return HS_OK;
}

}  // namespace
}  // namespace hs

namespace hs {

hs_err check_swap_in_args(const hs_swap_in_args* a, const char* who, int max_hot_size,
                          bool* empty) {
  *empty = false;
  if (a == nullptr) return fail(HS_ERR_ARG, "%s: args is NULL", who);
  if (a->batch < 0 || a->top_k < 0)
    return fail(HS_ERR_ARG, "%s: batch (%d) and top_k (%d) must be >= 0", who, a->batch,
                a->top_k);
  if (a->hot_size < 1 || a->hot_size > max_hot_size)
    return fail(HS_ERR_UNSUPPORTED, "%s: hot_size %d outside [1, %d]", who, a->hot_size,
                max_hot_size);
  if (a->top_k > a->hot_size)
    return fail(HS_ERR_UNSUPPORTED, "%s: top_k %d > hot_size %d", who, a->top_k, a->hot_size);
  if (a->row_bytes < 1) return fail(HS_ERR_ARG, "%s: row_bytes must be >= 1", who);
  if (a->flags & ~(HS_SEQ_LENS_I64 | HS_REQ_STATE_I64 | HS_OVERLAP_PREV))
    return fail(HS_ERR_ARG, "%s: unknown flags 0x%x", who, a->flags);
  if (a->batch == 0 || a->top_k == 0) {
    *empty = true;
    return HS_OK;
  }
  const struct {
    const void* p;
    const char* name;
  } required[] = {{a->topk_ids, "topk_ids"},   {a->seq_lens, "seq_lens"},
                  {a->req_state, "req_state"}, {a->slot_tokens, "slot_tokens"},
                  {a->slot_rows, "slot_rows"}, {a->lru, "lru"},
                  {a->pool_k, "pool_k"},       {a->hot_k, "hot_k"},
                  {a->out_rows, "out_rows"}};
  for (const auto& q : required)
    if (q.p == nullptr) return fail(HS_ERR_ARG, "%s: %s is NULL", who, q.name);
  if ((a->pool_v == nullptr) != (a->hot_v == nullptr))
    return fail(HS_ERR_ARG, "%s: pool_v and hot_v must both be set or both be NULL", who);
  const int64_t H = a->hot_size, K = a->top_k;
  if (a->topk_stride < K || a->out_stride < K)
    return fail(HS_ERR_ARG, "%s: topk_stride/out_stride must be >= top_k", who);
  if (a->slot_tokens_stride < H + 1 || a->slot_rows_stride < H + 1)
    return fail(HS_ERR_ARG, "%s: slot strides must be >= hot_size + 1", who);
  if (a->lru_stride < H) return fail(HS_ERR_ARG, "%s: lru_stride must be >= hot_size", who);
  if ((a->miss_src == nullptr) != (a->miss_dst == nullptr))
    return fail(HS_ERR_ARG, "%s: miss_src and miss_dst must both be set or both be NULL", who);
  if (a->miss_src != nullptr && (a->miss_count == nullptr || a->plan_stride < K))
    return fail(HS_ERR_ARG, "%s: the miss plan needs miss_count and plan_stride >= top_k", who);
  if (a->miss_mask != nullptr && a->mask_stride < K)
    return fail(HS_ERR_ARG, "%s: mask_stride must be >= top_k", who);
  if (a->pool_rows == nullptr && a->src_bt == nullptr)
    return fail(HS_ERR_ARG, "%s: pool_rows or src_bt is required", who);
  if (a->src_bt == nullptr &&
      (a->pool_rows_cols < 0 || a->pool_rows_stride < a->pool_rows_cols))
    return fail(HS_ERR_ARG, "%s: need 0 <= pool_rows_cols <= pool_rows_stride", who);
  if (a->src_bt != nullptr &&
      (a->src_block_size < 1 || a->src_bt_blocks < 0 || a->src_bt_stride < a->src_bt_blocks))
    return fail(HS_ERR_ARG, "%s: src_bt needs block size >= 1 and stride >= blocks", who);
  if (a->res_bt != nullptr &&
      (a->res_block_size < 1 || a->res_bt_blocks < 0 || a->res_bt_stride < a->res_bt_blocks))
    return fail(HS_ERR_ARG, "%s: res_bt needs block size >= 1 and stride >= blocks", who);
  if (a->max_seq_len < 0) return fail(HS_ERR_ARG, "%s: max_seq_len must be >= 0", who);
  if (a->num_states < 1 || a->pool_num_rows < 0 || a->hot_num_rows < 0)
    return fail(HS_ERR_ARG, "%s: num_states >= 1, pool/hot row counts >= 0", who);
  if (a->hot_num_rows > INT32_MAX)
    return fail(HS_ERR_UNSUPPORTED, "%s: hot_num_rows must fit int32", who);
  return HS_OK;
}

hs_err derive_swap_in(const hs_swap_in_args* a, const char* who, SwapInDerived* d) {
  const MemKind pk = classify(a->pool_k);
  const MemKind pv = a->pool_v ? classify(a->pool_v) : MemKind::kDevice;
  for (MemKind k : {pk, pv})
    if (k == MemKind::kUnregistered || k == MemKind::kUnknown)
      return fail(HS_ERR_ARG, "%s: pool memory must be device, managed or pinned host memory",
                  who);
  const MemKind hk = classify(a->hot_k);
  const MemKind hv = a->hot_v ? classify(a->hot_v) : MemKind::kDevice;
  for (MemKind k : {hk, hv})
    if (k != MemKind::kDevice && k != MemKind::kManaged)
      return fail(HS_ERR_ARG, "%s: hot buffers must be device memory", who);
  const uintptr_t align = reinterpret_cast<uintptr_t>(a->pool_k) |
                          reinterpret_cast<uintptr_t>(a->hot_k) |
                          reinterpret_cast<uintptr_t>(a->pool_v) |
                          reinterpret_cast<uintptr_t>(a->hot_v) |
                          static_cast<uintptr_t>(a->row_bytes);
  d->copy_width = (align & 15) == 0 ? 16 : ((align & 3) == 0 ? 4 : 1);
  d->pools_device = (pk == MemKind::kDevice || pk == MemKind::kManaged) &&
                    (pv == MemKind::kDevice || pv == MemKind::kManaged);
  const uint64_t cpr = static_cast<uint64_t>(a->row_bytes) / d->copy_width;
  if (cpr * static_cast<uint64_t>(a->top_k) >= (1ull << 32))
    return fail(HS_ERR_UNSUPPORTED, "%s: top_k * row chunks must be < 2^32", who);
  d->chunks_per_row = static_cast<uint32_t>(cpr);
  int eb = 1;  // bits of an entry index (K <= 2^eb)
  while ((1 << eb) < a->top_k) ++eb;
  d->entry_bits = eb;
  // The packed hash needs every valid id (< max_seq_len) below 2^(32 - eb) - 1.
  d->packed = a->max_seq_len > 0 &&
              static_cast<uint64_t>(a->max_seq_len) - 1 < (1ull << (32 - eb)) - 1;
  d->tables = a->src_bt != nullptr || a->res_bt != nullptr;
  const uint32_t sbs = a->src_bt != nullptr ? static_cast<uint32_t>(a->src_block_size) : 1u;
  const uint32_t rbs = a->res_bt != nullptr ? static_cast<uint32_t>(a->res_block_size) : 1u;
  d->div_src_bs = FastDiv{fastdiv_magic(sbs), sbs};
  d->div_res_bs = FastDiv{fastdiv_magic(rbs), rbs};
  return HS_OK;
}

hs_err ensure_smem(const void* fn, int device, int bytes) {
  struct Entry {
    const void* fn;
    int device;
    int bytes;
  };
  static std::mutex mu;
  static Entry table[256];
  static int n = 0;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < n; ++i)
    if (table[i].fn == fn && table[i].device == device) slot = i;
  if (slot >= 0 && table[slot].bytes >= bytes) return HS_OK;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  if (slot >= 0)
    table[slot].bytes = bytes;
  else if (n < 256)
    table[n++] = Entry{fn, device, bytes};
  return HS_OK;
}

}  // namespace hs

extern "C" hs_err hs_swap_in(const hs_swap_in_args* a, hs_stream_t stream) {
  hs::CallRange range("hs_swap_in");
  hs::clear_error();
  return hs::swap_in_launch(a, stream, -1, 0);
}

extern "C" hs_err hs_swap_in_timeout_selftest(const hs_swap_in_args* a, int32_t rank,
                                              int32_t which, hs_stream_t stream) {
  hs::clear_error();
  if (which != 0 && which != 1)
    return hs::fail(HS_ERR_ARG, "hs_swap_in_timeout_selftest: which must be 0 or 1");
  return hs::swap_in_launch(a, stream, rank < 0 ? -2 : rank, which);
}
