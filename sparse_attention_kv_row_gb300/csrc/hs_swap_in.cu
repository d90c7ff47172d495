// hs_swap_in.cu -- the HiSparse decode-time swap-in for sm_103a.
//
// Defined by SGLang jit_kernel/csrc/hisparse.cuh (load_cache_to_device_buffer
// and its kernel) with the invalid-entry rules, padding rows and corruption
// tripwires of vLLM csrc/libtorch_stable/hisparse_kernels.cu
// (hisparse_resolve_residency_kernel).  One CTA owns one batch row:
//
//   A  stage    the row's top-k ids, LRU order, slot tokens and slot rows into
//               shared memory with LDGSTS (coalesced, all in flight at once)
//               instead of one dependent gather per LRU position;
//   B  hash     insert valid ids into an open-addressing table (Knuth
//               multiplicative hash, linear probing, 2K..4K entries); the
//               smallest entry index per id wins (atomicMin), which makes the
//               first occurrence of a repeated id the canonical one;
//   C  walk     every LRU position probes its slot's token; a hit is claimed
//               by the lowest position (atomicMin), and the lowest position of
//               each slot is recorded to catch repeated slots;
//   D  compact  ballot/popc per warp + one warp-wide scan of chunk counts:
//               hits forward, evictables in LRU order;
//   E  misses   candidates in top-k order look up their pool row, then the
//               same ballot/scan assigns the m-th miss the m-th evictable slot;
//   F  write    LRU order [stale evictables][misses][hits], output row,
//               counters;
//   G  copy     (miss, 16-byte chunk) work items spread over all threads of
//               the CTA: read-only no-L1 loads from the pool (HBM or pinned
//               host memory), L2-only stores into the hot buffer.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "hs_device.cuh"
#include "hs_host.h"

namespace hs {
namespace {

constexpr int kThreads = 1024;
constexpr int kCopyUnroll = 4;

struct SwapInLayout {
  int hash_bits, hash_size;
  int o_keys, o_vals, o_ids, o_hitpos, o_out, o_tok, o_rows, o_slotpos, o_found, o_lru,
      o_hits, o_cnt, o_misc;
  int total;
};

__host__ __device__ inline int take(int* o, int bytes) {
  const int r = *o;
  *o += (bytes + 15) & ~15;
  return r;
}

// Shared-memory layout of one row.  After phase C the hash keys hold the
// per-entry pool rows (int64 [K]) and the hash values the per-miss entry index
// (int32 [K]); after phase C the slot-token array holds the evictable list.
__host__ __device__ inline SwapInLayout make_layout(int K, int H) {
  SwapInLayout L;
  int bits = 1;
  while ((1 << bits) < 2 * K) ++bits;
  L.hash_bits = bits;
  L.hash_size = 1 << bits;
  int o = 0;
  L.o_keys = take(&o, 4 * L.hash_size);
  L.o_vals = take(&o, 4 * L.hash_size);
  L.o_ids = take(&o, 4 * K + 16);
  L.o_hitpos = take(&o, 4 * K);
  L.o_out = take(&o, 4 * K);
  L.o_tok = take(&o, 4 * H + 16);
  L.o_rows = take(&o, 4 * (H + 1) + 16);
  L.o_slotpos = take(&o, 4 * H);
  L.o_found = take(&o, 2 * H);
  L.o_lru = take(&o, 2 * H + 16);
  L.o_hits = take(&o, 2 * H);
  const int chunks = ((H > K ? H : K) + 31) / 32;
  L.o_cnt = take(&o, 4 * chunks);
  L.o_misc = take(&o, 16);
  L.total = o;
  return L;
}

struct SwapInParams {
  int32_t top_k, hot_size;
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
  uint32_t chunks_per_row;  // row_bytes / copy width
  FastDiv div_chunks;
};

enum { kMiscFlags = 0, kMiscHits = 1, kMiscMisses = 2 };
constexpr int32_t kWant = INT_MAX;  // hitpos of a wanted, not yet hit entry
constexpr int32_t kDone = -1;       // hitpos of an entry that is never a hit

__device__ __forceinline__ uint32_t hash_of(int32_t key, int bits) {
  return (static_cast<uint32_t>(key) * 2654435761u) >> (32 - bits);
}

// Entry index stored for `key`, or -1 when the key is absent.
__device__ __forceinline__ int32_t hash_find(const int32_t* keys, const int32_t* vals,
                                             int32_t key, int bits) {
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t h = hash_of(key, bits);
  for (uint32_t n = 0; n <= mask; ++n) {
    const int32_t k = keys[h];
    if (k == key) return vals[h];
    if (k == -1) return -1;
    h = (h + 1u) & mask;
  }
  return -1;
}

template <int G>
struct Chunk;
template <>
struct Chunk<16> {
  using T = uint4;
  static __device__ __forceinline__ T ld(const unsigned char* p) { return ld_stream_v4(p); }
  static __device__ __forceinline__ void st(unsigned char* p, T v) { st_l2_v4(p, v); }
};
template <>
struct Chunk<4> {
  using T = uint32_t;
  static __device__ __forceinline__ T ld(const unsigned char* p) { return ld_stream_u32(p); }
  static __device__ __forceinline__ void st(unsigned char* p, T v) { st_l2_u32(p, v); }
};
template <>
struct Chunk<1> {
  using T = uint32_t;
  static __device__ __forceinline__ T ld(const unsigned char* p) { return ld_stream_u8(p); }
  static __device__ __forceinline__ void st(unsigned char* p, T v) { st_l2_u8(p, v); }
};

// Phase G: copy every applied miss row, work item = (miss m, chunk c).
template <int G>
__device__ __forceinline__ void copy_misses(const SwapInParams& p, const unsigned char* pool,
                                            unsigned char* hot, int M, const int32_t* missi,
                                            const int32_t* out_s, const int64_t* pr_s) {
  using C = Chunk<G>;
  const uint32_t cpr = p.chunks_per_row;
  const uint32_t total = static_cast<uint32_t>(M) * cpr;
  for (uint32_t w0 = threadIdx.x; w0 < total; w0 += kThreads * kCopyUnroll) {
    typename C::T v[kCopyUnroll];
    unsigned char* dst[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const uint32_t w = w0 + u * kThreads;
      dst[u] = nullptr;
      if (w < total) {
        const uint32_t m = cpr == 1 ? w : fast_div(w, p.div_chunks);
        const uint32_t c = w - m * cpr;
        const int32_t i = missi[m];
        const int32_t d = out_s[i];
        if (d >= 0) {
          const int64_t off = static_cast<int64_t>(c) * G;
          v[u] = C::ld(pool + pr_s[i] * p.row_bytes + off);
          dst[u] = hot + static_cast<int64_t>(d) * p.row_bytes + off;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (dst[u] != nullptr) C::st(dst[u], v[u]);
  }
}

template <typename SeqT, typename ReqT, int G>
__global__ void __launch_bounds__(kThreads, 1) swap_in_kernel(const SwapInParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int b = blockIdx.x;
  const int K = p.top_k;
  const int H = p.hot_size;
  const SwapInLayout L = make_layout(K, H);
  const unsigned lanes_before = (1u << lane) - 1u;

  // ---- A: stage the top-k row first; it does not depend on the state row.
  const int32_t* ids_g = p.topk_ids + static_cast<int64_t>(b) * p.topk_stride;
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L.o_ids +
                                            (reinterpret_cast<uintptr_t>(ids_g) & 15u));
  stage_bytes(ids, ids_g, 4LL * K, tid, kThreads);

  int32_t* out_g = p.out_rows + static_cast<int64_t>(b) * p.out_stride;
  const bool pad_nr = p.num_real != nullptr && b >= __ldg(p.num_real);
  const int64_t r = static_cast<int64_t>(__ldg(static_cast<const ReqT*>(p.req_state) + b));
  const int64_t Lb = static_cast<int64_t>(__ldg(static_cast<const SeqT*>(p.seq_lens) + b));

  if (pad_nr || r < 0 || r >= p.num_states) {  // padding row / bad state row
    cp_async_commit_wait_all();
    for (int i = tid; i < K; i += kThreads) out_g[i] = -1;
    if (tid == 0) {
      if (p.miss_count) p.miss_count[b] = 0;
      if (p.status) p.status[b] = (pad_nr || r < 0) ? 0 : HS_ST_BAD_STATE;
    }
    return;
  }

  const int32_t* rows_g = p.slot_rows + r * p.slot_rows_stride;
  if (Lb <= H) {  // fast path: the whole sequence sits in the hot buffer in order
    cp_async_commit_wait_all();
    __syncthreads();
    const int64_t count = Lb < K ? Lb : K;
    for (int i = tid; i < K; i += kThreads) {
      const int32_t t = ids[i];
      out_g[i] = (i < count && t >= 0 && t < Lb) ? __ldg(rows_g + t) : -1;
    }
    if (tid == 0) {
      if (p.miss_count) p.miss_count[b] = 0;
      if (p.status) p.status[b] = 0;
    }
    return;
  }

  int32_t* tokens_g = p.slot_tokens + r * p.slot_tokens_stride;
  int16_t* lru_g = p.lru + r * p.lru_stride;
  int32_t* tok = reinterpret_cast<int32_t*>(smem + L.o_tok +
                                            (reinterpret_cast<uintptr_t>(tokens_g) & 15u));
  int32_t* rows = reinterpret_cast<int32_t*>(smem + L.o_rows +
                                             (reinterpret_cast<uintptr_t>(rows_g) & 15u));
  int16_t* lru = reinterpret_cast<int16_t*>(smem + L.o_lru +
                                            (reinterpret_cast<uintptr_t>(lru_g) & 15u));
  stage_bytes(tok, tokens_g, 4LL * H, tid, kThreads);
  stage_bytes(rows, rows_g, 4LL * (H + 1), tid, kThreads);
  stage_bytes(lru, lru_g, 2LL * H, tid, kThreads);

  int32_t* keys = reinterpret_cast<int32_t*>(smem + L.o_keys);
  int32_t* vals = reinterpret_cast<int32_t*>(smem + L.o_vals);
  int32_t* hitpos = reinterpret_cast<int32_t*>(smem + L.o_hitpos);
  int32_t* out_s = reinterpret_cast<int32_t*>(smem + L.o_out);
  int32_t* slotpos = reinterpret_cast<int32_t*>(smem + L.o_slotpos);
  int16_t* found = reinterpret_cast<int16_t*>(smem + L.o_found);
  int16_t* hits = reinterpret_cast<int16_t*>(smem + L.o_hits);
  int32_t* cnt = reinterpret_cast<int32_t*>(smem + L.o_cnt);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.o_misc);
  for (int i = tid; i < L.hash_size; i += kThreads) {
    keys[i] = -1;
    vals[i] = INT_MAX;
  }
  for (int s = tid; s < H; s += kThreads) slotpos[s] = INT_MAX;
  if (tid < 4) misc[tid] = 0;
  cp_async_commit_wait_all();
  __syncthreads();

  // ---- B: hash the valid ids; the smallest entry index per id wins.
  const int bits = L.hash_bits;
  const uint32_t hmask = static_cast<uint32_t>(L.hash_size) - 1u;
  for (int i = tid; i < K; i += kThreads) {
    const int32_t t = ids[i];
    if (t >= 0 && t < Lb) {
      uint32_t h = hash_of(t, bits);
      for (uint32_t n = 0; n <= hmask; ++n) {
        const int32_t old = atomicCAS(&keys[h], -1, t);
        if (old == -1 || old == t) {
          atomicMin(&vals[h], i);
          break;
        }
        h = (h + 1u) & hmask;
      }
    }
  }
  __syncthreads();

  int32_t my_flags = 0;
  for (int i = tid; i < K; i += kThreads) {
    const int32_t t = ids[i];
    int32_t hp = kDone, o = -1;
    if (t >= 0 && t < Lb) {
      if (hash_find(keys, vals, t, bits) != i) {
        my_flags |= HS_ST_DUP_ID;  // a later copy of an id: -1
      } else if (t == Lb - 1) {
        o = rows[H];  // the newest token lives in slot H
      } else {
        hp = kWant;
      }
    }
    hitpos[i] = hp;
    out_s[i] = o;
  }
  __syncthreads();

  // ---- C: walk the LRU order; the lowest position claims each hit and each slot.
  for (int q = tid; q < H; q += kThreads) {
    const int s = lru[q];
    int f = -2;  // -2: slot out of range
    if (s >= 0 && s < H) {
      atomicMin(&slotpos[s], q);
      const int32_t tk = tok[s];
      f = tk >= 0 ? hash_find(keys, vals, tk, bits) : -1;
      if (f >= 0) atomicMin(&hitpos[f], q);
    }
    found[q] = static_cast<int16_t>(f);
  }
  __syncthreads();

  // ---- D: compact positions: hits forward, evictables in LRU order.
  const int pos_chunks = (H + 31) / 32;
  for (int base = 0; base < H; base += kThreads) {
    const int q = base + tid;
    bool hit = false;
    if (q < H) {
      const int f = found[q];
      hit = f >= 0 && hitpos[f] == q;
    }
    const unsigned m = __ballot_sync(kFullMask, hit);
    if (lane == 0 && base + warp * 32 < H) cnt[(base >> 5) + warp] = __popc(m);
  }
  __syncthreads();
  if (warp == 0) {
    const int nh = warp_scan_array(cnt, pos_chunks, lane);
    if (lane == 0) misc[kMiscHits] = nh;
  }
  __syncthreads();
  int32_t* evict = reinterpret_cast<int32_t*>(smem + L.o_tok);  // slot tokens are dead now
  for (int base = 0; base < H; base += kThreads) {
    const int q = base + tid;
    bool hit = false;
    int f = -2;
    if (q < H) {
      f = found[q];
      hit = f >= 0 && hitpos[f] == q;
    }
    const unsigned m = __ballot_sync(kFullMask, hit);
    if (q < H) {
      const int before = cnt[q >> 5] + __popc(m & lanes_before);
      const int s = lru[q];
      if (hit) {
        hits[before] = static_cast<int16_t>(s);
        out_s[f] = rows[s];
      } else {
        const bool bad = (f == -2) || slotpos[s] != q;
        if (bad) my_flags |= HS_ST_BAD_LRU_SLOT;
        evict[q - before] = (bad ? 0x10000 : 0) | (s & 0xFFFF);
      }
    }
  }
  __syncthreads();

  // ---- E: miss candidates in top-k order, pool-row check, slot assignment.
  int64_t* pr_s = reinterpret_cast<int64_t*>(smem + L.o_keys);  // hash is dead now
  int32_t* missi = reinterpret_cast<int32_t*>(smem + L.o_vals);
  const int64_t* pool_rows_g = p.pool_rows + r * p.pool_rows_stride;
  const int ent_chunks = (K + 31) / 32;
  for (int base = 0; base < K; base += kThreads) {
    const int i = base + tid;
    bool miss = false;
    if (i < K) {
      int64_t pr = -1;
      if (hitpos[i] == kWant) {
        const int32_t t = ids[i];
        pr = t < p.pool_rows_cols ? __ldg(pool_rows_g + t) : -1;
        if (pr >= 0 && pr < p.pool_num_rows) {
          miss = true;
        } else {
          pr = -1;
          my_flags |= HS_ST_BAD_POOL_ROW;
        }
      }
      pr_s[i] = pr;
    }
    const unsigned m = __ballot_sync(kFullMask, miss);
    if (lane == 0 && base + warp * 32 < K) cnt[(base >> 5) + warp] = __popc(m);
  }
  __syncthreads();
  if (warp == 0) {
    const int nm = warp_scan_array(cnt, ent_chunks, lane);
    if (lane == 0) misc[kMiscMisses] = nm;
  }
  __syncthreads();
  for (int base = 0; base < K; base += kThreads) {
    const int i = base + tid;
    const bool miss = i < K && pr_s[i] >= 0;
    const unsigned m = __ballot_sync(kFullMask, miss);
    if (miss) {
      const int mm = cnt[i >> 5] + __popc(m & lanes_before);
      missi[mm] = i;
      const int32_t e = evict[mm];
      const int s = static_cast<int16_t>(e & 0xFFFF);
      if (e >> 16) {
        out_s[i] = -1;
        my_flags |= HS_ST_BAD_LRU_SLOT;
      } else {
        const int32_t hr = rows[s];
        if (hr < 0 || hr >= p.hot_num_rows) {
          out_s[i] = -1;
          my_flags |= HS_ST_BAD_HOT_ROW;
        } else {
          out_s[i] = hr;
          tokens_g[s] = ids[i];
        }
      }
    }
  }
  if (my_flags) atomicOr(&misc[kMiscFlags], my_flags);
  __syncthreads();

  // ---- F: LRU writeback, output row, counters.
  const int nh = misc[kMiscHits];
  const int M = misc[kMiscMisses];
  const int E = H - nh;
  for (int q = tid; q < H; q += kThreads) {
    int s;
    if (q < E - M)
      s = static_cast<int16_t>(evict[M + q] & 0xFFFF);
    else if (q < E)
      s = static_cast<int16_t>(evict[q - (E - M)] & 0xFFFF);
    else
      s = hits[q - E];
    lru_g[q] = static_cast<int16_t>(s);
  }
  for (int i = tid; i < K; i += kThreads) out_g[i] = out_s[i];
  if (tid == 0) {
    if (p.miss_count) p.miss_count[b] = M;
    if (p.status) p.status[b] = misc[kMiscFlags];
    if (p.stats) {
      atomicAdd(p.stats, static_cast<unsigned long long>(nh));
      atomicAdd(p.stats + 1, static_cast<unsigned long long>(M));
    }
  }

  // ---- G: copy the missing rows.
  copy_misses<G>(p, p.pool_k, p.hot_k, M, missi, out_s, pr_s);
  if (p.pool_v != nullptr) copy_misses<G>(p, p.pool_v, p.hot_v, M, missi, out_s, pr_s);
}

using KernelFn = void (*)(const SwapInParams);

template <int G>
KernelFn pick_kernel(int flags) {
  const bool s64 = flags & HS_SEQ_LENS_I64, r64 = flags & HS_REQ_STATE_I64;
  if (s64 && r64) return swap_in_kernel<int64_t, int64_t, G>;
  if (s64) return swap_in_kernel<int64_t, int32_t, G>;
  if (r64) return swap_in_kernel<int32_t, int64_t, G>;
  return swap_in_kernel<int32_t, int32_t, G>;
}

// Raises the dynamic shared-memory limit of a kernel once per device to the
// largest size requested so far.
hs_err ensure_smem(KernelFn fn, int device, int bytes) {
  struct Entry {
    KernelFn fn;
    int device;
    int bytes;
  };
  static std::mutex mu;
  static Entry table[128];
  static int n = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i) {
    if (table[i].fn == fn && table[i].device == device) {
      if (table[i].bytes >= bytes) return HS_OK;
      const cudaError_t e =
          cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e != cudaSuccess)
        return fail(HS_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      table[i].bytes = bytes;
      return HS_OK;
    }
  }
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  if (n < 128) table[n++] = Entry{fn, device, bytes};
  return HS_OK;
}

}  // namespace
}  // namespace hs

extern "C" int64_t hs_swap_in_smem_bytes(int32_t top_k, int32_t hot_size) {
  if (top_k < 1 || hot_size < 1 || hot_size > 32767 || top_k > hot_size) return 0;
  return hs::make_layout(top_k, hot_size).total;
}

extern "C" hs_err hs_swap_in(const hs_swap_in_args* a, hs_stream_t stream) {
  using namespace hs;
  clear_error();
  if (a == nullptr) return fail(HS_ERR_ARG, "hs_swap_in: args is NULL");
  if (a->batch < 0 || a->top_k < 0)
    return fail(HS_ERR_ARG, "hs_swap_in: batch (%d) and top_k (%d) must be >= 0", a->batch,
                a->top_k);
  if (a->hot_size < 1 || a->hot_size > 32767)
    return fail(HS_ERR_UNSUPPORTED, "hs_swap_in: hot_size %d outside [1, 32767]", a->hot_size);
  if (a->top_k > a->hot_size)
    return fail(HS_ERR_UNSUPPORTED, "hs_swap_in: top_k %d > hot_size %d", a->top_k,
                a->hot_size);
  if (a->row_bytes < 1) return fail(HS_ERR_ARG, "hs_swap_in: row_bytes must be >= 1");
  if (a->flags & ~(HS_SEQ_LENS_I64 | HS_REQ_STATE_I64))
    return fail(HS_ERR_ARG, "hs_swap_in: unknown flags 0x%x", a->flags);
  if (a->batch == 0 || a->top_k == 0) return HS_OK;

  const struct {
    const void* p;
    const char* name;
  } required[] = {{a->topk_ids, "topk_ids"},   {a->seq_lens, "seq_lens"},
                  {a->req_state, "req_state"}, {a->slot_tokens, "slot_tokens"},
                  {a->slot_rows, "slot_rows"}, {a->lru, "lru"},
                  {a->pool_rows, "pool_rows"}, {a->pool_k, "pool_k"},
                  {a->hot_k, "hot_k"},         {a->out_rows, "out_rows"}};
  for (const auto& q : required)
    if (q.p == nullptr) return fail(HS_ERR_ARG, "hs_swap_in: %s is NULL", q.name);
  if ((a->pool_v == nullptr) != (a->hot_v == nullptr))
    return fail(HS_ERR_ARG, "hs_swap_in: pool_v and hot_v must both be set or both be NULL");
  const int64_t H = a->hot_size, K = a->top_k;
  if (a->topk_stride < K || a->out_stride < K)
    return fail(HS_ERR_ARG, "hs_swap_in: topk_stride/out_stride must be >= top_k");
  if (a->slot_tokens_stride < H + 1 || a->slot_rows_stride < H + 1)
    return fail(HS_ERR_ARG, "hs_swap_in: slot strides must be >= hot_size + 1");
  if (a->lru_stride < H) return fail(HS_ERR_ARG, "hs_swap_in: lru_stride must be >= hot_size");
  if (a->pool_rows_cols < 0 || a->pool_rows_stride < a->pool_rows_cols)
    return fail(HS_ERR_ARG, "hs_swap_in: need 0 <= pool_rows_cols <= pool_rows_stride");
  if (a->num_states < 1 || a->pool_num_rows < 0 || a->hot_num_rows < 0)
    return fail(HS_ERR_ARG, "hs_swap_in: num_states >= 1, pool/hot row counts >= 0");
  if (a->hot_num_rows > INT32_MAX)
    return fail(HS_ERR_UNSUPPORTED, "hs_swap_in: hot_num_rows must fit int32");

  DeviceInfo dev;
  hs_err err = current_device(&dev);
  if (err != HS_OK) return err;
  const SwapInLayout L = make_layout(a->top_k, a->hot_size);
  if (L.total > dev.max_smem_optin)
    return fail(HS_ERR_UNSUPPORTED,
                "hs_swap_in: top_k %d / hot_size %d need %d B of shared memory, the device "
                "allows %d B",
                a->top_k, a->hot_size, L.total, dev.max_smem_optin);

  const MemKind pk = classify(a->pool_k);
  const MemKind pv = a->pool_v ? classify(a->pool_v) : MemKind::kDevice;
  for (MemKind k : {pk, pv})
    if (k == MemKind::kUnregistered || k == MemKind::kUnknown)
      return fail(HS_ERR_ARG,
                  "hs_swap_in: pool memory must be device, managed or pinned host memory");
  const MemKind hk = classify(a->hot_k);
  const MemKind hv = a->hot_v ? classify(a->hot_v) : MemKind::kDevice;
  for (MemKind k : {hk, hv})
    if (k != MemKind::kDevice && k != MemKind::kManaged)
      return fail(HS_ERR_ARG, "hs_swap_in: hot buffers must be device memory");

  const uintptr_t align = reinterpret_cast<uintptr_t>(a->pool_k) |
                          reinterpret_cast<uintptr_t>(a->hot_k) |
                          reinterpret_cast<uintptr_t>(a->pool_v) |
                          reinterpret_cast<uintptr_t>(a->hot_v) |
                          static_cast<uintptr_t>(a->row_bytes);
  const int G = (align & 15) == 0 ? 16 : ((align & 3) == 0 ? 4 : 1);
  const uint64_t cpr = static_cast<uint64_t>(a->row_bytes) / G;
  if (cpr * static_cast<uint64_t>(K) >= (1ull << 32))
    return fail(HS_ERR_UNSUPPORTED, "hs_swap_in: top_k * row chunks must be < 2^32");

  SwapInParams p;
  p.top_k = a->top_k;
  p.hot_size = a->hot_size;
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
  p.chunks_per_row = static_cast<uint32_t>(cpr);
  p.div_chunks = FastDiv{fastdiv_magic(static_cast<uint32_t>(cpr)), static_cast<uint32_t>(cpr)};

  KernelFn fn = G == 16 ? pick_kernel<16>(a->flags)
                        : (G == 4 ? pick_kernel<4>(a->flags) : pick_kernel<1>(a->flags));
  err = ensure_smem(fn, dev.device, L.total);
  if (err != HS_OK) return err;
  fn<<<a->batch, kThreads, L.total, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "hs_swap_in launch: %s", cudaGetErrorString(e));
  return HS_OK;
}
