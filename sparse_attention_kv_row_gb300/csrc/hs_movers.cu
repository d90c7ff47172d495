// hs_movers.cu -- indexed KV-row movers for sm_103a, plus a streaming-read
// bandwidth probe.
//
//  store_kv   tokenspeed tokenspeed_kernel/ops/kvcache/triton.py, store_kv_cache:
//             k_dst[loc[t]] = k_src[t], v_dst[loc[t]] = v_src[t].
//  gather     vLLM csrc/libtorch_stable/hisparse_kernels.cu, hisparse_gather_plan_kernel /
//             hisparse_gather_compact_kernel: a resolving layer's miss plan replayed
//             onto a layer that shares its indices.
//  invalidate vLLM csrc/libtorch_stable/hisparse_kernels.cu,
//             hisparse_invalidate_written_slots_kernel: resident copies of
//             rewritten tokens are dropped from the slot-token table.
//  transfer   tokenspeed ... transfer_kv_per_layer(_mla) / transfer_kv_all_layer(_mla)
//             and SGLang jit_kernel/csrc/hisparse.cuh, transfer_cache_dsv4_mla_kernel:
//             for each index pair, the same row of every layer's cache.
//
// Work is flattened into (row) units -- (token, K|V) for store_kv and
// (pair, layer) for transfer, pair-major like the pages.  The register mover
// spreads one warp per unit over a persistent grid sized to the SM count; a
// warp moves its row in 16-byte chunks when source, destination and size
// allow it, else in 4-byte words, else bytes, with up to four chunks per lane
// in flight.  A transfer whose sources the caller declares device memory, with
// 16-byte row pitches and sizes, uses the bulk (TMA) mover instead: one
// thread per row in flight, global -> shared -> global (measured 61 % of HBM
// against 55 % for the register mover on the 61-layer transfer; the register
// mover stays for store_kv, where it was the faster of the two).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hs_device.cuh"
#include "hs_host.h"
#include "hs_swap_in_common.cuh"

namespace hs {
namespace {

constexpr int kMoverThreads = 256;
constexpr int kMoverBlocksPerSm = 8;
constexpr int kUnroll = 4;

// Copies `bytes` bytes from src to dst with one warp, choosing the widest chunk
// that all three of (src, dst, bytes) allow.  Stores are evict-first, or kept
// in L2 (kKeepL2) for rows an attention kernel reads next.
template <bool kKeepL2 = false>
__device__ __forceinline__ void warp_copy_row(unsigned char* dst, const unsigned char* src,
                                              int64_t bytes, int lane) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                       static_cast<uintptr_t>(bytes);
  if ((al & 15) == 0) {
    const int64_t n = bytes >> 4;
    for (int64_t c0 = lane; c0 < n; c0 += kWarp * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + u * kWarp;
        if (c < n) v[u] = ld_stream_v4(src + (c << 4));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + u * kWarp;
        if (c < n) {
          if (kKeepL2)
            st_l2_v4(dst + (c << 4), v[u]);
          else
            st_stream_v4(dst + (c << 4), v[u]);
        }
      }
    }
  } else if ((al & 3) == 0) {
    const int64_t n = bytes >> 2;
    for (int64_t c0 = lane; c0 < n; c0 += kWarp * kUnroll) {
      uint32_t v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + u * kWarp;
        if (c < n) v[u] = ld_stream_u32(src + (c << 2));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + u * kWarp;
        if (c < n) {
          if (kKeepL2)
            st_l2_u32(dst + (c << 2), v[u]);
          else
            st_stream_u32(dst + (c << 2), v[u]);
        }
      }
    }
  } else {
    for (int64_t c0 = lane; c0 < bytes; c0 += kWarp * kUnroll) {
      uint32_t v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + u * kWarp;
        if (c < bytes) v[u] = ld_stream_u8(src + c);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + u * kWarp;
        if (c < bytes) {
          if (kKeepL2)
            st_l2_u8(dst + c, v[u]);
          else
            st_stream_u8(dst + c, v[u]);
        }
      }
    }
  }
}

struct StoreKvParams {
  const unsigned char* k_src;
  const unsigned char* v_src;
  int64_t src_k_stride, src_v_stride;
  unsigned char* k_dst;
  unsigned char* v_dst;
  int64_t dst_stride, dst_rows;
  const int64_t* loc;
  int64_t n_tokens, row_bytes;
  int32_t* status;
};

// ------------------------------------------------------------------ bulk (TMA) mover
// For rows whose addresses and size are multiples of 16 bytes.  Thread t of a
// CTA owns slot t (row_bytes of shared memory) and mbarrier t and moves units
// u = blockIdx.x * blockDim.x + t, += gridDim.x * blockDim.x, one at a time:
// one bulk load global -> slot completed on the mbarrier (a bounded wait),
// then one bulk store slot -> global, which has read the slot before the
// slot's next load.  A thread issues a few instructions per row, and an SM
// holds ~190 KB of rows in flight.
constexpr int kBulkSmemTarget = 96 * 1024;  // shared memory per CTA, about
constexpr uint32_t kMoverPolls = 1u << 22;

__host__ __device__ inline int bulk_slots_offset(int threads) { return (threads * 8 + 15) & ~15; }

template <class Unit>
__device__ __forceinline__ void bulk_move(const Unit& unit, uint64_t units, uint32_t bytes,
                                          int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int t = threadIdx.x;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem) + t;
  unsigned char* slot = smem + bulk_slots_offset(blockDim.x) + static_cast<uint32_t>(t) * bytes;
  mbar_init(bar, 1);
  fence_mbar_init();
  uint32_t parity = 0;
  bool stored = false;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * blockDim.x + t;
  const unsigned char* src = nullptr;
  unsigned char* dst = nullptr;
  bool ok = u < units && unit(u, &src, &dst);
  while (u < units) {
    bool loading = false;
    if (ok) {
      const uintptr_t al = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
      if ((al & 15) != 0) {  // a layer base off 16 bytes: this row by words or bytes
        if ((al & 3) == 0) {
          for (uint32_t o = 0; o < bytes; o += 4) st_stream_u32(dst + o, ld_stream_u32(src + o));
        } else {
          for (uint32_t o = 0; o < bytes; ++o) st_stream_u8(dst + o, ld_stream_u8(src + o));
        }
      } else {
        if (stored) bulk_wait_read_all();
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(slot, src, bytes, bar);
        loading = true;
      }
    }
    // The next row's indices and addresses load while this row is in flight.
    const uint64_t nu = u + stride;
    const unsigned char* nsrc = nullptr;
    unsigned char* ndst = nullptr;
    const bool nok = nu < units && unit(nu, &nsrc, &ndst);
    if (loading) {
      if (!mbar_wait(bar, parity, kMoverPolls)) {
        if (status) atomicOr(status, HS_ST_TIMEOUT);
        mbar_wait(bar, parity, kMoverPolls, 16000000000ull);  // wait out the load in flight
        break;
      }
      parity ^= 1u;
      bulk_store(dst, slot, bytes);
      bulk_commit();
      stored = true;
    }
    u = nu;
    src = nsrc;
    dst = ndst;
    ok = nok;
  }
  if (stored) bulk_wait_read_all();  // every slot is read before shared memory is released
}

__global__ void __launch_bounds__(kMoverThreads) store_kv_kernel(const StoreKvParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kMoverThreads / kWarp);
  const int kv = p.v_src != nullptr ? 2 : 1;
  const int64_t units = p.n_tokens * kv;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * (kMoverThreads / kWarp) +
                   (threadIdx.x >> 5);
       u < units; u += warps) {
    const int64_t t = kv == 2 ? (u >> 1) : u;
    const bool is_v = kv == 2 && (u & 1);
    const int64_t d = __ldg(p.loc + t);
    if (d < 0 || d >= p.dst_rows) {
      if (lane == 0 && !is_v && p.status) atomicOr(p.status, HS_ST_BAD_INDEX);
      continue;
    }
    const unsigned char* src = is_v ? p.v_src + t * p.src_v_stride : p.k_src + t * p.src_k_stride;
    unsigned char* dst = (is_v ? p.v_dst : p.k_dst) + d * p.dst_stride;
    warp_copy_row(dst, src, p.row_bytes, lane);
  }
}

// Rows of 16-byte chunks, at most 512 * U bytes, every base and stride a
// multiple of 16 (the common KV layout).  One warp per unit; a lane's U chunks
// are loaded together with the unit's destination index -- the source row of
// token t is always in range, so its loads do not wait for the index check --
// which makes a unit one memory round trip instead of two.  At 32 registers 64
// warps fit on an SM, so a decode step's K+V scatter is in flight at once.
template <int U>
__global__ void __launch_bounds__(kMoverThreads, 8) store_kv_vec_kernel(const StoreKvParams p) {
  const int lane = threadIdx.x & 31;
  const bool has_v = p.v_src != nullptr;
  // Loop bounds re-read from the parameters and gridDim, not held in registers.
  for (uint32_t u = blockIdx.x * (kMoverThreads / kWarp) + (threadIdx.x >> 5);
       u < (static_cast<uint32_t>(p.n_tokens) << (has_v ? 1 : 0));  // < 2^31
       u += gridDim.x * (kMoverThreads / kWarp)) {
    const int left = static_cast<int>(p.row_bytes >> 4) - lane;  // lane's chunks: 32 * k < left
    const uint32_t t = has_v ? (u >> 1) : u;
    const bool is_v = has_v && (u & 1);
    const int64_t d = __ldg(p.loc + t);
    const unsigned char* src =
        (is_v ? p.v_src + t * p.src_v_stride : p.k_src + t * p.src_k_stride) + (lane << 4);
    uint4 v[U];
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (32 * k < left) v[k] = ld_stream_v4(src + 512 * k);
    if (d < 0 || d >= p.dst_rows) {
      if (lane == 0 && !is_v && p.status) atomicOr(p.status, HS_ST_BAD_INDEX);
      continue;
    }
    unsigned char* dst = (is_v ? p.v_dst : p.k_dst) + d * p.dst_stride + (lane << 4);
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (32 * k < left) st_stream_v4(dst + 512 * k, v[k]);
  }
}

struct TransferParams {
  const uint64_t* src_ptrs;
  const uint64_t* dst_ptrs;
  const int64_t* src_idx;
  const int64_t* dst_idx;
  int64_t pair_begin;      // first pair of this launch
  uint32_t units;          // pairs_in_launch * ptr_pairs  (< 2^32)
  uint32_t ptr_pairs;      // num_layers * (1 + has_v)
  FastDiv div_ptr_pairs;
  uint32_t pairs;          // pairs in this launch (bulk path: units are layer-major)
  FastDiv div_pairs;
  int64_t src_stride, dst_stride, src_rows, dst_rows, row_bytes;
  int32_t* status;
};

__global__ void __launch_bounds__(kMoverThreads) transfer_kernel(const TransferParams p) {
  const int lane = threadIdx.x & 31;
  const uint32_t warps = gridDim.x * (kMoverThreads / kWarp);
  for (uint32_t u = blockIdx.x * (kMoverThreads / kWarp) + (threadIdx.x >> 5); u < p.units;
       u += warps) {
    const uint32_t pair = p.ptr_pairs == 1 ? u : fast_div(u, p.div_ptr_pairs);
    const uint32_t layer = u - pair * p.ptr_pairs;
    const int64_t n = p.pair_begin + pair;
    const int64_t s = __ldg(p.src_idx + n);
    const int64_t d = __ldg(p.dst_idx + n);
    if (s < 0 || s >= p.src_rows || d < 0 || d >= p.dst_rows) {
      if (lane == 0 && layer == 0 && p.status) atomicOr(p.status, HS_ST_BAD_INDEX);
      continue;
    }
    const unsigned char* src =
        reinterpret_cast<const unsigned char*>(__ldg(p.src_ptrs + layer)) + s * p.src_stride;
    unsigned char* dst =
        reinterpret_cast<unsigned char*>(__ldg(p.dst_ptrs + layer)) + d * p.dst_stride;
    warp_copy_row(dst, src, p.row_bytes, lane);
  }
}

// Units of the bulk path are layer-major (u = pointer pair * pairs + pair):
// the rows in flight at any moment lie in one or two layers' buffers, not in
// every layer's, which spares the address translation caches.  Rows are
// independent, so the order is free.
struct TransferUnit {
  const TransferParams* p;
  __device__ __forceinline__ bool operator()(uint64_t u32, const unsigned char** src,
                                             unsigned char** dst) const {
    const uint32_t u = static_cast<uint32_t>(u32);
    const uint32_t layer = p->ptr_pairs == 1 ? 0u : div_any(u, p->div_pairs);
    const uint32_t pair = u - layer * p->pairs;
    const int64_t n = p->pair_begin + pair;
    const int64_t s = __ldg(p->src_idx + n);
    const int64_t d = __ldg(p->dst_idx + n);
    if (s < 0 || s >= p->src_rows || d < 0 || d >= p->dst_rows) {
      if (layer == 0 && p->status) atomicOr(p->status, HS_ST_BAD_INDEX);
      return false;
    }
    *src = reinterpret_cast<const unsigned char*>(__ldg(p->src_ptrs + layer)) + s * p->src_stride;
    *dst = reinterpret_cast<unsigned char*>(__ldg(p->dst_ptrs + layer)) + d * p->dst_stride;
    return true;
  }
};

__global__ void transfer_bulk_kernel(const TransferParams p) {
  bulk_move(TransferUnit{&p}, p.units, static_cast<uint32_t>(p.row_bytes), p.status);
}

struct GatherParams {
  const uint64_t* pool_ptrs;
  const uint64_t* hot_ptrs;
  uint32_t ptr_pairs;  // num_layers * (1 + has_v)
  int64_t pool_rows, hot_rows, row_bytes;
  const int64_t* miss_src;
  const int32_t* miss_dst;
  int64_t plan_stride;
  const int32_t* miss_count;
  int32_t top_k;
  int32_t* status;
  uint32_t chunks16;   // row_bytes / 16 when row_bytes is a multiple of 16, else 0
  FastDiv div_chunks16;
  FastDiv div_ptr_pairs;
  int32_t overlap;     // launched with programmatic stream serialization
};

constexpr int kGatherUnits = 256;  // (miss, pointer pair) units a block stages per round
constexpr int kGatherBlocksPerSm = 4;  // resident blocks of the replay (<= 64 registers)
constexpr int kGatherUnroll = 6;       // 16-byte chunks in flight per thread

// Block (row, y) replays misses [y*mb, (y+1)*mb) of its row, mb = ceil(n /
// gridDim.y): units u = (miss - first miss) * ptr_pairs + pointer pair, in
// rounds of kGatherUnits.  A round first stages each unit's source and
// destination row addresses in shared memory (its plan entries and layer
// pointers are independent loads: one round trip), then copies them: as flat
// (unit, 16-byte chunk) items, kGatherUnroll per thread with all loads before
// the stores, when every staged unit is 16-byte aligned; else one warp per unit.
__global__ void __launch_bounds__(kMoverThreads, kGatherBlocksPerSm)
    gather_misses_kernel(const GatherParams p) {
  constexpr int W = kMoverThreads / kWarp;
  __shared__ const unsigned char* s_src[kGatherUnits];
  __shared__ unsigned char* s_dst[kGatherUnits];
  // The next launch may start now: it reads nothing this kernel writes before
  // its own grid-dependency wait.
  grid_dep_launch_dependents();
  if (p.overlap) grid_dep_wait();  // the plan may come from the kernel before this one
  // The plan and the counts are read through L2 (ld.global.cg), not the
  // read-only path: with early start the swap-in that writes them is still
  // running when this grid begins, so they are not read-only for its lifetime.
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  int n = __ldcg(p.miss_count + row);
  n = n < 0 ? 0 : (n > p.top_k ? p.top_k : n);
  const uint32_t mb = (static_cast<uint32_t>(n) + gridDim.y - 1) / gridDim.y;
  const uint32_t m0 = blockIdx.y * mb;
  const uint32_t m1 = m0 + mb < static_cast<uint32_t>(n) ? m0 + mb : static_cast<uint32_t>(n);
  const uint32_t units = m1 > m0 ? (m1 - m0) * p.ptr_pairs : 0u;
  const int64_t* src_g = p.miss_src + row * p.plan_stride;
  const int32_t* dst_g = p.miss_dst + row * p.plan_stride;
  for (uint32_t u0 = 0; u0 < units; u0 += kGatherUnits) {
    const int nu = units - u0 < kGatherUnits ? static_cast<int>(units - u0) : kGatherUnits;
    __syncthreads();  // the previous round's copies are done with the staged units
    bool misaligned = false;
    if (tid < nu) {
      const uint32_t u = u0 + tid;
      const uint32_t k = p.ptr_pairs == 1 ? u : fast_div(u, p.div_ptr_pairs);
      const uint32_t pp = u - k * p.ptr_pairs;
      const int32_t d = __ldcg(dst_g + m0 + k);
      const int64_t sr = __ldcg(reinterpret_cast<const long long*>(src_g) + m0 + k);
      const uintptr_t pool = static_cast<uintptr_t>(__ldg(p.pool_ptrs + pp));
      const uintptr_t hot = static_cast<uintptr_t>(__ldg(p.hot_ptrs + pp));
      const unsigned char* from = nullptr;
      unsigned char* to = nullptr;
      if (d >= 0) {  // a miss given no hot row is skipped
        if (sr < 0 || sr >= p.pool_rows || d >= p.hot_rows) {
          if (pp == 0 && p.status) atomicOr(p.status, HS_ST_BAD_INDEX);
        } else {
          from = reinterpret_cast<const unsigned char*>(pool) + sr * p.row_bytes;
          to = reinterpret_cast<unsigned char*>(hot) + static_cast<int64_t>(d) * p.row_bytes;
          misaligned = ((reinterpret_cast<uintptr_t>(from) | reinterpret_cast<uintptr_t>(to)) & 15) != 0;
        }
      }
      s_src[tid] = from;
      s_dst[tid] = to;
    }
    // The staged units are visible to all, and every thread takes the same path.
    const bool any_misaligned = __syncthreads_or(misaligned) != 0;
    if (p.chunks16 != 0 && !any_misaligned) {
      const uint32_t items = static_cast<uint32_t>(nu) * p.chunks16;
      // An item in flight holds its data and its unit; the destination is
      // recomputed for the store, which keeps registers for more items.
      for (uint32_t w0 = tid; w0 < items; w0 += kMoverThreads * kGatherUnroll) {
        uint4 v[kGatherUnroll];
        uint32_t unit[kGatherUnroll];
#pragma unroll
        for (int j = 0; j < kGatherUnroll; ++j) {
          const uint32_t w = w0 + j * kMoverThreads;
          unit[j] = kGatherUnits;  // none
          if (w < items) {
            const uint32_t k = fast_div(w, p.div_chunks16);
            const unsigned char* from = s_src[k];
            if (from != nullptr) {
              v[j] = ld_stream_v4(from + ((w - k * p.chunks16) << 4));
              unit[j] = k;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kGatherUnroll; ++j) {
          const uint32_t k = unit[j];
          if (k == kGatherUnits) continue;
          const uint32_t w = w0 + j * kMoverThreads;
          st_l2_v4(s_dst[k] + ((w - k * p.chunks16) << 4), v[j]);
        }
      }
    } else {
      for (int k = tid >> 5; k < nu; k += W)
        if (s_src[k] != nullptr) warp_copy_row<true>(s_dst[k], s_src[k], p.row_bytes, tid & 31);
    }
  }
}

// Block (token q, chunk c) scans slots [c * kInvSlots, (c + 1) * kInvSlots) of
// token q's state row: each thread loads its kInvPer slots first, then clears
// the ones that hold the token, so a block costs one memory round trip.
constexpr int kInvThreads = 256;
constexpr int kInvPer = 4;
constexpr int kInvSlots = kInvThreads * kInvPer;
__global__ void __launch_bounds__(kInvThreads) invalidate_kernel(int32_t* slot_tokens, int64_t stride,
                                                                 int32_t hot_size, int64_t num_states,
                                                                 const int64_t* state_rows,
                                                                 const int32_t* tokens,
                                                                 int32_t* status, int32_t chunks) {
  const int64_t q = blockIdx.x / chunks;
  const int64_t c = blockIdx.x - q * chunks;
  const int64_t r = __ldg(state_rows + q);
  const int32_t t = __ldg(tokens + q);
  if (r < 0 || t < 0) return;
  if (r >= num_states) {
    if (c == 0 && threadIdx.x == 0 && status) atomicOr(status, HS_ST_BAD_INDEX);
    return;
  }
  int32_t* row = slot_tokens + r * stride;
  const int64_t s0 = c * kInvSlots + threadIdx.x;
  int32_t v[kInvPer];
#pragma unroll
  for (int u = 0; u < kInvPer; ++u) {
    const int64_t s = s0 + u * kInvThreads;
    v[u] = s < hot_size ? row[s] : -1;
  }
#pragma unroll
  for (int u = 0; u < kInvPer; ++u) {
    const int64_t s = s0 + u * kInvThreads;
    if (s < hot_size && v[u] == t) row[s] = -1;
  }
}

// The bounded wait of the swap-in's staging, run on an mbarrier that nothing
// arms: thread 0 initialises it and polls at most max_polls times, and the
// block reports the wait that ran out.  No copy is in flight on the barrier.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t max_polls, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, max_polls)) atomicOr(status, HS_ST_TIMEOUT);
}

__global__ void __launch_bounds__(512) probe_read_kernel(const uint4* src, int64_t n16,
                                                         unsigned long long* sink) {
  uint32_t acc = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream_v4(src + i);
    const uint4 b = ld_stream_v4(src + i + stride);
    const uint4 c = ld_stream_v4(src + i + 2 * stride);
    const uint4 d = ld_stream_v4(src + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^
           d.z ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = ld_stream_v4(src + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(kFullMask, acc, o);
  if ((threadIdx.x & 31) == 0 && acc != 0) atomicXor(sink, static_cast<unsigned long long>(acc));
}

// Threads (= slots) per CTA of a bulk mover for rows of `bytes`, and its
// shared memory; 0 threads when rows that large do not suit it.
int bulk_threads(int64_t bytes) {
  if (bytes < 16 || bytes > 16384 || bytes % 16 != 0) return 0;
  int t = static_cast<int>(kBulkSmemTarget / (bytes + 8));
  t = t < 32 ? 32 : (t > 512 ? 512 : t);
  return t & ~31;
}

template <class Params>
hs_err launch_bulk(void (*kernel)(Params), const Params& p, int64_t units, int64_t bytes,
                   const DeviceInfo& dev, hs_stream_t stream, const char* who) {
  const int threads = bulk_threads(bytes);
  const int smem = bulk_slots_offset(threads) + threads * static_cast<int>(bytes);
  hs_err err = ensure_smem(reinterpret_cast<const void*>(kernel), dev.device, smem);
  if (err != HS_OK) return err;
  // CTAs per SM for this (kernel, row size), queried once per device.
  static std::mutex mu;
  static struct { const void* fn; int device, bytes, per_sm; } seen[32];
  static int n_seen = 0;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_seen; ++i)
      if (seen[i].fn == reinterpret_cast<const void*>(kernel) && seen[i].device == dev.device &&
          seen[i].bytes == bytes)
        per_sm = seen[i].per_sm;
  }
  cudaError_t e = cudaSuccess;
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (e != cudaSuccess)
      return fail(HS_ERR_CUDA, "%s: occupancy query: %s", who, cudaGetErrorString(e));
    if (per_sm < 1) per_sm = 1;
    std::lock_guard<std::mutex> lock(mu);
    if (n_seen < 32)
      seen[n_seen++] = {reinterpret_cast<const void*>(kernel), dev.device,
                        static_cast<int>(bytes), per_sm};
  }
  int64_t grid = static_cast<int64_t>(dev.sm_count) * per_sm;
  const int64_t need = (units + threads - 1) / threads;
  if (grid > need) grid = need;
  kernel<<<static_cast<unsigned>(grid), threads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "%s launch: %s", who, cudaGetErrorString(e));
  return HS_OK;
}

int mover_grid(const DeviceInfo& dev, int64_t units) {
  const int64_t warps_per_block = kMoverThreads / kWarp;
  int64_t blocks = (units + warps_per_block - 1) / warps_per_block;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * kMoverBlocksPerSm;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

}  // namespace
}  // namespace hs

extern "C" hs_err hs_store_kv(const void* k_src, const void* v_src, int64_t src_k_stride,
                              int64_t src_v_stride, void* k_dst, void* v_dst, int64_t dst_stride,
                              int64_t dst_rows, const int64_t* loc, int64_t n_tokens,
                              int64_t row_bytes, int32_t* status, hs_stream_t stream) {
  hs::CallRange range("hs_store_kv");
  using namespace hs;
  clear_error();
  if (n_tokens < 0 || row_bytes < 1 || dst_rows < 0)
    return fail(HS_ERR_ARG, "hs_store_kv: need n_tokens >= 0, row_bytes >= 1, dst_rows >= 0");
  if (n_tokens == 0) return HS_OK;
  if (k_src == nullptr || k_dst == nullptr || loc == nullptr)
    return fail(HS_ERR_ARG, "hs_store_kv: k_src, k_dst and loc are required");
  if ((v_src == nullptr) != (v_dst == nullptr))
    return fail(HS_ERR_ARG, "hs_store_kv: v_src and v_dst must both be set or both be NULL");
  if (src_k_stride < row_bytes || dst_stride < row_bytes ||
      (v_src != nullptr && src_v_stride < row_bytes))
    return fail(HS_ERR_ARG, "hs_store_kv: strides must be >= row_bytes");
  DeviceInfo dev;
  hs_err err = current_device(&dev);
  if (err != HS_OK) return err;
  StoreKvParams p{static_cast<const unsigned char*>(k_src),
                  static_cast<const unsigned char*>(v_src),
                  src_k_stride,
                  src_v_stride,
                  static_cast<unsigned char*>(k_dst),
                  static_cast<unsigned char*>(v_dst),
                  dst_stride,
                  dst_rows,
                  loc,
                  n_tokens,
                  row_bytes,
                  status};
  const int64_t units = n_tokens * (v_src != nullptr ? 2 : 1);
  const uintptr_t al = reinterpret_cast<uintptr_t>(k_src) | reinterpret_cast<uintptr_t>(v_src) |
                       reinterpret_cast<uintptr_t>(k_dst) | reinterpret_cast<uintptr_t>(v_dst) |
                       static_cast<uintptr_t>(src_k_stride) |
                       static_cast<uintptr_t>(v_src != nullptr ? src_v_stride : 0) |
                       static_cast<uintptr_t>(dst_stride) | static_cast<uintptr_t>(row_bytes);
  const int grid = mover_grid(dev, units);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool vec = (al & 15) == 0 && units < (int64_t{1} << 31);
  if (vec && row_bytes <= 512)
    store_kv_vec_kernel<1><<<grid, kMoverThreads, 0, st>>>(p);
  else if (vec && row_bytes <= 1024)
    store_kv_vec_kernel<2><<<grid, kMoverThreads, 0, st>>>(p);
  else if (vec && row_bytes <= 2048)
    store_kv_vec_kernel<4><<<grid, kMoverThreads, 0, st>>>(p);
  else
    store_kv_kernel<<<grid, kMoverThreads, 0, st>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "hs_store_kv launch: %s", cudaGetErrorString(e));
  return HS_OK;
}

extern "C" hs_err hs_transfer_kv(const uint64_t* src_ptrs, const uint64_t* dst_ptrs,
                                 int32_t num_layers, int32_t has_v, const int64_t* src_idx,
                                 const int64_t* dst_idx, int64_t n, int64_t src_stride,
                                 int64_t dst_stride, int64_t src_rows, int64_t dst_rows,
                                 int64_t row_bytes, int32_t* status, hs_stream_t stream) {
  hs::CallRange range("hs_transfer_kv");
  using namespace hs;
  clear_error();
  if (n < 0 || num_layers < 0 || row_bytes < 1 || src_rows < 0 || dst_rows < 0)
    return fail(HS_ERR_ARG, "hs_transfer_kv: negative size or row_bytes < 1");
  if (has_v & ~(HS_XFER_HAS_V | HS_XFER_DEVICE_SOURCES))
    return fail(HS_ERR_ARG, "hs_transfer_kv: unknown flags 0x%x", has_v);
  const bool device_src = (has_v & HS_XFER_DEVICE_SOURCES) != 0;
  has_v &= HS_XFER_HAS_V;
  if (n == 0 || num_layers == 0) return HS_OK;
  if (src_ptrs == nullptr || dst_ptrs == nullptr || src_idx == nullptr || dst_idx == nullptr)
    return fail(HS_ERR_ARG, "hs_transfer_kv: pointer arrays and index arrays are required");
  if (src_stride < row_bytes || dst_stride < row_bytes)
    return fail(HS_ERR_ARG, "hs_transfer_kv: strides must be >= row_bytes");
  DeviceInfo dev;
  hs_err err = current_device(&dev);
  if (err != HS_OK) return err;
  const uint32_t ptr_pairs = static_cast<uint32_t>(num_layers) * (has_v ? 2u : 1u);
  // Units are 32-bit: launch at most floor((2^32 - 1) / ptr_pairs) pairs at a time.
  const int64_t max_pairs = static_cast<int64_t>(0xFFFFFFFFull / ptr_pairs);
  for (int64_t begin = 0; begin < n; begin += max_pairs) {
    const int64_t pairs = (n - begin) < max_pairs ? (n - begin) : max_pairs;
    TransferParams p;
    p.src_ptrs = src_ptrs;
    p.dst_ptrs = dst_ptrs;
    p.src_idx = src_idx;
    p.dst_idx = dst_idx;
    p.pair_begin = begin;
    p.units = static_cast<uint32_t>(pairs * ptr_pairs);
    p.ptr_pairs = ptr_pairs;
    p.div_ptr_pairs = FastDiv{fastdiv_magic(ptr_pairs), ptr_pairs};
    p.pairs = static_cast<uint32_t>(pairs);
    p.div_pairs = FastDiv{fastdiv_magic(p.pairs), p.pairs};
    p.src_stride = src_stride;
    p.dst_stride = dst_stride;
    p.src_rows = src_rows;
    p.dst_rows = dst_rows;
    p.row_bytes = row_bytes;
    p.status = status;
    // The layers' base pointers are on the device: the bulk mover copies a row
    // whose address is off 16 bytes by words instead.
    if (device_src && ((src_stride | dst_stride) & 15) == 0 && bulk_threads(row_bytes) > 0) {
      err = launch_bulk(transfer_bulk_kernel, p, p.units, row_bytes, dev, stream,
                        "hs_transfer_kv");
      if (err != HS_OK) return err;
      continue;
    }
    transfer_kernel<<<mover_grid(dev, p.units), kMoverThreads, 0,
                      reinterpret_cast<cudaStream_t>(stream)>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
      return fail(HS_ERR_CUDA, "hs_transfer_kv launch: %s", cudaGetErrorString(e));
  }
  return HS_OK;
}

extern "C" hs_err hs_probe_read(const void* src, int64_t bytes, unsigned long long* sink,
                                hs_stream_t stream) {
  using namespace hs;
  clear_error();
  if (src == nullptr || sink == nullptr || bytes < 0 || (bytes & 15) ||
      (reinterpret_cast<uintptr_t>(src) & 15))
    return fail(HS_ERR_ARG, "hs_probe_read: need a 16-byte aligned source and bytes %% 16 == 0");
  if (bytes == 0) return HS_OK;
  DeviceInfo dev;
  hs_err err = current_device(&dev);
  if (err != HS_OK) return err;
  probe_read_kernel<<<dev.sm_count * 4, 512, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), bytes >> 4, sink);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "hs_probe_read launch: %s", cudaGetErrorString(e));
  return HS_OK;
}

extern "C" hs_err hs_gather_misses(const uint64_t* pool_ptrs, const uint64_t* hot_ptrs,
                                   int32_t num_layers, int32_t flags, int64_t pool_num_rows,
                                   int64_t hot_num_rows, int64_t row_bytes,
                                   const int64_t* miss_src, const int32_t* miss_dst,
                                   int64_t plan_stride, const int32_t* miss_count, int32_t batch,
                                   int32_t top_k, int32_t* status, hs_stream_t stream) {
  hs::CallRange range("hs_gather_misses");
  using namespace hs;
  clear_error();
  if (batch < 0 || top_k < 0 || num_layers < 0 || row_bytes < 1 || pool_num_rows < 0 ||
      hot_num_rows < 0)
    return fail(HS_ERR_ARG, "hs_gather_misses: negative size or row_bytes < 1");
  if (flags & ~(HS_GATHER_HAS_V | HS_OVERLAP_PREV))
    return fail(HS_ERR_ARG, "hs_gather_misses: unknown flags 0x%x", flags);
  const bool has_v = (flags & HS_GATHER_HAS_V) != 0;
  if (batch == 0 || top_k == 0 || num_layers == 0) return HS_OK;
  if (pool_ptrs == nullptr || hot_ptrs == nullptr || miss_src == nullptr ||
      miss_dst == nullptr || miss_count == nullptr)
    return fail(HS_ERR_ARG, "hs_gather_misses: pointer arrays and the plan arrays are required");
  if (plan_stride < top_k) return fail(HS_ERR_ARG, "hs_gather_misses: plan_stride < top_k");
  const uint64_t pairs = static_cast<uint64_t>(num_layers) * (has_v ? 2u : 1u);
  if (pairs * static_cast<uint64_t>(top_k) >= (1ull << 32))
    return fail(HS_ERR_UNSUPPORTED, "hs_gather_misses: top_k * layers must be < 2^32");
  DeviceInfo dev;
  hs_err err = current_device(&dev);
  if (err != HS_OK) return err;
  GatherParams p;
  p.pool_ptrs = pool_ptrs;
  p.hot_ptrs = hot_ptrs;
  p.ptr_pairs = static_cast<uint32_t>(pairs);
  p.pool_rows = pool_num_rows;
  p.hot_rows = hot_num_rows;
  p.row_bytes = row_bytes;
  p.miss_src = miss_src;
  p.miss_dst = miss_dst;
  p.plan_stride = plan_stride;
  p.miss_count = miss_count;
  p.top_k = top_k;
  p.status = status;
  // The flat path counts (unit, chunk) items in 32 bits: kGatherUnits * chunks < 2^32.
  p.chunks16 = row_bytes % 16 == 0 && row_bytes / 16 <= (1ll << 23)
                   ? static_cast<uint32_t>(row_bytes / 16) : 0u;
  p.div_chunks16 = FastDiv{fastdiv_magic(p.chunks16 > 0 ? p.chunks16 : 1u),
                           p.chunks16 > 0 ? p.chunks16 : 1u};
  p.div_ptr_pairs = FastDiv{fastdiv_magic(p.ptr_pairs), p.ptr_pairs};
  p.overlap = (flags & HS_OVERLAP_PREV) != 0;
  // Enough blocks per row to cover the device even for a few rows, at most
  // one warp per (miss, layer) unit.
  constexpr int W = kMoverThreads / kWarp;
  const int64_t units = static_cast<int64_t>(top_k) * static_cast<int64_t>(pairs);
  int64_t y = static_cast<int64_t>(dev.sm_count) * kGatherBlocksPerSm / batch;
  const int64_t y_max = (units + W - 1) / W;
  if (y > y_max) y = y_max;
  if (y < 1) y = 1;
  if (y > 65535) y = 65535;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(batch), static_cast<unsigned>(y), 1);
  cfg.blockDim = dim3(kMoverThreads, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.overlap ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gather_misses_kernel, p);
  if (e != cudaSuccess)
    return fail(HS_ERR_CUDA, "hs_gather_misses launch: %s", cudaGetErrorString(e));
  return HS_OK;
}

extern "C" hs_err hs_invalidate_tokens(int32_t* slot_tokens, int64_t slot_tokens_stride,
                                       int32_t hot_size, int64_t num_states,
                                       const int64_t* state_rows, const int32_t* tokens,
                                       int64_t n_tokens, int32_t* status, hs_stream_t stream) {
  hs::CallRange range("hs_invalidate_tokens");
  using namespace hs;
  clear_error();
  if (n_tokens < 0 || hot_size < 0 || num_states < 0)
    return fail(HS_ERR_ARG, "hs_invalidate_tokens: negative size");
  if (n_tokens == 0 || hot_size == 0 || num_states == 0) return HS_OK;
  if (slot_tokens == nullptr || state_rows == nullptr || tokens == nullptr)
    return fail(HS_ERR_ARG, "hs_invalidate_tokens: slot_tokens, state_rows and tokens are required");
  if (slot_tokens_stride < static_cast<int64_t>(hot_size) + 1)
    return fail(HS_ERR_ARG, "hs_invalidate_tokens: slot_tokens_stride must be >= hot_size + 1");
  const int64_t chunks = (static_cast<int64_t>(hot_size) + kInvSlots - 1) / kInvSlots;
  if (n_tokens * chunks > 2147483647)
    return fail(HS_ERR_UNSUPPORTED, "hs_invalidate_tokens: n_tokens * ceil(hot_size / %d) must fit a grid",
                kInvSlots);
  invalidate_kernel<<<static_cast<unsigned>(n_tokens * chunks), kInvThreads, 0,
                      reinterpret_cast<cudaStream_t>(stream)>>>(
      slot_tokens, slot_tokens_stride, hot_size, num_states, state_rows, tokens, status,
      static_cast<int32_t>(chunks));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(HS_ERR_CUDA, "hs_invalidate_tokens launch: %s", cudaGetErrorString(e));
  return HS_OK;
}

extern "C" hs_err hs_wait_selftest(int32_t max_polls, int32_t* status, hs_stream_t stream) {
  using namespace hs;
  clear_error();
  if (max_polls < 0 || status == nullptr)
    return fail(HS_ERR_ARG, "hs_wait_selftest: needs max_polls >= 0 and a status word");
  wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t>(max_polls), status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(HS_ERR_CUDA, "hs_wait_selftest launch: %s", cudaGetErrorString(e));
  return HS_OK;
}
