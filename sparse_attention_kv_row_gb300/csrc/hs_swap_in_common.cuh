// hs_swap_in_common.cuh -- pieces shared by the two swap-in kernels (one
// cluster per row; one CTA per row and layer): the request hash, per-entry
// classification codes, bounded block-wide waits, copy chunks, and the host
// side's argument checks.
#pragma once

#include <climits>
#include <cstdint>

#include "hs_device.cuh"
#include "hs_host.h"

namespace hs {

constexpr int32_t kUnclaimed = INT_MAX;
constexpr uint32_t kMaxPolls = 1u << 22;    // bounded mbarrier waits (and at most 1 s each)
constexpr uint32_t kDrainPolls = 1u << 26;  // waiting out copies still in flight after a time-out
constexpr uint64_t kDrainNs = 16000000000ull;  // ... for at most 16 s

// Waits until the phase of `bar` with the given parity has completed: thread
// 0 polls (a bounded wait) while the other threads wait at the block barrier,
// which then makes the staged bytes visible to all of them.  (Threads polling
// a barrier that is not armed yet would take shared-memory bandwidth from the
// thread about to arm it.)  False in every thread when the wait ran out.
__device__ __forceinline__ bool block_wait(uint64_t* bar, uint32_t parity,
                                           uint32_t polls = kMaxPolls) {
  return __syncthreads_and(threadIdx.x == 0 ? mbar_wait(bar, parity, polls) : 1) != 0;
}

// Per-entry classification, stored as one byte per top-k entry.
enum : int8_t {
  kInvalid = 0, kRepeat = 1, kNewest = 2, kHit = 3, kBadPool = 4, kMiss = 5,
  kResident = 6,  // served from a resident block (block tables)
  kUnmapped = 7   // no source row through the source block table: treated as invalid
};

__device__ __forceinline__ uint32_t hash_of(int32_t key, int bits) {
  return (static_cast<uint32_t>(key) * 2654435761u) >> (32 - bits);
}

// Bit of `key` in a request filter of 2^bits bits (a second multiplicative hash).
__device__ __forceinline__ uint32_t filter_bit(int32_t key, int bits) {
  return (static_cast<uint32_t>(key) * 0x85EBCA6Bu) >> (32 - bits);
}

// The request hash: valid ids -> their canonical (smallest) top-k entry, by
// open addressing with linear probing in one shared-memory region of
// 4 * 2^bits bytes.  Packed form, used when the caller bounds every sequence
// so that each valid id is below 2^(32 - eb) - 1: 2^bits words
// `id << eb | entry`.  Wide form otherwise: 2^(bits - 1) pairs {id, entry}.
// Empty slots are all ones in both forms, so one fill clears either.
template <bool packed>
struct ReqHash {
  uint32_t* w;
  int bits, eb;

  static constexpr uint32_t kEmpty = 0xFFFFFFFFu;
  __device__ __forceinline__ int nbits() const { return packed ? bits : bits - 1; }
  __device__ __forceinline__ uint32_t mask() const { return (1u << nbits()) - 1u; }
  __device__ __forceinline__ uint32_t first(int32_t key) const { return hash_of(key, nbits()); }
  __device__ __forceinline__ int2* pairs() const { return reinterpret_cast<int2*>(w); }

  // Inserts (key, i); true when the key was already present.
  __device__ __forceinline__ bool insert(int32_t key, int32_t i) const {
    const uint32_t m = mask();
    uint32_t h = first(key);
    if (packed) {
      const uint32_t v = (static_cast<uint32_t>(key) << eb) | i;
      for (uint32_t n = 0; n <= m; ++n) {
        const uint32_t old = atomicCAS(&w[h], kEmpty, v);
        if (old == kEmpty) return false;
        if ((old >> eb) == static_cast<uint32_t>(key)) return true;
        h = (h + 1u) & m;
      }
      return false;
    }
    for (uint32_t n = 0; n <= m; ++n) {
      const int32_t old = atomicCAS(&pairs()[h].x, -1, key);
      if (old == -1) {
        pairs()[h].y = i;
        return false;
      }
      if (old == key) return true;
      h = (h + 1u) & m;
    }
    return false;
  }
  // Packed form: inserts (key, i) from slot h on; true when the key was already present.
  __device__ __forceinline__ bool insert_from(int32_t key, int32_t i, uint32_t h) const {
    const uint32_t m = mask();
    const uint32_t v = (static_cast<uint32_t>(key) << eb) | i;
    for (uint32_t n = 0; n < m; ++n) {
      const uint32_t old = atomicCAS(&w[h], kEmpty, v);
      if (old == kEmpty) return false;
      if ((old >> eb) == static_cast<uint32_t>(key)) return true;
      h = (h + 1u) & m;
    }
    return false;
  }
  // Lowers key's entry to i if i is smaller (the key is present).
  __device__ __forceinline__ void make_min(int32_t key, int32_t i) const {
    const uint32_t m = mask();
    uint32_t h = first(key);
    for (uint32_t n = 0; n <= m; ++n) {
      if (packed) {
        if ((w[h] >> eb) == static_cast<uint32_t>(key)) {
          atomicMin(&w[h], (static_cast<uint32_t>(key) << eb) | i);
          return;
        }
      } else if (pairs()[h].x == key) {
        atomicMin(&pairs()[h].y, i);
        return;
      }
      h = (h + 1u) & m;
    }
  }
  // Entry of `key` looked up from slot h on; -1 when absent.
  __device__ __forceinline__ int32_t find_from(int32_t key, uint32_t h) const {
    const uint32_t m = mask();
    if (packed) {
      const uint32_t emask = (1u << eb) - 1u;
      for (uint32_t n = 0; n <= m; ++n) {
        const uint32_t v = w[h];
        if (v == kEmpty) return -1;
        if ((v >> eb) == static_cast<uint32_t>(key)) return static_cast<int32_t>(v & emask);
        h = (h + 1u) & m;
      }
      return -1;
    }
    for (uint32_t n = 0; n <= m; ++n) {
      const int2 kv = pairs()[h];
      if (kv.x == key) return kv.y;
      if (kv.x == -1) return -1;
      h = (h + 1u) & m;
    }
    return -1;
  }
  __device__ __forceinline__ int32_t find(int32_t key) const { return find_from(key, first(key)); }
};

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

// The request map: valid id -> its canonical (smallest) top-k entry.
enum : int { kMapWide = 0, kMapPacked = 1, kMapDirect = 2 };

// The direct request map, used when the caller bounds the sequence length:
// one bit per token id of the row marks the requested ids; a word's prefix
// (set bits in the words before it) plus the popc of its lower bits is the
// id's dense rank among the requested ids; ent[rank] is the id's canonical
// (smallest) top-k entry.  A lookup is three shared loads and no probe loop.
struct DirectMap {
  uint32_t* bm;
  uint16_t* pre;
  int32_t* ent;
  // The rank of a requested id (its bit is set).
  __device__ __forceinline__ int rank(int32_t t, uint32_t w) const {
    return pre[t >> 5] + __popc(w & ((1u << (t & 31)) - 1u));
  }
  // Entry of a valid id, -1 when it is not requested.
  __device__ __forceinline__ int32_t find(int32_t t) const {
    const uint32_t w = bm[t >> 5];
    if (!((w >> (t & 31)) & 1u)) return -1;
    return ent[rank(t, w)];
  }
};

// ------------------------------------------------------------------ host side
// What the host derives once from a checked hs_swap_in_args.
struct SwapInDerived {
  int copy_width;          // 16, 4 or 1 bytes per copy chunk
  uint32_t chunks_per_row;
  int entry_bits;          // bits of a top-k entry index
  bool packed;             // the packed request hash is usable
  bool tables;             // block tables given
  bool pools_device;       // both pools in device (or managed) memory
  FastDiv div_src_bs, div_res_bs;
};

// Argument checks shared by every swap-in entry point (the messages name
// `who`), then the memory kinds of the pools and hot buffers and the derived
// values.  max_hot_size is the largest hot_size the caller's kernel handles.
hs_err check_swap_in_args(const hs_swap_in_args* a, const char* who, int max_hot_size,
                          bool* empty);
hs_err derive_swap_in(const hs_swap_in_args* a, const char* who, SwapInDerived* d);

// Hash-table size exponent: the smallest power of two >= mult * K.
__host__ __device__ inline int hash_bits_for(int K, int mult) {
  int bits = 2;  // the wide form keeps at least two pairs
  while ((1 << bits) < mult * K) ++bits;
  return bits;
}

// Raises a kernel's dynamic shared-memory limit once per device to the
// largest size requested so far.
hs_err ensure_smem(const void* fn, int device, int bytes);

// The one-CTA-per-(row, layer) swap-in (hs_swap_in_rows.cu) over `layers`
// checked argument blocks; fail_wait >= 0 makes that wait of every row give
// up at once (the time-out self-test), -1 none.
// The least shared memory that kernel needs per CTA (nothing staged, the
// smallest request hash).
int64_t swap_in_rows_min_smem(int K, int H, bool tables);
hs_err swap_in_rows_launch(const hs_swap_in_args* layers, int num_layers, hs_stream_t stream,
                           const char* who, int fail_wait);

}  // namespace hs
