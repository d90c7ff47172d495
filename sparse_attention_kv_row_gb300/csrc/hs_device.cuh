// hs_device.cuh -- device helpers for the swap-in and mover kernels (sm_103a):
// cache-hinted loads/stores as inline PTX, LDGSTS staging into shared memory,
// warp scans, and a 32-bit divider by multiply-high.
#pragma once

#include <cstdint>

namespace hs {

constexpr int kWarp = 32;
constexpr unsigned kFullMask = 0xFFFFFFFFu;

// ------------------------------------------------------------------ loads/stores
// Streaming reads of pool bytes: read-only path, no L1 allocation.  Used on
// device memory and on pinned host memory alike.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream_u8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Hot-buffer writes: cache in L2 only (the attention kernel reads them next).
__device__ __forceinline__ void st_l2_v4(void* p, uint4 v) {
  asm volatile("st.global.cg.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_l2_u32(void* p, uint32_t v) {
  asm volatile("st.global.cg.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_l2_u8(void* p, uint32_t v) {
  asm volatile("st.global.cg.u8 [%0], %1;" ::"l"(p), "h"((uint16_t)v) : "memory");
}

// Streaming writes for bulk movers (evict-first).
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_stream_u32(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_stream_u8(void* p, uint32_t v) {
  asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "h"((uint16_t)v) : "memory");
}

// ------------------------------------------------------------------ LDGSTS staging
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async_16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_8(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------ bulk copies
// One-dimensional bulk copies global -> shared through the tensor memory
// accelerator, completed on an mbarrier by transaction bytes.
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's earlier shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
          smem_addr(bar))
      : "memory");
}
// One arrival that also announces `bytes` more transaction bytes.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}
// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Each poll lets the thread sleep until the phase completes, for at most this
// long: a waiting thread issues a handful of instructions, not one poll every
// few cycles that takes issue slots from the warps still working.
constexpr uint32_t kPollSleepNs = 100000;
// Waits for the completion of phase `parity`: at most `max_polls` polls and at
// most `limit_ns` nanoseconds; false if the phase did not complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_polls,
                                          uint64_t limit_ns = 1000000000ull) {
  const uint64_t t0 = max_polls != 0 ? global_ns() : 0ull;
  for (uint32_t n = 0; n < max_polls; ++n) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kPollSleepNs)
        : "memory");
    if (done) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return false;
}
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// A hint to bring [src, src + bytes) of global memory into L2 (no data
// returned, nothing to wait for).  src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// A bulk copy shared -> global, in this thread's current bulk group.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src_smem)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until this thread's committed bulk stores have read their shared
// memory (the slots may be written again).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until this thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------ grid dependency
// Programmatic dependent launch: a grid launched with programmatic stream
// serialization may start before the preceding kernel in its stream has
// finished; `grid_dep_wait` blocks until that kernel has completed and its
// writes are visible (a no-op for a grid launched the ordinary way), and
// `grid_dep_launch_dependents` lets the next such grid start early.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

struct StagePending {
  int32_t off;  // byte offset in dst, or -1
  uint32_t val;
};
// A byte of a staged row's unaligned head or tail, loaded by one thread into a
// register and stored by stage_finish() after the row's wait, so that no
// thread stalls on the load in between.
__device__ __forceinline__ void stage_finish(void* dst, StagePending pend) {
  if (pend.off >= 0) static_cast<unsigned char*>(dst)[pend.off] = static_cast<unsigned char>(pend.val);
}

// Staging by one bulk copy: the 16-byte-aligned body of [src, src + nbytes)
// goes to dst (dst must be congruent to src modulo 16) through the tensor
// memory accelerator; the unaligned head and tail bytes are loaded by threads
// into a StagePending.
struct StageSplit {
  uint32_t head, body;
};
__device__ __forceinline__ StageSplit stage_split(const void* src, int64_t nbytes) {
  const uintptr_t s = reinterpret_cast<uintptr_t>(src);
  int64_t head = static_cast<int64_t>((16u - (s & 15u)) & 15u);
  if (head > nbytes) head = nbytes;
  return StageSplit{static_cast<uint32_t>(head),
                    static_cast<uint32_t>(((nbytes - head) >> 4) << 4)};
}
__device__ __forceinline__ StagePending stage_edges(const void* src, int64_t nbytes, StageSplit sp,
                                                    int tid) {
  const unsigned char* sc = static_cast<const unsigned char*>(src);
  const uint32_t tail = static_cast<uint32_t>(nbytes) - sp.head - sp.body;
  StagePending pend{-1, 0};
  if (static_cast<uint32_t>(tid) < sp.head) {
    pend.off = tid;
    pend.val = sc[tid];
  } else if (tid >= 32 && static_cast<uint32_t>(tid) < 32u + tail) {
    pend.off = static_cast<int32_t>(sp.head + sp.body + (tid - 32));
    pend.val = sc[pend.off];
  }
  return pend;
}
// Issued by one thread after the barrier was armed for the bodies' bytes.
__device__ __forceinline__ void stage_body(void* dst, const void* src, StageSplit sp,
                                           uint64_t* bar) {
  if (sp.body > 0)
    bulk_load(static_cast<char*>(dst) + sp.head, static_cast<const char*>(src) + sp.head, sp.body,
              bar);
}

// ------------------------------------------------------------------ scans
// Exclusive prefix over the 32 lanes; returns the warp total in *total.
__device__ __forceinline__ int warp_exclusive_scan(int v, int lane, int* total) {
  int x = v;
#pragma unroll
  for (int d = 1; d < kWarp; d <<= 1) {
    const int y = __shfl_up_sync(kFullMask, x, d);
    if (lane >= d) x += y;
  }
  *total = __shfl_sync(kFullMask, x, kWarp - 1);
  return x - v;
}

// In-place exclusive scan of cnt[0..n) (n <= 32 * 1024) by one warp; returns
// the grand total to every lane of that warp.
__device__ __forceinline__ int warp_scan_array(int* cnt, int n, int lane) {
  const int per = (n + kWarp - 1) / kWarp;
  const int begin = lane * per;
  const int end = min(n, begin + per);
  int local = 0;
  for (int i = begin; i < end; ++i) local += cnt[i];
  int total;
  int run = warp_exclusive_scan(local, lane, &total);
  for (int i = begin; i < end; ++i) {
    const int c = cnt[i];
    cnt[i] = run;
    run += c;
  }
  return total;
}

// ------------------------------------------------------------------ division
// floor(n / d) for 32-bit n by multiply-high with M = ceil(2^64 / d) (Lemire,
// Kaser, Kurz, "Faster remainder by direct computation", 2019): exact for every
// 32-bit n and 1 <= d < 2^32.  M is computed on the host.
struct FastDiv {
  uint64_t magic;
  uint32_t d;
};
__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
  return static_cast<uint32_t>(__umul64hi(f.magic, static_cast<uint64_t>(n)));
}
// floor(n / f.d), also for d == 1 (whose multiplier is not representable).
__device__ __forceinline__ uint32_t div_any(uint32_t n, FastDiv f) {
  return f.d == 1 ? n : fast_div(n, f);
}

}  // namespace hs

namespace hs {

// ------------------------------------------------------------------ clusters
// Thread-block cluster primitives (sm_90+ PTX): rank within the cluster, the
// shared-memory window of a peer CTA (DSMEM), and split arrive/wait barriers.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address, in the cluster shared window, of `p` (a local shared pointer) in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(p)), "r"(rank));
  return out;
}
__device__ __forceinline__ int32_t peer_ld(uint32_t addr) {
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void peer_st(uint32_t addr, int32_t v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void peer_min(uint32_t addr, int32_t v) {
  asm volatile("red.shared::cluster.min.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void peer_or(uint32_t addr, int32_t v) {
  asm volatile("red.shared::cluster.or.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrival without release semantics: pair it with fence_acq_rel_cluster() in
// the threads whose earlier writes peers must see (a release by every thread
// of a 1024-thread CTA was measured to cost about half a microsecond).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// ------------------------------------------------------------------ block scan
// Exclusive prefix sum of v over the block's threads in thread order; `wsum`
// is shared scratch of >= 33 ints.  Returns the prefix and, in *total, the
// block sum.  Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_sum(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < kWarp; d <<= 1) {
    const int y = __shfl_up_sync(kFullMask, x, d);
    if (lane >= d) x += y;
  }
  if (lane == kWarp - 1) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int t = lane < nwarps ? wsum[lane] : 0;
    int tot;
    const int ex = warp_exclusive_scan(t, lane, &tot);
    if (lane < nwarps) wsum[lane] = ex;
    if (lane == 0) wsum[32] = tot;
  }
  __syncthreads();
  const int r = wsum[warp] + x - v;
  *total = wsum[32];
  __syncthreads();  // wsum may be reused right away
  return r;
}

}  // namespace hs
