// hs_fp8.cu -- FP8 (E4M3) KV write for sm_103a.
//
// Defined by tokenspeed tokenspeed_kernel/ops/kvcache/triton.py,
// fused_fp8_set_kv_buffer and _fused_fp8_set_kv_buffer_kernel: each token's K
// and V rows [heads, head_dim] are multiplied by an inverse scale (fp32,
// 1/scale, when scales are given), converted to float8 e4m3 and scattered to
// cache slot cache_loc[t] = page * page_size + offset of a paged cache.
//
// The work is flattened into 16-byte input chunks: (token, K|V, head, chunk)
// with the chunk fastest, so consecutive threads read consecutive input bytes
// and write consecutive cache bytes.  A thread converts its chunk with the
// hardware's paired fp32 -> e4m3 conversion (round to nearest even, finite
// saturation) and stores 8 (bf16/fp16 input) or 4 (fp32 input) bytes.  Rows
// whose strides do not allow 16-byte chunks go element by element.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hs_device.cuh"
#include "hs_host.h"

namespace hs {
namespace {

constexpr int kFp8Threads = 256;
constexpr int kFp8BlocksPerSm = 8;
constexpr int kFp8Unroll = 2;  // units in flight per thread

struct Fp8Params {
  const unsigned char* in[2];  // K, V inputs
  int64_t stride_token[2], stride_head[2];  // bytes
  unsigned char* cache[2];
  int64_t c_page, c_off, c_head;  // bytes
  const float* scale[2];          // device fp32 [1] or NULL
  const int64_t* loc;
  int64_t num_slots;
  int32_t page_size;
  uint32_t chunks;         // chunks per (token, K|V, head) row
  uint32_t rows_per_tok;   // kv * heads
  uint32_t heads;
  FastDiv div_chunks, div_rows, div_heads, div_page;  // div_page: num_slots < 2^32
  int64_t t_begin;         // first token of this launch
  uint32_t units;          // launch tokens * rows_per_tok * chunks (< 2^32)
  int32_t* status;
};

// Two floats -> two e4m3 codes (low byte = a): round to nearest even,
// finite overflow and infinities saturate to the largest finite value.
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

template <int kDtype>  // HS_DT_F32, HS_DT_F16, HS_DT_BF16
__device__ __forceinline__ float load_elem(const unsigned char* p) {
  if constexpr (kDtype == HS_DT_F32) {
    return *reinterpret_cast<const float*>(p);
  } else if constexpr (kDtype == HS_DT_F16) {
    return __half2float(*reinterpret_cast<const __half*>(p));
  } else {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
}

// Elements per 16-byte chunk.
template <int kDtype>
__host__ __device__ constexpr int chunk_elems() {
  return kDtype == HS_DT_F32 ? 4 : 8;
}

// Converts one 16-byte input chunk and stores its E codes at d.
template <int kDtype>
__device__ __forceinline__ void convert_store(uint4 raw, float sc, bool scaled, unsigned char* d) {
  constexpr int E = chunk_elems<kDtype>();
  float x[E];
  if constexpr (kDtype == HS_DT_F32) {
    x[0] = __uint_as_float(raw.x);
    x[1] = __uint_as_float(raw.y);
    x[2] = __uint_as_float(raw.z);
    x[3] = __uint_as_float(raw.w);
  } else {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = static_cast<uint16_t>(w[i] & 0xFFFF);
      const uint16_t hi = static_cast<uint16_t>(w[i] >> 16);
      if constexpr (kDtype == HS_DT_F16) {
        x[2 * i] = __half2float(__ushort_as_half(lo));
        x[2 * i + 1] = __half2float(__ushort_as_half(hi));
      } else {
        x[2 * i] = __uint_as_float(static_cast<uint32_t>(lo) << 16);
        x[2 * i + 1] = __uint_as_float(static_cast<uint32_t>(hi) << 16);
      }
    }
  }
  if (scaled) {
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = x[i] * sc;  // one fp32 multiply per element
  }
  if constexpr (E == 8) {
    uint2 o;
    o.x = static_cast<uint32_t>(e4m3x2(x[0], x[1])) |
          (static_cast<uint32_t>(e4m3x2(x[2], x[3])) << 16);
    o.y = static_cast<uint32_t>(e4m3x2(x[4], x[5])) |
          (static_cast<uint32_t>(e4m3x2(x[6], x[7])) << 16);
    *reinterpret_cast<uint2*>(d) = o;
  } else {
    *reinterpret_cast<uint32_t*>(d) = static_cast<uint32_t>(e4m3x2(x[0], x[1])) |
                                      (static_cast<uint32_t>(e4m3x2(x[2], x[3])) << 16);
  }
}

// Rows whose heads are contiguous in the input and in the cache: one warp per
// (token, K|V), the token's slot computed once, every lane moving 16-byte
// chunks of the [heads x dim] row.  p.chunks = chunks per row, p.units =
// tokens x (1 + has_v).
template <int kDtype>
__global__ void __launch_bounds__(kFp8Threads, 6) fp8_row_kernel(const Fp8Params p) {
  constexpr int E = chunk_elems<kDtype>();
  constexpr int U = 4;  // chunks per lane in flight
  const int lane = threadIdx.x & 31;
  const float inv_k = p.scale[0] != nullptr ? 1.0f / __ldg(p.scale[0]) : 1.0f;
  const float inv_v = p.scale[1] != nullptr ? 1.0f / __ldg(p.scale[1]) : 1.0f;
  const uint32_t kvn = p.rows_per_tok / p.heads;  // 1 (K only) or 2
  const uint32_t warps = gridDim.x * (kFp8Threads / kWarp);
  for (uint32_t u = blockIdx.x * (kFp8Threads / kWarp) + (threadIdx.x >> 5); u < p.units;
       u += warps) {
    const bool is_v = kvn == 2 && (u & 1u);
    const int64_t t = p.t_begin + (kvn == 2 ? (u >> 1) : u);
    const int64_t L = __ldg(p.loc + t);
    const unsigned char* src = (is_v ? p.in[1] : p.in[0]) +
                               t * (is_v ? p.stride_token[1] : p.stride_token[0]);
    // The row's first round of chunks loads together with its slot index (the
    // source row of token t is always in range): one round trip, not two.
    uint4 raw[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t c = lane + j * kWarp;
      if (c < p.chunks) raw[j] = ld_stream_v4(src + static_cast<int64_t>(c) * 16);
    }
    if (L < 0 || L >= p.num_slots) {
      if (!is_v && lane == 0 && p.status) atomicOr(p.status, HS_ST_BAD_INDEX);
      continue;
    }
    const int64_t page = div_any(static_cast<uint32_t>(L), p.div_page);
    const int64_t off = L - page * p.page_size;
    unsigned char* dst = (is_v ? p.cache[1] : p.cache[0]) + page * p.c_page + off * p.c_off;
    const float sc = is_v ? inv_v : inv_k;
    const bool scaled = (is_v ? p.scale[1] : p.scale[0]) != nullptr;
    for (uint32_t c0 = lane;;) {
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + j * kWarp;
        if (c < p.chunks) convert_store<kDtype>(raw[j], sc, scaled, dst + static_cast<int64_t>(c) * E);
      }
      c0 += kWarp * U;
      if (c0 >= p.chunks) break;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + j * kWarp;
        if (c < p.chunks) raw[j] = ld_stream_v4(src + static_cast<int64_t>(c) * 16);
      }
    }
  }
}

// kVec: 16-byte input chunks and 8- or 4-byte stores (host checked the
// alignment); otherwise one element per unit.
template <int kDtype, bool kVec>
__global__ void __launch_bounds__(kFp8Threads) fp8_store_kernel(const Fp8Params p) {
  constexpr int E = kVec ? chunk_elems<kDtype>() : 1;
  constexpr int kInBytes = kDtype == HS_DT_F32 ? 4 : 2;
  // the inverse scales, divided in fp32 (IEEE division)
  const float inv_k = p.scale[0] != nullptr ? 1.0f / __ldg(p.scale[0]) : 1.0f;
  const float inv_v = p.scale[1] != nullptr ? 1.0f / __ldg(p.scale[1]) : 1.0f;
  const uint32_t stride = gridDim.x * blockDim.x;
  // kUnroll units per thread per round, all loads issued before any convert.
  for (uint32_t u0 = blockIdx.x * blockDim.x + threadIdx.x; u0 < p.units;
       u0 += stride * kFp8Unroll) {
    const unsigned char* src[kFp8Unroll];
    unsigned char* dst[kFp8Unroll];
    int64_t L[kFp8Unroll];
    uint32_t kvs[kFp8Unroll];
#pragma unroll
    for (int j = 0; j < kFp8Unroll; ++j) {
      // u = ((t' * rows_per_tok) + kv * heads + h) * chunks + c, t = t_begin + t'
      const uint32_t u = u0 + j * stride;
      L[j] = -1;
      src[j] = nullptr;
      dst[j] = nullptr;
      kvs[j] = 0;
      if (u >= p.units) continue;
      const uint32_t row = div_any(u, p.div_chunks);
      const uint32_t c = u - row * p.chunks;
      const uint32_t tt = div_any(row, p.div_rows);
      const uint32_t rk = row - tt * p.rows_per_tok;
      const int64_t t = p.t_begin + tt;
      const uint32_t kv = div_any(rk, p.div_heads);
      const uint32_t h = rk - kv * p.heads;
      kvs[j] = kv;
      L[j] = __ldg(p.loc + t);
      src[j] = (kv ? p.in[1] : p.in[0]) + t * (kv ? p.stride_token[1] : p.stride_token[0]) +
               static_cast<int64_t>(h) * (kv ? p.stride_head[1] : p.stride_head[0]) +
               static_cast<int64_t>(c) * E * kInBytes;
      dst[j] = (kv ? p.cache[1] : p.cache[0]) + static_cast<int64_t>(h) * p.c_head +
               static_cast<int64_t>(c) * E;
      if (rk == 0 && c == 0) kvs[j] |= 2u;  // the token's first unit reports a bad slot
    }
    uint4 raw[kFp8Unroll];
    float x1[kFp8Unroll];
#pragma unroll
    for (int j = 0; j < kFp8Unroll; ++j) {
      if (src[j] == nullptr) continue;
      if constexpr (kVec)
        raw[j] = ld_stream_v4(src[j]);
      else
        x1[j] = load_elem<kDtype>(src[j]);
    }
#pragma unroll
    for (int j = 0; j < kFp8Unroll; ++j) {
      if (src[j] == nullptr) continue;
      if (L[j] < 0 || L[j] >= p.num_slots) {
        if ((kvs[j] & 2u) && p.status) atomicOr(p.status, HS_ST_BAD_INDEX);
        continue;
      }
      const int64_t page = div_any(static_cast<uint32_t>(L[j]), p.div_page);
      const int64_t off = L[j] - page * p.page_size;
      unsigned char* d = dst[j] + page * p.c_page + off * p.c_off;
      const bool is_v = (kvs[j] & 1u) != 0;
      const float sc = is_v ? inv_v : inv_k;
      const bool scaled = (is_v ? p.scale[1] : p.scale[0]) != nullptr;
      if constexpr (!kVec) {
        *d = static_cast<unsigned char>(e4m3x2(scaled ? x1[j] * sc : x1[j], 0.0f) & 0xFF);
      } else {
        convert_store<kDtype>(raw[j], sc, scaled, d);
      }
    }
  }
}

}  // namespace
}  // namespace hs

extern "C" hs_err hs_fp8_store_kv(const void* k, const void* v, int32_t in_dtype,
                                  int64_t k_stride_token, int64_t k_stride_head,
                                  int64_t v_stride_token, int64_t v_stride_head, void* k_cache,
                                  void* v_cache, int64_t cache_stride_page,
                                  int64_t cache_stride_offset, int64_t cache_stride_head,
                                  int32_t page_size, int64_t num_slots, const int64_t* cache_loc,
                                  int64_t n_tokens, int32_t num_kv_heads, int32_t head_dim,
                                  const float* k_scale, const float* v_scale, int32_t* status,
                                  hs_stream_t stream) {
  hs::CallRange range("hs_fp8_store_kv");
  using namespace hs;
  clear_error();
  if (in_dtype != HS_DT_F32 && in_dtype != HS_DT_F16 && in_dtype != HS_DT_BF16)
    return fail(HS_ERR_ARG, "hs_fp8_store_kv: unknown input dtype %d", in_dtype);
  if (num_slots > 0xFFFFFFFFll)
    return fail(HS_ERR_UNSUPPORTED, "hs_fp8_store_kv: num_slots must be < 2^32");
  if (n_tokens < 0 || page_size < 1 || num_slots < 0 || num_kv_heads < 1 || head_dim < 1)
    return fail(HS_ERR_ARG, "hs_fp8_store_kv: need n_tokens >= 0, page_size >= 1, "
                            "num_slots >= 0, heads >= 1, head_dim >= 1");
  if (n_tokens == 0) return HS_OK;
  if (k == nullptr || k_cache == nullptr || cache_loc == nullptr)
    return fail(HS_ERR_ARG, "hs_fp8_store_kv: k, k_cache and cache_loc are required");
  if ((v == nullptr) != (v_cache == nullptr))
    return fail(HS_ERR_ARG, "hs_fp8_store_kv: v and v_cache must both be set or both be NULL");
  const int64_t esz = in_dtype == HS_DT_F32 ? 4 : 2;
  if (k_stride_head < head_dim || (v && v_stride_head < head_dim) ||
      cache_stride_head < head_dim || cache_stride_offset < 1 || cache_stride_page < 1)
    return fail(HS_ERR_ARG, "hs_fp8_store_kv: head strides must be >= head_dim, cache strides >= 1");
  DeviceInfo dev;
  hs_err err = current_device(&dev);
  if (err != HS_OK) return err;

  const int kv = v ? 2 : 1;
  const int E = in_dtype == HS_DT_F32 ? 4 : 8;
  uintptr_t in_al = reinterpret_cast<uintptr_t>(k) | static_cast<uintptr_t>(k_stride_token * esz) |
                    static_cast<uintptr_t>(k_stride_head * esz);
  uintptr_t out_al = reinterpret_cast<uintptr_t>(k_cache) |
                     static_cast<uintptr_t>(cache_stride_page) |
                     static_cast<uintptr_t>(cache_stride_offset) |
                     static_cast<uintptr_t>(cache_stride_head);
  if (v) {
    in_al |= reinterpret_cast<uintptr_t>(v) | static_cast<uintptr_t>(v_stride_token * esz) |
             static_cast<uintptr_t>(v_stride_head * esz);
    out_al |= reinterpret_cast<uintptr_t>(v_cache);
  }
  const bool vec = head_dim % E == 0 && (in_al & 15) == 0 && (out_al % E) == 0;
  const uint32_t chunks = static_cast<uint32_t>(vec ? head_dim / E : head_dim);
  const uint64_t rows_per_tok = static_cast<uint64_t>(kv) * static_cast<uint64_t>(num_kv_heads);
  const uint64_t per_tok = rows_per_tok * chunks;
  if (per_tok >= (1ull << 32))
    return fail(HS_ERR_UNSUPPORTED, "hs_fp8_store_kv: heads * head_dim too large");

  Fp8Params p;
  p.in[0] = static_cast<const unsigned char*>(k);
  p.in[1] = static_cast<const unsigned char*>(v ? v : k);
  p.stride_token[0] = k_stride_token * esz;
  p.stride_head[0] = k_stride_head * esz;
  p.stride_token[1] = (v ? v_stride_token : k_stride_token) * esz;
  p.stride_head[1] = (v ? v_stride_head : k_stride_head) * esz;
  p.cache[0] = static_cast<unsigned char*>(k_cache);
  p.cache[1] = static_cast<unsigned char*>(v ? v_cache : k_cache);
  p.c_page = cache_stride_page;
  p.c_off = cache_stride_offset;
  p.c_head = cache_stride_head;
  p.scale[0] = k_scale;
  p.scale[1] = v_scale;
  p.loc = cache_loc;
  p.num_slots = num_slots;
  p.page_size = page_size;
  p.chunks = chunks;
  p.rows_per_tok = static_cast<uint32_t>(rows_per_tok);
  p.heads = static_cast<uint32_t>(num_kv_heads);
  p.div_chunks = FastDiv{fastdiv_magic(chunks), chunks};
  p.div_rows = FastDiv{fastdiv_magic(p.rows_per_tok), p.rows_per_tok};
  p.div_heads = FastDiv{fastdiv_magic(p.heads), p.heads};
  p.div_page = FastDiv{fastdiv_magic(static_cast<uint32_t>(page_size)),
                       static_cast<uint32_t>(page_size)};
  p.status = status;
  using Fn = void (*)(const Fp8Params);
  // Heads contiguous in the input and in the cache: one warp per (token, K|V) row.
  const bool rows = vec && k_stride_head == head_dim && (!v || v_stride_head == head_dim) &&
                    cache_stride_head == head_dim;
  Fn fn;
  if (rows) {
    p.chunks = static_cast<uint32_t>(static_cast<int64_t>(num_kv_heads) * head_dim / E);
    fn = in_dtype == HS_DT_F32 ? fp8_row_kernel<HS_DT_F32>
                               : (in_dtype == HS_DT_F16 ? fp8_row_kernel<HS_DT_F16>
                                                        : fp8_row_kernel<HS_DT_BF16>);
    for (int64_t begin = 0; begin < n_tokens; begin += (1ll << 30)) {
      const int64_t nt = (n_tokens - begin) < (1ll << 30) ? (n_tokens - begin) : (1ll << 30);
      p.t_begin = begin;
      p.units = static_cast<uint32_t>(nt * kv);
      int64_t blocks = (static_cast<int64_t>(p.units) + kFp8Threads / kWarp - 1) /
                       (kFp8Threads / kWarp);
      const int64_t cap = static_cast<int64_t>(dev.sm_count) * kFp8BlocksPerSm;
      if (blocks > cap) blocks = cap;
      fn<<<static_cast<unsigned>(blocks), kFp8Threads, 0,
           reinterpret_cast<cudaStream_t>(stream)>>>(p);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess)
        return fail(HS_ERR_CUDA, "hs_fp8_store_kv launch: %s", cudaGetErrorString(e));
    }
    return HS_OK;
  }
  if (in_dtype == HS_DT_F32)
    fn = vec ? fp8_store_kernel<HS_DT_F32, true> : fp8_store_kernel<HS_DT_F32, false>;
  else if (in_dtype == HS_DT_F16)
    fn = vec ? fp8_store_kernel<HS_DT_F16, true> : fp8_store_kernel<HS_DT_F16, false>;
  else
    fn = vec ? fp8_store_kernel<HS_DT_BF16, true> : fp8_store_kernel<HS_DT_BF16, false>;
  // 32-bit unit indices: launch at most floor((2^32 - 1) / per_tok) tokens at a time.
  const int64_t max_tok = static_cast<int64_t>(0xFFFFFFFFull / per_tok);
  for (int64_t begin = 0; begin < n_tokens; begin += max_tok) {
    const int64_t nt = (n_tokens - begin) < max_tok ? (n_tokens - begin) : max_tok;
    p.t_begin = begin;
    p.units = static_cast<uint32_t>(static_cast<uint64_t>(nt) * per_tok);
    int64_t blocks = (static_cast<int64_t>(p.units) + kFp8Threads - 1) / kFp8Threads;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * kFp8BlocksPerSm;
    if (blocks > cap) blocks = cap;
    fn<<<static_cast<unsigned>(blocks), kFp8Threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
      return fail(HS_ERR_CUDA, "hs_fp8_store_kv launch: %s", cudaGetErrorString(e));
  }
  return HS_OK;
}
