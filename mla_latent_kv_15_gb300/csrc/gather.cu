// Paged context gather (gather_and_maybe_dequant_cache of the MLA pages'
// chunked-prefill context path, vllm/v1/attention/backends/mla/common.py,
// MLACommonImpl._compute_prefill_context): request b's latent rows at
// context positions seq_starts[b] + j, j < cu_seq_lens[b+1] - cu_seq_lens[b],
// fetched through the block table into dense rows cu_seq_lens[b] + j of a
// bf16 workspace; an e4m3 cache is dequantised on the way
// (bf16(float32(code) * kv_scale)).
//
// An HBM-bound copy: each CTA resolves 16 destination rows (request by
// binary search over cu_seq_lens, page through the block table), then its
// 256 threads move the rows with 16-byte loads (and 16-byte stores for a bf16
// cache, 32-byte stores of 16 dequantised values for an e4m3 one), so
// consecutive threads touch consecutive bytes of a row.  Grid-stride over
// row groups.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kGRows = 16;       // destination rows per CTA iteration
constexpr int kGThreads = 256;
constexpr int kChunks = kDqk * 2 / 16;   // 16-byte pieces of a bf16 row: 72
constexpr int kChunks8 = kDqk / 16;      // 16-byte pieces of an e4m3 row: 36 (32 output bytes each)

// Two e4m3 codes -> two floats (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four e4m3 codes (one 32-bit word, lowest byte first) -> four bf16 values
// bf16(float32(code) * scale), packed in two words.
__device__ __forceinline__ uint2 dequant4(uint32_t w, float scale) {
  const float2 a = e4m3x2_to_float2((uint16_t)(w & 0xFFFF)), b = e4m3x2_to_float2((uint16_t)(w >> 16));
  return make_uint2(bf16x2_bits(a.x * scale, a.y * scale), bf16x2_bits(b.x * scale, b.y * scale));
}

__device__ __forceinline__ void st_global_v8(void* p, uint2 a, uint2 b, uint2 c, uint2 d) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(b.x),
               "r"(b.y), "r"(c.x), "r"(c.y), "r"(d.x), "r"(d.y)
               : "memory");
}

template <bool kFp8>
__global__ void __launch_bounds__(kGThreads) gather_kernel(const uint8_t* __restrict__ cache, int64_t num_blocks,
                                                           int page_size, float kv_scale,
                                                           const int32_t* __restrict__ block_table, int max_pages,
                                                           const int32_t* __restrict__ cu,
                                                           const int32_t* __restrict__ starts, int batch,
                                                           uint8_t* __restrict__ dst, int64_t num_tokens,
                                                           int32_t* status) {
  __shared__ int64_t s_src[kGRows];   // source row, -1: zero-fill, -2: nothing to write
  const int64_t total_req = cu[batch];
  const int64_t total = total_req < num_tokens ? total_req : num_tokens;
  if (blockIdx.x == 0 && threadIdx.x == 0 && total_req > num_tokens && status) atomicOr(status, 8);
  const int64_t cap = (int64_t)max_pages * page_size;
  const int64_t groups = (total + kGRows - 1) / kGRows;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t r0 = g * kGRows;
    if (threadIdx.x < kGRows) {
      const int64_t r = r0 + threadIdx.x;
      int64_t src = -2;
      if (r < total) {
        // request b: the last one with cu[b] <= r
        int lo = 0, hi = batch - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (cu[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int64_t pos = (int64_t)(starts ? starts[b] : 0) + (r - cu[b]);
        src = -1;
        if (pos < 0 || pos >= cap) {
          if (status) atomicOr(status, 2);
        } else {
          const int64_t page = block_table[(int64_t)b * max_pages + pos / page_size];
          if (page < 0 || page >= num_blocks) {
            if (status) atomicOr(status, 4);
          } else {
            src = page * page_size + pos % page_size;
          }
        }
      }
      s_src[threadIdx.x] = src;
    }
    __syncthreads();
    if (kFp8) {
      // 16 codes in (one 16-byte load), 32 bytes out (one 32-byte store when
      // dst is 32-byte aligned, else two 16-byte stores)
      const bool a32 = (reinterpret_cast<uintptr_t>(dst) & 31) == 0;
      for (int c = threadIdx.x; c < kGRows * kChunks8; c += kGThreads) {
        const int i = c / kChunks8, k = c - i * kChunks8;
        const int64_t src = s_src[i];
        if (src == -2) continue;
        uint4 codes = make_uint4(0, 0, 0, 0);
        if (src >= 0) codes = __ldg(reinterpret_cast<const uint4*>(cache + src * kDqk) + k);
        const float sc = src >= 0 ? kv_scale : 0.f;
        uint8_t* out = dst + (r0 + i) * (kDqk * 2) + k * 32;
        const uint2 v0 = dequant4(codes.x, sc), v1 = dequant4(codes.y, sc), v2 = dequant4(codes.z, sc),
                    v3 = dequant4(codes.w, sc);
        if (a32) {
          st_global_v8(out, v0, v1, v2, v3);
        } else {
          reinterpret_cast<uint4*>(out)[0] = make_uint4(v0.x, v0.y, v1.x, v1.y);
          reinterpret_cast<uint4*>(out)[1] = make_uint4(v2.x, v2.y, v3.x, v3.y);
        }
      }
    } else {
      for (int c = threadIdx.x; c < kGRows * kChunks; c += kGThreads) {
        const int i = c / kChunks, k = c - i * kChunks;
        const int64_t src = s_src[i];
        if (src == -2) continue;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (src >= 0) v = __ldg(reinterpret_cast<const uint4*>(cache + src * (kDqk * 2)) + k);
        reinterpret_cast<uint4*>(dst + (r0 + i) * (kDqk * 2))[k] = v;
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_gather(const void* cache, int64_t num_blocks, int page_size, int cache_fp8, float kv_scale,
                          const int32_t* block_table, int max_pages, const int32_t* cu_seq_lens,
                          const int32_t* seq_starts, int batch, void* dst, int64_t num_tokens, int32_t* status,
                          cudaStream_t s) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || sms <= 0)
    sms = 148;
  const int64_t groups = (num_tokens + kGRows - 1) / kGRows;
  const int64_t cap = (int64_t)sms * 8;   // eight 256-thread CTAs per SM
  const unsigned grid = (unsigned)(groups < cap ? groups : cap);
  const uint8_t* c = static_cast<const uint8_t*>(cache);
  uint8_t* d = static_cast<uint8_t*>(dst);
  if (cache_fp8)
    gather_kernel<true><<<grid, kGThreads, 0, s>>>(c, num_blocks, page_size, kv_scale, block_table, max_pages,
                                                   cu_seq_lens, seq_starts, batch, d, num_tokens, status);
  else
    gather_kernel<false><<<grid, kGThreads, 0, s>>>(c, num_blocks, page_size, kv_scale, block_table, max_pages,
                                                    cu_seq_lens, seq_starts, batch, d, num_tokens, status);
  return cudaGetLastError();
}

}  // namespace mla
