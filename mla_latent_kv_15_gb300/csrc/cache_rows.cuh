// The row write of concat_and_cache_mla (page "vllm/v1/attention/backends/
// mla/common.py", MLACommonImpl.forward: the cache update that precedes the
// attention of a step) and the query's scaled_fp8_quant (same page, the
// decode's query quantisation), shared by the kernels of cache_write.cu and
// the extra blocks of the plan kernel (mla_decode_step, mla_decode_fp8q_step).
//
// One warp per token.  A bf16 row is 72 16-byte vectors (64 of kv_c, 8 of
// k_pe) moved with 16-byte loads and stores.  For an e4m3 cache every value is
// divided by kv_scale in float32 (IEEE division) and converted with
// round-to-nearest-even and satfinite, so the codes are bit-identical to a
// correctly rounded reference.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {

__device__ __forceinline__ uint32_t fp8x4(const float (&x)[4]) {
  uint32_t r = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    r |= (uint32_t)__nv_cvt_float_to_fp8(x[k], __NV_SATFINITE, __NV_E4M3) << (8 * k);
  return r;
}

// e4m3 codes of eight bf16 values: RNE-satfinite of f32(x) / f32(scale) (IEEE
// division), as scaled_fp8_quant with a static scale.
__device__ __forceinline__ uint2 quantize8(const uint4 src, float scale) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&src);
  float lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float2 f0 = __bfloat1622float2(h[k]);
    const float2 f1 = __bfloat1622float2(h[2 + k]);
    lo[2 * k] = __fdiv_rn(f0.x, scale);
    lo[2 * k + 1] = __fdiv_rn(f0.y, scale);
    hi[2 * k] = __fdiv_rn(f1.x, scale);
    hi[2 * k + 1] = __fdiv_rn(f1.y, scale);
  }
  return make_uint2(fp8x4(lo), fp8x4(hi));
}

// Vector v (eight values) of the query into its e4m3 [q_abs | q_pe] row:
// the first rows * 64 vectors are q_abs's, the next rows * 8 q_pe's.
__device__ __forceinline__ void quantize_query_vec(const QuantArgs& qa, int64_t v) {
  const int64_t na = qa.rows * (kLkv / 8);
  int64_t r;
  int c;
  const __nv_bfloat16* src;
  if (v < na) {
    r = v / (kLkv / 8);
    c = (int)(v - r * (kLkv / 8)) * 8;
    src = static_cast<const __nv_bfloat16*>(qa.q_abs) + r * kLkv + c;
  } else {
    const int64_t u = v - na;
    r = u / (kRope / 8);
    const int cr = (int)(u - r * (kRope / 8)) * 8;
    src = static_cast<const __nv_bfloat16*>(qa.q_pe) + r * kRope + cr;
    c = kLkv + cr;
  }
  *reinterpret_cast<uint2*>(qa.q8 + r * kDqk + c) = quantize8(*reinterpret_cast<const uint4*>(src), qa.q_scale);
}

// Token `tok`'s row into its slot (a slot outside [0, num_slots) is padding:
// nothing is written); `lane` is the thread's lane in the token's warp.
template <bool kFp8>
__device__ __forceinline__ void write_cache_row(const CacheWriteArgs& w, int64_t tok, int lane) {
  const auto* kv_c = static_cast<const __nv_bfloat16*>(w.kv_c);
  const auto* k_pe = static_cast<const __nv_bfloat16*>(w.k_pe);
  const int64_t slot = w.slots[tok];
  if (slot < 0 || slot >= w.num_slots) return;
  for (int v = lane; v < 72; v += 32) {
    const uint4 src = v < 64 ? reinterpret_cast<const uint4*>(kv_c + tok * kLkv)[v]
                             : reinterpret_cast<const uint4*>(k_pe + tok * kRope)[v - 64];
    if (!kFp8) {
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(w.cache) + slot * kDqk)[v] = src;
    } else {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&src);
      float lo[4], hi[4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float2 f0 = __bfloat1622float2(h[k]);
        const float2 f1 = __bfloat1622float2(h[2 + k]);
        lo[2 * k] = __fdiv_rn(f0.x, w.kv_scale);
        lo[2 * k + 1] = __fdiv_rn(f0.y, w.kv_scale);
        hi[2 * k] = __fdiv_rn(f1.x, w.kv_scale);
        hi[2 * k + 1] = __fdiv_rn(f1.y, w.kv_scale);
      }
      uint2 v2;
      v2.x = fp8x4(lo);
      v2.y = fp8x4(hi);
      reinterpret_cast<uint2*>(static_cast<uint8_t*>(w.cache) + slot * kDqk)[v] = v2;
    }
  }
}

}  // namespace mla
