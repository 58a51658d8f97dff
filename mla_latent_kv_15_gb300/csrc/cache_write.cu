// concat_and_cache_mla: write the latent rows [kv_c | k_pe] of new tokens into
// the paged cache at their slots (page "vllm/v1/attention/backends/mla/
// common.py", MLACommonImpl.forward: the cache update that precedes the
// attention of a step).
//
// One warp per token.  A bf16 row is 72 16-byte vectors (64 of kv_c, 8 of
// k_pe) moved with 16-byte loads and stores.  For an e4m3 cache every value is
// divided by kv_scale in float32 (IEEE division) and converted with
// round-to-nearest-even and satfinite, so the codes are bit-identical to a
// correctly rounded reference.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {
namespace {

__device__ __forceinline__ uint32_t fp8x4(const float (&x)[4]) {
  uint32_t r = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    r |= (uint32_t)__nv_cvt_float_to_fp8(x[k], __NV_SATFINITE, __NV_E4M3) << (8 * k);
  return r;
}

template <bool kFp8>
__global__ void __launch_bounds__(256) cache_write_kernel(const __nv_bfloat16* __restrict__ kv_c,
                                                          const __nv_bfloat16* __restrict__ k_pe,
                                                          const int64_t* __restrict__ slots, int64_t num_tokens,
                                                          void* __restrict__ cache, int64_t num_slots,
                                                          float kv_scale) {
  // Launched as a programmatic dependent: only the launch overlaps the
  // previous kernel (which may still read the cache or have written the
  // inputs); every CTA waits for it before touching memory, so the grid also
  // completes after it.  The next kernel may then be launched at once (its
  // prologue overlaps this write; it waits for this grid before reading).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t tok = blockIdx.x * 8LL + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= num_tokens) return;
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) return;
  for (int v = lane; v < 72; v += 32) {
    const uint4 src = v < 64 ? reinterpret_cast<const uint4*>(kv_c + tok * kLkv)[v]
                             : reinterpret_cast<const uint4*>(k_pe + tok * kRope)[v - 64];
    if (!kFp8) {
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(cache) + slot * kDqk)[v] = src;
    } else {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&src);
      float lo[4], hi[4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float2 f0 = __bfloat1622float2(h[k]);
        const float2 f1 = __bfloat1622float2(h[2 + k]);
        lo[2 * k] = __fdiv_rn(f0.x, kv_scale);
        lo[2 * k + 1] = __fdiv_rn(f0.y, kv_scale);
        hi[2 * k] = __fdiv_rn(f1.x, kv_scale);
        hi[2 * k + 1] = __fdiv_rn(f1.y, kv_scale);
      }
      uint2 w;
      w.x = fp8x4(lo);
      w.y = fp8x4(hi);
      reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + slot * kDqk)[v] = w;
    }
  }
}

// scaled_fp8_quant with a static scale over `rows` rows of `width` values
// (width a multiple of 8; row pitches in elements, multiples of 8 for x and
// of 8 for out): eight values per thread per step (16-byte load, 8-byte
// store), grid-stride.
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const __nv_bfloat16* __restrict__ x, int64_t x_stride,
                                                           int64_t rows, int width, float scale,
                                                           uint8_t* __restrict__ out, int64_t out_stride) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int vpr = width / 8;
  const int64_t nvec = rows * vpr;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = v / vpr;
    const int c = (int)(v - r * vpr) * 8;
    const uint4 src = *reinterpret_cast<const uint4*>(x + r * x_stride + c);
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
    *reinterpret_cast<uint2*>(out + r * out_stride + c) = make_uint2(fp8x4(lo), fp8x4(hi));
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* x, int64_t x_stride, int64_t rows, int width, float scale, void* out,
                                int64_t out_stride, cudaStream_t s) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || sms <= 0)
    sms = 148;
  const int64_t nvec = rows * (width / 8);
  int64_t blocks = (nvec + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_fp8_kernel, static_cast<const __nv_bfloat16*>(x), x_stride, rows,
                                     width, scale, static_cast<uint8_t*>(out), out_stride);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_cache_write(const void* kv_c, const void* k_pe, const int64_t* slots, int64_t num_tokens,
                               void* cache, int64_t num_slots, int cache_fp8, float kv_scale, cudaStream_t s) {
  const int64_t blocks = (num_tokens + 7) / 8;
  const auto* c = static_cast<const __nv_bfloat16*>(kv_c);
  const auto* p = static_cast<const __nv_bfloat16*>(k_pe);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cache_fp8 ? cudaLaunchKernelEx(&cfg, cache_write_kernel<true>, c, p, slots, num_tokens, cache,
                                                 num_slots, kv_scale)
                            : cudaLaunchKernelEx(&cfg, cache_write_kernel<false>, c, p, slots, num_tokens, cache,
                                                 num_slots, kv_scale);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
