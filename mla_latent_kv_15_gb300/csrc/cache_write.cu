// concat_and_cache_mla and scaled_fp8_quant kernels (the row write and the
// eight-value quantisation themselves are in cache_rows.cuh).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "cache_rows.cuh"
#include "common.cuh"

namespace mla {
namespace {

template <bool kFp8>
__global__ void __launch_bounds__(256) cache_write_kernel(const CacheWriteArgs w) {
  // Launched as a programmatic dependent: only the launch overlaps the
  // previous kernel (which may still read the cache or have written the
  // inputs); every CTA waits for it before touching memory, so the grid also
  // completes after it.  The next kernel may then be launched at once (its
  // prologue overlaps this write; it waits for this grid before reading).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t tok = blockIdx.x * 8LL + (threadIdx.x >> 5);
  if (tok < w.num_tokens) write_cache_row<kFp8>(w, tok, threadIdx.x & 31);
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
    *reinterpret_cast<uint2*>(out + r * out_stride + c) =
        quantize8(*reinterpret_cast<const uint4*>(x + r * x_stride + c), scale);
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

cudaError_t launch_cache_write(const CacheWriteArgs& w, cudaStream_t s) {
  const int64_t blocks = (w.num_tokens + 7) / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = w.fp8 ? cudaLaunchKernelEx(&cfg, cache_write_kernel<true>, w)
                        : cudaLaunchKernelEx(&cfg, cache_write_kernel<false>, w);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
