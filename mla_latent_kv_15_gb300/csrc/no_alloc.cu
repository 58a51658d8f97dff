// mla_decode_no_alloc: the decode for callers that cannot allocate device
// memory.  Some callers cannot call cudaMalloc (or any allocating routine)
// around a decode step: code that runs while a CUDA graph is being captured,
// serving loops that must not touch the allocator mid-step, or runtimes whose
// memory is handed out by a host framework that owns every device buffer.
// They pass their inputs and outputs as usual; the split-KV scratch comes
// from a fixed device array that belongs to this library instead of a
// caller-provided workspace.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/mla.h"
#include "common.cuh"

namespace mla {
int report_error(int code, const char* msg);
}

namespace {

constexpr size_t kScratchBytes = MLA_NO_ALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  It is a module-scope device variable: every GPU that
// loads this code holds it until the process exits.  Host code must never
// hand the name `g_scratch` to a kernel (on the host it is only a stand-in
// for the device variable); the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up on first use).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mla::report_error(MLA_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return mla::report_error(MLA_ERR_UNSUPPORTED, "device index above 63");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static decode scratch failed: %s",
               cudaGetErrorString(e));
      return mla::report_error(MLA_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

// Copies (and on request clears) the device error word of the last
// allocation-free decode on the current device: the first int of the static
// scratch, where the decode's plan header keeps it.
extern "C" int mla_decode_no_alloc_status(int* status, int clear, void* stream) {
  if (!status) return mla::report_error(MLA_ERR_INVALID_ARG, "null pointer argument");
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(status, ws, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "reading the allocation-free decode's error word failed: %s", cudaGetErrorString(e));
    return mla::report_error(MLA_ERR_CUDA, msg);
  }
  return MLA_OK;
}

extern "C" int mla_decode_no_alloc(const void* q_abs, const void* q_pe, const void* cache, int64_t num_blocks,
                                   int page_size, int cache_dtype, float kv_scale, const int32_t* block_table,
                                   int max_pages_per_seq, const int32_t* seq_lens, int batch,
                                   const int32_t* query_start_loc, int total_q, int num_heads, float scale,
                                   int num_splits, void* out, float* lse, void* stream) {
  if (batch > 0 && total_q > 0 && num_heads > 0 && num_splits >= 0) {
    const size_t need = mla_decode_workspace_size(batch, total_q, num_heads, num_splits);
    if (need > kScratchBytes) {
      char msg[256];
      snprintf(msg, sizeof msg,
               "this batch needs %zu bytes of decode scratch but the static scratch holds %zu; "
               "use mla_decode with a caller workspace",
               need, kScratchBytes);
      return mla::report_error(MLA_ERR_WORKSPACE, msg);
    }
  }
  if (batch == 0 || total_q == 0)  // nothing to do: mla_decode returns before touching the device
    return mla_decode(q_abs, q_pe, cache, num_blocks, page_size, cache_dtype, kv_scale, block_table,
                      max_pages_per_seq, seq_lens, batch, query_start_loc, total_q, num_heads, scale, num_splits,
                      out, lse, nullptr, 0, stream);
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != MLA_OK) return rc;
  // Nothing in the scratch has to start at zero: the plan kernel rewrites
  // every field that the decode and combine kernels read (status word
  // included) before they run, on the same stream.
  return mla_decode(q_abs, q_pe, cache, num_blocks, page_size, cache_dtype, kv_scale, block_table,
                    max_pages_per_seq, seq_lens, batch, query_start_loc, total_q, num_heads, scale, num_splits, out,
                    lse, ws, kScratchBytes, stream);
}
