// C-ABI entry points of libmla.so (declared in include/mla.h): host-side
// argument validation, TMA descriptor encoding and kernel launches.  Nothing
// here allocates device memory; every buffer belongs to the caller.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/mla.h"
#include "common.cuh"
#include "tmap.cuh"

namespace {

thread_local std::string g_last_error;
thread_local cudaEvent_t g_timing_start = nullptr, g_timing_stop = nullptr;
// bounded-wait test settings of the calling thread (mla_set_decode_wait_test)
thread_local int g_test_skip_tile = 0;
thread_local unsigned long long g_wait_limit_ns = 1000000000ull;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return MLA_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}

bool valid_page_size(int ps) { return ps == 16 || ps == 32 || ps == 64 || ps == 128 || ps == 256; }

}  // namespace

namespace mla {
// Lets entry points defined in other translation units report an error
// through mla_last_error().
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace mla

namespace {

// Checks of a cache write's arguments (mla_cache_write, mla_decode_step);
// fills *w when they pass (num_tokens == 0 passes and writes nothing).
int cache_write_args(const void* kv_c, const void* k_pe, const int64_t* slot_mapping, int64_t num_tokens, void* cache,
                     int64_t num_blocks, int page_size, int cache_dtype, float kv_scale, mla::CacheWriteArgs* w) {
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)num_tokens);
  if (cache_dtype != MLA_BF16 && cache_dtype != MLA_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "cache_dtype must be MLA_BF16 or MLA_FP8_E4M3 (got %d)", cache_dtype);
  if (page_size <= 0 || num_blocks <= 0)
    return fail(MLA_ERR_INVALID_ARG, "page_size and num_blocks must be positive");
  if (cache_dtype == MLA_FP8_E4M3 && !(std::isfinite(kv_scale) && kv_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "kv_scale must be finite and > 0 for an fp8 cache");
  *w = mla::CacheWriteArgs{kv_c, k_pe, slot_mapping, num_tokens, cache, num_blocks * page_size, kv_scale,
                           cache_dtype == MLA_FP8_E4M3};
  if (num_tokens == 0) return ok();
  if (!kv_c || !k_pe || !slot_mapping || !cache) return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(kv_c, 16) || !aligned(k_pe, 16) || !aligned(cache, 16) || !aligned(slot_mapping, 8))
    return fail(MLA_ERR_INVALID_ARG, "kv_c, k_pe and cache must be 16-byte aligned, slot_mapping 8-byte aligned");
  return ok();
}

}  // namespace

extern "C" {

const char* mla_last_error(void) { return g_last_error.c_str(); }

int mla_set_decode_timing_events(void* start, void* stop) {
  g_timing_start = start && stop ? static_cast<cudaEvent_t>(start) : nullptr;
  g_timing_stop = start && stop ? static_cast<cudaEvent_t>(stop) : nullptr;
  return ok();
}

int mla_set_decode_wait_test(int skip_first_tile, unsigned long long wait_limit_ns) {
  if (wait_limit_ns == 0) wait_limit_ns = 1000000000ull;
  if (wait_limit_ns < 100000ull || wait_limit_ns > 1000000000ull)
    return fail(MLA_ERR_INVALID_ARG, "wait_limit_ns must be 0 (default 1 s) or in [1e5, 1e9]");
  g_test_skip_tile = skip_first_tile != 0;
  g_wait_limit_ns = wait_limit_ns;
  return ok();
}

int mla_device_sm_count(void) {
  int n = sm_count();
  if (n <= 0) return fail(MLA_ERR_CUDA, "cannot query the current device");
  return n;
}

int mla_cache_write(const void* kv_c, const void* k_pe, const int64_t* slot_mapping, int64_t num_tokens,
                    void* cache, int64_t num_blocks, int page_size, int cache_dtype, float kv_scale,
                    void* stream) {
  mla::CacheWriteArgs w;
  const int rc = cache_write_args(kv_c, k_pe, slot_mapping, num_tokens, cache, num_blocks, page_size, cache_dtype,
                                  kv_scale, &w);
  if (rc != MLA_OK || num_tokens == 0) return rc;
  cudaError_t e = mla::launch_cache_write(w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cache write launch");
  return ok();
}

size_t mla_decode_workspace_size(int batch, int total_q, int num_heads, int max_splits) {
  if (batch <= 0 || total_q <= 0 || num_heads <= 0 || max_splits < 0) return 0;
  return mla::workspace_layout(batch, total_q, num_heads, max_splits).total;
}

}  // extern "C"

namespace {

// The decode of mla_decode (q8 == nullptr: bf16 q_abs and q_pe) and of
// mla_decode_fp8q (q8: e4m3 [q_abs | q_pe] rows with q_scale, e4m3 cache).
int decode_impl(const void* q_abs, const void* q_pe, const void* q8, float q_scale, const void* cache,
                int64_t num_blocks, int page_size, int cache_dtype, float kv_scale, const int32_t* block_table,
                int max_pages_per_seq, const int32_t* seq_lens, int batch, const int32_t* query_start_loc,
                int total_q, int num_heads, float scale, int num_splits, void* out, float* lse, void* workspace,
                size_t workspace_bytes, void* stream, const mla::CacheWriteArgs* write = nullptr,
                const mla::QuantArgs* quant = nullptr) {
  if (batch < 0 || total_q < 0) return fail(MLA_ERR_INVALID_ARG, "batch and total_q must be >= 0");
  if (num_heads < 1 || num_heads > 1024) return fail(MLA_ERR_INVALID_ARG, "num_heads must be in [1, 1024]");
  if (batch == 0 || total_q == 0) return ok();
  if (!query_start_loc && total_q != batch)
    return fail(MLA_ERR_INVALID_ARG, "without query_start_loc every request has one query token (total_q == batch)");
  if ((q8 ? !q8 : (!q_abs || !q_pe)) || !cache || !block_table || !seq_lens || !out || !workspace)
    return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  if ((q8 ? !aligned(q8, 16) : (!aligned(q_abs, 16) || !aligned(q_pe, 16))) || !aligned(cache, 16) ||
      !aligned(out, 16))
    return fail(MLA_ERR_INVALID_ARG, "the query, cache and out must be 16-byte aligned");
  if (q8 && cache_dtype != MLA_FP8_E4M3)
    return fail(MLA_ERR_UNSUPPORTED, "an e4m3 query needs an e4m3 cache");
  if (q8 && !(std::isfinite(q_scale) && q_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "q_scale must be finite and > 0");
  if (q8 && !(std::isnormal(q_scale * kv_scale)))
    return fail(MLA_ERR_INVALID_ARG, "q_scale * kv_scale must be a normal float (the scores' code-product factor)");
  if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || (query_start_loc && !aligned(query_start_loc, 4)) ||
      (lse && !aligned(lse, 4)))
    return fail(MLA_ERR_INVALID_ARG, "block_table, seq_lens, query_start_loc and lse must be 4-byte aligned");
  if (!aligned(workspace, 256)) return fail(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (!valid_page_size(page_size))
    return fail(MLA_ERR_UNSUPPORTED, "page_size must be 16, 32, 64, 128 or 256 (got %d)", page_size);
  if (num_blocks <= 0 || num_blocks * (int64_t)page_size >= (int64_t)1 << 31)
    return fail(MLA_ERR_INVALID_ARG, "num_blocks * page_size must be in [1, 2^31)");
  if (max_pages_per_seq <= 0) return fail(MLA_ERR_INVALID_ARG, "max_pages_per_seq must be positive");
  if ((int64_t)total_q * num_heads >= ((int64_t)1 << 31) - 1024)
    return fail(MLA_ERR_INVALID_ARG, "total_q * num_heads must be below 2^31");
  if (cache_dtype != MLA_BF16 && cache_dtype != MLA_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "cache_dtype must be MLA_BF16 or MLA_FP8_E4M3 (got %d)", cache_dtype);
  if (cache_dtype == MLA_FP8_E4M3 && !(std::isfinite(kv_scale) && kv_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "kv_scale must be finite and > 0 for an fp8 cache");
  if (!std::isfinite(scale) || scale == 0.f) return fail(MLA_ERR_INVALID_ARG, "scale must be finite and nonzero");
  if (num_splits < 0 || num_splits > 4096) return fail(MLA_ERR_INVALID_ARG, "num_splits must be in [0, 4096]");

  const mla::WorkspaceLayout L = mla::workspace_layout(batch, total_q, num_heads, num_splits);
  if (workspace_bytes < L.total)
    return fail(MLA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu required", workspace_bytes, L.total);
  const int sms = sm_count();
  if (sms < 2) return fail(MLA_ERR_CUDA, "cannot query the current device");
  const int clusters = sms / 2 < mla::kMaxClusters ? sms / 2 : mla::kMaxClusters;

  const uint64_t rows = (uint64_t)total_q * num_heads;
  const uint64_t kv_rows = (uint64_t)num_blocks * page_size;
  // Each CTA of a pair reads latent columns [256r, 256r+256) and rope columns
  // [512+32r, 512+32r+32): tensor maps for the latent boxes and the rope boxes
  // of the query and of the cache.
  CUtensorMap tm_q, tm_qr, tm_kv, tm_kvr;
  const uint32_t kv_box_rows = page_size < mla::kTile ? page_size : mla::kTile;
  bool enc;
  if (q8) {
    // e4m3 query rows and cache rows (576 bytes wide): 128-byte latent boxes
    // (128-B swizzle) and 32-byte rope boxes (32-B swizzle)
    enc = mla::encode_tmap_2d(&tm_q, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, mla::kDqk, rows, mla::kDqk, 128, 64,
                              CU_TENSOR_MAP_SWIZZLE_128B) &&
          mla::encode_tmap_2d(&tm_qr, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, mla::kDqk, rows, mla::kDqk, 32, 64,
                              CU_TENSOR_MAP_SWIZZLE_32B) &&
          mla::encode_tmap_2d(&tm_kv, cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, mla::kDqk, kv_rows, mla::kDqk, 128,
                              kv_box_rows, CU_TENSOR_MAP_SWIZZLE_128B) &&
          mla::encode_tmap_2d(&tm_kvr, cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, mla::kDqk, kv_rows, mla::kDqk, 32,
                              kv_box_rows, CU_TENSOR_MAP_SWIZZLE_32B);
  } else {
    // bf16 q_abs (64-dim boxes, 128-B swizzle) and q_pe (32-dim boxes, 64-B swizzle)
    enc = mla::encode_tmap_2d(&tm_q, q_abs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, mla::kLkv, rows, mla::kLkv * 2, 64, 64,
                              CU_TENSOR_MAP_SWIZZLE_128B) &&
          mla::encode_tmap_2d(&tm_qr, q_pe, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, mla::kRope, rows, mla::kRope * 2, 32,
                              64, CU_TENSOR_MAP_SWIZZLE_64B);
    if (cache_dtype == MLA_BF16)
      enc = enc &&
            mla::encode_tmap_2d(&tm_kv, cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, mla::kDqk, kv_rows, mla::kDqk * 2,
                                64, kv_box_rows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            mla::encode_tmap_2d(&tm_kvr, cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, mla::kDqk, kv_rows, mla::kDqk * 2,
                                32, kv_box_rows, CU_TENSOR_MAP_SWIZZLE_64B);
    else  // e4m3 codes land unswizzled and are expanded on chip
      enc = enc &&
            mla::encode_tmap_2d(&tm_kv, cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, mla::kDqk, kv_rows, mla::kDqk, 64,
                                kv_box_rows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            mla::encode_tmap_2d(&tm_kvr, cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, mla::kDqk, kv_rows, mla::kDqk, 32,
                                kv_box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  // the epilogue stores whole 32-row x 64-dim pieces of the output and of the
  // split partials with TMA (128-B swizzle, as they are staged on chip)
  const mla::Plan plan = mla::plan_from_workspace(workspace, L);
  CUtensorMap tm_out, tm_part;
  enc = enc &&
        mla::encode_tmap_2d(&tm_out, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, mla::kLkv, rows, mla::kLkv * 2, 64, 32,
                            CU_TENSOR_MAP_SWIZZLE_128B) &&
        mla::encode_tmap_2d(&tm_part, plan.part_o, CU_TENSOR_MAP_DATA_TYPE_UINT16, mla::kLkv,
                            (uint64_t)L.max_units * mla::kRows, mla::kLkv * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!enc) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor layout");

  mla::DecodeArgs a{};
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.qsl = query_start_loc;
  a.batch = batch;
  a.num_heads = num_heads;
  a.max_pages = max_pages_per_seq;
  a.page_size = page_size;
  a.num_blocks = (int)num_blocks;
  a.total_rows = (int)rows;
  // an e4m3 row holds value / kv_scale: the scale folds into the scores and the output
  const float kvs = cache_dtype == MLA_FP8_E4M3 ? kv_scale : 1.f;
  // the kernel works with a positive scale; a negative one negates q instead
  a.scale_log2 = std::fabs(scale) * 1.4426950408889634f * kvs;
  if (q8) {
    // the e4m3-query kernel turns its code-product sums into real partial
    // scores (x q_scale x kv_scale) before the exchange
    a.qk_scale = q_scale * kv_scale;
    a.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  }
  a.neg_q = scale < 0.f;
  a.out_scale = kvs;
  a.out = out;
  a.lse = lse;
  a.wait_limit_ns = g_wait_limit_ns;
  a.debug_skip_tile = g_test_skip_tile;
  a.plan = plan;

  cudaStream_t s = (cudaStream_t)stream;
  // small head counts with one query token per request (total_q == batch):
  // 32-row groups and the decode variant with small receive buffers and a
  // deeper cache ring.  Groups never outnumber the batch then: a request with
  // Sq tokens gives ceil(Sq * N / 32) <= Sq groups.
  const int small_rows = !q8 && cache_dtype == MLA_BF16 && num_heads <= 32 && total_q == batch;
  const int variant = q8 ? 3 : (cache_dtype == MLA_FP8_E4M3 ? 1 : (small_rows ? 2 : 0));
  cudaError_t e = mla::launch_plan(seq_lens, query_start_loc, batch, num_heads, max_pages_per_seq, page_size,
                                   num_splits, clusters, small_rows ? 32 : mla::kRows, a.plan, write, quant, sms,
                                   s);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  const bool timed = g_timing_start && g_timing_stop;
  if (timed && (e = cudaEventRecord(g_timing_start, s)) != cudaSuccess) return cuda_fail(e, "timing event");
  e = mla::launch_decode(tm_q, tm_qr, tm_kv, tm_kvr, tm_out, tm_part, variant, a, clusters, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (timed && (e = cudaEventRecord(g_timing_stop, s)) != cudaSuccess) return cuda_fail(e, "timing event");
  e = mla::launch_combine(a, L.max_groups, sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return ok();
}

}  // namespace

extern "C" {

int mla_decode(const void* q_abs, const void* q_pe, const void* cache, int64_t num_blocks, int page_size,
               int cache_dtype, float kv_scale, const int32_t* block_table, int max_pages_per_seq,
               const int32_t* seq_lens, int batch, const int32_t* query_start_loc, int total_q, int num_heads,
               float scale, int num_splits, void* out, float* lse, void* workspace, size_t workspace_bytes,
               void* stream) {
  return decode_impl(q_abs, q_pe, nullptr, 0.f, cache, num_blocks, page_size, cache_dtype, kv_scale, block_table,
                     max_pages_per_seq, seq_lens, batch, query_start_loc, total_q, num_heads, scale, num_splits, out,
                     lse, workspace, workspace_bytes, stream);
}

int mla_decode_step(const void* kv_c, const void* k_pe, const int64_t* slot_mapping, int64_t num_new_tokens,
                    const void* q_abs, const void* q_pe, void* cache, int64_t num_blocks, int page_size,
                    int cache_dtype, float kv_scale, const int32_t* block_table, int max_pages_per_seq,
                    const int32_t* seq_lens, int batch, const int32_t* query_start_loc, int total_q, int num_heads,
                    float scale, int num_splits, void* out, float* lse, void* workspace, size_t workspace_bytes,
                    void* stream) {
  mla::CacheWriteArgs w;
  const int rc = cache_write_args(kv_c, k_pe, slot_mapping, num_new_tokens, cache, num_blocks, page_size,
                                  cache_dtype, kv_scale, &w);
  if (rc != MLA_OK) return rc;
  if (batch == 0 || total_q == 0)   // no decode: the write alone
    return mla_cache_write(kv_c, k_pe, slot_mapping, num_new_tokens, cache, num_blocks, page_size, cache_dtype,
                           kv_scale, stream);
  return decode_impl(q_abs, q_pe, nullptr, 0.f, cache, num_blocks, page_size, cache_dtype, kv_scale, block_table,
                     max_pages_per_seq, seq_lens, batch, query_start_loc, total_q, num_heads, scale, num_splits, out,
                     lse, workspace, workspace_bytes, stream, num_new_tokens > 0 ? &w : nullptr);
}

int mla_decode_fp8q_step(const void* kv_c, const void* k_pe, const int64_t* slot_mapping, int64_t num_new_tokens,
                         const void* q_abs, const void* q_pe, float q_scale, void* q_fp8, void* cache,
                         int64_t num_blocks, int page_size, float kv_scale, const int32_t* block_table,
                         int max_pages_per_seq, const int32_t* seq_lens, int batch, const int32_t* query_start_loc,
                         int total_q, int num_heads, float scale, int num_splits, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream) {
  mla::CacheWriteArgs w;
  int rc = cache_write_args(kv_c, k_pe, slot_mapping, num_new_tokens, cache, num_blocks, page_size, MLA_FP8_E4M3,
                            kv_scale, &w);
  if (rc != MLA_OK) return rc;
  if (batch == 0 || total_q == 0)   // no decode: the write alone
    return mla_cache_write(kv_c, k_pe, slot_mapping, num_new_tokens, cache, num_blocks, page_size, MLA_FP8_E4M3,
                           kv_scale, stream);
  if (!q_abs || !q_pe || !q_fp8) return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q_abs, 16) || !aligned(q_pe, 16) || !aligned(q_fp8, 16))
    return fail(MLA_ERR_INVALID_ARG, "q_abs, q_pe and q_fp8 must be 16-byte aligned");
  if (!(std::isfinite(q_scale) && q_scale > 0.f)) return fail(MLA_ERR_INVALID_ARG, "q_scale must be finite and > 0");
  if (total_q < 0 || num_heads < 1 || num_heads > 1024)
    return fail(MLA_ERR_INVALID_ARG, "total_q must be >= 0 and num_heads in [1, 1024]");
  const mla::QuantArgs qa{q_abs, q_pe, (int64_t)total_q * num_heads, q_scale, static_cast<uint8_t*>(q_fp8)};
  return decode_impl(nullptr, nullptr, q_fp8, q_scale, cache, num_blocks, page_size, MLA_FP8_E4M3, kv_scale,
                     block_table, max_pages_per_seq, seq_lens, batch, query_start_loc, total_q, num_heads, scale,
                     num_splits, out, lse, workspace, workspace_bytes, stream, num_new_tokens > 0 ? &w : nullptr,
                     &qa);
}

int mla_decode_fp8q(const void* q_fp8, float q_scale, const void* cache, int64_t num_blocks, int page_size,
                    float kv_scale, const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                    int batch, const int32_t* query_start_loc, int total_q, int num_heads, float scale,
                    int num_splits, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(nullptr, nullptr, q_fp8, q_scale, cache, num_blocks, page_size, MLA_FP8_E4M3, kv_scale,
                     block_table, max_pages_per_seq, seq_lens, batch, query_start_loc, total_q, num_heads, scale,
                     num_splits, out, lse, workspace, workspace_bytes, stream);
}

int mla_decode_status(const void* workspace, int* status, void* stream) {
  if (!workspace || !status) return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(status, workspace, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  return ok();
}

int mla_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, int64_t rows, int dim,
                     int o_dtype, void* out, float* lse_out, void* stream) {
  if (rows < 0) return fail(MLA_ERR_INVALID_ARG, "rows must be >= 0");
  if (dim <= 0 || dim % 8 != 0 || dim > 4096) return fail(MLA_ERR_INVALID_ARG, "dim must be a multiple of 8 in [8, 4096]");
  if (o_dtype != MLA_BF16 && o_dtype != MLA_FP32)
    return fail(MLA_ERR_INVALID_ARG, "o_dtype must be MLA_BF16 or MLA_FP32 (got %d)", o_dtype);
  if (rows == 0) return ok();
  if (!o_a || !lse_a || !o_b || !lse_b || !out) return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(out, 16))
    return fail(MLA_ERR_INVALID_ARG, "o_a, o_b and out must be 16-byte aligned");
  if (!aligned(lse_a, 4) || !aligned(lse_b, 4) || (lse_out && !aligned(lse_out, 4)))
    return fail(MLA_ERR_INVALID_ARG, "LSE arrays must be 4-byte aligned");
  if (lse_out && (lse_out == lse_a || lse_out == lse_b))
    return fail(MLA_ERR_INVALID_ARG, "lse_out must not alias lse_a or lse_b");
  const int sms = sm_count();   // of the current device, per call
  if (sms < 1) return fail(MLA_ERR_CUDA, "cannot query the current device");
  cudaError_t e = mla::launch_merge_states(o_a, lse_a, o_b, lse_b, rows, dim, o_dtype == MLA_BF16, out, lse_out,
                                           sms, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return ok();
}

}  // extern "C"

namespace {

// Shared body of the two per-head projections: validation of what both have
// in common, tensor maps, launch.
int head_proj(const char* name, const void* x, int64_t x_stride, const void* w, int64_t T, int N, int d_in,
              int d_out, void* y, void* stream) {
  if (T < 0) return fail(MLA_ERR_INVALID_ARG, "%s: num_tokens must be >= 0", name);
  if (T > 65535LL * 128) return fail(MLA_ERR_UNSUPPORTED, "%s: num_tokens must be <= 8388480", name);
  if (N < 1 || N > 1024) return fail(MLA_ERR_INVALID_ARG, "%s: num_heads must be in [1, 1024]", name);
  if (T == 0) return ok();
  if (!x || !w || !y) return fail(MLA_ERR_INVALID_ARG, "%s: null pointer argument", name);
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16))
    return fail(MLA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", name);
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x), yb = reinterpret_cast<uintptr_t>(y);
  const uintptr_t xe = xb + (uintptr_t)((T * N - 1) * x_stride + d_in) * 2, ye = yb + (uintptr_t)(T * N * d_out) * 2;
  if (xb < ye && yb < xe) return fail(MLA_ERR_INVALID_ARG, "%s: the output must not overlap the input", name);
  CUtensorMap tm_x, tm_w;
  if (!mla::encode_tmap_3d(&tm_x, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)d_in, (uint64_t)N, (uint64_t)T,
                           (uint64_t)x_stride * 2, (uint64_t)x_stride * 2 * N, 64, 1,
                           (uint32_t)mla::head_proj_x_rows(T),
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
      !mla::encode_tmap_2d(&tm_w, w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)d_out, (uint64_t)N * d_in,
                           (uint64_t)d_out * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(MLA_ERR_CUDA, "%s: tensor map encoding failed", name);
  cudaError_t e = mla::launch_head_proj(tm_x, tm_w, y, T, N, d_in, d_out, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}

}  // namespace

extern "C" {

int mla_q_absorb(const void* q_nope, int64_t q_row_stride, const void* w_uk_t, int64_t num_tokens, int num_heads,
                 int nope_dim, void* ql_nope, void* stream) {
  if (nope_dim < 64 || nope_dim > 1024 || nope_dim % 64 != 0)
    return fail(MLA_ERR_UNSUPPORTED, "mla_q_absorb: nope_dim must be a multiple of 64 in [64, 1024] (got %d)",
                nope_dim);
  if (q_row_stride < nope_dim || q_row_stride % 8 != 0 || q_row_stride > (1LL << 24))
    return fail(MLA_ERR_INVALID_ARG, "mla_q_absorb: q_row_stride must be >= nope_dim, a multiple of 8 and <= 2^24");
  return head_proj("mla_q_absorb", q_nope, q_row_stride, w_uk_t, num_tokens, num_heads, nope_dim, mla::kLkv,
                   ql_nope, stream);
}

int mla_v_up_proj(const void* o_lat, const void* w_uv, int64_t num_tokens, int num_heads, int v_head_dim, void* out,
                  void* stream) {
  const bool ok_dim = (v_head_dim >= 64 && v_head_dim <= 256 && v_head_dim % 64 == 0) || v_head_dim == 512 ||
                      v_head_dim == 1024;
  if (!ok_dim)
    return fail(MLA_ERR_UNSUPPORTED, "mla_v_up_proj: v_head_dim must be 64, 128, 192, 256, 512 or 1024 (got %d)",
                v_head_dim);
  return head_proj("mla_v_up_proj", o_lat, mla::kLkv, w_uv, num_tokens, num_heads, mla::kLkv, v_head_dim, out,
                   stream);
}

int mla_gather_cache(const void* cache, int64_t num_blocks, int page_size, int cache_dtype, float kv_scale,
                     const int32_t* block_table, int max_pages_per_seq, const int32_t* cu_seq_lens,
                     const int32_t* seq_starts, int batch, void* dst, int64_t num_tokens, int32_t* status,
                     void* stream) {
  if (num_tokens < 0 || batch < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens and batch must be >= 0");
  if (cache_dtype != MLA_BF16 && cache_dtype != MLA_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "cache_dtype must be MLA_BF16 or MLA_FP8_E4M3 (got %d)", cache_dtype);
  if (num_tokens == 0 || batch == 0) return ok();
  if (page_size < 1 || num_blocks < 1 || max_pages_per_seq < 1)
    return fail(MLA_ERR_INVALID_ARG, "page_size, num_blocks and max_pages_per_seq must be positive");
  if (cache_dtype == MLA_FP8_E4M3 && !(std::isfinite(kv_scale) && kv_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "kv_scale must be finite and > 0 for an fp8 cache");
  if (!cache || !block_table || !cu_seq_lens || !dst) return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(cache, 16) || !aligned(dst, 16)) return fail(MLA_ERR_INVALID_ARG, "cache and dst must be 16-byte aligned");
  if (!aligned(block_table, 4) || !aligned(cu_seq_lens, 4) || (seq_starts && !aligned(seq_starts, 4)) ||
      (status && !aligned(status, 4)))
    return fail(MLA_ERR_INVALID_ARG, "block_table, cu_seq_lens, seq_starts and status must be 4-byte aligned");
  cudaError_t e = mla::launch_gather(cache, num_blocks, page_size, cache_dtype == MLA_FP8_E4M3, kv_scale,
                                     block_table, max_pages_per_seq, cu_seq_lens, seq_starts, batch, dst,
                                     num_tokens, status, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  return ok();
}

int mla_quantize_fp8(const void* x, int64_t x_stride, int64_t rows, int width, float scale, void* out,
                     int64_t out_stride, void* stream) {
  if (rows < 0) return fail(MLA_ERR_INVALID_ARG, "rows must be >= 0");
  if (width <= 0 || width % 8 != 0) return fail(MLA_ERR_INVALID_ARG, "width must be a positive multiple of 8");
  if (x_stride < width || x_stride % 8 != 0 || out_stride < width || out_stride % 8 != 0)
    return fail(MLA_ERR_INVALID_ARG, "strides must be multiples of 8 and at least width");
  if (!(std::isfinite(scale) && scale > 0.f)) return fail(MLA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (rows == 0) return ok();
  if (!x || !out) return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(x, 16) || !aligned(out, 8)) return fail(MLA_ERR_INVALID_ARG, "x must be 16-byte and out 8-byte aligned");
  cudaError_t e = mla::launch_quantize_fp8(x, x_stride, rows, width, scale, out, out_stride, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return ok();
}

int mla_proj_status(int* status, int clear, void* stream) {
  if (!status) return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  cudaError_t e = mla::head_proj_status(status, clear, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "projection status read");
  return ok();
}

}  // extern "C"
