/*
 * mla.h -- C ABI of libmla.so: absorbed ("data-movement friendly") Multi-head
 * Latent Attention decode over a paged latent KV cache, for NVIDIA GB300
 * (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers to dense, row-major tensors
 *    (no strides) that the caller allocates and owns.  The library keeps no
 *    pointer after a call returns and allocates no memory: scratch memory
 *    comes from the caller (`workspace`).
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Every call is asynchronous with respect to the host: it only
 *    enqueues kernels on `stream`.
 *  - Return value: MLA_OK (0) or a negative mla_status.  Arguments are
 *    validated on the host BEFORE anything is enqueued; on an error nothing
 *    is launched and mla_last_error() describes the problem.  Device-side
 *    data (slot ids, block-table entries, sequence lengths) cannot be checked
 *    on the host; how each call treats bad values is stated below.
 *  - Latent widths are fixed by the model family: Lkv = 512 (kv_c / q_abs /
 *    output), R = 64 (k_pe / q_pe), cache row = Lkv + R = 576 elements
 *    (vllm/v1/attention/backends/mla/common.py, module docstring, "More
 *    Extent Definitions", DeepSeek-V3 values).
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size or enum    */
  MLA_ERR_UNSUPPORTED = -2, /* valid request outside what the kernels cover  */
  MLA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed             */
  MLA_ERR_WORKSPACE = -4    /* workspace missing or smaller than required   */
};

enum mla_dtype {
  MLA_BF16 = 0,     /* bfloat16                                        */
  MLA_FP8_E4M3 = 1, /* OCP FP8 E4M3 ("fn": no inf, max 448)            */
  MLA_FP32 = 2      /* float32 (merge inputs/outputs only)              */
};

/* Device error word bits written by mla_decode (see mla_decode_status). */
enum mla_device_error {
  MLA_DEVERR_TIMEOUT = 1,       /* a bounded on-chip wait gave up          */
  MLA_DEVERR_BAD_SEQ_LEN = 2,   /* seq_len > max_pages_per_seq*page_size   */
  MLA_DEVERR_BAD_BLOCK = 4,     /* block-table entry outside [0,num_blocks) */
  MLA_DEVERR_BAD_QSL = 8        /* query_start_loc inconsistent with total_q */
};

/*
 * mla_cache_write -- concat_and_cache_mla: store the latent rows of new tokens
 * in the paged cache (page "vllm/v1/attention/backends/mla/common.py",
 * MLACommonImpl.forward, the cache update before the attention; page
 * "vllm.model_executor.layers.attention.mla_attention", MLAAttention.forward
 * and do_kv_cache_update).
 *
 *   kv_c          [num_tokens, 512] bf16, 16-byte aligned
 *   k_pe          [num_tokens, 64]  bf16, 16-byte aligned
 *   slot_mapping  [num_tokens] int64: flattened cache row of each token,
 *                 slot = block * page_size + offset_in_block; a negative slot
 *                 marks a padding token and is skipped.  Slots >= num_blocks *
 *                 page_size are skipped as well (device data is not checked
 *                 on the host).
 *   cache         [num_blocks, page_size, 576] of cache_dtype, 16-byte aligned;
 *                 row `slot` receives [kv_c | k_pe].
 *   cache_dtype   MLA_BF16: the bf16 bits are copied unchanged.
 *                 MLA_FP8_E4M3: each value x is stored as e4m3(x / kv_scale),
 *                 float32 divide, round to nearest even, finite overflow
 *                 saturated to +-448 (kv_scale = abs-max / 448 as in
 *                 calc_kv_scales; dequantisation multiplies by kv_scale).
 *   kv_scale      > 0 and finite for fp8; ignored for bf16.
 * num_tokens == 0 is a no-op.  One launch.
 */
MLA_API int mla_cache_write(const void* kv_c, const void* k_pe, const int64_t* slot_mapping, int64_t num_tokens,
                    void* cache, int64_t num_blocks, int page_size, int cache_dtype, float kv_scale,
                    void* stream);

/*
 * mla_decode_workspace_size -- bytes of device workspace mla_decode needs for
 * a batch of `batch` requests, `total_q` query tokens in all, `num_heads`
 * heads, and a split count num_splits <= max_splits (pass 0 when only the
 * automatic split is used).  Depends on sizes only, never on device data, so
 * a buffer sized once serves every later step of the same shape (and every
 * CUDA-graph replay).
 */
MLA_API size_t mla_decode_workspace_size(int batch, int total_q, int num_heads, int max_splits);

/*
 * mla_decode -- absorbed MLA decode (forward_mqa): for every query row
 * (token t, head h) attend, as MQA, over the request's latent rows
 * [kv_c | k_pe] reached through its block table, and return the 512-wide
 * latent output and the natural-log LSE (common.py docstring,
 * "Data-Movement Friendly Approach"; mla_attention.py MLACommonImpl.forward_mqa
 * returns (o, lse)):
 *
 *   s_j   = scale * (q_abs[t,h] . kv_c_j + q_pe[t,h] . k_pe_j)
 *   out   = sum_j softmax(s)_j * kv_c_j          lse = ln sum_j exp(s_j)
 *
 * over keys j < L(t) = seq_len[b] - Sq_b + 1 + t_local: with Sq_b query tokens
 * a request's t-th verify token sees its context plus the new tokens up to
 * itself (rocm_aiter_mla.py, AiterMLAImpl.forward_mqa, multi-token verify).
 * Long contexts are split across CTAs and recombined with the LSE merge
 * (merge_attn_states).  Rows with L(t) <= 0 (e.g. seq_len 0 padding requests)
 * get out = 0 and lse = -inf.
 *
 *   q_abs            [total_q, num_heads, 512] bf16 (ql_nope = q_nope . W_UK)
 *   q_pe             [total_q, num_heads, 64]  bf16
 *   cache            [num_blocks, page_size, 576] of cache_dtype (bf16 or e4m3)
 *   kv_scale         fp8 dequantisation scale (row value = code * kv_scale);
 *                    ignored for bf16
 *   block_table      [batch, max_pages_per_seq] int32: physical block of each
 *                    logical page; token j of request b is row
 *                    block_table[b, j / page_size] * page_size + j % page_size
 *   seq_lens         [batch] int32: tokens of each request INCLUDING its query
 *                    tokens of this step
 *   query_start_loc  [batch + 1] int32 prefix sums of per-request query counts
 *                    (query_start_loc[0] = 0, [batch] = total_q), or NULL for
 *                    one query token per request (then total_q == batch)
 *   num_heads        1..1024
 *   scale            softmax scale, passed explicitly (1/sqrt(P+R) for MLA);
 *                    finite and nonzero
 *   num_splits       0: split long contexts automatically to balance all SMs;
 *                    k > 0: cut every (request, 128-row group) into
 *                    min(k, tiles) contiguous pieces of near-equal length
 *   out              [total_q, num_heads, 512] bf16
 *   lse              [total_q, num_heads] float32, or NULL
 *   workspace        >= mla_decode_workspace_size(batch, total_q, num_heads,
 *                    num_splits) bytes, 256-byte aligned; scratch only
 *   page_size        16, 32, 64, 128 or 256
 * All device pointers 16-byte aligned.  Launches: a scheduler kernel, the
 * decode kernel and a combine kernel.  Device data errors (seq_len beyond
 * the block table, block ids outside the cache) do not fault: the affected
 * rows read zeros and a bit of mla_device_error is set in the workspace's
 * status word (mla_decode_status).
 */
MLA_API int mla_decode(const void* q_abs, const void* q_pe, const void* cache, int64_t num_blocks, int page_size,
               int cache_dtype, float kv_scale, const int32_t* block_table, int max_pages_per_seq,
               const int32_t* seq_lens, int batch, const int32_t* query_start_loc, int total_q,
               int num_heads, float scale, int num_splits, void* out, float* lse, void* workspace,
               size_t workspace_bytes, void* stream);

/*
 * mla_decode_step -- one decode step: mla_cache_write of the step's new rows
 * (kv_c [num_new_tokens, 512] bf16, k_pe [num_new_tokens, 64] bf16 into the
 * slots slot_mapping [num_new_tokens] int64, a negative slot is padding),
 * then mla_decode over the updated cache: the same results as the two calls
 * in that order, with the same argument rules.  The rows are written by
 * extra blocks of the scheduler's launch, which run beside the split plan,
 * so the write costs the step no launch of its own.  num_new_tokens == 0
 * writes nothing; batch == 0 or total_q == 0 only writes.
 */
MLA_API int mla_decode_step(const void* kv_c, const void* k_pe, const int64_t* slot_mapping, int64_t num_new_tokens,
                            const void* q_abs, const void* q_pe, void* cache, int64_t num_blocks, int page_size,
                            int cache_dtype, float kv_scale, const int32_t* block_table, int max_pages_per_seq,
                            const int32_t* seq_lens, int batch, const int32_t* query_start_loc, int total_q,
                            int num_heads, float scale, int num_splits, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * mla_decode_status -- copy the device error word of the last mla_decode that
 * used `workspace` (OR of mla_device_error bits; 0 = clean) to *status.
 * Synchronises `stream`.  The word is cleared by every mla_decode.
 */
MLA_API int mla_decode_status(const void* workspace, int* status, void* stream);

/*
 * mla_merge_states -- merge_attn_states: combine two partial attention
 * results over disjoint key sets (common.py docstring, "Chunked Prefill";
 * MLACommonImpl._compute_prefill_context):
 *
 *   lse = ln(exp(lse_a) + exp(lse_b))
 *   out = exp(lse_a - lse) * o_a + exp(lse_b - lse) * o_b
 *
 * A side with lse = -inf (no keys) gets weight 0; both -inf gives out = 0,
 * lse = -inf.
 *   o_a, o_b, out   [rows, dim] of o_dtype (MLA_BF16 or MLA_FP32)
 *   lse_a, lse_b    [rows] float32 natural-log LSE
 *   lse_out         [rows] float32, or NULL; must not alias lse_a or lse_b
 *   dim             multiple of 8, <= 4096
 * rows == 0 is a no-op.  out may alias o_a or o_b.  One launch.
 */
MLA_API int mla_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, int64_t rows,
                     int dim, int o_dtype, void* out, float* lse_out, void* stream);

/*
 * mla_set_decode_timing_events -- profiling aid.  While both events are
 * non-NULL, every later mla_decode call of the calling thread records `start`
 * immediately before and `stop` immediately after its decode kernel, on the
 * call's stream, so the kernel can be timed alone with cudaEventElapsedTime.
 * The events (cudaEvent_t passed as void*) belong to the caller.  Passing NULL
 * for either turns the recording off.  Always returns MLA_OK.
 */
MLA_API int mla_set_decode_timing_events(void* start, void* stop);

/*
 * mla_decode_no_alloc -- mla_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart of this entry point; it exists for
 * callers that are not allowed to call cudaMalloc or any other allocating
 * routine around a decode step (for example while a CUDA graph is being
 * captured, or in a runtime whose host framework owns every device buffer).
 *
 * Arguments and results are those of mla_decode without `workspace` and
 * `workspace_bytes`: inputs and outputs still come from the caller.  The
 * split-KV scratch is a fixed device array of MLA_NO_ALLOC_SCRATCH_BYTES
 * (96 MiB) inside the library; every GPU that loads the library holds it until
 * the process exits.  A batch whose scratch need
 * (mla_decode_workspace_size(batch, total_q, num_heads, num_splits)) exceeds
 * it is rejected with MLA_ERR_WORKSPACE before anything is enqueued.  The
 * first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  No call
 * allocates memory.
 *
 * All calls share the one array and it keeps the last call's contents, so
 * calls that may overlap on the GPU (different streams, different host
 * threads) race: serialise them on one stream.  The device error word of
 * these calls lives in the shared array; mla_decode_no_alloc_status reads it.
 */
#define MLA_NO_ALLOC_SCRATCH_BYTES ((size_t)96 << 20)
MLA_API int mla_decode_no_alloc(const void* q_abs, const void* q_pe, const void* cache, int64_t num_blocks,
                                int page_size, int cache_dtype, float kv_scale, const int32_t* block_table,
                                int max_pages_per_seq, const int32_t* seq_lens, int batch,
                                const int32_t* query_start_loc, int total_q, int num_heads, float scale,
                                int num_splits, void* out, float* lse, void* stream);

/*
 * mla_decode_no_alloc_status -- the device error word (OR of mla_device_error
 * bits; 0 = clean) of the last mla_decode_no_alloc on the current device,
 * copied to *status; cleared afterwards if `clear` is non-zero.  Like
 * mla_decode_no_alloc it has no counterpart on the pages: it gives the
 * callers that cannot allocate the same view of bad block-table entries,
 * bad sequence lengths and expired on-chip waits that mla_decode_status gives
 * workspace callers.  Synchronises `stream`; allocates nothing.
 */
MLA_API int mla_decode_no_alloc_status(int* status, int clear, void* stream);

/*
 * mla_q_absorb -- query absorption of the decode branch (page
 * "vllm/v1/attention/backends/mla/common.py", MLACommonImpl.forward: the
 * no-rope part of every head's query is multiplied by that head's W_UK_T with
 * a batched matmul over heads; the module docstring's ql_nope in the
 * "Data-Movement Friendly Approach"):
 *
 *   ql_nope[t, n, l] = sum_p q_nope[t, n, p] * w_uk_t[n, p, l]
 *
 * written as [num_tokens, num_heads, 512] bf16, the q_abs layout mla_decode
 * reads.  Products accumulate in float32 on the tensor cores; the result is
 * rounded to bf16 (nearest even).
 *   q_nope        bf16, row (t, n) at q_nope + (t * num_heads + n) * q_row_stride
 *                 elements; q_row_stride >= nope_dim and a multiple of 8 (192
 *                 reads the first 128 columns of q = [q_nope | q_pe]);
 *                 16-byte aligned
 *   w_uk_t        [num_heads, nope_dim, 512] bf16, dense (W_UK_T in the (N, P, L)
 *                 order process_weights_after_loading stores), 16-byte aligned
 *   ql_nope       [num_tokens, num_heads, 512] bf16, dense, 16-byte aligned;
 *                 must not overlap q_nope
 *   nope_dim      multiple of 64 in [64, 1024] (DeepSeek-V3: 128)
 *   num_heads     [1, 1024]; num_tokens in [0, 8388480]; 0 is a no-op.
 * One launch (a programmatic dependent of the previous kernel on `stream`).
 * Device-side timeouts set MLA_DEVERR_TIMEOUT in the word mla_proj_status reads.
 */
MLA_API int mla_q_absorb(const void* q_nope, int64_t q_row_stride, const void* w_uk_t, int64_t num_tokens,
                         int num_heads, int nope_dim, void* ql_nope, void* stream);

/*
 * mla_v_up_proj -- the value up-projection after the latent decode (page
 * "vllm/v1/attention/backends/mla/common.py", MLACommonBaseImpl._v_up_proj:
 * every head's latent output is multiplied by that head's W_UV with a batched
 * matmul over heads; the module docstring's last step of the "Data-Movement
 * Friendly Approach"):
 *
 *   out[t, n, v] = sum_l o_lat[t, n, l] * w_uv[n, l, v]
 *
 * written as [num_tokens, num_heads, v_head_dim] bf16 (= the [T, N * V] input
 * of the output projection).  float32 accumulation, bf16 result (nearest even).
 *   o_lat         [num_tokens, num_heads, 512] bf16, dense (mla_decode's out),
 *                 16-byte aligned
 *   w_uv          [num_heads, 512, v_head_dim] bf16, dense (W_UV in the (N, L, V)
 *                 order process_weights_after_loading stores), 16-byte aligned
 *   out           [num_tokens, num_heads, v_head_dim] bf16, dense, 16-byte
 *                 aligned; must not overlap o_lat
 *   v_head_dim    multiple of 64 in [64, 256], or 512 or 1024 (DeepSeek-V3: 128)
 *   num_heads     [1, 1024]; num_tokens in [0, 8388480]; 0 is a no-op.
 * One launch, as for mla_q_absorb.
 */
MLA_API int mla_v_up_proj(const void* o_lat, const void* w_uv, int64_t num_tokens, int num_heads, int v_head_dim,
                          void* out, void* stream);

/*
 * mla_proj_status -- copy the device error word of the projection kernels
 * (mla_q_absorb, mla_v_up_proj; OR of mla_device_error bits, 0 = clean) to
 * *status, then clear it if `clear` is non-zero.  The word is shared by every
 * projection launched in the process on the current device.  Synchronises
 * `stream`.
 */
MLA_API int mla_proj_status(int* status, int clear, void* stream);

/*
 * mla_decode_fp8q -- mla_decode with an e4m3 query over an e4m3 cache: the
 * decode branch's fp8 path (common.py, MLACommonImpl.forward: with an fp8
 * cache the absorbed query and q_pe are quantised by scaled_fp8_quant with
 * layer._q_scale, and the kernels get q_scale and k_scale; the scores'
 * factor is scale * q_scale * k_scale, as FlashInferImpl.get_xqa_bmm1_scale
 * forms it).  The score products run on the fp8 tensor cores (e4m3 x e4m3,
 * float32 accumulation); P.V stays bf16 x bf16 (values expanded exactly).
 *   q_fp8     [total_q, num_heads, 576] e4m3 codes, rows [q_abs | q_pe]
 *             quantised with q_scale (mla_quantize_fp8), 16-byte aligned
 *   q_scale   finite and > 0, with q_scale * kv_scale a normal float32
 *   the cache must be e4m3 (kv_scale finite and > 0); every other argument,
 *   the output, the LSE, the workspace and the error behaviour are those of
 *   mla_decode.
 */
MLA_API int mla_decode_fp8q(const void* q_fp8, float q_scale, const void* cache, int64_t num_blocks, int page_size,
                            float kv_scale, const int32_t* block_table, int max_pages_per_seq,
                            const int32_t* seq_lens, int batch, const int32_t* query_start_loc, int total_q,
                            int num_heads, float scale, int num_splits, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * mla_decode_fp8q_step -- one e4m3-query step: mla_cache_write of the step's
 * new rows into the e4m3 cache, mla_quantize_fp8 of q_abs [total_q,
 * num_heads, 512] and q_pe [total_q, num_heads, 64] (bf16, dense) with
 * q_scale into q_fp8 [total_q, num_heads, 576] (e4m3 codes of [q_abs | q_pe],
 * written by this call), then mla_decode_fp8q: the same results as those
 * calls in that order, with the same argument rules.  The cache rows and the
 * query codes are written by extra blocks of the scheduler's launch, beside
 * the split plan.  num_new_tokens == 0 writes no cache row; batch == 0 or
 * total_q == 0 only writes the cache rows.
 */
MLA_API int mla_decode_fp8q_step(const void* kv_c, const void* k_pe, const int64_t* slot_mapping,
                                 int64_t num_new_tokens, const void* q_abs, const void* q_pe, float q_scale,
                                 void* q_fp8, void* cache, int64_t num_blocks, int page_size, float kv_scale,
                                 const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                                 int batch, const int32_t* query_start_loc, int total_q, int num_heads, float scale,
                                 int num_splits, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * mla_quantize_fp8 -- scaled_fp8_quant with a static per-tensor scale, as the
 * decode branch applies it to the absorbed query and q_pe when the cache is
 * fp8 (common.py, MLACommonImpl.forward: scaled_fp8_quant(..., layer._q_scale)):
 *
 *   out[r * out_stride + c] = e4m3(float32(x[r * x_stride + c]) / float32(scale))
 *
 * for r < rows, c < width (float32 divide, round to nearest even, finite
 * overflow saturated to +-448; the cache write's rule).  The strides let
 * q_abs and q_pe go straight into the [q_abs | q_pe] rows mla_decode_fp8q reads.
 *   x      bf16, 16-byte aligned, x_stride (elements) a multiple of 8
 *   out    e4m3 codes, 8-byte aligned, out_stride (elements) a multiple of 8
 *   width  a multiple of 8, <= both strides;  rows >= 0 (0 is a no-op)
 *   scale  finite and > 0.  One launch.
 */
MLA_API int mla_quantize_fp8(const void* x, int64_t x_stride, int64_t rows, int width, float scale, void* out,
                             int64_t out_stride, void* stream);

/*
 * mla_gather_cache -- gather_and_maybe_dequant_cache of the chunked-prefill
 * context path (common.py, MLACommonImpl._compute_prefill_context, with the
 * chunk metadata of MLACommonMetadataBuilder): copy the latent rows of a
 * context chunk of every request out of the paged cache into a dense bf16
 * workspace.
 *
 *   dst[cu_seq_lens[b] + j] = row at context position seq_starts[b] + j of
 *                             request b, j < cu_seq_lens[b+1] - cu_seq_lens[b],
 *   row at position p = cache[block_table[b, p / page_size], p % page_size]
 *
 * A bf16 cache is copied bit for bit; an e4m3 cache is dequantised to
 * bf16(float32(code) * kv_scale) (float32 product, round to nearest even).
 *   cache         [num_blocks, page_size, 576] of cache_dtype, 16-byte aligned;
 *                 page_size >= 1 (chunk starts need not be page aligned)
 *   block_table   [batch, max_pages_per_seq] int32
 *   cu_seq_lens   [batch + 1] int32 on the device, cu_seq_lens[0] = 0,
 *                 non-decreasing
 *   seq_starts    [batch] int32 on the device, or NULL (every chunk starts at
 *                 position 0)
 *   dst           [num_tokens, 576] bf16, 16-byte aligned; num_tokens is its
 *                 capacity in rows (>= cu_seq_lens[batch]); rows past
 *                 cu_seq_lens[batch] are not written
 *   status        one int32 on the device, or NULL: OR of mla_device_error
 *                 bits -- MLA_DEVERR_BAD_SEQ_LEN: a position outside the
 *                 block table; MLA_DEVERR_BAD_BLOCK: a page id outside
 *                 [0, num_blocks); MLA_DEVERR_BAD_QSL: cu_seq_lens[batch] >
 *                 num_tokens (rows past num_tokens are dropped).  Rows whose
 *                 position or page is bad are written as zeros.  The word is
 *                 OR-ed into, never cleared.
 * num_tokens == 0 or batch == 0 is a no-op.  One launch.
 */
MLA_API int mla_gather_cache(const void* cache, int64_t num_blocks, int page_size, int cache_dtype, float kv_scale,
                             const int32_t* block_table, int max_pages_per_seq, const int32_t* cu_seq_lens,
                             const int32_t* seq_starts, int batch, void* dst, int64_t num_tokens, int32_t* status,
                             void* stream);

/*
 * mla_set_decode_wait_test -- test aid for the failure detection of the
 * decode kernels (the pages have no counterpart).  Every mbarrier wait inside
 * a decode is bounded in wall time; when one runs out, the CTA records
 * MLA_DEVERR_TIMEOUT in the device error word and unwinds without hanging.
 * After this call, later mla_decode / mla_decode_fp8q / mla_decode_no_alloc
 * calls of the calling thread bound every wait by `wait_limit_ns` (0 = the
 * default 1 s; otherwise 1e5..1e9), and with skip_first_tile != 0 the first
 * CTA of the grid never loads its first cache tile, so the wait for that tile
 * runs out.  The decode still returns; its outputs are then undefined and the
 * error word reports the timeout.  Call with (0, 0) to restore the defaults.
 */
MLA_API int mla_set_decode_wait_test(int skip_first_tile, unsigned long long wait_limit_ns);

/* Human-readable description of the calling thread's last error ("" if none). */
MLA_API const char* mla_last_error(void);

/* Streaming multiprocessors of the current device (the decode grid is sized
 * from it), or a negative mla_status. */
MLA_API int mla_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
