// Per-head projections around the absorbed decode, on tcgen05:
//
//   y[t, n, :] = x[t, n, :] @ W[n]        W[n]: [d_in, d_out] row-major
//
// which is both batched GEMMs of the MLA pages' "data-movement friendly"
// path (vllm/v1/attention/backends/mla/common.py):
//   * query absorption (MLACommonImpl.forward, decode branch):
//     ql_nope = bmm(q_nope, W_UK_T), W_UK_T stored (N, P, Lkv);
//   * the value up-projection (MLACommonBaseImpl._v_up_proj):
//     out = bmm(o_latent, W_UV), W_UV stored (N, Lkv, V).
//
// One CTA computes a 128-token x bn-column tile of one head: D[t][j] in TMEM
// (lane = token, column = output dim), A = the token rows of x (K-major,
// 128-byte swizzled boxes of 64 input dims), B = W[n] (output dims
// contiguous: the MN-major operand form), K staged 64 input dims at a time
// through a TMA ring deep enough to hold a whole head's weights at decode
// batch sizes, so every load of a CTA is in flight at once.  The op streams
// every weight once and is HBM-bound for decode batch sizes.  With fewer
// than 128 tokens the x box holds only round_up(T, 16) rows; the MMA rows
// past it read other bytes of the CTA's shared memory and their results are
// never stored.  Weights do not depend on the previous kernel, so the first
// weight loads are issued before the grid-dependency wait.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {
namespace {
using namespace ptx;

constexpr int kPM = 128;                               // tokens per CTA (MMA M)
constexpr int kPK = 64;                                // input dims per stage
constexpr int kPStagesMax = 8;
constexpr int kPThreads = 192;                         // TMA warp, MMA warp, 4 epilogue warps
constexpr uint32_t kXBoxMax = kPM * kPK * 2;           // 16 KB: 128 token rows x 64 dims
constexpr uint32_t kWBox = kPK * 64 * 2;               // 8 KB: 64 input rows x 64 output dims
constexpr uint32_t kRingBudget = 96 * 1024;            // ring bytes: two CTAs share an SM
constexpr uint32_t kSmemPerSm = 233472;                // shared memory of an SM (228 KB)

__device__ unsigned int g_proj_error;                  // OR of MLA_DEVERR_* bits

struct ProjBars {
  uint64_t full[kPStagesMax];
  uint64_t empty[kPStagesMax];
  uint64_t d_full;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void proj_abort(ProjBars* bars) {
  atomicOr(&g_proj_error, 1u);  // MLA_DEVERR_TIMEOUT
  *reinterpret_cast<volatile int*>(&bars->abort) = 1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kPThreads, 1)
    head_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     __nv_bfloat16* __restrict__ y, int T, int N, int d_in, int d_out, int bn, int stages,
                     int xrows) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t xbox = (uint32_t)xrows * kPK * 2;
  const uint32_t stage_bytes = xbox + (uint32_t)(bn / 64) * kWBox;
  ProjBars* bars = reinterpret_cast<ProjBars*>(smem + stages * stage_bytes + (kXBoxMax > xbox ? kXBoxMax - xbox : 0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x;
  const int j0 = blockIdx.y * bn;
  const int t0 = blockIdx.z * kPM;
  const int kc = d_in / kPK;
  const uint32_t tcols = bn <= 64 ? 64 : bn <= 128 ? 128 : 256;

  const int npre = kc < stages ? kc : stages;  // chunks the ring holds from the start
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->d_full), 1);
    bars->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    // Launched as a programmatic dependent: the weights are not written by
    // the previous kernel, so their first loads go out before the wait; x may
    // be that kernel's output and y may still be read by it, so the x loads
    // (and through them the MMAs and the stores) wait for its completion.
    for (int c = 0; c < npre; ++c) {
      const uint32_t st = smem_u32(smem + c * stage_bytes);
      const uint32_t full = smem_u32(&bars->full[c]);
      mbar_expect_tx(full, stage_bytes);
      for (int b = 0; b < bn / 64; ++b)
        tma_load_2d(st + xbox + b * kWBox, &tm_w, j0 + 64 * b, n * d_in + c * kPK, full);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int c = 0; c < npre; ++c)
      tma_load_3d(smem_u32(smem + c * stage_bytes), &tm_x, c * kPK, n, t0, smem_u32(&bars->full[c]));
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;
  // The next kernel on the stream may launch now (its CTAs take idle SMs and
  // run their prologue); it still waits for this grid's completion before
  // it reads anything this grid writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = npre;
      for (int c = npre; c < kc; ++c) {
        const int slot = c % stages, round = c / stages;
        if (round > 0 && !mbar_wait(smem_u32(&bars->empty[slot]), (round - 1) & 1)) {
          proj_abort(bars);
          break;
        }
        if (*abort_flag) break;
        const uint32_t st = smem_u32(smem + slot * stage_bytes);
        const uint32_t full = smem_u32(&bars->full[slot]);
        mbar_expect_tx(full, stage_bytes);
        tma_load_3d(st, &tm_x, c * kPK, n, t0, full);
        for (int b = 0; b < bn / 64; ++b)
          tma_load_2d(st + xbox + b * kWBox, &tm_w, j0 + 64 * b, n * d_in + c * kPK, full);
        issued = c + 1;
      }
      // every copy this thread issued has landed before the CTA may exit
      for (int c = issued > stages ? issued - stages : 0; c < issued; ++c)
        if (!mbar_wait(smem_u32(&bars->full[c % stages]), (c / stages) & 1)) proj_abort(bars);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kPM, bn, 0, 1);  // A K-major tokens, B MN-major weights
      for (int c = 0; c < kc; ++c) {
        const int slot = c % stages;
        if (!mbar_wait(smem_u32(&bars->full[slot]), (c / stages) & 1)) {
          proj_abort(bars);
          break;
        }
        if (*abort_flag) break;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + slot * stage_bytes);
        const uint64_t xd = smem_desc(st, 16, 1024, kSwizzle128B);
        const uint64_t wd = smem_desc(st + xbox, kWBox, 1024, kSwizzle128B);
        // 16 input dims per MMA: 32 bytes along a swizzled x row, 16 rows (2 KB) of a weight box
#pragma unroll
        for (int k = 0; k < kPK / 16; ++k)
          mma_ss(tmem, xd + ((k * 32) >> 4), wd + ((k * 2048) >> 4), idesc, (c > 0 || k > 0) ? 1u : 0u);
        mma_commit(smem_u32(&bars->empty[slot]));
      }
      // arrives once every MMA issued above has completed; the tensor memory
      // is released only after that
      mma_commit(smem_u32(&bars->d_full));
      if (!mbar_wait(smem_u32(&bars->d_full), 0)) proj_abort(bars);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // the TMEM lane quarter this warp may read
    const int t = t0 + 32 * q + lane;
    const bool done = mbar_wait(smem_u32(&bars->d_full), 0);
    if (!done) proj_abort(bars);
    tc_fence_after();
    if (done && !*abort_flag) {
      __nv_bfloat16* dst = y + ((size_t)t * N + n) * d_out + j0;
      for (int c0 = 0; c0 < bn; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + c0, r);
        tmem_wait_ld();
        if (t < T) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            d4[v] = make_uint4(pack_bf16x2(r[8 * v], r[8 * v + 1]), pack_bf16x2(r[8 * v + 2], r[8 * v + 3]),
                               pack_bf16x2(r[8 * v + 4], r[8 * v + 5]), pack_bf16x2(r[8 * v + 6], r[8 * v + 7]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

}  // namespace

// Rows of the x box: the token count rounded up to 16, at most one 128-token tile.
int head_proj_x_rows(int64_t T) { return T >= kPM ? kPM : (int)((T + 15) / 16 * 16); }

namespace {

struct ProjShape {
  int bn;        // output columns per CTA (MMA N)
  int xrows;     // rows of the x box
  int stages;    // ring depth
  size_t smem;   // dynamic shared memory per CTA
};

int proj_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || n <= 0)
    return 148;
  return n;
}

// The op is HBM-bound: the widest column tile whose grid still gives most
// SMs two CTAs (one CTA's prologue and epilogue then run under the other's
// loads; measured on the DeepSeek-V3 shapes, 128 heads x 64 tokens: the
// up-projection 7.95 us with 128 CTAs of 128 columns, 6.9 us with 256 of
// 64; the absorption 7.3 us with 256 CTAs of 256 columns, 8.6 us with 512 of
// 128, which no longer fit on the GPU at once), and a ring of at most
// ~96 KB so that two CTAs share an SM.
ProjShape proj_shape(int64_t T, int N, int d_in, int d_out) {
  ProjShape p;
  const int64_t tiles = (T + kPM - 1) / kPM;
  const int64_t want = 3LL * proj_sm_count() / 2;
  p.bn = 64;
  for (int cand = 256; cand >= 128; cand /= 2)
    if (d_out % cand == 0 && (int64_t)N * (d_out / cand) * tiles >= want) {
      p.bn = cand;
      break;
    }
  p.xrows = head_proj_x_rows(T);
  const int kc = d_in / kPK;
  const uint32_t xbox = (uint32_t)p.xrows * kPK * 2;
  const uint32_t stage = xbox + (uint32_t)(p.bn / 64) * kWBox;
  int st = (int)(kRingBudget / stage);
  st = st > kPStagesMax ? kPStagesMax : st;
  st = st > kc ? kc : st;
  p.stages = st < 1 ? 1 : st;
  // + the part of a full 128-row box the last stage's MMA rows reach past the ring
  p.smem = 1024 + (size_t)p.stages * stage + (kXBoxMax - xbox) + sizeof(ProjBars);
  // never more CTAs on an SM than its 512 tensor-memory columns hold (an
  // allocation beyond them would wait for another CTA to finish)
  const uint32_t tcols = p.bn <= 64 ? 64 : p.bn <= 128 ? 128 : 256;
  const size_t floor_smem = kSmemPerSm / (512 / tcols + 1);   // + the 1 KB each CTA reserves
  if (p.smem < floor_smem) p.smem = floor_smem;
  return p;
}

}  // namespace

cudaError_t launch_head_proj(const CUtensorMap& tm_x, const CUtensorMap& tm_w, void* y, int64_t T, int N, int d_in,
                             int d_out, cudaStream_t s) {
  const ProjShape p = proj_shape(T, N, d_in, d_out);
  const int bn = p.bn, xrows = p.xrows, stages = p.stages;
  const size_t smem = p.smem;
  // set on every call: the attribute belongs to the current device
  cudaError_t e = cudaFuncSetAttribute(head_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(1024 + kRingBudget + kXBoxMax + sizeof(ProjBars) + 1024));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)N, (unsigned)(d_out / bn), (unsigned)((T + kPM - 1) / kPM));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, head_proj_kernel, tm_x, tm_w, static_cast<__nv_bfloat16*>(y), (int)T, N,
                                     d_in, d_out, bn, stages, xrows);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t head_proj_status(int* status, int clear, cudaStream_t s) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_proj_error, sizeof v, 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_proj_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *status = (int)v;
  return e;
}

}  // namespace mla
