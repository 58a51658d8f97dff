// LSE merge kernels (merge_attn_states of the MLA pages: combine partial
// attention results over disjoint key sets by their log-sum-exp).
//
//  * combine_kernel: after a split-KV decode, merges the k partials of every
//    split group (fp16 codes with a power-of-two scale per 32-dim chunk, fp32
//    LSE) into the final bf16 output and LSE, and zero-fills groups that see
//    no key (o = 0, lse = -inf).
//  * merge2_kernel: the public two-way merge (mla_merge_states).
//
// Both stream with 16-byte vector loads over a grid sized in multiples of the
// SM count (of the current device, queried by the caller on every call).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace mla {
namespace {

// acc[0..7] += w * the eight fp16 codes in v (a partial's codes times w x its scale)
__device__ __forceinline__ void accumulate(float* acc, float w, const uint4 v) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __half22float2(h[k]);
    acc[2 * k] = fmaf(w, f.x, acc[2 * k]);
    acc[2 * k + 1] = fmaf(w, f.y, acc[2 * k + 1]);
  }
}

// Merge of the split groups' partials.  The work item is (group, rows
// 4y..4y+3); 64 threads take an item, 16 per row and 32 dims per thread
// (dims 128c + 8s .. 128c + 8s + 7 for c = 0..3 of thread s, so that every
// load instruction of a warp reads whole 256-byte runs), and a block of 256
// threads holds four items at once.
// The kernel is bound by the latency of its loads: every load of an item's
// pieces is issued before any use, and the next item's group record loads
// while the current one merges.  One wave of blocks (as many as are
// resident on every SM at once) strides over the items.
__global__ void __launch_bounds__(256, 2) combine_kernel(const DecodeArgs a) {
  const Plan& P = a.plan;
  constexpr int kQuads = kRows / 4;   // items per group
  // pieces whose loads are all in flight at once: with the balanced split a
  // group spans at most three CTA-pair spans unless it is longer than two
  constexpr int kFew = 3;
  constexpr int kChunks = kLkv / 32;  // scales per partial row
  const int VG = (int)gridDim.x * 4;  // item slots of the grid
  const int cap = P.max_groups * kQuads;
  // The plan's records are complete before this grid starts: the decode
  // kernel lets it launch only after its own wait for the plan grid.  So the
  // header and the first record are read before the wait for the decode
  // grid, which only the partials need.
  int item = (int)blockIdx.x * 4 + (int)(threadIdx.x >> 6);
  GroupRec gnext{};
  if (item < cap) gnext = P.groups[item / kQuads];
  const int items = min(cap, P.header->num_groups * kQuads);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel on the stream may launch (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
  const int sub = threadIdx.x & 15;              // dims 128 c + 8 sub .. + 7, c = 0..3
  const int d0 = sub * 8;
  const int quad_row = (threadIdx.x >> 4) & 3;   // row of the item
  for (; item < items; item += VG) {
    const GroupRec gr = gnext;
    if (item + VG < items) gnext = P.groups[(item + VG) / kQuads];
    if (gr.pieces == 1) continue;  // written directly by the decode kernel
    const int r = (item % kQuads) * 4 + quad_row;
    if (r >= gr.nrows || gr.row0 + r >= a.total_rows) continue;
    const int R = gr.row0 + r;
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
    float lse = -INFINITY;
    if (gr.pieces <= kFew) {
      // the usual case: every load of every piece issued before any use
      float l[kFew], sc[kFew][4];
      uint4 x[kFew][4];
#pragma unroll
      for (int i = 0; i < kFew; ++i) {
        l[i] = -INFINITY;
        if (i < gr.pieces) {
          const size_t at = (size_t)(gr.ubase + i) * kRows + r;
          l[i] = P.part_lse[at];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            sc[i][c] = P.part_scale[at * kChunks + 4 * c + (sub >> 2)];
            x[i][c] = *reinterpret_cast<const uint4*>(P.part_o + at * kLkv + 128 * c + d0);
          }
        }
      }
      float mx = l[0];
#pragma unroll
      for (int i = 1; i < kFew; ++i) mx = fmaxf(mx, l[i]);
      if (mx != -INFINITY) {
        float wsum = 0.f;
#pragma unroll
        for (int i = 0; i < kFew; ++i) {
          if (i < gr.pieces) {
            const float w = __expf(l[i] - mx);
            wsum += w;
#pragma unroll
            for (int c = 0; c < 4; ++c) accumulate(acc + 8 * c, w * sc[i][c], x[i][c]);
          }
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] *= inv;
        lse = mx + __logf(wsum);
      }
    } else {
      // more pieces than registers (num_splits > kFew): one piece at a time
      float mx = -INFINITY;
      for (int i = 0; i < gr.pieces; ++i) mx = fmaxf(mx, P.part_lse[(size_t)(gr.ubase + i) * kRows + r]);
      if (mx != -INFINITY) {
        float wsum = 0.f;
        for (int i = 0; i < gr.pieces; ++i) {
          const size_t at = (size_t)(gr.ubase + i) * kRows + r;
          const float w = __expf(P.part_lse[at] - mx);
          wsum += w;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            accumulate(acc + 8 * c, w * P.part_scale[at * kChunks + 4 * c + (sub >> 2)],
                       *reinterpret_cast<const uint4*>(P.part_o + at * kLkv + 128 * c + d0));
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] *= inv;
        lse = mx + __logf(wsum);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 v;
      __nv_bfloat162 h;
      h = __floats2bfloat162_rn(acc[8 * c + 0], acc[8 * c + 1]); v.x = *reinterpret_cast<uint32_t*>(&h);
      h = __floats2bfloat162_rn(acc[8 * c + 2], acc[8 * c + 3]); v.y = *reinterpret_cast<uint32_t*>(&h);
      h = __floats2bfloat162_rn(acc[8 * c + 4], acc[8 * c + 5]); v.z = *reinterpret_cast<uint32_t*>(&h);
      h = __floats2bfloat162_rn(acc[8 * c + 6], acc[8 * c + 7]); v.w = *reinterpret_cast<uint32_t*>(&h);
      *reinterpret_cast<uint4*>(out + (size_t)R * kLkv + 128 * c + d0) = v;
    }
    if (a.lse && sub == 0) a.lse[R] = lse;
  }
}

template <bool kBf16>
__device__ __forceinline__ void load8(const void* base, size_t idx, float (&x)[8]) {
  if (kBf16) {
    const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + idx);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

template <bool kBf16>
__device__ __forceinline__ void store8(void* base, size_t idx, const float (&x)[8]) {
  if (kBf16) {
    uint4 v;
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
      w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + idx) = v;
  } else {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + idx);
    p[0] = make_float4(x[0], x[1], x[2], x[3]);
    p[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
}

// One thread per 8 consecutive elements of a row; grid-stride over all vectors.
template <bool kBf16>
__global__ void __launch_bounds__(256) merge2_kernel(const void* __restrict__ o_a, const float* __restrict__ lse_a,
                                                     const void* __restrict__ o_b, const float* __restrict__ lse_b,
                                                     int64_t rows, int dim, void* out, float* lse_out) {
  const int vpr = dim / 8;
  const int64_t nvec = rows * vpr;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = v / vpr;
    const size_t idx = (size_t)r * dim + (size_t)(v - r * vpr) * 8;
    const float la = lse_a[r], lb = lse_b[r];
    const float mx = fmaxf(la, lb);
    float x[8], y[8];
    load8<kBf16>(o_a, idx, x);
    load8<kBf16>(o_b, idx, y);
    float res[8];
    float lse;
    if (mx == -INFINITY) {
#pragma unroll
      for (int k = 0; k < 8; ++k) res[k] = 0.f;
      lse = -INFINITY;
    } else {
      const float wa = __expf(la - mx), wb = __expf(lb - mx);
      const float inv = 1.f / (wa + wb);
#pragma unroll
      for (int k = 0; k < 8; ++k) res[k] = (wa * x[k] + wb * y[k]) * inv;
      lse = mx + __logf(wa + wb);
    }
    store8<kBf16>(out, idx, res);
    if (lse_out && v - r * vpr == 0) lse_out[r] = lse;
  }
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, int max_groups, int sm_count, cudaStream_t s) {
  // one wave: as many blocks as are resident on every SM at once (a block
  // beyond that would start only when another ends), or fewer when the plan
  // cannot hold as many items
  static const int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_kernel, 256, 0) != cudaSuccess || n < 1) n = 1;
    return n;
  }();
  cudaLaunchConfig_t cfg = {};
  const long long max_items = (long long)max_groups * (kRows / 4);
  long long blocks = (long long)(sm_count > 0 ? sm_count : 1) * per_sm;
  if (blocks * 4 > max_items) blocks = (max_items + 3) / 4;   // four items per block at once
  if (blocks < 1) blocks = 1;
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                                int64_t rows, int dim, int o_is_bf16, void* out, float* lse_out, int sm_count,
                                cudaStream_t s) {
  const int64_t nvec = rows * (dim / 8);
  int64_t blocks = (nvec + 255) / 256;
  const int64_t cap = (int64_t)(sm_count > 0 ? sm_count : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (o_is_bf16)
    merge2_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(o_a, lse_a, o_b, lse_b, rows, dim, out, lse_out);
  else
    merge2_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(o_a, lse_a, o_b, lse_b, rows, dim, out, lse_out);
  return cudaGetLastError();
}

}  // namespace mla
