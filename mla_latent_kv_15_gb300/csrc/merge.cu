// LSE merge kernels (merge_attn_states of the MLA pages: combine partial
// attention results over disjoint key sets by their log-sum-exp).
//
//  * combine_kernel: after a split-KV decode, merges the k fp32 partials of
//    every split group into the final bf16 output and LSE, and zero-fills
//    groups that see no key (o = 0, lse = -inf).
//  * merge2_kernel: the public two-way merge (mla_merge_states).
//
// Both are HBM-bound streaming kernels: 16-byte vector loads, one warp-slice
// of 64 threads per 512-wide row, a grid sized in multiples of the SM count
// (of the current device, queried by the caller on every call).
#include <cuda_bf16.h>

#include "common.cuh"

namespace mla {
namespace {

// Merge of the split groups' partials.  One wave of blocks (the grid is a
// few blocks per SM) strides over the work items (group, rows 4y..4y+3), 64
// threads per row and 8 dims per thread; the next item's group record is
// loaded while the current item is merged, so each item costs one round
// trip to memory (a grid of one block per item ran in several waves of
// blocks that each waited for two dependent loads).
__global__ void __launch_bounds__(256) combine_kernel(const DecodeArgs a) {
  // launched as a programmatic dependent of the decode kernel: wait for it
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel on the stream may launch (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const Plan& P = a.plan;
  const int items = P.header->num_groups * (kRows / 4);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
  const int sub = threadIdx.x & 63;        // 8 dims per thread
  const int d0 = sub * 8;
  int item = blockIdx.x;
  GroupRec gnext{};
  if (item < items) gnext = P.groups[item / (kRows / 4)];
  for (; item < items; item += gridDim.x) {
    const GroupRec gr = gnext;
    if (item + (int)gridDim.x < items) gnext = P.groups[(item + gridDim.x) / (kRows / 4)];
    if (gr.pieces == 1) continue;  // written directly by the decode kernel
    const int r = (item % (kRows / 4)) * 4 + (threadIdx.x >> 6);
    if (r >= gr.nrows) continue;
    const int R = gr.row0 + r;
    if (R >= a.total_rows) continue;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float lse = -INFINITY;
    constexpr int kFew = 4;
    if (gr.pieces <= kFew) {
      // the usual case: every load of every piece issued before any use
      float l[kFew];
      float4 x0[kFew], x1[kFew];
#pragma unroll
      for (int i = 0; i < kFew; ++i) {
        l[i] = -INFINITY;
        if (i < gr.pieces) {
          const size_t slot = (size_t)(gr.ubase + i);
          l[i] = P.part_lse[slot * kRows + r];
          const float4* src = reinterpret_cast<const float4*>(P.part_o + (slot * kRows + r) * kLkv + d0);
          x0[i] = src[0];
          x1[i] = src[1];
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
            acc[0] += w * x0[i].x; acc[1] += w * x0[i].y; acc[2] += w * x0[i].z; acc[3] += w * x0[i].w;
            acc[4] += w * x1[i].x; acc[5] += w * x1[i].y; acc[6] += w * x1[i].z; acc[7] += w * x1[i].w;
          }
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] *= inv;
        lse = mx + __logf(wsum);
      }
    } else {
      float mx = -INFINITY;
      for (int i = 0; i < gr.pieces; ++i) mx = fmaxf(mx, P.part_lse[(size_t)(gr.ubase + i) * kRows + r]);
      if (mx != -INFINITY) {
        float wsum = 0.f;
        for (int i = 0; i < gr.pieces; ++i) {
          const size_t slot = (size_t)(gr.ubase + i);
          const float w = __expf(P.part_lse[slot * kRows + r] - mx);
          wsum += w;
          const float4* src = reinterpret_cast<const float4*>(P.part_o + (slot * kRows + r) * kLkv + d0);
          const float4 x0 = src[0], x1 = src[1];
          acc[0] += w * x0.x; acc[1] += w * x0.y; acc[2] += w * x0.z; acc[3] += w * x0.w;
          acc[4] += w * x1.x; acc[5] += w * x1.y; acc[6] += w * x1.z; acc[7] += w * x1.w;
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] *= inv;
        lse = mx + __logf(wsum);
      }
    }
    uint4 v;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(acc[0], acc[1]); v.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[2], acc[3]); v.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[4], acc[5]); v.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[6], acc[7]); v.w = *reinterpret_cast<uint32_t*>(&h);
    *reinterpret_cast<uint4*>(out + (size_t)R * kLkv + d0) = v;
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
  cudaLaunchConfig_t cfg = {};
  // one wave: four blocks per SM, or fewer when the plan cannot hold as many items
  const long long max_items = (long long)max_groups * (kRows / 4);
  long long blocks = (long long)(sm_count > 0 ? sm_count : 1) * 4;
  if (blocks > max_items) blocks = max_items;
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
