// LSE merge kernels (merge_attn_states of the MLA pages: combine partial
// attention results over disjoint key sets by their log-sum-exp).
//
//  * combine_kernel: after a split-KV decode, merges the k partials of every
//    split group (fp16 codes with a power-of-two scale per 32-dim chunk, fp32
//    LSE) into the final bf16 output and LSE, and zero-fills groups that see
//    no key (o = 0, lse = -inf).
//  * merge2_kernel: the public two-way merge (mla_merge_states).
//
// Both are HBM-bound streaming kernels: 16-byte vector loads, one warp-slice
// of 64 threads per 512-wide row, a grid sized in multiples of the SM count
// (of the current device, queried by the caller on every call).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace mla {
namespace {

// Merge of the split groups' partials.  One wave of blocks (the grid is as
// many blocks as fit on every SM at once) strides over the work items (group,
// rows 4y..4y+3), 64 threads per row and 8 dims per thread.  The kernel is
// bound by round trips to memory, not by bytes, so every round issues as many
// loads as it can: two consecutive items of a block are merged together when
// their pieces number at most kFew in all, and the group records of the next
// round are loaded while the current one is merged.
// acc += w * the eight fp16 codes in v (a partial's codes times w x its scale)
__device__ __forceinline__ void accumulate(float (&acc)[8], float w, const uint4 v) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __half22float2(h[k]);
    acc[2 * k] = fmaf(w, f.x, acc[2 * k]);
    acc[2 * k + 1] = fmaf(w, f.y, acc[2 * k + 1]);
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const DecodeArgs a) {
  const Plan& P = a.plan;
  constexpr int kQuads = kRows / 4;   // items per group
  constexpr int kFew = 4;             // pieces whose loads are all in flight at once
  const int G = (int)gridDim.x;
  const int cap = P.max_groups * kQuads;
  // The plan's records are complete before this grid starts: the decode
  // kernel lets it launch only after its own wait for the plan grid.  So the
  // header and the first records are read before the wait for the decode
  // grid, which only the partials need.
  int item = blockIdx.x;
  GroupRec ga{}, gb{};
  if (item < cap) ga = P.groups[item / kQuads];
  if (item + G < cap) gb = P.groups[(item + G) / kQuads];
  const int items = min(cap, P.header->num_groups * kQuads);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel on the stream may launch (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
  const int sub = threadIdx.x & 63;        // 8 dims per thread
  const int d0 = sub * 8;
  constexpr int kChunks = kLkv / 32;       // scales per partial row
  const int chunk = d0 / 32;               // the thread's scale
  const int quad_row = threadIdx.x >> 6;   // row of the item
  // pieces loaded for a group: none when the decode kernel wrote it directly
  auto loads = [](const GroupRec& g) { return g.pieces == 1 ? 0 : g.pieces; };
  // the item's row R (or -1 when there is nothing to write for this thread)
  auto row_of = [&](const GroupRec& g, int it) {
    const int r = (it % kQuads) * 4 + quad_row;
    if (g.pieces == 1 || r >= g.nrows || g.row0 + r >= a.total_rows) return -1;
    return g.row0 + r;
  };
  auto store = [&](int R, const float (&acc)[8], float lse) {
    uint4 v;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(acc[0], acc[1]); v.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[2], acc[3]); v.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[4], acc[5]); v.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[6], acc[7]); v.w = *reinterpret_cast<uint32_t*>(&h);
    *reinterpret_cast<uint4*>(out + (size_t)R * kLkv + d0) = v;
    if (a.lse && sub == 0) a.lse[R] = lse;
  };
  while (item < items) {
    const GroupRec g0 = ga, g1 = gb;
    const int i0 = item, i1 = item + G;
    const int n0 = loads(g0), n1 = i1 < items ? loads(g1) : 0;
    const bool pair = i1 < items && n0 + n1 <= kFew;
    // the records of the next round
    item += pair ? 2 * G : G;
    if (pair) {
      ga = item < items ? P.groups[item / kQuads] : GroupRec{};
    } else {
      ga = gb;
    }
    gb = item + G < items ? P.groups[(item + G) / kQuads] : GroupRec{};
    const int R0 = row_of(g0, i0);
    const int R1 = pair ? row_of(g1, i1) : -1;
    const int r0 = R0 - g0.row0, r1 = R1 - g1.row0;

    if (n0 > kFew) {
      // more pieces than registers (num_splits > kFew): one piece at a time
      if (R0 < 0) continue;
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      float lse = -INFINITY;
      float mx = -INFINITY;
      for (int i = 0; i < g0.pieces; ++i) mx = fmaxf(mx, P.part_lse[(size_t)(g0.ubase + i) * kRows + r0]);
      if (mx != -INFINITY) {
        float wsum = 0.f;
        for (int i = 0; i < g0.pieces; ++i) {
          const size_t slot = (size_t)(g0.ubase + i);
          const float w = __expf(P.part_lse[slot * kRows + r0] - mx);
          wsum += w;
          const size_t at = slot * kRows + r0;
          accumulate(acc, w * P.part_scale[at * kChunks + chunk],
                     *reinterpret_cast<const uint4*>(P.part_o + at * kLkv + d0));
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] *= inv;
        lse = mx + __logf(wsum);
      }
      store(R0, acc, lse);
      continue;
    }

    // every load of both items issued before any use: entries [0, n0) are
    // the first item's pieces, [n0, n0 + n1) the second's
    float l[kFew], sc[kFew];
    uint4 x[kFew];
#pragma unroll
    for (int i = 0; i < kFew; ++i) {
      l[i] = -INFINITY;
      size_t at = ~(size_t)0;
      if (R0 >= 0 && i < n0)
        at = (size_t)(g0.ubase + i) * kRows + r0;
      else if (R1 >= 0 && i >= n0 && i < n0 + n1)
        at = (size_t)(g1.ubase + i - n0) * kRows + r1;
      if (at != ~(size_t)0) {
        l[i] = P.part_lse[at];
        sc[i] = P.part_scale[at * kChunks + chunk];
        x[i] = *reinterpret_cast<const uint4*>(P.part_o + at * kLkv + d0);
      }
    }
    // LSE merge of entries [lo, hi) into row R
    auto merge = [&](int lo, int hi, int R) {
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kFew; ++i)
        if (i >= lo && i < hi) mx = fmaxf(mx, l[i]);
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      float lse = -INFINITY;
      if (mx != -INFINITY) {
        float wsum = 0.f;
#pragma unroll
        for (int i = 0; i < kFew; ++i) {
          if (i >= lo && i < hi) {
            const float w = __expf(l[i] - mx);
            wsum += w;
            accumulate(acc, w * sc[i], x[i]);
          }
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] *= inv;
        lse = mx + __logf(wsum);
      }
      store(R, acc, lse);
    };
    if (R0 >= 0) merge(0, n0, R0);
    if (R1 >= 0) merge(n0, n0 + n1, R1);
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
