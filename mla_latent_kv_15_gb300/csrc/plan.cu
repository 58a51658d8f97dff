// Split-KV scheduler: builds the work-unit plan of one mla_decode call on the
// device (no host synchronisation, so the whole decode can be captured in a
// CUDA graph).
//
// Query rows of a request are flattened as t*N + h and cut into groups of up
// to 128 rows (the tcgen05 M of the decode kernel; 32 for its small-rows
// variant, used when every request has one query token and N <= 32, where
// a group count never exceeds the batch size).  Every group reads the
// keys its last row may see, L = seq_len - Sq + 1 + t (multi-token causal
// rule of the AITER MLA backend's verify path), in 64-key tiles.  Groups are
// laid end to end on one flattened tile axis which is either
//   * cut into near-equal spans, one per CTA pair (automatic: pair c gets
//     positions [floor(c T / C), floor((c+1) T / C)) of the T on the axis,
//     a group straddling a boundary is split there), or
//   * with num_splits = k, every group is cut into min(k, tiles) near-equal
//     pieces and pieces go to the pair whose span holds their midpoint.
// Pieces of a split group write partials that the combine kernel merges
// with the LSE rule of merge_attn_states.
#include "cache_rows.cuh"
#include "common.cuh"

namespace mla {

namespace {

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Threads of the plan block: a small block keeps its barriers short (a
// batch of up to this many requests is one pass of every phase).
constexpr int kPlanThreads = 256;
constexpr int kPlanSmemGroups = 1024;   // staged plans: at most this many groups
// Fixed cost of a work unit in tiles of decode time: loading the group's
// query into tensor memory, refilling the pipeline and the epilogue (a fit of
// every CTA's end time on the DeepSeek-V3-shaped batch: ~4 us per unit
// against ~1.2 us per 64-key tile; 3 and 4 measured alike, 2 and 5 worse).  Each group is
// placed on the balanced axis behind this many virtual tiles, so that CTA
// pairs starting more groups get fewer real tiles.
constexpr int kUnitCostTiles = 3;
constexpr int kPlanSmemUnits = 2048;    // and units

// Exclusive scan over the block (blockDim.x == kPlanThreads) with one
// barrier: every warp scans its values and publishes its total; after the
// barrier each warp adds the totals of the warps before it.  Consecutive
// scans alternate between the two rows of `sums`, so a warp may start the
// next scan while another still reads this one's totals (no warp gets two
// scans ahead: each scan has a barrier).  *total gets the block's sum.
__device__ __forceinline__ int block_excl_scan(int v, int* total, int (&sums)[2][kPlanThreads / 32], int& row) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v);
  int* buf = sums[row];
  row ^= 1;
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kPlanThreads / 32; ++w) {
    const int x = buf[w];
    before += w < warp ? x : 0;
    all += x;
  }
  *total = all;
  return incl - v + before;
}

// floor(a / b) for a >= 0, b > 0 and a + b < 2^31: a float estimate (within
// a few units while a < 2^24) corrected with integer products; an integer
// division is a long chain of dependent instructions, and the plan is one
// chain of them.
__device__ __forceinline__ int divf(int a, int b) {
  int q = __float2int_rz(__fdividef((float)a, (float)b));
  while (q * b > a) --q;          // the estimate is within a few units
  while ((q + 1) * b <= a) ++q;
  return q;
}

// floor(a * b / c) for a, b >= 0 and c > 0: a 32-bit division whenever the
// product fits (a 64-bit division is a long chain of dependent instructions)
__device__ __forceinline__ int muldiv(int a, int b, int c) {
  const unsigned long long p = (unsigned long long)(unsigned)a * (unsigned)b;
  if (p <= 0xffffffffull) return (int)((unsigned)p / (unsigned)c);
  return (int)(p / (unsigned long long)c);
}

// kStaged: the group records and unit clusters live in shared memory while
// the plan is built (each phase reads what other threads wrote in the
// previous one) and are copied out at the end; for plans that fit.
// kMode: blocks 1.. of the launch do the step's other small jobs while block
// 0 builds the plan, so they cost the step no launch of their own: the new
// cache rows (blocks 1 .. write_blocks, 8 tokens a block; 1 bf16 cache,
// 2 e4m3 cache) and, in mode 3 (e4m3 cache), the query's quantisation (the
// remaining blocks, grid-stride over its 8-value vectors).
template <bool kStaged, int kMode>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ seq_lens,
                                                    const int32_t* __restrict__ qsl, int batch, int N,
                                                    int max_pages, int page_size, int num_splits, int C,
                                                    int GR, Plan P, const CacheWriteArgs w, const QuantArgs qa,
                                                    int write_blocks) {
  if constexpr (kMode != 0) {
    if (blockIdx.x > 0) {
      // as the cache-write kernel: wait for the kernel before, then let the
      // next one launch (the decode waits for this whole grid)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      const int b = (int)blockIdx.x - 1;
      if (b < write_blocks) {
        const int64_t tok = b * 8LL + (threadIdx.x >> 5);
        if (tok < w.num_tokens) write_cache_row<kMode >= 2>(w, tok, threadIdx.x & 31);
        return;
      }
      if constexpr (kMode == 3) {
        const int64_t nvec = qa.rows * (kDqk / 8);
        const int64_t stride = (int64_t)(gridDim.x - 1 - write_blocks) * kPlanThreads;
        for (int64_t v = (int64_t)(b - write_blocks) * kPlanThreads + threadIdx.x; v < nvec; v += stride)
          quantize_query_vec(qa, v);
      }
      return;
    }
  }
  __shared__ int s_flags;
  __shared__ int s_span[kMaxClusters + 1];   // first axis position of every span
  __shared__ GroupRec s_groups[kStaged ? kPlanSmemGroups : 1];
  __shared__ int s_ucl[kStaged ? kPlanSmemUnits : 1];
  __shared__ int s_kbase[kStaged ? kPlanSmemGroups : 1];   // seq_len - Sq + 1 - q0 of each group's request
  __shared__ int s_sums[2][kPlanThreads / 32];
  int sums_row = 0;
  GroupRec* grp = kStaged ? s_groups : P.groups;
  int* ucl = kStaged ? s_ucl : P.unit_cluster;
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent of the kernel before it on the
  // stream, so only its launch overlaps that kernel's tail: it waits for that
  // grid (which may have written seq_lens or query_start_loc, or still read
  // an earlier plan) before touching memory. The decode kernel waits only for
  // this grid, which therefore also orders it after everything earlier.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the decode kernel may launch now: its prologue (barriers, TMEM, cluster
  // sync) overlaps the plan; it waits for this grid before reading the plan
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) s_flags = 0;
  __syncthreads();
  const long long kv_cap = (long long)max_pages * page_size;
  const int gshift = __ffs(GR) - 1;   // GR is a power of two

  // 1. groups of every request
  int carry = 0;
  for (int base = 0; base < batch; base += kPlanThreads) {
    const int b = base + tid;
    int sq = 0, ng = 0, q0 = 0;
    long long seq = 0;
    if (b < batch) {
      // all of the request's loads at once
      q0 = qsl ? qsl[b] : b;
      sq = qsl ? qsl[b + 1] - q0 : 1;
      seq = seq_lens[b];
      if (sq < 0) sq = 0;
      ng = (int)(((long long)sq * N + GR - 1) >> gshift);
    }
    int total;
    const int gb = block_excl_scan(ng, &total, s_sums, sums_row) + carry;
    if (b < batch && ng > 0) {
      if (seq > kv_cap) {
        atomicOr(&s_flags, 2);  // MLA_DEVERR_BAD_SEQ_LEN
        seq = kv_cap;
      }
      const int kbase = (int)(seq - sq + 1 - q0);
      const int rows_b = sq * N;
      for (int g = 0; g < ng && gb + g < P.max_groups; ++g) {
        if (kStaged) s_kbase[gb + g] = kbase;
        GroupRec r;
        r.b = b;
        r.row0 = q0 * N + g * GR;
        r.nrows = min(GR, rows_b - g * GR);
        const int t_last = divf(g * GR + r.nrows - 1, N);
        long long L = seq - sq + 1 + t_last;
        if (L < 0) L = 0;
        if (L > kv_cap) L = kv_cap;
        r.lmax = (int)L;
        r.tiles = (int)((L + kTile - 1) / kTile);
        r.pieces = 0;
        r.ubase = 0;
        r.tpos = 0;
        grp[gb + g] = r;
      }
    }
    carry += total;
  }
  int G = carry;
  if (G > P.max_groups) {  // query_start_loc disagrees with total_q: plan nothing
    if (tid == 0) atomicOr(&s_flags, 8);  // MLA_DEVERR_BAD_QSL
    G = 0;
  }
  __syncthreads();

  // 2. positions on the balanced axis: every group with keys spans its
  //    virtual unit-cost tiles, then its real tiles
  carry = 0;
  for (int base = 0; base < G; base += kPlanThreads) {
    const int g = base + tid;
    const int tl = g < G ? grp[g].tiles : 0;
    const int t = tl > 0 ? tl + kUnitCostTiles : 0;
    int total;
    const int pos = block_excl_scan(t, &total, s_sums, sums_row) + carry;
    if (g < G) grp[g].tpos = pos;
    carry += total;
  }
  const int T = carry;
  // Span c of the axis is [floor(c T / Cs), floor((c+1) T / Cs)) with
  // Cs = min(C, T) spans, none of them empty.  With T = a Cs + b, the start
  // of span c is c a + floor(c b / Cs) (c b < Cs^2: a short division); the
  // span of a position is a float estimate corrected against the starts.
  const int Cs = T < C ? (T > 0 ? T : 1) : C;
  const bool small_axis = T < (1 << 24);
  const int sa = small_axis ? divf(T, Cs) : T / Cs;
  const int sb = T - sa * Cs;
  const int W = T > 0 ? (T >= C ? sa + (sb > 0) : 1) : 1;   // ceil(T / C) positions per span
  for (int c = tid; c <= Cs; c += kPlanThreads) s_span[c] = c * sa + divf(c * sb, Cs);
  const float span_per_pos = T > 0 ? __fdividef((float)Cs, (float)T) : 0.f;
  auto span_start = [&](int c) { return s_span[c]; };
  auto span_of = [&](int p) {
    int c = min(Cs - 1, max(0, (int)((float)p * span_per_pos)));
    while (c > 0 && s_span[c] > p) --c;
    while (c < Cs - 1 && s_span[c + 1] <= p) ++c;
    return c;
  };
  __syncthreads();

  // 3. pieces per group, unit bases
  carry = 0;
  for (int base = 0; base < G; base += kPlanThreads) {
    const int g = base + tid;
    int pieces = 0;
    if (g < G) {
      const GroupRec r = grp[g];
      if (r.tiles > 0) {
        const int s0 = r.tpos + kUnitCostTiles;   // first real tile on the axis
        if (num_splits > 0)
          pieces = min(num_splits, r.tiles);
        else
          pieces = span_of(s0 + r.tiles - 1) - span_of(s0) + 1;   // spans the group's real tiles touch
      }
    }
    int total;
    const int ub = block_excl_scan(pieces, &total, s_sums, sums_row) + carry;
    if (g < G) {
      grp[g].pieces = pieces;
      grp[g].ubase = ub;
    }
    carry += total;
  }
  int U = carry;
  if (U > P.max_units) {  // cannot happen for a workspace sized for num_splits
    __syncthreads();
    for (int g = tid; g < G; g += kPlanThreads) grp[g].pieces = 0;
    if (tid == 0) atomicOr(&s_flags, 8);
    U = 0;
  }
  __syncthreads();

  // 4. units
  for (int g = tid; g < G; g += kPlanThreads) {
    const GroupRec r = grp[g];
    const int s0 = r.tpos + kUnitCostTiles;       // first real tile on the axis
    int kbase = 0;
    if (kStaged) {
      kbase = s_kbase[g];
    } else if (r.pieces > 0) {
      const int sq = qsl ? qsl[r.b + 1] - qsl[r.b] : 1;
      const int q0 = qsl ? qsl[r.b] : r.b;
      const long long seq = min((long long)seq_lens[r.b], kv_cap);
      kbase = (int)(seq - sq + 1 - q0);
    }
    const int c0 = num_splits > 0 || r.pieces == 0 ? 0 : span_of(s0);   // the span of the group's first piece
    for (int i = 0; i < r.pieces; ++i) {
      UnitRec u;
      int cl;
      u.b = r.b;
      u.row0 = r.row0;
      u.nrows = r.nrows;
      u.lmax = r.lmax;
      u.kbase = kbase;
      if (num_splits > 0) {
        u.tile_begin = muldiv(i, r.tiles, r.pieces);
        u.tile_end = muldiv(i + 1, r.tiles, r.pieces);
        cl = min(C - 1, span_of(s0 + (u.tile_begin + u.tile_end) / 2));
      } else {
        cl = c0 + i;
        u.tile_begin = max(s0, span_start(cl)) - s0;
        u.tile_end = min(s0 + r.tiles, span_start(cl + 1)) - s0;
      }
      u.slot = r.pieces > 1 ? r.ubase + i : -1;
      P.units[r.ubase + i] = u;
      ucl[r.ubase + i] = cl;
    }
  }
  __syncthreads();

  // 5. first unit of every cluster (unit clusters are non-decreasing)
  for (int u = tid; u < U; u += kPlanThreads) {
    const int c = ucl[u];
    const int cp = u > 0 ? ucl[u - 1] : -1;
    for (int k = cp + 1; k <= c; ++k) P.cluster_begin[k] = u;
    if (kStaged) P.unit_cluster[u] = c;
  }
  if (kStaged)
    for (int g = tid; g < G; g += kPlanThreads) P.groups[g] = grp[g];
  if (tid == 0) {
    const int last = U > 0 ? ucl[U - 1] : -1;
    for (int k = last + 1; k <= kMaxClusters; ++k) P.cluster_begin[k] = U;
    PlanHeader h;
    h.status = s_flags;
    h.num_groups = G;
    h.num_units = U;
    h.num_clusters = C;
    h.total_tiles = T;
    h.tiles_per_cluster = W;
    h.pad[0] = h.pad[1] = 0;
    *P.header = h;
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* qsl, int batch, int num_heads, int max_pages,
                        int page_size, int num_splits, int num_clusters, int group_rows, Plan plan,
                        const CacheWriteArgs* write, const QuantArgs* quant, int sm_count, cudaStream_t s) {
  const bool writes = write && write->num_tokens > 0;
  const int write_blocks = writes ? (int)((write->num_tokens + 7) / 8) : 0;
  int quant_blocks = 0;
  if (quant) {
    // grid-stride, the whole launch in one wave: four blocks per SM (each
    // holds the plan's shared memory), less the plan and write blocks
    const int64_t want = (quant->rows * (kDqk / 8) + kPlanThreads - 1) / kPlanThreads;
    int64_t cap = 4LL * (sm_count > 0 ? sm_count : 1) - 1 - write_blocks;
    if (cap < (sm_count > 0 ? sm_count : 1)) cap = sm_count > 0 ? sm_count : 1;
    quant_blocks = (int)(want < cap ? (want > 0 ? want : 1) : cap);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1u + (unsigned)write_blocks + (unsigned)quant_blocks);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool staged = plan.max_groups <= kPlanSmemGroups && plan.max_units <= kPlanSmemUnits;
  const int mode = quant ? 3 : (writes ? (write->fp8 ? 2 : 1) : 0);
  if (quant && writes && !write->fp8) return cudaErrorInvalidValue;   // an e4m3 query goes with an e4m3 cache
  const CacheWriteArgs w = writes ? *write : CacheWriteArgs{};
  const QuantArgs qa = quant ? *quant : QuantArgs{};
  using Kernel = void (*)(const int32_t*, const int32_t*, int, int, int, int, int, int, int, Plan,
                          const CacheWriteArgs, const QuantArgs, int);
  static const Kernel kernels[2][4] = {
      {plan_kernel<false, 0>, plan_kernel<false, 1>, plan_kernel<false, 2>, plan_kernel<false, 3>},
      {plan_kernel<true, 0>, plan_kernel<true, 1>, plan_kernel<true, 2>, plan_kernel<true, 3>}};
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernels[staged][mode], seq_lens, qsl, batch, num_heads, max_pages,
                                     page_size, num_splits, num_clusters, group_rows, plan, w, qa, write_blocks);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
