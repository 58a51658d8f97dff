// Absorbed MLA decode on sm_103a: tcgen05 tensor cores, TMEM accumulators,
// TMA page gathers, and a CTA pair that splits the latent width.
//
// Math (vllm/v1/attention/backends/mla/common.py, module docstring,
// "Data-Movement Friendly Approach"): for every query row (token t, head h)
//   s_j = scale * ([q_abs | q_pe] . [kv_c_j | k_pe_j]),  o = softmax(s) . kv_c
// over the keys its causal window allows (multi-token verify rule of the AITER
// MLA backend: L = seq_len - Sq + 1 + t).
//
// Design (one work unit = <=128 query rows of one request x a tile range):
//  * All query rows of a unit form the M = 128 dimension of both MMAs
//      S = Q . K^T   (M=128 rows, N=64 keys,  K=576)
//      O += P . V    (M=128 rows, N=dims,     K=64 keys),   V = kv_c.
//  * O for 128 rows x 512 dims in fp32 would fill all of TMEM, so a CLUSTER
//    OF TWO CTAs splits the latent width: CTA r owns output dims
//    [256r, 256r+256) and the matching slice of the score contraction
//    (CTA0: kv_c[0:256]; CTA1: kv_c[256:512] + k_pe).  Each CTA TMA-loads only
//    its own columns of every cached row, so every cache byte is read from
//    HBM once.  The two partial score tiles are exchanged through
//    distributed shared memory (st.async with mbarrier transaction counts)
//    and summed; both CTAs then run the identical online softmax.
//  * TMEM (512 columns): O half [0,256), Q slice as the A operand of the score
//    MMA [256,416), S [416,480), P (bf16, A operand of P.V) [480,512).
//  * Warp roles: warp 0 TMA producer, warp 1 MMA issuer (+TMEM owner),
//    warps 2-5 softmax / exchange / O rescale / epilogue (one query row per
//    thread, the row's TMEM lane).
//  * Online softmax in the exp2 domain with lazy rescaling: O and l are
//    rescaled only when a row's running max grows by more than 8 (log2
//    units); the final o = O / l and lse = (m + log2 l) ln 2 are exact for
//    any reference m.
//  * Split units write fp32 partials (normalised o and lse) that the combine
//    kernel merges (merge_attn_states rule).
//  * Every mbarrier wait is bounded (1 s); on expiry the CTA raises its abort
//    flag and the error word, skips all further waits and runs to the end
//    without touching memory outside its buffers.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kStages = 4;                       // cache-tile ring depth
constexpr int kBoxBytes = 64 * 128;              // 64 rows x 64 bf16 (128 B, swizzled)
constexpr int kStageBytes = 5 * kBoxBytes;       // up to 5 column boxes per CTA
constexpr int kXBytes = kRows * kTile * 4;       // one partial score tile (fp32)
constexpr int kNumThreads = 192;

constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemQ = 256;
constexpr uint32_t kTmemS = 416;
constexpr uint32_t kTmemP = 480;
constexpr float kRescaleThreshold = 8.0f;        // log2 units

struct __align__(8) Barriers {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t q_ready;
  uint64_t s_full;
  uint64_t s_free;
  uint64_t p_full;
  uint64_t o_done;
  uint64_t x_full[2];
  uint64_t x_free[2];
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + 2 * kXBytes + sizeof(Barriers);

struct Ctx {
  Barriers* bars;
  int* status;
};

__device__ __forceinline__ void raise_error(const Ctx& c, int bit) {
  c.bars->abort = 1;
  atomicOr(c.status, bit);
}

// Bounded wait; once the CTA has aborted every wait returns at once.
__device__ __forceinline__ void wait_bar(const Ctx& c, uint64_t* bar, uint32_t parity) {
  if (*(volatile int*)&c.bars->abort) return;
  if (!mbar_wait(smem_u32(bar), parity)) raise_error(c, 1);
}
__device__ __forceinline__ void wait_bar_cluster(const Ctx& c, uint64_t* bar, uint32_t parity) {
  if (*(volatile int*)&c.bars->abort) return;
  if (!mbar_wait_cluster(smem_u32(bar), parity)) raise_error(c, 1);
}

__device__ __forceinline__ void named_bar_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int kCacheFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kNumThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qpe,
                  const __grid_constant__ CUtensorMap tm_kv, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* stages = smem;
  uint8_t* xbuf = smem + kStages * kStageBytes;
  Barriers* bars = reinterpret_cast<Barriers*>(xbuf + 2 * kXBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = (int)cluster_id_x();
  const int nkb = rank == 0 ? 4 : 5;               // column boxes of this CTA
  const Plan& P = a.plan;
  Ctx ctx{bars, &P.header->status};

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->kv_full[i]), 1);
      mbar_init(smem_u32(&bars->kv_empty[i]), 1);
    }
    mbar_init(smem_u32(&bars->q_ready), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->s_free), 4);
    mbar_init(smem_u32(&bars->p_full), 4);
    mbar_init(smem_u32(&bars->o_done), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->x_full[i]), 1);
      mbar_init(smem_u32(&bars->x_free[i]), 4);
    }
    mbar_init(smem_u32(&bars->mma_drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_qpe);
    tma_prefetch_desc(&tm_kv);
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  const int ubeg = P.cluster_begin[cluster];
  const int uend = P.cluster_begin[cluster + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t item = 0;
      const int sub_rows = a.page_size < kTile ? a.page_size : kTile;
      const int nsub = kTile / sub_rows;
      const int oob_row = a.num_blocks * a.page_size;  // first row past the cache: reads zeros
      for (int u = ubeg; u < uend; ++u) {
        const UnitRec ur = P.units[u];
        const GroupRec gr = P.groups[ur.group];
        for (int half = 0; half < 2; ++half, ++item) {
          const uint32_t slot = item % kStages, round = item / kStages;
          wait_bar(ctx, &bars->kv_empty[slot], (round & 1) ^ 1);
          const uint32_t st = smem_u32(stages + slot * kStageBytes);
          const uint32_t full = smem_u32(&bars->kv_full[slot]);
          mbar_expect_tx(full, nkb * kBoxBytes);
          const int y = gr.row0 + 64 * half;
          for (int i = 0; i < 4; ++i) tma_load_2d(st + i * kBoxBytes, &tm_q, 256 * rank + 64 * i, y, full);
          if (rank == 1) tma_load_2d(st + 4 * kBoxBytes, &tm_qpe, 0, y, full);
        }
        const int32_t* bt = a.block_table + (size_t)gr.b * a.max_pages;
        for (int j = ur.tile_begin; j < ur.tile_end; ++j, ++item) {
          const uint32_t slot = item % kStages, round = item / kStages;
          wait_bar(ctx, &bars->kv_empty[slot], (round & 1) ^ 1);
          const uint32_t st = smem_u32(stages + slot * kStageBytes);
          const uint32_t full = smem_u32(&bars->kv_full[slot]);
          mbar_expect_tx(full, nkb * kBoxBytes);
          for (int sb = 0; sb < nsub; ++sb) {
            const int key = j * kTile + sb * sub_rows;
            const int lp = key / a.page_size;
            int y = oob_row;                 // sub-pages past the group's last key are not read
            if (key < gr.lmax && lp < a.max_pages) {
              const int blk = bt[lp];
              if (blk >= 0 && blk < a.num_blocks)
                y = blk * a.page_size + key % a.page_size;
              else
                atomicOr(ctx.status, 4);
            }
            const uint32_t dst = st + sb * sub_rows * 128;
            for (int i = 0; i < nkb; ++i) {
              const int x = rank == 0 ? 64 * i : (i < 4 ? 256 + 64 * i : 512);
              tma_load_2d(dst + i * kBoxBytes, &tm_kv, x, y, full);
            }
          }
        }
      }
      // drain: every issued load has landed before the CTA may exit
      const uint32_t first = item > kStages ? item - kStages : 0;
      for (uint32_t k = first; k < item; ++k) {
        if (*(volatile int*)&bars->abort) {
          // bounded even after an abort: the loads still target our own buffers
          mbar_wait(smem_u32(&bars->kv_full[k % kStages]), (k / kStages) & 1);
        } else {
          wait_bar(ctx, &bars->kv_full[k % kStages], (k / kStages) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, kTile, 0, 0);   // K-major keys
      const uint32_t id_pv = idesc_bf16_f32(128, 256, 0, 1);    // MN-major values
      uint32_t item = 0, it = 0, units_done = 0;
      for (int u = ubeg; u < uend; ++u) {
        const UnitRec ur = P.units[u];
        const int ntiles = ur.tile_end - ur.tile_begin;
        item += 2;  // the two Q items are consumed by the softmax warps
        wait_bar(ctx, &bars->q_ready, units_done & 1);
        tc_fence_after();
        uint32_t prev_slot = 0;
        for (int jj = 0; jj < ntiles; ++jj, ++item, ++it) {
          const uint32_t slot = item % kStages, round = item / kStages;
          wait_bar(ctx, &bars->kv_full[slot], round & 1);
          wait_bar(ctx, &bars->s_free, (it & 1) ^ 1);
          tc_fence_after();
          const uint32_t st = smem_u32(stages + slot * kStageBytes);
          for (int i = 0; i < nkb; ++i)
            for (int k = 0; k < 4; ++k)
              mma_ts(tbase + kTmemS, tbase + kTmemQ + i * 32 + k * 8,
                     smem_desc(st + i * kBoxBytes + k * 32, 16, 1024, kSwizzle128B), id_s, (i | k) != 0);
          mma_commit(smem_u32(&bars->s_full));
          if (jj > 0) {
            wait_bar(ctx, &bars->p_full, (it - 1) & 1);
            tc_fence_after();
            const uint32_t pst = smem_u32(stages + prev_slot * kStageBytes);
            for (int k = 0; k < 4; ++k)
              mma_ts(tbase + kTmemO, tbase + kTmemP + k * 8,
                     smem_desc(pst + k * 2048, kBoxBytes, 1024, kSwizzle128B), id_pv, (jj > 1) || (k > 0));
            mma_commit(smem_u32(&bars->o_done));
            mma_commit(smem_u32(&bars->kv_empty[prev_slot]));
          }
          prev_slot = slot;
        }
        if (ntiles > 0) {
          wait_bar(ctx, &bars->p_full, (it - 1) & 1);
          tc_fence_after();
          const uint32_t pst = smem_u32(stages + prev_slot * kStageBytes);
          for (int k = 0; k < 4; ++k)
            mma_ts(tbase + kTmemO, tbase + kTmemP + k * 8, smem_desc(pst + k * 2048, kBoxBytes, 1024, kSwizzle128B),
                   id_pv, (ntiles > 1) || (k > 0));
          mma_commit(smem_u32(&bars->o_done));
          mma_commit(smem_u32(&bars->kv_empty[prev_slot]));
        }
        ++units_done;
      }
      // every issued MMA has completed before TMEM is released
      mma_commit(smem_u32(&bars->mma_drain));
      mbar_wait(smem_u32(&bars->mma_drain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- softmax / exchange / epilogue
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = q4 * 32 + lane;          // query row of this thread in the unit
    const uint32_t tl = tbase + ((uint32_t)(q4 * 32) << 16);
    const int tid128 = threadIdx.x - 64;
    const uint32_t x_local[2] = {smem_u32(xbuf), smem_u32(xbuf + kXBytes)};
    const uint32_t x_remote[2] = {mapa(x_local[0], peer), mapa(x_local[1], peer)};
    const uint32_t xfull_remote[2] = {mapa(smem_u32(&bars->x_full[0]), peer), mapa(smem_u32(&bars->x_full[1]), peer)};
    const uint32_t xfree_remote[2] = {mapa(smem_u32(&bars->x_free[0]), peer), mapa(smem_u32(&bars->x_free[1]), peer)};
    const uint32_t xrow_off = (uint32_t)row * (kTile * 4);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);

    uint32_t item = 0, it = 0, od = 0;
    for (int u = ubeg; u < uend; ++u) {
      const UnitRec ur = P.units[u];
      const GroupRec gr = P.groups[ur.group];
      const int b = gr.b;
      const int sq = a.qsl ? a.qsl[b + 1] - a.qsl[b] : 1;
      const int q0 = a.qsl ? a.qsl[b] : b;
      const int R = gr.row0 + row;
      const bool valid = row < gr.nrows && R < a.total_rows;
      int Lr = 0;
      if (valid) {
        const int tloc = R / a.num_heads - q0;
        Lr = a.seq_lens[b] - sq + 1 + tloc;
        Lr = Lr < 0 ? 0 : (Lr > gr.lmax ? gr.lmax : Lr);
      }

      // Q slice -> TMEM (A operand of the score MMA)
      {
        const uint32_t my = item + (row >= 64 ? 1 : 0);
        const uint32_t slot = my % kStages, round = my / kStages;
        wait_bar(ctx, &bars->kv_full[slot], round & 1);
        __syncwarp();
        const int k = row & 63;
        const uint32_t base = smem_u32(stages + slot * kStageBytes) + k * 128;
        for (int i = 0; i < nkb; ++i) {
          uint32_t q[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = lds128(base + i * kBoxBytes + ((c ^ (k & 7)) << 4));
            q[4 * c + 0] = v.x;
            q[4 * c + 1] = v.y;
            q[4 * c + 2] = v.z;
            q[4 * c + 3] = v.w;
          }
          tmem_st32(tl + kTmemQ + i * 32, q);
        }
        tmem_wait_st();
        tc_fence_before();
        named_bar_softmax();
        if (tid128 == 0) {
          mbar_arrive(smem_u32(&bars->kv_empty[item % kStages]));
          mbar_arrive(smem_u32(&bars->kv_empty[(item + 1) % kStages]));
          mbar_arrive(smem_u32(&bars->q_ready));
        }
        item += 2;
      }

      float m = -INFINITY, l = 0.f;
      const int ntiles = ur.tile_end - ur.tile_begin;
      for (int jj = 0; jj < ntiles; ++jj, ++item, ++it) {
        const int key0 = (ur.tile_begin + jj) * kTile;
        float s[kTile];
        wait_bar(ctx, &bars->s_full, it & 1);
        __syncwarp();
        tc_fence_after();
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tl + kTmemS, r0);
          tmem_ld32(tl + kTmemS + 32, r1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            s[c] = __uint_as_float(r0[c]);
            s[32 + c] = __uint_as_float(r1[c]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->s_free));

        // exchange partial scores with the peer CTA
        const int xb = it & 1;
        const uint32_t xu = it >> 1;
        wait_bar_cluster(ctx, &bars->x_free[xb], (xu & 1) ^ 1);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_async_v4(x_remote[xb] + xrow_off + ((c ^ (row & 15)) << 4), __float_as_uint(s[4 * c]),
                      __float_as_uint(s[4 * c + 1]), __float_as_uint(s[4 * c + 2]), __float_as_uint(s[4 * c + 3]),
                      xfull_remote[xb]);
        if (tid128 == 0) mbar_expect_tx(smem_u32(&bars->x_full[xb]), kXBytes);
        wait_bar_cluster(ctx, &bars->x_full[xb], xu & 1);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint4 v = lds128(x_local[xb] + xrow_off + ((c ^ (row & 15)) << 4));
          s[4 * c + 0] += __uint_as_float(v.x);
          s[4 * c + 1] += __uint_as_float(v.y);
          s[4 * c + 2] += __uint_as_float(v.z);
          s[4 * c + 3] += __uint_as_float(v.w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(xfree_remote[xb]);

        // online softmax (exp2 domain)
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          const float v = (key0 + c < Lr) ? s[c] * a.scale_log2 : -INFINITY;
          s[c] = v;
          tmax = fmaxf(tmax, v);
        }
        float alpha = 1.f;
        if (tmax > m + kRescaleThreshold) {
          alpha = fast_exp2(m - tmax);  // m = -inf -> 0
          l *= alpha;
          m = tmax;
        }
        const float mref = m == -INFINITY ? 0.f : m;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float p0 = fast_exp2(s[2 * c] - mref);
          const float p1 = fast_exp2(s[2 * c + 1] - mref);
          l += p0 + p1;
          pk[c] = pack_bf16x2(p0, p1);
        }
        if (jj > 0) {
          wait_bar(ctx, &bars->o_done, od & 1);
          ++od;
          __syncwarp();
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            for (int ch = 0; ch < 8; ++ch) {
              uint32_t o[32];
              tmem_ld32(tl + kTmemO + ch * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tmem_st32(tl + kTmemO + ch * 32, o);
            }
          }
        }
        tmem_st32(tl + kTmemP, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
      }

      // epilogue
      if (ntiles > 0) {
        wait_bar(ctx, &bars->o_done, od & 1);
        ++od;
      }
      __syncwarp();
      tc_fence_after();
      const float inv = l > 0.f ? a.out_scale / l : 0.f;
      const float lse_nat = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t o[32];
        tmem_ld32(tl + kTmemO + ch * 32, o);
        tmem_wait_ld();
        if (!valid) continue;
        const int d0 = 256 * rank + 32 * ch;
        if (ur.slot < 0) {
          uint4* dst = reinterpret_cast<uint4*>(out + (size_t)R * kLkv + d0);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(P.part_o + ((size_t)ur.slot * kRows + row) * kLkv + d0);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                 __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        }
      }
      if (valid && rank == 0) {
        if (ur.slot < 0) {
          if (a.lse) a.lse[R] = lse_nat;
        } else {
          P.part_lse[(size_t)ur.slot * kRows + row] = lse_nat;
        }
      }
      tc_fence_before();
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  cluster_sync();  // no CTA leaves while its peer may still write into it
}

}  // namespace

size_t decode_smem_bytes(int) { return kSmemBytes; }

cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_qpe, const CUtensorMap& tm_kv,
                          int cache_dtype, const DecodeArgs& a, int num_clusters, cudaStream_t s) {
  (void)cache_dtype;
  auto kern = decode_kernel<0>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<2 * num_clusters, kNumThreads, kSmemBytes, s>>>(tm_q, tm_qpe, tm_kv, a);
  return cudaGetLastError();
}

}  // namespace mla
