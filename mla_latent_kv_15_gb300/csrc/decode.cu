// Absorbed MLA decode on sm_103a: tcgen05 tensor cores, TMEM accumulators,
// TMA page gathers, and a CTA pair that splits the 576-wide contraction of the
// scores and the 512-wide output.
//
// Math (vllm/v1/attention/backends/mla/common.py, module docstring,
// "Data-Movement Friendly Approach"): for every query row (token t, head h)
//   s_j = scale * ([q_abs | q_pe] . [kv_c_j | k_pe_j]),  o = softmax(s) . kv_c
// over the keys its causal window allows (multi-token verify rule of the AITER
// MLA backend: L = seq_len - Sq + 1 + t).
//
// Design (one work unit = <=128 query rows of one request x a tile range):
//  * The query rows of a unit form the M = 128 dimension of every MMA.
//  * A cluster of two CTAs shares each 64-key tile.  CTA r owns
//      - dims [256r, 256r+256) of the latent output, O += P . V;
//      - half of the score contraction: the same 256 latent dims plus rope
//        dims [32r, 32r+32), i.e. cache columns [256r, 256r+256) and
//        [512+32r, 512+32r+32).  It loads exactly those columns of every
//        cached row (the pair reads each cached byte once) and keeps the
//        matching 288 query dims in TMEM as the A operand.
//    Each CTA computes a partial score tile S_r (18 MMAs, N = 64 keys), stores
//    it into the peer's shared memory (st.async over the cluster network), and
//    adds the peer's partial to its own.  Nothing is computed twice.
//  * Exchange format: 16-bit block fixed point.  Per row and half tile (32
//    keys) the sender takes the range [lo, hi] of its partials over the keys
//    the row may see and sends 16-bit codes of (s - c) / step, c = (lo + hi)
//    / 2, step = half range / 32766, with c and step as an 8-byte header.
//    The absolute error is at most 1.5 steps whatever the magnitude of the
//    partials (fp16 would lose 2^-11 of |s|, a problem once partials reach
//    hundreds).  The receiver folds c into the row's maximum and the
//    exponent's offset.
//  * The next tile's codes go out while the current tile is processed: the
//    first half between the decoding steps of the received codes, the rest
//    after the exponentials, so the network transfer overlaps the arithmetic.
//    Partials
//    land in a ring of four receive buffers that needs no return handshake:
//    a CTA writes tile i+1 into the buffer of tile i-3 only after it has
//    received tile i-1 from the peer, and the peer sent tile i-1 only after
//    all its softmax threads had read tile i-3.  The code part of a buffer is
//    chunk-major ([8 chunks][rows][16 B]), so the 32 lanes of a warp write
//    512 contiguous bytes of the peer's shared memory per st.async.
//  * TMEM (512 columns): O half [0,256), Q slice [256,400), S [400,464),
//    bf16 P (A operand of P.V) [464,496).  With an e4m3 query the Q slice
//    holds codes, four per column, and fills only [256,328).
//  * e4m3 query over an e4m3 cache: the score MMAs are fp8 x fp8
//    (kind::f8f6f4, K = 32) straight on the landed e4m3 boxes; only the
//    value dims are widened to bf16 for P.V, after the tile's score MMAs
//    are done with the codes; the partial scores are multiplied by
//    q_scale * kv_scale before the exchange.
//  * Warp roles: a TMA producer, a score-MMA issuer (+TMEM owner), a P.V-MMA
//    issuer, eight softmax / exchange / O rescale / epilogue warps (two
//    threads per query row, each a key half of every tile and an output
//    half of O) and, for an e4m3 cache, four warps that expand e4m3 tiles to
//    bf16 (see Roles).  Separate score and P.V issuers let the two MMA
//    accumulation chains overlap in the tensor pipe.
//  * The producer looks up a tile's block-table entries before it waits for
//    the tile's ring slot, so a freed slot is refilled at once; cache tiles
//    are loaded with an L2 evict-first policy.
//  * Online softmax in the exp2 domain with lazy rescaling: O and l are
//    rescaled only when a row's running max grows by more than 8 (log2
//    units); the final o = O / l and lse = (m + log2 l) ln 2 are exact for
//    any reference m.  The exponentials are computed with the current
//    reference while the row's two halves exchange their tile maxima, and
//    again only if the maximum moved.  CTA 0 writes the LSE.
//  * Split units write partials that the combine kernel merges
//    (merge_attn_states rule): the normalised o as fp16 codes with a
//    power-of-two scale per 32-dim chunk (the chunk's largest magnitude
//    lands in [2^14, 2^15): 11 significant bits at any magnitude, half the
//    bytes of fp32) and the lse in fp32.  The epilogue stages each warp's
//    32 rows through 4 KB of shared memory (two receive buffers the peer
//    cannot be writing at that point) so that its global stores are whole
//    128-byte lines; with a bf16 cache and 128-row units a whole 32-row
//    piece leaves by one TMA store, which drains while the warp goes on to
//    the next unit.
//  * A unit's plan record is one 32-byte line, prefetched into L1 during the
//    epilogue of the unit before.
//  * Waits take a completed phase at once and otherwise suspend on the
//    barrier (1 us hints).  Every mbarrier wait is bounded (1 s unless the
//    launch asks for less); on
//    expiry the CTA raises its abort flag and the error word, skips its local
//    waits and runs to the end without touching memory outside its buffers.
//    Waits for the peer's partial scores stay bounded waits even then (at most
//    1 ms each once aborted), so no store of the peer is still in flight into
//    this CTA's shared memory when it exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kBox = 64 * 128;                    // 64 rows x 64 bf16 (128 B rows, 128-B swizzle)
constexpr int kVBoxes = 4;                        // the CTA's 256 latent dims: values and scores
constexpr int kRopeBox = 64 * 64;                 // 64 rows x 32 bf16 rope dims (64 B rows, 64-B swizzle)
constexpr int kRopeOff = kVBoxes * kBox;          // rope half-box after the four latent boxes
constexpr int kStageBytes = kRopeOff + kRopeBox;  // 36 KB: every cached column the CTA reads
static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of the 128-B swizzle");
// e4m3 cache, bf16 query (variant 1): the CTA's e4m3 tile lands unswizzled in
// the top of its bf16 slot (four 64 x 64-byte boxes, then the 64 x 32-byte
// rope half-box) and is expanded in place into the bf16 layout above.
constexpr int kFp8Box = 64 * 64;
constexpr int kFp8RopeBox = 64 * 32;
constexpr int kFp8TileBytes = kVBoxes * kFp8Box + kFp8RopeBox;   // 18 KB
constexpr int kFp8InPlace = kStageBytes - kFp8TileBytes;
// e4m3 query and cache (variant 3): each item lands as two 128-dim boxes (64
// rows x 128 e4m3, 128-B swizzle) and one 32-dim rope box (64 rows x 32 e4m3,
// 32-B swizzle) that the fp8 score MMAs read directly, in the top 18 KB of
// the slot; the value dims (the two 128-dim boxes) are then expanded to bf16
// into boxes 0-3 of the slot, once the tile's score MMAs are done.
constexpr int kQ8Box = 64 * 128;
constexpr int kQ8RopeBox = 64 * 32;
constexpr int kQ8Bytes = 2 * kQ8Box + kQ8RopeBox;
constexpr int kQ8InPlace = kStageBytes - kQ8Bytes;
static_assert(kQ8InPlace % 1024 == 0 && kQ8InPlace + kQ8Bytes == kStageBytes, "e4m3 landing area");
// Kernel variants: 0 bf16 cache; 1 e4m3 cache (expanded in place in the bf16
// ring); 3 e4m3 query and e4m3 cache (fp8 score MMAs, values expanded for
// P.V); 2 bf16 cache with at most 32 query rows per unit (small head counts:
// the receive ring shrinks to 32-row buffers and the cache ring gets a fifth
// stage).
template <int kVariant>
struct Layout {
  static constexpr int kStages = kVariant == 2 ? 5 : 4;
  static constexpr int kXRows = kVariant == 2 ? 32 : kRows;        // rows of a receive buffer
  static constexpr int kXChunk = kXRows * 16;                      // one 16-byte chunk of every row
  static constexpr int kXHdr = 8 * kXChunk;                        // row headers after the 8 code chunks
  static constexpr int kXBytes = kXHdr + kXRows * 16;              // codes + (centre, step) per row half
};
constexpr int kXBuffers = 4;                      // receive ring (4: reuse needs no handshake)
constexpr uint32_t kXRowBytes = 2 * (kTile + 8);  // exchanged bytes per row and tile: two halves, codes + header
// Warp roles.  Warps 0-7: softmax / exchange / O rescale / epilogue, two
// threads per query row (warp w: TMEM lanes 32(w%4).., key half and output
// half w/4).  Warp 8: TMA producer; 9: score-MMA issuer (and TMEM owner);
// 10: P.V-MMA issuer; 11 idle; e4m3 cache: 12-15 expand e4m3 tiles to bf16.
template <int kVariant>
struct Roles {
  static constexpr int kThreads = (kVariant == 1 || kVariant == 3) ? 512 : 384;
};
constexpr int kSoftmaxWarps = 8;
// e4m3 cache: register budget per thread of each warpgroup (two softmax
// groups, the producer/issuer group, the expansion group) within the 512 x 128
// the CTA is launched with
constexpr uint32_t kRegsSoftmax8 = 168, kRegsIssue8 = 96, kRegsExpand8 = 80;
static_assert(128 * (2 * kRegsSoftmax8 + kRegsIssue8 + kRegsExpand8) <= 512 * 128, "register split");
constexpr int kWarpProducer = 8, kWarpScore = 9, kWarpPV = 10, kWarpExpand0 = 12;
constexpr int kQCols = 144;                       // 288 query dims as packed bf16 pairs

constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemQ = 256;
constexpr uint32_t kTmemS = kTmemQ + kQCols;      // 400
constexpr uint32_t kTmemP = kTmemS + kTile;       // 464
constexpr float kRescaleThreshold = 8.0f;         // log2 units
// Exchange codes: c + (u - 32768) * step, u in [1, 65535].  A float of value
// 12582912 + u (1.5 * 2^23 + u) holds u in its low 16 bits.
constexpr float kCodeMagic = 12582912.0f + 32768.0f;
constexpr float kCodeRange = 32766.0f;            // |code| <= 32766 leaves a margin for rounding
constexpr uint64_t kAbortWaitNs = 1000000ull;     // bound of a peer wait once the CTA has aborted

static_assert(kTmemP + kTile / 2 <= 512, "TMEM columns");

constexpr int kMaxStages = 5;
constexpr int kMaxSub = 4;   // sub-pages of a tile (pages of 16 rows)

struct __align__(8) Barriers {
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];  // 2 arrivals: score issuer + P.V issuer (or 2 from the softmax for query items)
  uint64_t stg_full[kMaxStages];  // e4m3 tile landed in the upper part of its ring slot
  uint64_t kx_free[kMaxStages];   // variant 3: the slot's score MMAs are done (its e4m3 boxes may be overwritten)
  uint64_t q_ready;
  uint64_t s_full;
  uint64_t s_free;
  uint64_t p_full;
  uint64_t p_free;
  uint64_t o_full;
  uint64_t x_full[kXBuffers];   // peer's partial scores landed (transaction count)
  uint64_t s_drain;
  uint64_t p_drain;
  uint32_t tmem_base;
  int abort;
};

// the two threads of a row exchange their tile maxima (two parities) and,
// at the end of a unit, their row sums: [2][2][128] + [2][128] floats
constexpr int kPairFloats = 2 * 2 * kRows + 2 * kRows;

template <int kVariant>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Layout<kVariant>::kStages * kStageBytes +
         kXBuffers * (size_t)Layout<kVariant>::kXBytes + sizeof(Barriers) + 16 + kPairFloats * sizeof(float);
}
static_assert(smem_bytes<0>() <= 232448 && smem_bytes<1>() <= 232448 && smem_bytes<2>() <= 232448 &&
                  smem_bytes<3>() <= 232448,
              "shared memory per CTA");
static_assert(Layout<0>::kStages <= kMaxStages && Layout<1>::kStages <= kMaxStages &&
                  Layout<2>::kStages <= kMaxStages && Layout<3>::kStages <= kMaxStages,
              "barrier arrays");
static_assert(Layout<0>::kXBytes % 16 == 0 && Layout<2>::kXBytes % 16 == 0, "receive buffers 16-byte aligned");

struct Ctx {
  Barriers* bars;
  int* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ void raise_error(const Ctx& c, int bit) {
  c.bars->abort = 1;
  atomicOr(c.status, bit);
}

// Bounded waits on this CTA's own pipeline; once the CTA has aborted they
// return at once.
__device__ __forceinline__ void wait_bar(const Ctx& c, uint64_t* bar, uint32_t parity) {
  // a completed phase is taken at once (aborted or not); the abort flag is
  // read only when the wait would block
  if (mbar_try_wait(smem_u32(bar), parity)) return;
  if (*(volatile int*)&c.bars->abort) return;
  if (!mbar_wait(smem_u32(bar), parity, c.limit_ns)) raise_error(c, 1);
}
// Bounded wait for the peer's partial scores.  It is kept after an abort
// (with a 1 ms bound): the peer's stores into this CTA's receive buffers must
// land before the CTA exits.
__device__ __forceinline__ void wait_bar_cluster(const Ctx& c, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(smem_u32(bar), parity)) return;
  const bool aborted = *(volatile int*)&c.bars->abort;
  const uint64_t lim = aborted && c.limit_ns > kAbortWaitNs ? kAbortWaitNs : c.limit_ns;
  if (!mbar_wait_cluster(smem_u32(bar), parity, lim)) raise_error(c, 1);
}

__device__ __forceinline__ void named_bar_softmax() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// the two warps holding the halves of the same rows (warps q and q + 4)
__device__ __forceinline__ void named_bar_pair(int q) { asm volatile("bar.sync %0, 64;" ::"r"(3 + q) : "memory"); }
__device__ __forceinline__ void named_bar_expand() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// three-input max (one instruction on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// packed pair arithmetic (one f32x2 instruction for two fp32 lanes)
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n .reg .b64 x, y;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n add.rn.f32x2 x, x, y;\n"
      " mov.b64 {%0, %1}, x;\n}" : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fma2(float& r0, float& r1, float a0, float a1, float b, float c) {
  asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %4};\n mov.b64 z, {%5, %5};\n"
      " fma.rn.f32x2 x, x, y, z;\n mov.b64 {%0, %1}, x;\n}" : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// acc = d * b + acc for a pair (vector addend)
__device__ __forceinline__ void fma2v(float& acc0, float& acc1, float d0, float d1, float b) {
  asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %4};\n mov.b64 z, {%0, %1};\n"
      " fma.rn.f32x2 z, x, y, z;\n mov.b64 {%0, %1}, z;\n}" : "+f"(acc0), "+f"(acc1) : "f"(d0), "f"(d1), "f"(b));
}

// three-input min
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Maximum of 32 values (NaN entries are ignored: max returns the other operand).
__device__ __forceinline__ float max_tree32(const float (&x)[32]) {
  float m[11];
#pragma unroll
  for (int c = 0; c < 10; ++c) m[c] = fmax3(x[3 * c], x[3 * c + 1], x[3 * c + 2]);
  m[10] = fmaxf(x[30], x[31]);
  return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmax3(m[6], m[7], fmax3(m[8], m[9], m[10])));
}

// Maximum and minimum over the first n of 32 values (n < 32: the last,
// ragged tile of a row; the other values are left out); NaN if n <= 0.
__device__ __forceinline__ void range_first_n(const float (&x)[kTile / 2], int n, float& hi, float& lo) {
  const float nan = __int_as_float(0x7fffffff);
  float h[11], l[11];
#pragma unroll
  for (int c = 0; c < 10; ++c) {
    const float a = 3 * c < n ? x[3 * c] : nan, b = 3 * c + 1 < n ? x[3 * c + 1] : nan,
                d = 3 * c + 2 < n ? x[3 * c + 2] : nan;
    h[c] = fmax3(a, b, d);
    l[c] = fmin3(a, b, d);
  }
  const float a = 30 < n ? x[30] : nan, b = 31 < n ? x[31] : nan;
  h[10] = fmaxf(a, b);
  l[10] = fminf(a, b);
  hi = fmax3(fmax3(h[0], h[1], h[2]), fmax3(h[3], h[4], h[5]), fmax3(h[6], h[7], fmax3(h[8], h[9], h[10])));
  lo = fmin3(fmin3(l[0], l[1], l[2]), fmin3(l[3], l[4], l[5]), fmin3(l[6], l[7], fmin3(l[8], l[9], l[10])));
}

__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 v, uint32_t (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[j] & 0xFFFF), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[j] >> 16), __NV_E4M3);
    const float2 flo = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 fhi = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    o[2 * j] = pack_bf16x2(flo.x, flo.y);
    o[2 * j + 1] = pack_bf16x2(fhi.x, fhi.y);
  }
}

// Expand one e4m3 tile (four 64 x 64-byte latent boxes and one 64 x 32-byte
// rope box, row-major, at the top of the ring slot) into the bf16 layouts the
// MMAs read (what bf16 TMA loads would have written: 128-byte-swizzled
// latent boxes, a 64-byte-swizzled rope box), in place: every thread first
// reads its share of the whole tile, then all write.  e4m3 -> f16 -> f32 ->
// bf16 is exact: every e4m3 value is a bf16 value.  Runs on the 128 threads of
// the expansion warps; 9 chunks of 16 codes each.
__device__ __forceinline__ void expand_e4m3_tile(uint32_t stage, int t) {
  constexpr int kPer = kFp8TileBytes / 16 / 128;
  static_assert(kPer == 9, "8 latent chunks and 1 rope chunk per thread");
  uint4 v[kPer];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = t + 128 * k;
    const int q = i & 3, r = (i >> 2) & 63, p = i >> 8;   // chunk in the row, row (key), box
    v[k] = lds128(stage + kFp8InPlace + p * kFp8Box + r * 64 + q * 16);
  }
  // rope: row t >> 1, chunk t & 1
  v[8] = lds128(stage + kFp8InPlace + kVBoxes * kFp8Box + (t >> 1) * 32 + (t & 1) * 16);
  named_bar_expand();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = t + 128 * k;
    const int q = i & 3, r = (i >> 2) & 63, p = i >> 8;
    uint32_t o[8];
    e4m3x16_to_bf16(v[k], o);
    const uint32_t row = stage + p * kBox + r * 128;
    sts128(row + (((2 * q) ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
    sts128(row + (((2 * q + 1) ^ (r & 7)) << 4), o[4], o[5], o[6], o[7]);
  }
  {
    const int r = t >> 1, q = t & 1;                      // 16 rope dims 16q.. of row r -> 64-B swizzled chunks 2q, 2q+1
    uint32_t o[8];
    e4m3x16_to_bf16(v[8], o);
    const uint32_t row = stage + kRopeOff + r * 64;
    const int sw = (r >> 1) & 3;
    sts128(row + (((2 * q) ^ sw) << 4), o[0], o[1], o[2], o[3]);
    sts128(row + (((2 * q + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
  }
}

template <int kVariant>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Roles<kVariant>::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qr,
                  const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kvr,
                  const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_part,
                  const DecodeArgs a) {
  constexpr int kCacheFp8 = kVariant == 1 || kVariant == 3;
  constexpr bool kQ8 = kVariant == 3;       // e4m3 query: fp8 x fp8 score MMAs
  // the epilogue's pieces leave by TMA stores (bf16 cache, 128-row units:
  // measured 1 % faster there; the e4m3 variants' softmax warps spill more
  // with it and the e4m3-query one ran 10 % slower)
  constexpr bool kTmaStore = kVariant == 0;
  constexpr int kStages = Layout<kVariant>::kStages;
  constexpr int kXBytes = Layout<kVariant>::kXBytes;
  constexpr int kXRows = Layout<kVariant>::kXRows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* stages = smem;
  uint8_t* x_recv = stages + kStages * kStageBytes;      // receive ring
  Barriers* bars = reinterpret_cast<Barriers*>(x_recv + kXBuffers * kXBytes);
  float* pairbuf = reinterpret_cast<float*>(((uintptr_t)(bars + 1) + 15) & ~(uintptr_t)15);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = (int)cluster_id_x();
  const Plan& P = a.plan;
  Ctx ctx{bars, &P.header->status, a.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->kv_full[i]), 1);
      mbar_init(smem_u32(&bars->kv_empty[i]), 2);
    }
    for (int i = 0; i < kMaxStages; ++i) mbar_init(smem_u32(&bars->stg_full[i]), 1);
    for (int i = 0; i < kMaxStages; ++i) mbar_init(smem_u32(&bars->kx_free[i]), 1);
    mbar_init(smem_u32(&bars->q_ready), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->s_free), kSoftmaxWarps);
    mbar_init(smem_u32(&bars->p_full), kSoftmaxWarps);
    mbar_init(smem_u32(&bars->p_free), 1);
    mbar_init(smem_u32(&bars->o_full), 1);
    for (int i = 0; i < kXBuffers; ++i) mbar_init(smem_u32(&bars->x_full[i]), 1);
    mbar_init(smem_u32(&bars->s_drain), 1);
    mbar_init(smem_u32(&bars->p_drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpScore) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_qr);
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_kvr);
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  // everything above overlaps the plan kernel (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the combine kernel may launch now (its blocks take SMs as CTAs of this
  // grid finish; it waits for the whole grid before reading the partials)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int ubeg = P.cluster_begin[cluster];
  const int uend = P.cluster_begin[cluster + 1];

  // Role bodies; the dispatch below differs per cache type: with an e4m3
  // cache each warpgroup first sets its register budget, so the compiler
  // allocates every role's code against that budget.
  auto producer = [&]() {
    // ------------------------------------------------------------ producer
    // Lane 0 streams everything with TMA: bf16 tiles straight into the ring;
    // e4m3 tiles into the top of the ring slot, which the expansion warps
    // turn into the bf16 layout the MMAs read.  Each CTA loads its 256
    // latent columns [256r, 256r+256) and its 32 rope columns
    // [512+32r, 512+32r+32) of every cached row.
    const bool leader = lane == 0;
    if (leader) {
      uint32_t item = 0;
      const int sub_rows = a.page_size < kTile ? a.page_size : kTile;
      const int nsub = kTile / sub_rows;
      const int oob_row = a.num_blocks * a.page_size;  // first row past the cache: reads zeros
      const int xl = 256 * (int)rank, xr = kLkv + 32 * (int)rank;   // first latent / rope column of the CTA
      // cache lines are read once per pair: evict them first, so that the
      // split-KV partials, queries and block tables stay in L2
      const uint64_t pol = l2_policy_evict_first();
      for (int u = ubeg; u < uend; ++u) {
        const UnitRec ur = P.units[u];
        const UnitRec& gr = ur;
        const int32_t* bt = a.block_table + (size_t)gr.b * a.max_pages;
        // loads the CTA's columns of tile j (all sub-pages) into dst, counting on `full`:
        //   bf16:           4 latent boxes of 64 x 128 B, then the 64 x 64-B rope box
        //   e4m3 (v1):      4 latent boxes of 64 x 64 B, then the 64 x 32-B rope box
        //   e4m3 query (v3): 2 latent boxes of 64 x 128 B, then the 64 x 32-B rope box
        // cache row of sub-page sb of tile j (a block-table lookup)
        auto lookup = [&](int j, int sb) {
          const int key = j * kTile + sb * sub_rows;
          const int lp = key / a.page_size;
          int y = oob_row;                   // sub-pages past the group's last key are not read
          if (key < gr.lmax && lp < a.max_pages) {
            const int blk = bt[lp];
            if (blk >= 0 && blk < a.num_blocks)
              y = blk * a.page_size + key % a.page_size;
            else
              atomicOr(ctx.status, 4);
          }
          return y;
        };
        const int ntiles = ur.tile_end - ur.tile_begin;
        // the CTA's 288 query dims for rows 0-63, then 64-127
        for (int half = 0; half < 2; ++half, ++item) {
          if (!leader) continue;
          const uint32_t slot = item % kStages, round = item / kStages;
          wait_bar(ctx, &bars->kv_empty[slot], (round & 1) ^ 1);
          const uint32_t st = smem_u32(stages + slot * kStageBytes);
          const int y = gr.row0 + 64 * half;
          if constexpr (kQ8) {
            // e4m3 query rows [q_abs | q_pe] (576 wide): the CTA's two
            // 128-dim latent boxes and its 32-dim rope box
            const uint32_t full = smem_u32(&bars->stg_full[slot]);
            mbar_expect_tx(full, kQ8Bytes);
            for (int p = 0; p < 2; ++p) tma_load_2d(st + kQ8InPlace + p * kQ8Box, &tm_q, xl + 128 * p, y, full);
            tma_load_2d(st + kQ8InPlace + 2 * kQ8Box, &tm_qr, xr, y, full);
            // kv_full's phases count every item of the slot
            mbar_arrive(smem_u32(&bars->kv_full[slot]));
          } else {
            // bf16 q_abs boxes (64 dims) and the q_pe half (32 dims, 64-B swizzle)
            const uint32_t full = smem_u32(&bars->kv_full[slot]);
            mbar_expect_tx(full, kStageBytes);
            for (int p = 0; p < kVBoxes; ++p) tma_load_2d(st + p * kBox, &tm_q, xl + 64 * p, y, full);
            tma_load_2d(st + kRopeOff, &tm_qr, 32 * (int)rank, y, full);
            // e4m3 cache: a query item also completes a phase of the slot's
            // stg_full, so its phases count every item of the slot
            if (kCacheFp8) mbar_arrive(smem_u32(&bars->stg_full[slot]));
          }
        }
        for (int jj = 0; jj < ntiles; ++jj, ++item) {
          // test aid: CTA 0 of cluster 0 never loads its first cache tile, so
          // a consumer's bounded wait for it runs out
          if (a.debug_skip_tile && cluster == 0 && rank == 0 && u == ubeg && jj == 0) continue;
          const uint32_t slot = item % kStages, round = item / kStages;
          {
            // The block-table lookups precede the slot wait, so their
            // latency overlaps it and the tile is issued the moment the slot
            // frees (measured 5-9 % faster kernels on the DeepSeek-V3-shaped
            // and multi-token batches)
            int ys[kMaxSub];
#pragma unroll
            for (int sb = 0; sb < kMaxSub; ++sb) {
              if (sb >= nsub) break;
              ys[sb] = lookup(ur.tile_begin + jj, sb);
            }
            wait_bar(ctx, &bars->kv_empty[slot], (round & 1) ^ 1);
            if constexpr (!kCacheFp8) {
              const uint32_t full = smem_u32(&bars->kv_full[slot]);
              mbar_expect_tx(full, kStageBytes);
              const uint32_t dst = smem_u32(stages + slot * kStageBytes);
#pragma unroll
              for (int sb = 0; sb < kMaxSub; ++sb) {
                if (sb >= nsub) break;
                for (int p = 0; p < kVBoxes; ++p)
                  tma_load_2d_hint(dst + p * kBox + sb * sub_rows * 128, &tm_kv, xl + 64 * p, ys[sb], full, pol);
                tma_load_2d_hint(dst + kRopeOff + sb * sub_rows * 64, &tm_kvr, xr, ys[sb], full, pol);
              }
            } else if constexpr (kQ8) {
              const uint32_t full = smem_u32(&bars->stg_full[slot]);
              mbar_expect_tx(full, kQ8Bytes);
              const uint32_t dst = smem_u32(stages + slot * kStageBytes + kQ8InPlace);
#pragma unroll
              for (int sb = 0; sb < kMaxSub; ++sb) {
                if (sb >= nsub) break;
                for (int p = 0; p < 2; ++p)
                  tma_load_2d_hint(dst + p * kQ8Box + sb * sub_rows * 128, &tm_kv, xl + 128 * p, ys[sb], full, pol);
                tma_load_2d_hint(dst + 2 * kQ8Box + sb * sub_rows * 32, &tm_kvr, xr, ys[sb], full, pol);
              }
            } else {
              const uint32_t full = smem_u32(&bars->stg_full[slot]);
              mbar_expect_tx(full, kFp8TileBytes);
              const uint32_t dst = smem_u32(stages + slot * kStageBytes + kFp8InPlace);
#pragma unroll
              for (int sb = 0; sb < kMaxSub; ++sb) {
                if (sb >= nsub) break;
                for (int p = 0; p < kVBoxes; ++p)
                  tma_load_2d_hint(dst + p * kFp8Box + sb * sub_rows * 64, &tm_kv, xl + 64 * p, ys[sb], full, pol);
                tma_load_2d_hint(dst + kVBoxes * kFp8Box + sb * sub_rows * 32, &tm_kvr, xr, ys[sb], full, pol);
              }
            }
          }
        }
      }
      // drain: every issued load has landed before the CTA may exit (with an
      // e4m3 query every item's loads complete on stg_full)
      if (leader) {
        const uint32_t first = item > kStages ? item - kStages : 0;
        for (uint32_t k = first; k < item; ++k)
          mbar_wait(smem_u32(kQ8 ? &bars->stg_full[k % kStages] : &bars->kv_full[k % kStages]), (k / kStages) & 1,
                    a.wait_limit_ns);
      }
    }
    __syncwarp();
  };
  auto score_issuer = [&]() {
    // ---------------------------------------------------- score-MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, kTile, 0, 0);   // K-major keys, N = 64
      constexpr uint64_t kStageDesc = kStageBytes >> 4;
      // latent boxes: 128-B swizzle, 8-row groups 1024 B apart; rope box:
      // 64-B swizzle, 8-row groups 512 B apart
      const uint64_t kv_desc0 = smem_desc(smem_u32(stages), 16, 1024, kSwizzle128B);
      const uint64_t kr_desc0 = smem_desc(smem_u32(stages + kRopeOff), 16, 512, kSwizzle64B);
      const uint32_t d = tbase + kTmemS;
      const uint32_t qa = tbase + kTmemQ;      // latent box p, 16-dim step k: column p*32 + k*8; rope: 128 + k*8
      uint32_t item = 0, it = 0, units_done = 0;
      for (int u = ubeg; u < uend; ++u, ++units_done) {
        const UnitRec ur = P.units[u];
        const int ntiles = ur.tile_end - ur.tile_begin;
        item += 2;  // query items are consumed by the softmax warps
        wait_bar(ctx, &bars->q_ready, units_done & 1);
        if constexpr (kQ8) {
          // the query items' slots get their kx_free phase too (after every
          // earlier MMA, like the tile items' commits)
          mma_commit(smem_u32(&bars->kx_free[(item - 2) % kStages]));
          mma_commit(smem_u32(&bars->kx_free[(item - 1) % kStages]));
        }
        for (int jj = 0; jj < ntiles; ++jj, ++item, ++it) {
          const uint32_t slot = item % kStages, round = item / kStages;
          if constexpr (kQ8) {
            // fp8 x fp8: the e4m3 boxes are read as they landed, 9 MMAs of K = 32
            // (8 over the two 128-dim latent boxes, 1 over the 32-dim rope box)
            wait_bar(ctx, &bars->stg_full[slot], round & 1);
            wait_bar(ctx, &bars->s_free, (it & 1) ^ 1);
            tc_fence_after();
            constexpr uint32_t id_s8 = idesc_e4m3_f32(128, kTile);
            const uint32_t base8 = smem_u32(stages + slot * kStageBytes + kQ8InPlace);
            const uint64_t kd8 = smem_desc(base8, 16, 1024, kSwizzle128B);
            const uint64_t kr8 = smem_desc(base8 + 2 * kQ8Box, 16, 256, kSwizzle32B);
#pragma unroll
            for (int p = 0; p < 2; ++p)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ts_f8(d, qa + 32 * p + 8 * k, kd8 + ((p * kQ8Box + k * 32) >> 4), id_s8, (p | k) ? 1u : 0u);
            mma_ts_f8(d, qa + 64, kr8, id_s8, 1u);
            mma_commit(smem_u32(&bars->s_full));
            mma_commit(smem_u32(&bars->kv_empty[slot]));
            mma_commit(smem_u32(&bars->kx_free[slot]));
            continue;
          }
          wait_bar(ctx, &bars->kv_full[slot], round & 1);
          wait_bar(ctx, &bars->s_free, (it & 1) ^ 1);
          tc_fence_after();
          const uint64_t kd = kv_desc0 + slot * kStageDesc;
          const uint64_t kr = kr_desc0 + slot * kStageDesc;
#pragma unroll
          for (int p = 0; p < kVBoxes; ++p)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts(d, qa + p * 32 + k * 8, kd + ((p * kBox + k * 32) >> 4), id_s, (p | k) ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < 2; ++k) mma_ts(d, qa + 128 + k * 8, kr + ((k * 32) >> 4), id_s, 1u);
          mma_commit(smem_u32(&bars->s_full));
          mma_commit(smem_u32(&bars->kv_empty[slot]));
        }
      }
      mma_commit(smem_u32(&bars->s_drain));
      mbar_wait(smem_u32(&bars->s_drain), 0, a.wait_limit_ns);
    }
    __syncwarp();
  };
  auto pv_issuer = [&]() {
    // ------------------------------------------------------ P.V-MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_pv = idesc_bf16_f32(128, 256, 0, 1);    // MN-major values, N = 256
      // values = the CTA's output dims = boxes 0-3 of its stage; 16-key steps are 2048 B apart
      const uint64_t v_desc0 = smem_desc(smem_u32(stages), kBox, 1024, kSwizzle128B);
      constexpr uint64_t kStageDesc = kStageBytes >> 4;
      uint32_t item = 0, it = 0;
      for (int u = ubeg; u < uend; ++u) {
        const UnitRec ur = P.units[u];
        const int ntiles = ur.tile_end - ur.tile_begin;
        item += 2;
        for (int jj = 0; jj < ntiles; ++jj, ++item, ++it) {
          const uint32_t slot = item % kStages, round = item / kStages;
          wait_bar(ctx, &bars->kv_full[slot], round & 1);
          wait_bar(ctx, &bars->p_full, it & 1);
          tc_fence_after();
          const uint64_t vd = v_desc0 + slot * kStageDesc;
          const uint32_t pa = tbase + kTmemP;
          mma_ts(tbase + kTmemO, pa, vd, id_pv, jj > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 1; k < kTile / 16; ++k) mma_ts(tbase + kTmemO, pa + 8 * k, vd + ((k * 2048) >> 4), id_pv, 1);
          mma_commit(smem_u32(&bars->p_free));
          mma_commit(smem_u32(&bars->kv_empty[slot]));
        }
        mma_commit(smem_u32(&bars->o_full));
      }
      mma_commit(smem_u32(&bars->p_drain));
      mbar_wait(smem_u32(&bars->p_drain), 0, a.wait_limit_ns);
    }
    __syncwarp();
  };
  auto expander = [&]() {
    // -------------------------------------------------------- e4m3 expansion
    const int te = threadIdx.x - 32 * kWarpExpand0;   // 0..127
    uint32_t item = 0;
    for (int u = ubeg; u < uend; ++u) {
      const UnitRec ur = P.units[u];
      const int ntiles = ur.tile_end - ur.tile_begin;
      item += 2;  // the query items are loaded by the producer
      for (int jj = 0; jj < ntiles; ++jj, ++item) {
        const uint32_t slot = item % kStages, round = item / kStages;
        wait_bar(ctx, &bars->stg_full[slot], round & 1);
        if constexpr (kQ8) {
          // Variant 3: the value dims (the two 128-dim e4m3 boxes = the CTA's
          // 256 output dims) become the bf16 boxes 0-3 of the slot, which
          // overlap the e4m3 boxes: read everything, wait until the tile's
          // score MMAs are done with the e4m3 boxes, then write.
          const uint32_t st = smem_u32(stages + slot * kStageBytes);
          uint4 v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = te + 128 * k;
            const int q = i & 7, r = (i >> 3) & 63, b = i >> 9;   // 16-byte chunk, row (key), e4m3 box
            v[k] = lds128(st + kQ8InPlace + b * kQ8Box + r * 128 + ((q ^ (r & 7)) << 4));
          }
          wait_bar(ctx, &bars->kx_free[slot], round & 1);
          named_bar_expand();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = te + 128 * k;
            const int q = i & 7, r = (i >> 3) & 63, b = i >> 9;
            // 16 values: output dims 128 b + 16 q + [0, 16) -> bf16 box 2b + q/4, chunks 2(q%4), 2(q%4)+1
            uint32_t o[8];
            e4m3x16_to_bf16(v[k], o);
            const uint32_t rowa = st + (2 * b + (q >> 2)) * kBox + r * 128;
            const int c0 = 2 * (q & 3);
            sts128(rowa + ((c0 ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
            sts128(rowa + (((c0 + 1) ^ (r & 7)) << 4), o[4], o[5], o[6], o[7]);
          }
        } else {
          expand_e4m3_tile(smem_u32(stages + slot * kStageBytes), te);
        }
        fence_proxy_async_smem();    // bf16 writes visible to the MMAs
        named_bar_expand();
        if (te == 0) {
          mbar_arrive(smem_u32(&bars->kv_full[slot]));
        }
      }
    }
  };
  auto softmax = [&]() {
    // ------------------------------------- softmax / exchange / rescale / epilogue
    // Two threads per query row: warp w handles TMEM lanes 32(w%4).. (the
    // rows), keys [32h, 32h+32) of every tile and O columns [128h, 128h+128)
    // with h = w / 4.  Both halves of a row keep the same running maximum:
    // they exchange their tile maxima through shared memory every tile.
    constexpr int kHalf = kTile / 2;         // keys of a tile per thread
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int hh = warp >> 2;                // key half / output half
    const int row = q4 * 32 + lane;          // query row of this thread in the unit
    const uint32_t tl = tbase + ((uint32_t)(q4 * 32) << 16);
    const int tid = threadIdx.x;             // 0..255
    // receive buffers: codes chunk-major, [8][kXRows][16 B] (chunk c = keys
    // 8c..8c+7, so half h owns chunks 4h..4h+3; the 32 lanes of a warp write
    // and read 512 contiguous bytes per instruction), then the headers
    // [2][kXRows][8 B]
    constexpr uint32_t kXChunk = (uint32_t)Layout<kVariant>::kXChunk;
    constexpr uint32_t kXHdr = (uint32_t)Layout<kVariant>::kXHdr;
    const uint32_t xcode = (uint32_t)row * 16 + 4 * (uint32_t)hh * kXChunk;
    const uint32_t xhdr = kXHdr + (uint32_t)(hh * kXRows + row) * 8;
    const uint32_t xrecv0 = smem_u32(x_recv);
    const uint32_t xrecv_peer0 = mapa(xrecv0, peer);
    const uint32_t xfull_peer0 = mapa(smem_u32(&bars->x_full[0]), peer);
    float* pmax = pairbuf;                   // [parity][half][row]
    float* psum = pairbuf + 4 * kRows;       // [half][row]
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    int nrows_cur = 0;                       // rows of the current unit (the exchanged ones)

    // Load this half's partial scores of tile `t` from TMEM into `dst` and
    // free the S columns; `hi` and `lo` get their largest and smallest value
    // (the reducing TMEM loads of sm_103a compute them on the way).
    auto load_s = [&](uint32_t t, float (&dst)[kHalf], float& hi, float& lo) {
      wait_bar(ctx, &bars->s_full, t & 1);
      __syncwarp();
      tc_fence_after();
      uint32_t r[kHalf];
      tmem_ld32_max(tl + kTmemS + kHalf * hh, r, hi);
      tmem_ld32_min(tl + kTmemS + kHalf * hh, r, lo);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < kHalf; ++c) dst[c] = __uint_as_float(r[c]);
      if constexpr (kQ8) {
        // sums of code products -> real partial scores (both halves in the same units)
#pragma unroll
        for (int c = 0; c < kHalf; ++c) dst[c] *= a.qk_scale;
        hi *= a.qk_scale;
        lo *= a.qk_scale;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->s_free));
    };
    // Send this half's partial scores of tile `t` (valid rows only) straight
    // into the peer's receive buffer as 16-bit block fixed point: codes of
    // (s - c) / step over the `nvis` of its 32 keys the row may see, c the
    // middle of their range [lo, hi] and step = half the range / 32766 (the
    // range of a full half comes from the loads, a ragged one's is recomputed
    // over its visible keys), then the header (c, step) of the half.  16-byte
    // st.async stores that count against the peer's barrier (this keeps the
    // exchange off the TMA engine that streams the cache tiles).
    // The encoding of a half: c, step, 1/step and the FMA offset.
    struct Enc {
      float ctr, step, inv, off;
    };
    auto make_enc = [&](const float (&src)[kHalf], int nvis, float hi, float lo) {
      if (nvis < kHalf) range_first_n(src, nvis, hi, lo);
      if (!(hi >= lo)) hi = lo = 0.f;      // no visible key in this half
      Enc e;
      e.ctr = 0.5f * (hi + lo);
      const float half = fmaxf(fmaxf(hi - e.ctr, e.ctr - lo), 1e-30f);
      e.step = half * (1.f / kCodeRange);
      e.inv = __fdividef(kCodeRange, half);
      // code + 32768 = s * inv + (magic - c * inv), rounded to an integer by
      // the FMA (within 1.5 steps of the exact code)
      e.off = kCodeMagic - e.ctr * e.inv;
      return e;
    };
    // chunk c (keys 8c..8c+7 of the half) of tile t, valid rows only
    auto send_chunk = [&](uint32_t t, const float (&src)[kHalf], const Enc& e, int c) {
      if (row < nrows_cur) {
        const uint32_t b = t % kXBuffers;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float f0, f1;
          fma2(f0, f1, src[8 * c + 2 * j], src[8 * c + 2 * j + 1], e.inv, e.off);
          w[j] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x5410);
        }
        st_async_v4(xrecv_peer0 + b * kXBytes + xcode + c * kXChunk, w[0], w[1], w[2], w[3], xfull_peer0 + b * 8);
      }
    };
    auto send_hdr = [&](uint32_t t, const Enc& e) {
      if (row < nrows_cur) {
        const uint32_t b = t % kXBuffers;
        st_async_v2(xrecv_peer0 + b * kXBytes + xhdr, __float_as_uint(e.ctr), __float_as_uint(e.step),
                    xfull_peer0 + b * 8);
      }
    };
    auto send_s = [&](uint32_t t, const float (&src)[kHalf], int nvis, float hi, float lo) {
      const Enc e = make_enc(src, nvis, hi, lo);
#pragma unroll
      for (int c = 0; c < kHalf / 8; ++c) send_chunk(t, src, e, c);
      send_hdr(t, e);
    };
    // Add the peer's partial scores of this half of tile `t`, less the
    // half's centre c, into `acc`; returns c (the caller folds it into the
    // maximum and the exponent) and sets `amax` to the largest sum (computed
    // before the barrier, where it overlaps the wait).  `between(c)` runs
    // after chunk c is decoded (the caller sends the next tile's first
    // chunks there, so the network transfer overlaps the decoding).
    auto recv_s = [&](uint32_t t, float (&acc)[kHalf], uint32_t nbytes, float& amax, auto&& between) -> float {
      const uint32_t b = t % kXBuffers, use = t / kXBuffers;
      if (tid == 0) mbar_expect_tx(smem_u32(&bars->x_full[b]), nbytes);
      wait_bar_cluster(ctx, &bars->x_full[b], use & 1);
      __syncwarp();
      float ctr = 0.f;
      if (row < kXRows) {
        const uint2 h = lds64(xrecv0 + b * kXBytes + xhdr);
        ctr = __uint_as_float(h.x);
        const float step = __uint_as_float(h.y);
        const uint32_t base = xrecv0 + b * kXBytes + xcode;
#pragma unroll
        for (int c = 0; c < kHalf / 8; ++c) {
          const uint4 v = lds128(base + c * kXChunk);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float f0 = __uint_as_float(__byte_perm(w[j], 0x4B40u, 0x5410));   // 12582912 + u
            float f1 = __uint_as_float(__byte_perm(w[j], 0x4B40u, 0x5432));
            add2(f0, f1, -kCodeMagic, -kCodeMagic);                           // the code, exactly
            fma2v(acc[8 * c + 2 * j], acc[8 * c + 2 * j + 1], f0, f1, step);
          }
          between(c);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kHalf / 8; ++c) between(c);
      }
      amax = max_tree32(acc);
      // every row of buffer b is read before any thread sends its row of a
      // later tile: a received tile then proves the peer is done with the
      // buffer three tiles back, whatever the row counts of the units
      named_bar_softmax();
      return ctr;
    };
    // A unit's record is one 32-byte line; the epilogue of the unit before
    // prefetches it into L1, so the load at the unit's start is short.
    auto prefetch_unit = [&](int u) {
      asm volatile("prefetch.global.L1 [%0];" ::"l"(P.units + u));
    };
    if (ubeg < uend) prefetch_unit(ubeg);

    uint32_t item = 0, it = 0, units_done = 0;
    for (int u = ubeg; u < uend; ++u, ++units_done) {
      const UnitRec ur = P.units[u];
      const UnitRec& gr = ur;
      nrows_cur = gr.nrows;
      const int R = gr.row0 + row;
      const bool valid = row < gr.nrows && R < a.total_rows;
      // Keys the row may see (multi-token causal window).  Padding rows (past
      // the group) are never stored: they are not masked and never rescale
      // O, so they cost a warp no work beyond the valid rows'.
      int Lr = 0x7fffffff;
      if (valid) {
        Lr = ur.kbase + R / a.num_heads;
        Lr = Lr < 0 ? 0 : (Lr > gr.lmax ? gr.lmax : Lr);
      }
      // the warp needs masking only on tiles that reach past its shortest valid row
      const int lmin_warp = __reduce_min_sync(0xffffffffu, Lr);
      const uint32_t nbytes = (uint32_t)gr.nrows * kXRowBytes;

      // the CTA's 288 query dims -> TMEM (A operand of the score MMAs); the
      // two halves of a row write different columns
      const uint32_t my = item + (row >= 64 ? 1 : 0);
      const int k = row & 63;
      const uint32_t sbase = smem_u32(stages + (my % kStages) * kStageBytes);
      if constexpr (kQ8) {
        // e4m3 query: the nine 32-dim K steps of the CTA's 288 dims (eight
        // from its two 128-dim latent boxes, one from its 32-dim rope box),
        // four codes per TMEM column, in the order the score issuer walks
        // them; half h writes latent box h (and h = 1 the rope box)
        wait_bar(ctx, &bars->stg_full[my % kStages], (my / kStages) & 1);
        __syncwarp();
        const uint32_t base = sbase + kQ8InPlace;
        const uint32_t sgn = a.neg_q ? 0x80808080u : 0u;   // a negative scale negates q
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint4 v0 = lds128(base + hh * kQ8Box + k * 128 + (((2 * kk) ^ (k & 7)) << 4));
          const uint4 v1 = lds128(base + hh * kQ8Box + k * 128 + (((2 * kk + 1) ^ (k & 7)) << 4));
          const uint32_t w[8] = {v0.x ^ sgn, v0.y ^ sgn, v0.z ^ sgn, v0.w ^ sgn,
                                 v1.x ^ sgn, v1.y ^ sgn, v1.z ^ sgn, v1.w ^ sgn};
          tmem_st8(tl + kTmemQ + 32 * hh + 8 * kk, w);
        }
        if (hh == 1) {
          // rope box: 32-byte rows, 32-B swizzle (16-byte chunk c of row k at c ^ ((k >> 2) & 1))
          const uint32_t rb = base + 2 * kQ8Box + k * 32;
          const int sw = (k >> 2) & 1;
          const uint4 v0 = lds128(rb + ((0 ^ sw) << 4));
          const uint4 v1 = lds128(rb + ((1 ^ sw) << 4));
          const uint32_t w[8] = {v0.x ^ sgn, v0.y ^ sgn, v0.z ^ sgn, v0.w ^ sgn,
                                 v1.x ^ sgn, v1.y ^ sgn, v1.z ^ sgn, v1.w ^ sgn};
          tmem_st8(tl + kTmemQ + 64, w);
        }
      } else {
        // bf16 query: half h writes latent boxes 2h, 2h+1 (and h = 1 the q_pe half)
        wait_bar(ctx, &bars->kv_full[my % kStages], (my / kStages) & 1);
        __syncwarp();
        const uint32_t sgn = a.neg_q ? 0x80008000u : 0u;   // a negative scale negates q
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int p = 2 * hh + pp;
          uint32_t q[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = lds128(sbase + p * kBox + k * 128 + ((c ^ (k & 7)) << 4));
            q[4 * c + 0] = v.x ^ sgn;
            q[4 * c + 1] = v.y ^ sgn;
            q[4 * c + 2] = v.z ^ sgn;
            q[4 * c + 3] = v.w ^ sgn;
          }
          tmem_st32(tl + kTmemQ + p * 32, q);
        }
        if (hh == 1) {
          // q_pe half: 64-byte rows, 64-B swizzle (chunk c of row k at c ^ ((k >> 1) & 3))
          uint32_t h[16];
          const int sw = (k >> 1) & 3;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = lds128(sbase + kRopeOff + k * 64 + ((c ^ sw) << 4));
            h[4 * c + 0] = v.x ^ sgn;
            h[4 * c + 1] = v.y ^ sgn;
            h[4 * c + 2] = v.z ^ sgn;
            h[4 * c + 3] = v.w ^ sgn;
          }
          tmem_st16(tl + kTmemQ + 128, h);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      named_bar_softmax();
      if (tid == 0) {
        for (int qi = 0; qi < 2; ++qi) {      // two arrivals: the slot's count covers both issuers
          mbar_arrive(smem_u32(&bars->kv_empty[(item + qi) % kStages]));
          mbar_arrive(smem_u32(&bars->kv_empty[(item + qi) % kStages]));
        }
        mbar_arrive(smem_u32(&bars->q_ready));
      }
      item += 2;

      // the previous unit's TMA stores have read their scratch (receive
      // buffers the peer may write once this unit's first tiles go out)
      if constexpr (kTmaStore)
        if (lane == 0) bulk_wait_group_read<0>();

      float m = -INFINITY, l = 0.f;          // l: this half's share of the row sum
      const int ntiles = ur.tile_end - ur.tile_begin;
      // keys of this half of tile jj the row may see (32 on every tile before its last)
      auto nvis = [&](int jj) { return Lr - (ur.tile_begin + jj) * kTile - kHalf * hh; };
      float cur[kHalf], nxt[kHalf];
      if (ntiles > 0) {
        float hi, lo;
        load_s(it, cur, hi, lo);
        send_s(it, cur, nvis(0), hi, lo);
      }
      // One tile: `cur` holds this tile's own partials, `nxt` receives the
      // next tile's.  With a bf16 cache the loop runs two tiles per trip with
      // the arrays swapping roles, so no copy moves `nxt` into `cur`.
      auto tile = [&](int jj, float (&cur)[kHalf], float (&nxt)[kHalf]) {
        // The next tile's partials are loaded first and sent in pieces while
        // this tile is processed: chunks 0-1 between the decoding steps of
        // this tile's received partials, chunks 2-3 and the header after its
        // exponentials, so the network transfer overlaps the arithmetic.
        const bool has_next = jj + 1 < ntiles;
        Enc en{};
        if (has_next) {
          float hi, lo;
          load_s(it + 1, nxt, hi, lo);
          en = make_enc(nxt, nvis(jj + 1), hi, lo);
        }
        float hmax;
        // cur = own + peer partial - cpeer
        const float cpeer = recv_s(it, cur, nbytes, hmax, [&](int c) {
          if (has_next && c < 2) send_chunk(it + 1, nxt, en, c);
        });

        // mask on ragged tiles (and take the max again), the max of the
        // unscaled scores of both halves (the scale is positive), then
        // exp2(scale * s - m) as one FMA
        const int key0 = (ur.tile_begin + jj) * kTile + kHalf * hh;
        if (key0 + kHalf > lmin_warp) {
#pragma unroll
          for (int c = 0; c < kHalf; ++c) cur[c] = (key0 + c < Lr) ? cur[c] : -INFINITY;
          hmax = max_tree32(cur);
        }
        // P with the current reference, computed before the halves agree on
        // the tile maximum so that their barrier overlaps the exponentials;
        // recomputed if the maximum moves past the lazy threshold (the first
        // tile of a unit, or a new largest score)
        uint32_t pk[kHalf / 2];
        float lsum;
        auto exp_tile = [&](float mref) {
          const float kexp = fmaf(cpeer, a.scale_log2, -mref);   // exponent offset of this half
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < kHalf / 2; ++c) {
            float x0, x1;
            fma2(x0, x1, cur[2 * c], cur[2 * c + 1], a.scale_log2, kexp);
            const float p0 = fast_exp2(x0);
            const float p1 = fast_exp2(x1);
            add2(ls[2 * (c & 1)], ls[2 * (c & 1) + 1], p0, p1);
            pk[c] = pack_bf16x2(p0, p1);
          }
          lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
        };
        // the halves' maxima are exchanged through shared memory; the parity
        // alternates so that a write never meets a read of the previous tile
        float* pm = pmax + (it & 1) * 2 * kRows;
        const float own = (hmax + cpeer) * a.scale_log2;
        pm[hh * kRows + row] = own;
        exp_tile(m == -INFINITY ? 0.f : m);
        named_bar_pair(q4);
        const float tmax = fmaxf(own, pm[(1 - hh) * kRows + row]);
        float alpha = 1.f;
        if (valid && tmax > m + kRescaleThreshold) {
          alpha = fast_exp2(m - tmax);  // m = -inf -> 0
          l *= alpha;
          m = tmax;
          exp_tile(m);
        }
        l += lsum;
        if (has_next) {
          send_chunk(it + 1, nxt, en, 2);
          send_chunk(it + 1, nxt, en, 3);
          send_hdr(it + 1, en);
        }

        // P and O may be touched once the P.V of the previous tile has completed
        wait_bar(ctx, &bars->p_free, (it & 1) ^ 1);
        __syncwarp();
        tc_fence_after();
        if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t o[32];
            const uint32_t oc = tl + kTmemO + 128 * hh + ch * 32;
            tmem_ld32(oc, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(oc, o);
          }
        }
        tmem_st16(tl + kTmemP + (kHalf / 2) * hh, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
      };
      if constexpr (kCacheFp8) {
        // e4m3 cache: one tile per trip (the unrolled form measured 8 %
        // slower for these variants)
        for (int jj = 0; jj < ntiles; ++jj, ++item, ++it) {
          tile(jj, cur, nxt);
#pragma unroll
          for (int c = 0; c < kHalf; ++c) cur[c] = nxt[c];
        }
      } else {
        int jj = 0;
        for (; jj + 1 < ntiles; jj += 2) {
          tile(jj, cur, nxt);
          ++item, ++it;
          tile(jj + 1, nxt, cur);
          ++item, ++it;
        }
        if (jj < ntiles) {
          tile(jj, cur, nxt);
          ++item, ++it;
        }
      }

      if (u + 1 < uend) prefetch_unit(u + 1);

      // epilogue: the row sum of both halves, then the output
      psum[hh * kRows + row] = l;
      named_bar_pair(q4);
      const float lt = l + psum[(1 - hh) * kRows + row];
      wait_bar(ctx, &bars->o_full, units_done & 1);
      __syncwarp();
      tc_fence_after();
      const float inv = lt > 0.f ? a.out_scale / lt : 0.f;
      const float lse_nat = lt > 0.f ? (m + __log2f(lt)) * 0.6931471805599453f : -INFINITY;
      // The rows leave through shared memory so that every store writes
      // whole 128-byte lines (a thread owns a row: direct stores would write
      // one 32-byte sector of 32 different lines per instruction).  The
      // scratch of warp (q, h) is 4 KB of the receive buffer of the tile
      // before last (h = 0) or of the last tile (h = 1): both are read, and
      // the peer writes into them only after it has received the next
      // unit's first tile, which this CTA sends after its epilogue.
      const uint32_t scr = xrecv0 + ((it + 2 + (uint32_t)hh) % kXBuffers) * kXBytes + (uint32_t)q4 * 4096u;
      // Room for the warp's 4 KB: always with 128-row buffers; a 32-row
      // buffer (units of at most 32 rows) holds the one warp quadrant that
      // has rows.
      static_assert(kXRows == kRows ? 4 * 4096 <= kXBytes : 4096 <= kXBytes, "epilogue scratch");
      const bool store = __any_sync(0xffffffffu, valid) && (kXRows == kRows || q4 == 0);
      const int d0 = 256 * (int)rank + 128 * hh;
      // row r of the warp (lane r's row) is stored
      auto row_ok = [&](int r) { return q4 * 32 + r < gr.nrows && gr.row0 + q4 * 32 + r < a.total_rows; };
      // the thread's 128 bytes -> scratch row `lane` (16-byte chunks rotated by the row: no bank conflicts)
      auto stage = [&](const uint32_t (&w)[32]) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          sts128(scr + lane * 128 + ((c ^ (lane & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        __syncwarp();
      };
      // scratch -> global, 8 lanes per 128-byte row, 4 rows per instruction;
      // `dst(r)` is the first byte of row r's 128 bytes
      auto drain = [&](auto dst) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3), c = lane & 7;
          const uint4 v = lds128(scr + r * 128 + ((c ^ (r & 7)) << 4));
          if (row_ok(r)) *reinterpret_cast<uint4*>(dst(r) + 16 * c) = v;
        }
        __syncwarp();
      };
      // A warp whose 32 rows all belong to the unit (and every warp writing
      // split partials, whose slot rows are its own) hands each staged 4 KB
      // piece to a TMA store and goes on while it drains; the scratch is
      // written again only once the store has read it (before the next
      // piece, and before this warp's first send of the next unit: the peer
      // writes into these buffers only after that).  The 128-row receive
      // buffers keep the 1024-byte alignment of the 128-B swizzle.
      static_assert(!kTmaStore || kXRows == kRows, "TMA stores need the 128-row receive buffers");
      const bool full_rows = q4 * 32 + 32 <= gr.nrows && gr.row0 + q4 * 32 + 32 <= a.total_rows;
      bool pending = false;
      auto put = [&](const CUtensorMap* tm, int x, int y) {
        fence_proxy_async_smem();      // this lane's staged bytes, visible to the bulk copy
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tm, x, y, scr);
          bulk_commit_group();
        }
        pending = true;
      };
      auto reclaim = [&]() {
        if (pending) {
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
          pending = false;
        }
      };
      // two 32-column loads of O per wait
#pragma unroll 1
      for (int cp = 0; cp < 2; ++cp) {
        uint32_t oa[32], ob[32];
        tmem_ld32(tl + kTmemO + 128 * hh + cp * 64, oa);
        tmem_ld32(tl + kTmemO + 128 * hh + cp * 64 + 32, ob);
        tmem_wait_ld();
        if (!store) continue;
        reclaim();
        if (ur.slot < 0) {
          // bf16 output: the 64 dims are one 128-byte row piece
#pragma unroll
          for (int v = 0; v < 16; ++v)
            oa[v] = pack_bf16x2(__uint_as_float(oa[2 * v]) * inv, __uint_as_float(oa[2 * v + 1]) * inv);
#pragma unroll
          for (int v = 0; v < 16; ++v)
            oa[16 + v] = pack_bf16x2(__uint_as_float(ob[2 * v]) * inv, __uint_as_float(ob[2 * v + 1]) * inv);
          stage(oa);
          if (kTmaStore && full_rows)
            put(&tm_out, d0 + 64 * cp, gr.row0 + q4 * 32);
          else
            drain([&](int r) {
              return reinterpret_cast<uint8_t*>(out + (size_t)(gr.row0 + q4 * 32 + r) * kLkv + d0 + 64 * cp);
            });
        } else if constexpr (kVariant == 2) {
          // partial (see below); one maximum over both halves, the same scale
          // stored for both: this variant's code measured faster in this form
          float mx = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(oa[c])), fabsf(__uint_as_float(ob[c]))));
          const int ebits = (int)(__float_as_uint(mx * inv) >> 23);
          const int mexp = min(253, 268 - ebits);
          const float mul = inv * __int_as_float(mexp << 23);
#pragma unroll
          for (int v = 0; v < 16; ++v)
            oa[v] = pack_f16x2(__uint_as_float(oa[2 * v]) * mul, __uint_as_float(oa[2 * v + 1]) * mul);
#pragma unroll
          for (int v = 0; v < 16; ++v)
            oa[16 + v] = pack_f16x2(__uint_as_float(ob[2 * v]) * mul, __uint_as_float(ob[2 * v + 1]) * mul);
          stage(oa);
          drain([&](int r) {
            return reinterpret_cast<uint8_t*>(P.part_o + ((size_t)ur.slot * kRows + q4 * 32 + r) * kLkv + d0 + 64 * cp);
          });
          if (valid) {
            const float sc = __int_as_float((254 - mexp) << 23);
            *reinterpret_cast<float2*>(P.part_scale + ((size_t)ur.slot * kRows + row) * (kLkv / 32) +
                                       (d0 + 64 * cp) / 32) = make_float2(sc, sc);
          }
        } else {
          // partial: fp16 codes of o * 2^j per 32-dim chunk, 2^j chosen from
          // the chunk's largest magnitude so that it lands in [2^14, 2^15)
          // (within [2^-126, 2^126] for tiny chunks), and the scale 2^-j
          float* scale = P.part_scale + ((size_t)ur.slot * kRows + row) * (kLkv / 32) + (d0 + 64 * cp) / 32;
          auto encode = [&](const uint32_t (&o)[32], int at) {
            float mx = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) mx = fmaxf(mx, fabsf(__uint_as_float(o[c])));
            const int ebits = (int)(__float_as_uint(mx * inv) >> 23);  // biased exponent of the largest |o|
            const int mexp = min(253, 268 - ebits);                       // biased exponent of 2^j
            const float mul = inv * __int_as_float(mexp << 23);
#pragma unroll
            for (int v = 0; v < 16; ++v)
              oa[at + v] = pack_f16x2(__uint_as_float(o[2 * v]) * mul, __uint_as_float(o[2 * v + 1]) * mul);
            if (valid) scale[at / 16] = __int_as_float((254 - mexp) << 23);
          };
          encode(oa, 0);
          encode(ob, 16);
          stage(oa);
          if constexpr (kTmaStore)
            put(&tm_part, d0 + 64 * cp, ur.slot * kRows + q4 * 32);
          else
            drain([&](int r) {
              return reinterpret_cast<uint8_t*>(P.part_o + ((size_t)ur.slot * kRows + q4 * 32 + r) * kLkv + d0 +
                                                64 * cp);
            });
        }
      }
      if (valid && rank == 0 && hh == 0) {
        if (ur.slot < 0) {
          if (a.lse) a.lse[R] = lse_nat;
        } else {
          P.part_lse[(size_t)ur.slot * kRows + row] = lse_nat;
        }
      }
      tc_fence_before();
    }
    if constexpr (kTmaStore)
      if (lane == 0) bulk_wait_all();   // every TMA store of the warp is complete
  };

  if constexpr (kCacheFp8) {
    // 512 threads (128 registers each at launch): each warpgroup sets its budget
    if (warp < kSoftmaxWarps) {
      setmaxnreg_inc<kRegsSoftmax8>();
      softmax();
    } else if (warp < kWarpExpand0) {
      setmaxnreg_dec<kRegsIssue8>();
      if (warp == kWarpProducer)
        producer();
      else if (warp == kWarpScore)
        score_issuer();
      else if (warp == kWarpPV)
        pv_issuer();
    } else {
      setmaxnreg_dec<kRegsExpand8>();
      expander();
    }
  } else {
    if (warp < kSoftmaxWarps)
      softmax();
    else if (warp == kWarpProducer)
      producer();
    else if (warp == kWarpScore)
      score_issuer();
    else if (warp == kWarpPV)
      pv_issuer();
  }

  __syncthreads();
  if (warp == kWarpScore) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  cluster_sync();  // no CTA leaves while its peer may still write into it
}

}  // namespace

size_t decode_smem_bytes(int variant) {
  return variant == 1 ? smem_bytes<1>()
                      : (variant == 2 ? smem_bytes<2>() : (variant == 3 ? smem_bytes<3>() : smem_bytes<0>()));
}

cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_qr, const CUtensorMap& tm_kv,
                          const CUtensorMap& tm_kvr, const CUtensorMap& tm_out, const CUtensorMap& tm_part,
                          int variant, const DecodeArgs& a, int num_clusters, cudaStream_t s) {
  const size_t smem = decode_smem_bytes(variant);
  auto kern = variant == 1 ? decode_kernel<1>
                           : (variant == 2 ? decode_kernel<2> : (variant == 3 ? decode_kernel<3> : decode_kernel<0>));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the prologue (barriers, TMEM, cluster
  // sync) overlaps the plan kernel; the kernel waits for it before reading the plan
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_clusters);
  cfg.blockDim = dim3(variant == 1 || variant == 3 ? Roles<1>::kThreads : Roles<0>::kThreads);
  static_assert(Roles<1>::kThreads == Roles<3>::kThreads && Roles<0>::kThreads == Roles<2>::kThreads, "roles");
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tm_q, tm_qr, tm_kv, tm_kvr, tm_out, tm_part, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
