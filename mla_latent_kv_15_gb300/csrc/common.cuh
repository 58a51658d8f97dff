// Shared definitions of the MLA decode library: fixed widths, the split-KV
// plan that lives in the caller's workspace, and the launchers each
// translation unit exports to the C-ABI layer (api.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mla {

constexpr int kLkv = 512;          // latent width (kv_c, q_abs, output)
constexpr int kRope = 64;          // decoupled rope width (k_pe, q_pe)
constexpr int kDqk = kLkv + kRope; // cache row width
constexpr int kRows = 128;         // query rows per work unit (tcgen05 M)
constexpr int kTile = 64;          // keys per tile (S MMA N, P.V MMA K)
constexpr int kMaxClusters = 128;  // upper bound of CTA pairs in the decode grid

// Work-unit plan written by the scheduler kernel into the workspace.
//   group  = up to 128 consecutive query rows (flattened t*N + h) of one request
//   unit   = a contiguous tile range of one group, processed by one CTA pair
struct PlanHeader {
  int status;        // OR of mla_device_error bits
  int num_groups;
  int num_units;
  int num_clusters;
  int total_tiles;
  int tiles_per_cluster;
  int pad[2];
};

struct GroupRec {    // 32 bytes
  int b;             // request
  int row0;          // first flattened query row (t*N + h)
  int nrows;         // rows in this group (<= 128)
  int lmax;          // keys visible to the group's last row (>= 0)
  int pieces;        // units the group was cut into (0: no keys)
  int ubase;         // index of its first unit
  int tiles;         // ceil(lmax / kTile)
  int tpos;          // position of its first tile on the flattened tile axis
};

// Everything a CTA pair needs to run a unit, in one 32-byte record (one
// line, no dependent loads).
struct UnitRec {     // 32 bytes
  int tile_begin;
  int tile_end;
  int slot;          // partial-result slot (== unit index) or -1: write the final output
  int b;             // request
  int row0;          // first flattened query row of the group (t*N + h)
  int nrows;         // rows in the group
  int lmax;          // keys visible to the group's last row
  int kbase;         // seq_len - Sq + 1 - q0: row R sees min(kbase + R / N, lmax) keys
};
static_assert(sizeof(UnitRec) == 32, "unit record: one aligned 32-byte piece");

struct Plan {
  PlanHeader* header;
  GroupRec* groups;
  UnitRec* units;
  int* unit_cluster;     // cluster index of each unit
  int* cluster_begin;    // [kMaxClusters + 1] first unit of each cluster
  // split partials: row r of unit u holds fp16 codes of o / 2^e, one
  // power-of-two scale 2^e per 32-dim chunk (e from the chunk's largest
  // magnitude, so every finite o keeps fp16's 11 significant bits)
  uint16_t* part_o;      // [max_units][128][512] fp16 codes
  float* part_scale;     // [max_units][128][16] 2^e of each 32-dim chunk
  float* part_lse;       // [max_units][128]
  int max_groups;
  int max_units;
};

struct WorkspaceLayout {
  size_t header, groups, units, unit_cluster, cluster_begin, part_o, part_scale, part_lse, total;
  int max_groups, max_units;
};

// Byte offsets of each plan array for a batch shape (host and device agree).
inline WorkspaceLayout workspace_layout(int batch, int total_q, int num_heads, int max_splits) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  WorkspaceLayout L{};
  long long rows = (long long)total_q * num_heads;
  long long mg = (rows + 127LL * batch) / kRows + 1;
  long long mu = mg * (max_splits > 1 ? max_splits : 1) + kMaxClusters;
  L.max_groups = (int)mg;
  L.max_units = (int)mu;
  size_t off = 0;
  L.header = off;        off = up(off + sizeof(PlanHeader));
  L.groups = off;        off = up(off + sizeof(GroupRec) * (size_t)mg);
  L.units = off;         off = up(off + sizeof(UnitRec) * (size_t)mu);
  L.unit_cluster = off;  off = up(off + sizeof(int) * (size_t)mu);
  L.cluster_begin = off; off = up(off + sizeof(int) * (kMaxClusters + 1));
  L.part_o = off;        off = up(off + sizeof(uint16_t) * (size_t)mu * kRows * kLkv);
  L.part_scale = off;    off = up(off + sizeof(float) * (size_t)mu * kRows * (kLkv / 32));
  L.part_lse = off;      off = up(off + sizeof(float) * (size_t)mu * kRows);
  L.total = off;
  return L;
}

inline Plan plan_from_workspace(void* ws, const WorkspaceLayout& L) {
  char* p = static_cast<char*>(ws);
  Plan P;
  P.header = reinterpret_cast<PlanHeader*>(p + L.header);
  P.groups = reinterpret_cast<GroupRec*>(p + L.groups);
  P.units = reinterpret_cast<UnitRec*>(p + L.units);
  P.unit_cluster = reinterpret_cast<int*>(p + L.unit_cluster);
  P.cluster_begin = reinterpret_cast<int*>(p + L.cluster_begin);
  P.part_o = reinterpret_cast<uint16_t*>(p + L.part_o);
  P.part_scale = reinterpret_cast<float*>(p + L.part_scale);
  P.part_lse = reinterpret_cast<float*>(p + L.part_lse);
  P.max_groups = L.max_groups;
  P.max_units = L.max_units;
  return P;
}

// Everything the decode kernel needs besides its tensor maps.
struct DecodeArgs {
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* qsl;       // may be null: one query token per request
  int batch;
  int num_heads;
  int max_pages;
  int page_size;
  int num_blocks;
  int total_rows;           // total_q * num_heads: bound of every output row
  float scale_log2;         // |scale| * log2(e) (* kv_scale for fp8), > 0
  int neg_q;                // scale < 0: the kernel negates the query instead
  float out_scale;          // kv_scale for fp8, 1 for bf16
  float qk_scale;           // e4m3 query: q_scale * kv_scale (code products -> scores)
  void* out;                // bf16 [T*N, 512]
  float* lse;               // [T*N] or null
  unsigned long long wait_limit_ns;   // bound of every on-chip wait (1 s)
  int debug_skip_tile;      // test aid: CTA 0 of cluster 0 never loads its first cache tile
  Plan plan;
};

// The new rows of a step for concat_and_cache_mla: token t's kv_c (512 bf16)
// and k_pe (64 bf16) go to cache slot slots[t] (a slot outside
// [0, num_slots) is padding); an e4m3 cache stores value / kv_scale.
struct CacheWriteArgs {
  const void* kv_c;
  const void* k_pe;
  const int64_t* slots;
  int64_t num_tokens;
  void* cache;
  int64_t num_slots;
  float kv_scale;
  int fp8;
};

// The query of an e4m3-query step: q_abs [rows, 512] and q_pe [rows, 64] bf16
// (rows = total_q * num_heads, dense) into q8 [rows, 576] e4m3 codes of
// value / q_scale.
struct QuantArgs {
  const void* q_abs;
  const void* q_pe;
  int64_t rows;
  float q_scale;
  uint8_t* q8;
};

// ---- launchers (return cudaError_t of the launch)
// group_rows: query rows per group, a power of two (128; 32 for the small-rows decode variant)
// write: the step's cache rows, quant: the step's query quantisation, both
// done by extra blocks of the same launch (nullptr: none; quant needs an
// e4m3 cache write or none)
cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* qsl, int batch, int num_heads, int max_pages,
                        int page_size, int num_splits, int num_clusters, int group_rows, Plan plan,
                        const CacheWriteArgs* write, const QuantArgs* quant, int sm_count, cudaStream_t s);
// variant: 0 bf16 cache, 1 e4m3 cache, 2 bf16 cache with <= 32-row groups
// (plan built with group_rows = 32), 3 e4m3 query and e4m3 cache.  Tensor
// maps: the query's latent columns (64-dim boxes; 128-dim e4m3 boxes for
// variant 3) and its rope columns (32-dim boxes), the cache's latent columns
// and its rope columns, boxes as wide (rows: min(page, 64) for the cache, 64
// for the query); for the epilogue's stores, the bf16 output rows and the
// fp16 partial rows (64-dim x 32-row boxes, 128-B swizzle).
cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_qr, const CUtensorMap& tm_kv,
                          const CUtensorMap& tm_kvr, const CUtensorMap& tm_out, const CUtensorMap& tm_part,
                          int variant, const DecodeArgs& a, int num_clusters, cudaStream_t s);
// sm_count: of the current device (the combine runs one wave of blocks)
cudaError_t launch_combine(const DecodeArgs& a, int max_groups, int sm_count, cudaStream_t s);
cudaError_t launch_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                                int64_t rows, int dim, int o_is_bf16, void* out, float* lse_out, int sm_count,
                                cudaStream_t s);
cudaError_t launch_cache_write(const CacheWriteArgs& w, cudaStream_t s);
size_t decode_smem_bytes(int variant);
// y[t, n, :] = x[t, n, :] @ W[n] (tensor maps: x 3-D {d_in, N, T} boxes
// 64 x 1 x head_proj_x_rows(T), W 2-D {d_out, N*d_in} boxes 64x64, both
// 128-byte swizzled)
cudaError_t launch_head_proj(const CUtensorMap& tm_x, const CUtensorMap& tm_w, void* y, int64_t T, int N, int d_in,
                             int d_out, cudaStream_t s);
int head_proj_x_rows(int64_t T);
cudaError_t launch_quantize_fp8(const void* x, int64_t x_stride, int64_t rows, int width, float scale, void* out,
                                int64_t out_stride, cudaStream_t s);
cudaError_t launch_gather(const void* cache, int64_t num_blocks, int page_size, int cache_fp8, float kv_scale,
                          const int32_t* block_table, int max_pages, const int32_t* cu_seq_lens,
                          const int32_t* seq_starts, int batch, void* dst, int64_t num_tokens, int32_t* status,
                          cudaStream_t s);
cudaError_t head_proj_status(int* status, int clear, cudaStream_t s);

}  // namespace mla
