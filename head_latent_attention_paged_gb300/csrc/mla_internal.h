// Internal declarations shared by the host API and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mla_decode.h"

namespace mla {

constexpr int kDc = 512;          // latent width
constexpr int kDr = 64;           // RoPE key width
constexpr int kDqk = kDc + kDr;   // 576: one cached row
constexpr int kDnope = 192;
constexpr int kDv = 256;
constexpr int kTile = MLA_TILE_TOKENS;   // 64 cached rows per tile
constexpr int kChunkElems = 64;           // one 128-byte swizzle row of bf16
constexpr int kChunks = kDqk / kChunkElems;  // 9
constexpr int kChunkBytes = kTile * 128;     // 8 KB: 64 rows x 128 B
constexpr int kTileBytes = kChunks * kChunkBytes;  // 73,728
constexpr int kFp8RowBytes = kDqk + kDqk / 32;     // 594
constexpr int kFp4CodeBytes = kDqk / 2;            // 288: two e2m1 codes per byte
constexpr int kFp4RowBytes = kFp4CodeBytes + kDqk / 16;   // 324
constexpr int kMaxHeads = 32;     // TMEM: q_hat 288 + S 64 + O^T 4 x 32 columns
// Dense multi-token mode: G query tokens of one request share a row set of
// G * H <= 48 rows (TMEM: latent q_hat 256 + S 64 + O^T 4 x 48 columns; the
// RoPE part of q_hat is a shared-memory operand).
constexpr int kMaxRows = 48;
constexpr int kMaxStreams = 1 << 20;   // row sets per plan
// Up to this many row sets the decode kernel keeps their tile and cost
// prefixes in shared memory (when they fit beside its buffers); beyond, a
// one-block pre-pass writes them to the workspace.
constexpr int kSmemStreams = 256;
constexpr int kMaxSmemBytes = 232448;   // dynamic shared memory per CTA (227 KB)
constexpr int kMaxCtas = 65536;   // decode grid limit (split-KV by length)
// 72 KB bf16 tiles in flight per CTA.  An FP4 tile of quantised rows
// (20,736 B) is copied into the tail of the stage it is dequantised into;
// FP8 tiles (38,016 B) have a ring of their own beside two bf16 stages.
constexpr int kStages = 3;
constexpr int kFp8Stages = 2;
constexpr int kFp8RawSlots = 2;
constexpr int kFp8TileBytes = kTile * kFp8RowBytes;  // 38,016

enum DecodeMode : int {
  kModeDenseBf16 = 0,
  kModeSparseBf16 = 1,
  kModeDenseFp8 = 2,
  kModeDenseFp4 = 3,
  kModeDenseMulti = 4,   // bf16, q_len > 1: draft tokens of a request share each staged tile
  kModeDenseFp4Multi = 5,   // the same over an FP4 cache
  kModeDenseFp8Multi = 6,   // the same over an FP8 cache
};

struct DecodeParams {
  const uint16_t* q_hat;        // bf16 [S][H][576]
  const uint8_t* kv;            // cache base (bytes)
  const int32_t* block_table;   // [B][max_pages]
  const int32_t* seq_lens;      // [B]
  const int32_t* topk_idx;      // [S][width] or null
  float* part_o;                // [slots][H][512]
  float* part_lse;              // [slots][H]
  float* o_lat;                 // [S][H][512] output
  float* lse;                   // [S][H] output
  uint32_t* status;
  int32_t batch, q_len, heads, heads_pad;  // heads_pad: N of the PV MMA (multiple of 16, >= rows)
  int32_t group;                // query tokens per row set (1, or G >= 2 in the multi-token mode)
  int32_t rows;                 // rows of a full row set: group * heads
  int32_t page_size, num_pages, max_pages, topk_width, causal;
  int32_t num_streams, num_ctas;
  int32_t stream_cost;          // a stream's fixed cost in the work split (stream_cost_of_mode)
  int32_t* prefix_ws;           // int32 [2][S + 1] tile and cost prefixes written by the
                                // pre-pass, or null: the decode kernel computes them itself
  float scale_log2;             // sm_scale * log2(e)
};

struct DecodeLayout {   // dynamic shared memory layout of the decode kernel
  int32_t off_stage, off_raw, off_p, off_qrope, off_ctrl, total;
  int32_t prefix_in_smem;   // 1: the row-set prefixes follow the control block
};

DecodeLayout decode_layout(int heads, int heads_pad, int num_streams, int mode);
int decode_smem_bytes(int heads, int heads_pad, int num_streams, int mode);

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap* kv_map, int mode,
                          cudaStream_t stream);

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  const int32_t* seq_lens;
  float* o_lat;
  float* lse;
  int32_t batch, q_len, heads, page_size, max_pages, topk_width, causal;
  int32_t group, rows;          // as in DecodeParams
  int32_t num_streams, num_ctas, stream_cost;
  const int32_t* prefix_ws;     // the pre-pass's prefixes (as in DecodeParams), or null
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
// One block: the tile and cost prefixes over the row sets into p.prefix_ws.
cudaError_t launch_prefix(const DecodeParams& p, cudaStream_t stream);

// o = W_UV[h]^T o_lat per (head, 128 output dims, row block), a programmatic
// dependent of the launch before it; sm_count sizes the row blocks (16, 32
// or 64 rows) so the grid fits the SMs where it can.
cudaError_t launch_uv_proj_tma(const CUtensorMap* w_map, const float* o_lat, uint16_t* out,
                               int rows, int heads, int sm_count, cudaStream_t stream);
// The merge and the up-projection in one launch (a programmatic dependent
// of the decode): out = W_UV[h]^T o for every row, o the decode's o_lat row
// or, for a split row set, the merge of its partials (also written to
// p.o_lat and p.lse, the bits the merge kernel gives).
cudaError_t launch_merge_uv(const CUtensorMap* w_map, const CombineParams& p, uint16_t* out,
                            int sm_count, cudaStream_t stream);

struct AppendParams {
  const uint16_t* new_rows;     // bf16 [rows][576]
  const int32_t* positions;     // [rows] token index to write, -1 = none
  const int32_t* block_table;   // [rows][max_pages]
  uint8_t* kv;                  // cache base (bytes)
  uint32_t* status;             // nullable
  int32_t rows, page_size, num_pages, max_pages;
  int32_t kv_dtype;             // MLA_KV_BF16, MLA_KV_FP8_E4M3_E8M0 or MLA_KV_FP4_E2M1_E8M0
  float rope_theta;             // > 0: rotate k_rope to the row's position first
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// q_hat[r][h] = [bf16(W_UK[h] q[r][h][:192]) || q[r][h][192:256]] on the
// tensor cores; w_map: W_UK as [H * 512 rows][192] bf16, boxes of 64 x 128.
cudaError_t launch_q_absorb(const CUtensorMap* w_map, const uint16_t* q, uint16_t* q_hat,
                            int rows, int heads, cudaStream_t stream);

// Sets a kernel's maximum dynamic shared memory once per device (the
// attribute belongs to the current device's context).
cudaError_t set_smem_attr_once(const void* func, int slot, int bytes);

// The current CUDA context (nullptr if none or unknown).
void* current_context();

// Host steps shared by the entry points (MLA_* return codes).
int plan_check(const mla_plan* plan);
// Everything mla_decode_run checks before it queues any work.
int check_run_args(const mla_plan* plan, const void* q, const void* w_uk, const void* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk_idx,
                   const void* workspace, size_t workspace_bytes, const float* o_lat,
                   const float* lse);
int launch_attention(const mla_plan& plan, const void* q_hat, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk_idx,
                     uint8_t* ws, float* o_lat, float* lse, cudaStream_t st);
int launch_merge(const mla_plan& plan, const int32_t* seq_lens, const uint8_t* ws,
                 const void* w_uv, float* o_lat, float* lse, void* out, cudaStream_t st);

// Row set s covers request b and query tokens j0 .. j0 + nq - 1 (the group
// of `group` consecutive draft tokens; group = 1 outside the multi-token
// mode).  Its rows are (token j0 + jj, head h) for jj < nq, h < H, i.e. the
// contiguous rows (b * q_len + j0) * H .. + nq * H of q_hat and o_lat.
struct StreamGeom {
  int32_t b, j0, nq;
};
__host__ __device__ inline StreamGeom stream_geom(int32_t s, int32_t q_len, int32_t group) {
  const int32_t ng = (q_len + group - 1) / group;
  StreamGeom g;
  g.b = s / ng;
  g.j0 = (s - g.b * ng) * group;
  g.nq = q_len - g.j0 < group ? q_len - g.j0 : group;
  return g;
}

// Query tokens per row set for a problem: the multi-token mode groups
// min(q_len, 48 / H) draft tokens of a request when that is at least 2
// (dense bf16 and FP4 caches; the FP8 kernel's shared memory has no room
// for the RoPE query operand beside its raw-tile ring).
__host__ __device__ inline int32_t row_set_group(int32_t q_len, int32_t heads, int32_t kv_dtype,
                                                 int32_t topk_width) {
  (void)kv_dtype;   // every cache type groups draft rows (the sparse top-k lists do not)
  if (topk_width > 0 || q_len < 2) return 1;
  const int32_t g = kMaxRows / heads;
  const int32_t gq = g < q_len ? g : q_len;
  return gq >= 2 ? gq : 1;
}

// Tiles of one (request, query token) row set; identical on host and device.
__host__ __device__ inline int32_t stream_len(int32_t seq_len, int32_t q_len, int32_t j,
                                              int32_t causal, int32_t topk_width,
                                              int32_t max_tokens) {
  if (topk_width > 0) return topk_width;
  int32_t t = seq_len < 0 ? 0 : (seq_len > max_tokens ? max_tokens : seq_len);
  if (causal) {
    int32_t v = t - q_len + j + 1;
    t = v < 0 ? 0 : (v > t ? t : v);
  }
  return t;
}

// Work split.  Every tile gets a cost position: a stream with n > 0 tiles
// spans sc + n * kTileCost cost units, its fixed overhead sc (query load into
// TMEM, epilogue, the pipeline refill behind them) first, then one kTileCost
// slot per tile, so tile k of a stream starting at cost pc sits at pc + sc +
// k * kTileCost.  CTA c takes the tiles whose position lies in [c*U/C,
// (c+1)*U/C) for U the total cost: a CTA that opens more streams gets fewer
// tiles.  The overhead was measured at about three tile times in the kernels
// over bf16 caches and about two in those over quantised caches, whose tiles
// take longer.
constexpr int32_t kTileCost = 4;
constexpr int32_t kStreamCostBf16 = 13;
constexpr int32_t kStreamCostQuant = 8;
constexpr int32_t kStreamCostMax = 13;

__host__ __device__ inline int32_t stream_cost_of_mode(int mode) {
  return (mode == kModeDenseFp8 || mode == kModeDenseFp4 || mode == kModeDenseFp4Multi ||
          mode == kModeDenseFp8Multi)
             ? kStreamCostQuant
             : kStreamCostBf16;
}

__host__ __device__ inline int32_t stream_cost(int32_t ntiles, int32_t sc) {
  return ntiles > 0 ? sc + ntiles * kTileCost : 0;
}

__host__ __device__ inline int64_t tile_cost_pos(int64_t stream_cost_start, int32_t k, int32_t sc) {
  return stream_cost_start + sc + static_cast<int64_t>(k) * kTileCost;
}

// CTAs the work is split over: the plan's count, but at most one per tile
// (a cost range of at least kTileCost units per CTA leaves no CTA between a
// row set's first and last tile owners without a tile of it).
__host__ __device__ inline int32_t work_ctas(int32_t plan_ctas, int32_t total_tiles) {
  return total_tiles < 1 ? 1 : (plan_ctas < total_tiles ? plan_ctas : total_tiles);
}

// CTA that owns cost position x when `total` cost units are split over
// `ctas` CTAs as [c*total/ctas, (c+1)*total/ctas).
__host__ __device__ inline int32_t tile_owner(int64_t x, int64_t total, int32_t ctas) {
  return static_cast<int32_t>(((x + 1) * ctas - 1) / total);
}

}  // namespace mla
