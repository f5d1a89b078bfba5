// Host side of the C ABI declared in include/mla_decode.h: argument
// validation, the launch plan, TMA descriptors and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "mla_internal.h"

using namespace mla;

namespace {

constexpr int kAbiVersion = 20100;   // 2.1.0
constexpr int64_t kAlign = 256;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor map: `rows` rows of `cols` elements (row stride
// `row_bytes`), box of box_cols x box_rows, 128-byte swizzle.  Encoded maps
// are kept in a small table keyed by every argument, so a decode step that
// reuses its cache and weights does no encoding on the host.
struct MapKey {
  const void* base;
  uint64_t cols, rows, row_bytes;
  uint32_t box_cols, box_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && cols == o.cols && rows == o.rows && row_bytes == o.row_bytes &&
           box_cols == o.box_cols && box_rows == o.box_rows;
  }
};
constexpr int kMapCacheSize = 32;
std::mutex g_map_mutex;
MapKey g_map_keys[kMapCacheSize];
CUtensorMap g_maps[kMapCacheSize];
int g_map_count = 0, g_map_next = 0;

bool make_map_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  const MapKey key{base, cols, rows, row_bytes, box_cols, box_rows};
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_map_count; ++i)
      if (g_map_keys[i] == key) {
        *map = g_maps[i];
        return true;
      }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  const int slot = g_map_count < kMapCacheSize ? g_map_count++ : (g_map_next++ % kMapCacheSize);
  g_map_keys[slot] = key;
  g_maps[slot] = *map;
  return true;
}

}  // namespace

namespace mla {

// The current CUDA context (a driver handle, queried through the runtime's
// entry-point lookup so the library needs no link-time driver dependency).
// Per-context caches compare it to notice a context that was replaced.
void* current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(ptr);
  });
  CUcontext ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

cudaError_t set_smem_attr_once(const void* func, int slot, int bytes) {
  constexpr int kDevices = 64, kSlots = 16;
  static std::mutex mu;
  static int done[kDevices][kSlots] = {};
  static void* ctx_of[kDevices][kSlots] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevices || slot < 0 || slot >= kSlots)
    return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx != nullptr && ctx_of[dev][slot] == ctx && done[dev][slot] >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) {
    done[dev][slot] = ctx_of[dev][slot] == ctx ? (bytes > done[dev][slot] ? bytes : done[dev][slot]) : bytes;
    ctx_of[dev][slot] = ctx;
  }
  return err;
}

}  // namespace mla

namespace {

int group_of(const mla_problem& pr) {
  return row_set_group(pr.q_len, pr.num_heads, pr.kv_dtype, pr.topk_width);
}

int decode_mode(const mla_problem& pr) {
  if (pr.kv_dtype == MLA_KV_FP8_E4M3_E8M0)
    return group_of(pr) >= 2 ? kModeDenseFp8Multi : kModeDenseFp8;
  if (pr.kv_dtype == MLA_KV_FP4_E2M1_E8M0)
    return group_of(pr) >= 2 ? kModeDenseFp4Multi : kModeDenseFp4;
  if (pr.topk_width > 0) return kModeSparseBf16;
  return group_of(pr) >= 2 ? kModeDenseMulti : kModeDenseBf16;
}

// row sets: one per (request, group of draft tokens)
int32_t num_row_sets(const mla_problem& pr) {
  const int32_t g = group_of(pr);
  return pr.batch * ((pr.q_len + g - 1) / g);
}

// The cache shape and options every entry point shares (the append needs
// no more than this).
int validate_cache_shape(const mla_problem* pr) {
  if (pr == nullptr) return MLA_ERR_INVALID_ARGUMENT;
  if (pr->batch < 0 || pr->num_pages < 1 || pr->max_pages_per_seq < 1)
    return MLA_ERR_INVALID_ARGUMENT;
  if (pr->kv_lora_rank != kDc || pr->rope_dim != kDr || pr->nope_dim != kDnope ||
      pr->v_head_dim != kDv)
    return MLA_ERR_UNSUPPORTED;
  if (pr->page_size != 16 && pr->page_size != 32 && pr->page_size != 64 && pr->page_size != 128)
    return MLA_ERR_UNSUPPORTED;
  if (pr->kv_dtype != MLA_KV_BF16 && pr->kv_dtype != MLA_KV_FP8_E4M3_E8M0 &&
      pr->kv_dtype != MLA_KV_FP4_E2M1_E8M0)
    return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(pr->num_pages) * pr->page_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(pr->max_pages_per_seq) * pr->page_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

int validate_problem(const mla_problem* pr) {
  if (pr == nullptr) return MLA_ERR_INVALID_ARGUMENT;
  if (pr->batch < 0 || pr->q_len < 1 || pr->num_heads < 1 || pr->num_pages < 1 ||
      pr->max_pages_per_seq < 1 || pr->topk_width < 0 || !(pr->causal == 0 || pr->causal == 1) ||
      !std::isfinite(pr->sm_scale) || pr->sm_scale <= 0.f)
    return MLA_ERR_INVALID_ARGUMENT;
  if (pr->kv_lora_rank != kDc || pr->rope_dim != kDr || pr->nope_dim != kDnope ||
      pr->v_head_dim != kDv)
    return MLA_ERR_UNSUPPORTED;
  if (pr->page_size != 16 && pr->page_size != 32 && pr->page_size != 64 && pr->page_size != 128)
    return MLA_ERR_UNSUPPORTED;
  if (pr->num_heads > kMaxHeads) return MLA_ERR_UNSUPPORTED;
  if (pr->topk_width % 128 != 0) return MLA_ERR_UNSUPPORTED;
  if (pr->kv_dtype != MLA_KV_BF16 && pr->kv_dtype != MLA_KV_FP8_E4M3_E8M0 &&
      pr->kv_dtype != MLA_KV_FP4_E2M1_E8M0)
    return MLA_ERR_UNSUPPORTED;
  if (pr->kv_dtype != MLA_KV_BF16 && pr->topk_width > 0) return MLA_ERR_UNSUPPORTED;
  {  // row sets (draft tokens grouped where the multi-token mode applies)
    const int64_t g = group_of(*pr);
    if (static_cast<int64_t>(pr->batch) * ((pr->q_len + g - 1) / g) > kMaxStreams)
      return MLA_ERR_UNSUPPORTED;
  }
  if (static_cast<int64_t>(pr->num_pages) * pr->page_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(pr->max_pages_per_seq) * pr->page_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(pr->batch) * pr->q_len * pr->num_heads > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  {  // the kernels' cost prefix over row sets is 32-bit
    const int64_t longest = pr->topk_width > 0
                                ? pr->topk_width
                                : static_cast<int64_t>(pr->max_pages_per_seq) * pr->page_size;
    const int64_t per_stream = (longest + kTile - 1) / kTile * kTileCost + kStreamCostMax;
    if (static_cast<int64_t>(pr->batch) * pr->q_len * per_stream > INT32_MAX)
      return MLA_ERR_UNSUPPORTED;
  }
  return MLA_OK;
}

int64_t stream_tiles_host(const mla_problem& pr, const int32_t* seq_lens) {
  int64_t total = 0;
  const int32_t max_tokens = pr.max_pages_per_seq * pr.page_size;
  const int32_t g = group_of(pr);
  const int32_t S = num_row_sets(pr);
  for (int32_t s = 0; s < S; ++s) {
    const StreamGeom gm = stream_geom(s, pr.q_len, g);
    const int32_t len = stream_len(seq_lens[gm.b], pr.q_len, gm.j0 + gm.nq - 1, pr.causal,
                                   pr.topk_width, max_tokens);
    total += (len + kTile - 1) / kTile;
  }
  return total;
}

// Whether the row-set prefixes of the work split come from the pre-pass
// (too many row sets for the decode kernel's shared memory).
bool prefix_in_workspace(const mla_plan& plan) {
  const mla_problem& pr = plan.problem;
  const int rows = group_of(pr) * pr.num_heads;
  return !decode_layout(pr.num_heads, (rows + 15) / 16 * 16, plan.num_streams, decode_mode(pr))
              .prefix_in_smem;
}

void fill_combine_params(const mla_plan& plan, const uint8_t* ws, const int32_t* seq_lens,
                         float* o_lat, float* lse, CombineParams* out) {
  const mla_problem& pr = plan.problem;
  CombineParams& p = *out;
  p.part_o = reinterpret_cast<const float*>(ws + plan.ws_partial_o);
  p.part_lse = reinterpret_cast<const float*>(ws + plan.ws_partial_lse);
  p.seq_lens = seq_lens;
  p.o_lat = o_lat;
  p.lse = lse;
  p.batch = pr.batch;
  p.q_len = pr.q_len;
  p.heads = pr.num_heads;
  p.page_size = pr.page_size;
  p.max_pages = pr.max_pages_per_seq;
  p.topk_width = pr.topk_width;
  p.causal = pr.causal;
  p.group = group_of(pr);
  p.rows = p.group * pr.num_heads;
  p.num_streams = plan.num_streams;
  p.num_ctas = plan.num_ctas;
  p.stream_cost = stream_cost_of_mode(decode_mode(pr));
  p.prefix_ws = prefix_in_workspace(plan) ? reinterpret_cast<const int32_t*>(ws + plan.ws_prefix)
                                          : nullptr;
}

int absorb(const mla_plan& plan, const void* q, const void* w_uk, void* q_hat, cudaStream_t st) {
  const mla_problem& pr = plan.problem;
  const int rows = pr.batch * pr.q_len;
  if (rows == 0) return MLA_OK;
  CUtensorMap w_map;
  if (!make_map_bf16(&w_map, w_uk, kDnope, static_cast<uint64_t>(pr.num_heads) * kDc, kDnope * 2,
                     64, 128))
    return MLA_ERR_CUDA;
  const cudaError_t err = launch_q_absorb(&w_map, static_cast<const uint16_t*>(q),
                                          static_cast<uint16_t*>(q_hat), rows, pr.num_heads, st);
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

namespace mla {
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, uint64_t* waited_ns,
                                 cudaStream_t stream);

int plan_check(const mla_plan* plan) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARGUMENT;
  const int rc = validate_problem(&plan->problem);
  if (rc != MLA_OK) return rc;
  if (plan->num_streams != num_row_sets(plan->problem) || plan->num_ctas < 1 || plan->sm_count < 1 ||
      plan->num_ctas > kMaxCtas || plan->num_slots != plan->num_streams + plan->num_ctas - 1 ||
      plan->ws_partial_o < 0 || plan->ws_partial_lse < plan->ws_partial_o ||
      plan->ws_q_hat < plan->ws_partial_lse || plan->ws_prefix < plan->ws_q_hat ||
      plan->ws_status < plan->ws_prefix + 8 * (static_cast<int64_t>(plan->num_streams) + 1) || plan->ws_status + 4 > plan->workspace_bytes)
    return MLA_ERR_INVALID_ARGUMENT;
  return MLA_OK;
}

int check_run_args(const mla_plan* plan, const void* q, const void* w_uk, const void* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk_idx,
                   const void* workspace, size_t workspace_bytes, const float* o_lat,
                   const float* lse) {
  const int rc = plan_check(plan);
  if (rc != MLA_OK) return rc;
  const mla_problem& pr = plan->problem;
  if (!q || !kv_cache || !block_table || !seq_lens || !workspace || !o_lat || !lse)
    return MLA_ERR_INVALID_ARGUMENT;
  if ((pr.topk_width > 0) != (topk_idx != nullptr)) return MLA_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < static_cast<size_t>(plan->workspace_bytes)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(q) || (w_uk && !aligned16(w_uk)) || !aligned16(kv_cache) ||
      !aligned16(workspace) || !aligned16(o_lat) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (topk_idx && (reinterpret_cast<uintptr_t>(topk_idx) & 3u)))
    return MLA_ERR_MISALIGNED;
  return MLA_OK;
}

int launch_attention(const mla_plan& plan, const void* q_hat, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk_idx,
                     uint8_t* ws, float* o_lat, float* lse, cudaStream_t st) {
  const mla_problem& pr = plan.problem;
  if (plan.num_streams == 0) return MLA_OK;
  const int mode = decode_mode(pr);
  CUtensorMap kv_map;
  std::memset(&kv_map, 0, sizeof(kv_map));   // FP8 / FP4 caches are read with bulk copies
  if (mode != kModeDenseFp8 && mode != kModeDenseFp4 && mode != kModeDenseFp4Multi &&
      mode != kModeDenseFp8Multi &&
      !make_map_bf16(&kv_map, kv_cache, kDqk, static_cast<uint64_t>(pr.num_pages) * pr.page_size,
                     kDqk * 2, kChunkElems,
                     mode == kModeSparseBf16 ? 1 : (pr.page_size < kTile ? pr.page_size : kTile)))
    return MLA_ERR_CUDA;
  DecodeParams p;
  p.q_hat = static_cast<const uint16_t*>(q_hat);
  p.kv = static_cast<const uint8_t*>(kv_cache);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.topk_idx = topk_idx;
  p.part_o = reinterpret_cast<float*>(ws + plan.ws_partial_o);
  p.part_lse = reinterpret_cast<float*>(ws + plan.ws_partial_lse);
  p.o_lat = o_lat;
  p.lse = lse;
  p.status = reinterpret_cast<uint32_t*>(ws + plan.ws_status);
  p.batch = pr.batch;
  p.q_len = pr.q_len;
  p.heads = pr.num_heads;
  p.group = group_of(pr);
  p.rows = p.group * pr.num_heads;
  p.heads_pad = (p.rows + 15) / 16 * 16;
  p.page_size = pr.page_size;
  p.num_pages = pr.num_pages;
  p.max_pages = pr.max_pages_per_seq;
  p.topk_width = pr.topk_width;
  p.causal = pr.causal;
  p.num_streams = plan.num_streams;
  p.num_ctas = plan.num_ctas;
  p.stream_cost = stream_cost_of_mode(mode);
  p.scale_log2 = pr.sm_scale * 1.4426950408889634f;
  p.prefix_ws = nullptr;
  if (prefix_in_workspace(plan)) {
    p.prefix_ws = reinterpret_cast<int32_t*>(ws + plan.ws_prefix);
    if (launch_prefix(p, st) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return launch_decode(p, &kv_map, mode, st) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int launch_merge(const mla_plan& plan, const int32_t* seq_lens, const uint8_t* ws,
                 const void* w_uv, float* o_lat, float* lse, void* out, cudaStream_t st) {
  if (plan.num_streams == 0) return MLA_OK;
  CombineParams cp;
  fill_combine_params(plan, ws, seq_lens, o_lat, lse, &cp);
  // without W_UV: the merge over all SMs (one block per row of a row set);
  // with it: the merge inside the up-projection's blocks (per head, 128
  // output dims and a row block).  Either is a programmatic dependent of the
  // decode launch.
  cudaError_t err;
  if (w_uv == nullptr) {
    err = launch_combine(cp, st);
  } else {
    const mla_problem& pr = plan.problem;
    CUtensorMap w_map;
    if (!make_map_bf16(&w_map, w_uv, kDv, static_cast<uint64_t>(pr.num_heads) * kDc, kDv * 2, 64,
                       64))
      return MLA_ERR_CUDA;
    err = launch_merge_uv(&w_map, cp, static_cast<uint16_t*>(out), plan.sm_count, st);
  }
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla

extern "C" {

int mla_version(void) { return kAbiVersion; }

const char* mla_strerror(int code) {
  switch (code) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MLA_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA call or kernel launch failed";
    default: return "unknown error";
  }
}

int mla_decode_plan(const mla_problem* problem, const int32_t* seq_lens_host, int32_t sm_count,
                    int32_t split_tokens, mla_plan* plan_out, size_t* workspace_bytes) {
  int rc = validate_problem(problem);
  if (rc != MLA_OK) return rc;
  if (plan_out == nullptr || sm_count < 1 || split_tokens < 0 || split_tokens % kTile != 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (split_tokens > 0 && seq_lens_host == nullptr) return MLA_ERR_INVALID_ARGUMENT;
  mla_plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.problem = *problem;
  pl.split_tokens = split_tokens;
  pl.sm_count = sm_count;
  const mla_problem& pr = pl.problem;
  pl.num_streams = num_row_sets(pr);
  const int rows = group_of(pr) * pr.num_heads;   // rows of a full row set
  const int heads_pad = (rows + 15) / 16 * 16;
  int64_t tiles = 0;
  if (seq_lens_host != nullptr) {
    for (int b = 0; b < pr.batch; ++b)
      if (seq_lens_host[b] < 0) return MLA_ERR_INVALID_ARGUMENT;
    tiles = stream_tiles_host(pr, seq_lens_host);
  }
  pl.planned_tiles = tiles;
  int64_t ctas = sm_count;
  if (split_tokens > 0) {
    // split-KV by length: about split_tokens tokens per CTA
    const int64_t per = split_tokens / kTile;
    ctas = (tiles + per - 1) / per;
    if (ctas < 1) ctas = 1;
    if (ctas > kMaxCtas) return MLA_ERR_UNSUPPORTED;
  } else if (seq_lens_host != nullptr) {
    ctas = tiles < 1 ? 1 : (tiles < sm_count ? tiles : sm_count);
  }
  pl.num_ctas = static_cast<int32_t>(ctas);
  pl.num_slots = pl.num_streams + pl.num_ctas - 1;
  if (pl.num_slots < 1) pl.num_slots = 1;
  pl.smem_bytes = decode_smem_bytes(pr.num_heads, heads_pad, pl.num_streams, decode_mode(pr));
  pl.prefix_pass = decode_layout(pr.num_heads, heads_pad, pl.num_streams, decode_mode(pr))
                       .prefix_in_smem ? 0 : 1;
  if (pl.smem_bytes > kMaxSmemBytes) return MLA_ERR_UNSUPPORTED;
  int64_t off = 0;
  pl.ws_partial_o = off;
  off = align_up(off + static_cast<int64_t>(pl.num_slots) * rows * kDc * 4, kAlign);
  pl.ws_partial_lse = off;
  off = align_up(off + static_cast<int64_t>(pl.num_slots) * rows * 4, kAlign);
  pl.ws_q_hat = off;
  off = align_up(off + static_cast<int64_t>(pr.batch) * pr.q_len * pr.num_heads * kDqk * 2, kAlign);
  pl.ws_prefix = off;
  off = align_up(off + 8 * (static_cast<int64_t>(pl.num_streams) + 1), kAlign);
  pl.ws_status = off;
  off = align_up(off + 4, kAlign);
  pl.workspace_bytes = off;
  *plan_out = pl;
  if (workspace_bytes != nullptr) *workspace_bytes = static_cast<size_t>(off);
  return MLA_OK;
}

int mla_q_absorb(const mla_plan* plan, const void* q, const void* w_uk, void* q_hat,
                 mla_stream_t stream) {
  int rc = plan_check(plan);
  if (rc != MLA_OK) return rc;
  if (!q || !w_uk || !q_hat) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(w_uk) || !aligned16(q_hat)) return MLA_ERR_MISALIGNED;
  return absorb(*plan, q, w_uk, q_hat, reinterpret_cast<cudaStream_t>(stream));
}

int mla_decode_run(const mla_plan* plan, const void* q, const void* w_uk, const void* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk_idx,
                   void* workspace, size_t workspace_bytes, float* o_lat, float* lse,
                   mla_stream_t stream) {
  int rc = check_run_args(plan, q, w_uk, kv_cache, block_table, seq_lens, topk_idx, workspace,
                          workspace_bytes, o_lat, lse);
  if (rc != MLA_OK) return rc;
  if (plan->num_streams == 0) return MLA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void* q_hat = q;
  if (w_uk != nullptr) {   // absorb the queries into the workspace first
    q_hat = ws + plan->ws_q_hat;
    rc = absorb(*plan, q, w_uk, ws + plan->ws_q_hat, st);
    if (rc != MLA_OK) return rc;
  }
  return launch_attention(*plan, q_hat, kv_cache, block_table, seq_lens, topk_idx, ws, o_lat, lse,
                          st);
}

int mla_combine(const mla_plan* plan, const int32_t* seq_lens, const void* workspace,
                size_t workspace_bytes, const void* w_uv, float* o_lat, float* lse, void* out,
                mla_stream_t stream) {
  int rc = plan_check(plan);
  if (rc != MLA_OK) return rc;
  if (!seq_lens || !workspace || !o_lat || !lse || (w_uv && !out)) return MLA_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < static_cast<size_t>(plan->workspace_bytes)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace) || !aligned16(o_lat) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (w_uv && (!aligned16(w_uv) || !aligned16(out))) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return MLA_ERR_MISALIGNED;
  return launch_merge(*plan, seq_lens, static_cast<const uint8_t*>(workspace), w_uv, o_lat, lse,
                      out, reinterpret_cast<cudaStream_t>(stream));
}

int mla_decode_step(const mla_plan* plan, const void* q, const void* w_uk, const void* kv_cache,
                    const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk_idx,
                    void* workspace, size_t workspace_bytes, const void* w_uv, float* o_lat,
                    float* lse, void* out, mla_stream_t stream) {
  int rc = check_run_args(plan, q, w_uk, kv_cache, block_table, seq_lens, topk_idx, workspace,
                          workspace_bytes, o_lat, lse);
  if (rc != MLA_OK) return rc;
  if (!w_uv || !out) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned16(w_uv) || !aligned16(out)) return MLA_ERR_MISALIGNED;
  if (plan->num_streams == 0) return MLA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void* q_hat = q;
  if (w_uk != nullptr) {
    q_hat = ws + plan->ws_q_hat;
    rc = absorb(*plan, q, w_uk, ws + plan->ws_q_hat, st);
    if (rc != MLA_OK) return rc;
  }
  rc = launch_attention(*plan, q_hat, kv_cache, block_table, seq_lens, topk_idx, ws, o_lat, lse, st);
  if (rc != MLA_OK) return rc;
  return launch_merge(*plan, seq_lens, ws, w_uv, o_lat, lse, out, st);
}

int mla_uv_proj(const float* o_lat, const void* w_uv, void* out, int32_t rows, int32_t num_heads,
                mla_stream_t stream) {
  if (!o_lat || !w_uv || !out || rows < 0 || num_heads < 1 || num_heads > 128)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_MISALIGNED;
  if (rows == 0) return MLA_OK;
  CUtensorMap w_map;
  if (!make_map_bf16(&w_map, w_uv, kDv, static_cast<uint64_t>(num_heads) * kDc, kDv * 2, 64, 64))
    return MLA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  const cudaError_t err = launch_uv_proj_tma(&w_map, o_lat, static_cast<uint16_t*>(out), rows,
                                             num_heads, sms, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_cache_append(const mla_problem* problem, const void* new_rows, const int32_t* positions,
                     const int32_t* block_table, float rope_theta, void* kv_cache,
                     uint32_t* status, mla_stream_t stream) {
  const int rc = validate_cache_shape(problem);
  if (rc != MLA_OK) return rc;
  if (!new_rows || !positions || !block_table || !kv_cache) return MLA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(rope_theta) || rope_theta < 0.f || (rope_theta > 0.f && rope_theta <= 1.f))
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned16(new_rows) || !aligned16(kv_cache) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (status && (reinterpret_cast<uintptr_t>(status) & 3u)))
    return MLA_ERR_MISALIGNED;
  AppendParams p;
  p.new_rows = static_cast<const uint16_t*>(new_rows);
  p.positions = positions;
  p.block_table = block_table;
  p.kv = static_cast<uint8_t*>(kv_cache);
  p.status = status;
  p.rows = problem->batch;
  p.page_size = problem->page_size;
  p.num_pages = problem->num_pages;
  p.max_pages = problem->max_pages_per_seq;
  p.kv_dtype = problem->kv_dtype;
  p.rope_theta = rope_theta;
  const cudaError_t err = launch_append(p, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_selftest_bounded_wait(uint32_t* status, int64_t limit_ns, uint64_t* waited_ns,
                              mla_stream_t stream) {
  if (status == nullptr || limit_ns < 1 || limit_ns > 1000000000) return MLA_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(status) & 3u) ||
      (waited_ns && (reinterpret_cast<uintptr_t>(waited_ns) & 7u)))
    return MLA_ERR_MISALIGNED;
  const cudaError_t err = launch_wait_selftest(status, static_cast<uint64_t>(limit_ns), waited_ns,
                                               reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_get_status(const mla_plan* plan, const void* workspace, uint32_t* bits, mla_stream_t stream) {
  if (!plan || !workspace || !bits) return MLA_ERR_INVALID_ARGUMENT;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  if (cudaMemcpyAsync(&host, ws + plan->ws_status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  *bits = host;
  return MLA_OK;
}

int mla_clear_status(const mla_plan* plan, void* workspace, mla_stream_t stream) {
  if (!plan || !workspace) return MLA_ERR_INVALID_ARGUMENT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return cudaMemsetAsync(ws + plan->ws_status, 0, 4, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // extern "C"
