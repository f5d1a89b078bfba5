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

constexpr int kAbiVersion = 10000;   // 1.0.0
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
// `row_bytes`), box of box_cols x box_rows, 128-byte swizzle.
bool make_map_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int group_of(const mla_problem& pr) {
  return row_set_group(pr.q_len, pr.num_heads, pr.kv_dtype, pr.topk_width);
}

int decode_mode(const mla_problem& pr) {
  if (pr.kv_dtype == MLA_KV_FP8_E4M3_E8M0) return kModeDenseFp8;
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
    const int64_t per_stream = (longest + kTile - 1) / kTile * kTileCost + kStreamCost;
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
}

int plan_check(const mla_plan* plan) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARGUMENT;
  const int rc = validate_problem(&plan->problem);
  if (rc != MLA_OK) return rc;
  if (plan->num_streams != num_row_sets(plan->problem) || plan->num_ctas < 1)
    return MLA_ERR_INVALID_ARGUMENT;
  return MLA_OK;
}

}  // namespace

namespace mla {
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, uint64_t* waited_ns,
                                 cudaStream_t stream);
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
                    mla_plan* plan_out) {
  int rc = validate_problem(problem);
  if (rc != MLA_OK) return rc;
  if (plan_out == nullptr || sm_count < 1) return MLA_ERR_INVALID_ARGUMENT;
  mla_plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.problem = *problem;
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
  if (seq_lens_host != nullptr) ctas = tiles < 1 ? 1 : (tiles < sm_count ? tiles : sm_count);
  pl.num_ctas = static_cast<int32_t>(ctas);
  pl.num_slots = pl.num_streams + pl.num_ctas - 1;
  if (pl.num_slots < 1) pl.num_slots = 1;
  pl.smem_bytes = decode_smem_bytes(pr.num_heads, heads_pad, pl.num_streams, decode_mode(pr));
  if (pl.smem_bytes > 232448) return MLA_ERR_UNSUPPORTED;
  int64_t off = 0;
  pl.ws_partial_o = off;
  off = align_up(off + static_cast<int64_t>(pl.num_slots) * rows * kDc * 4, kAlign);
  pl.ws_partial_lse = off;
  off = align_up(off + static_cast<int64_t>(pl.num_slots) * rows * 4, kAlign);
  pl.ws_counters = off;
  off = align_up(off + static_cast<int64_t>(pl.num_streams) * 4, kAlign);
  pl.ws_status = off;
  off = align_up(off + 4, kAlign);
  pl.workspace_bytes = off;
  *plan_out = pl;
  return MLA_OK;
}

int mla_q_absorb(const mla_plan* plan, const void* q_nope, const void* q_rope, const void* w_uk,
                 void* q_hat, mla_stream_t stream) {
  int rc = plan_check(plan);
  if (rc != MLA_OK) return rc;
  if (!q_nope || !q_rope || !w_uk || !q_hat) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_hat))
    return MLA_ERR_MISALIGNED;
  const cudaError_t err = launch_q_absorb(
      static_cast<const uint16_t*>(q_nope), static_cast<const uint16_t*>(q_rope),
      static_cast<const uint16_t*>(w_uk), static_cast<uint16_t*>(q_hat),
      plan->problem.batch * plan->problem.q_len, plan->problem.num_heads,
      reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_run(const mla_plan* plan, const void* q_hat, const void* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk_idx,
                   void* workspace, float* o_lat, float* lse, mla_stream_t stream) {
  int rc = plan_check(plan);
  if (rc != MLA_OK) return rc;
  const mla_problem& pr = plan->problem;
  if (!q_hat || !kv_cache || !block_table || !seq_lens || !workspace || !o_lat || !lse)
    return MLA_ERR_INVALID_ARGUMENT;
  if ((pr.topk_width > 0) != (topk_idx != nullptr)) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_hat) || !aligned16(kv_cache) || !aligned16(workspace) || !aligned16(o_lat) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (topk_idx && (reinterpret_cast<uintptr_t>(topk_idx) & 3u)))
    return MLA_ERR_MISALIGNED;
  if (plan->num_streams == 0) return MLA_OK;
  const int mode = decode_mode(pr);
  CUtensorMap kv_map;
  std::memset(&kv_map, 0, sizeof(kv_map));   // FP8 / FP4 caches are read with bulk copies
  if (mode != kModeDenseFp8 && mode != kModeDenseFp4 &&
      !make_map_bf16(&kv_map, kv_cache, kDqk, static_cast<uint64_t>(pr.num_pages) * pr.page_size,
                     kDqk * 2, kChunkElems, pr.page_size < kTile ? pr.page_size : kTile))
    return MLA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p;
  p.q_hat = static_cast<const uint16_t*>(q_hat);
  p.kv = static_cast<const uint8_t*>(kv_cache);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.topk_idx = topk_idx;
  p.part_o = reinterpret_cast<float*>(ws + plan->ws_partial_o);
  p.part_lse = reinterpret_cast<float*>(ws + plan->ws_partial_lse);
  p.o_lat = o_lat;
  p.lse = lse;
  p.status = reinterpret_cast<uint32_t*>(ws + plan->ws_status);
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
  p.num_streams = plan->num_streams;
  p.num_ctas = plan->num_ctas;
  p.scale_log2 = pr.sm_scale * 1.4426950408889634f;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err = launch_decode(p, &kv_map, mode, st);
  if (err != cudaSuccess) return MLA_ERR_CUDA;
  // split row sets: merge their partials (all SMs, dependent launch)
  CombineParams cp;
  fill_combine_params(*plan, ws, seq_lens, o_lat, lse, &cp);
  err = launch_combine(cp, st);
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_combine(const mla_plan* plan, const int32_t* seq_lens, const void* workspace, float* o_lat,
                float* lse, mla_stream_t stream) {
  int rc = plan_check(plan);
  if (rc != MLA_OK) return rc;
  if (!seq_lens || !workspace || !o_lat || !lse) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned16(workspace) || !aligned16(o_lat) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_MISALIGNED;
  CombineParams p;
  fill_combine_params(*plan, static_cast<const uint8_t*>(workspace), seq_lens, o_lat, lse, &p);
  const cudaError_t err = launch_combine(p, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
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
  const cudaError_t err = launch_uv_proj_tma(&w_map, o_lat, static_cast<uint16_t*>(out), rows,
                                             num_heads, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_cache_append(const mla_problem* problem, const void* new_rows, const int32_t* positions,
                     const int32_t* block_table, void* kv_cache, uint32_t* status,
                     mla_stream_t stream) {
  const int rc = validate_problem(problem);
  if (rc != MLA_OK) return rc;
  if (!new_rows || !positions || !block_table || !kv_cache) return MLA_ERR_INVALID_ARGUMENT;
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
