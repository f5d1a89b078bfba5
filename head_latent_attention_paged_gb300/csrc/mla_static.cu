// mla_decode_run_static: the decode pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they decode: code
// running while a CUDA graph is being captured or replayed, runtimes that
// hand out only the input and output buffers they manage themselves, or
// allocators that forbid growth after start-up.  This entry point needs no
// workspace from them: its scratch (split partials and the status word)
// lives in one fixed-size array in device memory that belongs to this
// library.
//
// Properties of that array, for users:
//   * Size kStaticScratchBytes (16 MiB).  Every GPU that loads the library
//     holds it until the process exits.
//   * One array per device, shared by every call on that device.  Calls that
//     overlap on the GPU (different streams without ordering between them)
//     race on it and give undefined results; order them on one stream.
//   * It keeps the previous call's contents.  Each call clears the parts
//     that must start at zero (the reserved words and the status word)
//     on the caller's stream before launching.
//   * Every argument is checked before anything is queued, so a rejected
//     call leaves the array as it was.
//   * The first call on a device looks up the array's device address (a
//     runtime query, no allocation) with that device current, and looks it
//     up again when the device's current context is a different one (after
//     a device reset, or under another context).  Make that first call
//     before any stream capture begins.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mla_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_mla_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};

// Device address of this device's scratch array, looked up once per device
// and context.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* ctx = mla::current_context();
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr || ctx == nullptr || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_mla_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" MLA_API int mla_decode_run_static(const mla_plan* plan, const void* q_hat,
                                             const void* kv_cache, const int32_t* block_table,
                                             const int32_t* seq_lens, const int32_t* topk_idx,
                                             float* o_lat, float* lse, uint32_t* status,
                                             mla_stream_t stream) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARGUMENT;
  if (plan->workspace_bytes <= 0 ||
      static_cast<uint64_t>(plan->workspace_bytes) > kStaticScratchBytes)
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u)) return MLA_ERR_MISALIGNED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MLA_ERR_CUDA;
  // every check mla_decode_run makes, before anything touches the array
  int rc = mla::check_run_args(plan, q_hat, nullptr, kv_cache, block_table, seq_lens, topk_idx,
                               scratch, kStaticScratchBytes, o_lat, lse);
  if (rc != MLA_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  // The status word must start at zero; it sits at the end of the workspace
  // layout, after the row-set prefixes (cleared with it; the decode launch
  // writes them when it uses them).
  if (cudaMemsetAsync(ws + plan->ws_prefix, 0,
                      static_cast<size_t>(plan->workspace_bytes - plan->ws_prefix),
                      st) != cudaSuccess)
    return MLA_ERR_CUDA;
  rc = mla::launch_attention(*plan, q_hat, kv_cache, block_table, seq_lens, topk_idx, ws, o_lat,
                             lse, st);
  if (rc != MLA_OK) return rc;
  rc = mla::launch_merge(*plan, seq_lens, ws, nullptr, o_lat, lse, nullptr, st);
  if (rc != MLA_OK) return rc;
  if (status != nullptr &&
      cudaMemcpyAsync(status, ws + plan->ws_status, 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
