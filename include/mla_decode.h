/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) paged MLA latent-cache decode
 * library (libmla_gb300.so).
 *
 * The operation: Multi-head Latent Attention decode over a paged, low-rank
 * latent KV cache.  Each cached token of a layer holds a shared 512-dim latent
 * c_kv and a decoupled 64-dim RoPE key, not per-head K/V (GLM-4.7-Flash
 * record, phantomic12 inference-research: the MLA family paragraph and the
 * configuration clause kv_lora_rank 512 / qk_rope_head_dim 64 /
 * qk_nope_head_dim 192 / v_head_dim 256; 576 bf16 values = 1,152 bytes per
 * token and layer, 54,144 bytes per token over 47 layers).  The per-head
 * query is absorbed into the 576-dim latent space through W_UK (the kv_b_proj
 * up-projection), scored against every visible cached row, softmaxed, the
 * weighted latent rows are summed (o_lat) and finally up-projected through
 * W_UV:
 *
 *     q_hat[h]  = [W_UK[h] q_nope[h] || q_rope[h]]                 (576)
 *     s[h,t]    = sm_scale * q_hat[h] . row[t]                      row = [c_kv || k_rope]
 *     lse[h]    = ln sum_t exp(s[h,t])
 *     o_lat[h]  = sum_t exp(s[h,t] - lse[h]) c_kv[t]                 (512)
 *     o[h]      = W_UV[h]^T o_lat[h]                                 (256)
 *
 * Paged cache: logical position t of request b is slot t % P of physical page
 * block_table[b][t / P]; P is 64 or 128 (fix: Add glm4_moe_lite to MLA
 * detection, the note that CUTLASS_MLA enforces block_size=128; GLM-4.7-Flash
 * record: decode kernels are instantiated per KV cache page-block size and a
 * planner hard-codes 64), or 16 or 32 for compressed layers (same record:
 * the page block size block_size / compress_ratio).  The call split plan / run mirrors the
 * planner + kernel split of the FlashInfer MLA decode the record describes.
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer.  The library allocates no device memory;
 *     `mla_plan` is a plain struct the caller keeps.
 *   - Device pointers are CUDA device addresses on the current device and
 *     must be 16-byte aligned (TMA and bulk copies require it).
 *   - Every call that takes a stream is asynchronous on that stream
 *     (NULL = the legacy default stream) unless stated otherwise.
 *   - Return value 0 is success; a negative MLA_ERR_* code means nothing was
 *     launched (argument errors) or a launch failed (MLA_ERR_CUDA).  No
 *     exception or abort crosses the ABI.
 *   - Data errors found on the device (a block-table entry outside
 *     [0, num_pages), a sparse index outside [-1, visible window)) never
 *     fault: the offending rows are masked out and a sticky bit is set in the
 *     status word read by mla_get_status.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* mla_stream_t;

/* return codes */
#define MLA_OK 0
#define MLA_ERR_INVALID_ARGUMENT (-1)   /* null pointer, negative or inconsistent size */
#define MLA_ERR_UNSUPPORTED (-2)        /* a shape or option this library does not implement */
#define MLA_ERR_MISALIGNED (-3)         /* a device pointer not 16-byte aligned */
#define MLA_ERR_WORKSPACE_TOO_SMALL (-4)
#define MLA_ERR_CUDA (-5)               /* a CUDA runtime / driver call or launch failed */

/* latent-cache element formats */
#define MLA_KV_BF16 0
/* 576 float8_e4m3 values followed by 18 float8_e8m0 scales (one per 32
 * consecutive values, value = e4m3 * 2^(scale - 127)) per token: 594 bytes
 * per token, a page of P tokens is P contiguous rows.  All 576 dims are
 * quantised, RoPE dims included (GLM-4.7-Flash record, engine-kernel
 * constraint (2): FP8 latent with per-token inlined e8m0 scales, one per 32
 * e4m3 values). */
#define MLA_KV_FP8_E4M3_E8M0 1
/* 576 float4_e2m1 values packed two per byte (value 2i in the low nibble of
 * byte i: 288 bytes) followed by 36 float8_e8m0 scales (one per 16
 * consecutive values, value = e2m1 * 2^(scale - 127)) per token: 324 bytes
 * per token, a page of P tokens is P contiguous rows.  e2m1: sign, 2
 * exponent bits (bias 1), 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4,
 * 6.  The record gives only 288 bytes per token for its 512-value row
 * (GLM-4.7-Flash record, engine-kernel constraint (2): the FP4 variant of the
 * inlined-scale latent); 256 code bytes + 32 scale bytes is read as one e8m0
 * scale per 16 values, and the layout follows the FP8 variant's. */
#define MLA_KV_FP4_E2M1_E8M0 2

/* status-word bits (sticky until mla_clear_status) */
#define MLA_STATUS_BAD_PAGE 0x1u     /* a block-table entry outside [0, num_pages) was masked */
#define MLA_STATUS_BAD_INDEX 0x2u    /* a sparse index outside [-1, window) was masked */
#define MLA_STATUS_TIMEOUT 0x4u      /* an internal pipeline wait hit its time limit */

#define MLA_TILE_TOKENS 64           /* cached rows per pipeline tile */

/* One decode step of one layer.  All sizes are element counts. */
typedef struct {
  int32_t batch;            /* B: requests */
  int32_t q_len;            /* Q: query tokens per request (speculative drafts), >= 1 */
  int32_t num_heads;        /* H: query heads, 1..32 */
  int32_t kv_lora_rank;     /* must be 512 */
  int32_t rope_dim;         /* must be 64 */
  int32_t nope_dim;         /* must be 192 (only read by mla_q_absorb) */
  int32_t v_head_dim;       /* must be 256 */
  int32_t page_size;        /* P: 16, 32, 64 or 128 */
  int32_t num_pages;        /* physical pages in the cache pool */
  int32_t max_pages_per_seq;/* row stride of block_table */
  int32_t kv_dtype;         /* MLA_KV_BF16, MLA_KV_FP8_E4M3_E8M0 or MLA_KV_FP4_E2M1_E8M0
                               (the quantised formats: dense only, topk_width 0) */
  int32_t topk_width;       /* 0: dense; else sparse row width, a multiple of 128
                               (vllm API docs, vllm.models.glm5next.common.model,
                               Glm5NextModel.__init__: top-k is tiled in 128
                               columns and padded slots stay masked) */
  int32_t causal;           /* 1: query token j sees positions <= T_b - Q + j;
                               0: every query token sees all T_b positions */
  float sm_scale;           /* softmax scale on q_hat . row; 1/sqrt(192 + 64) for GLM-4.7-Flash */
} mla_problem;

/* Filled by mla_decode_plan; treat as opaque, keep it alive while in use. */
typedef struct {
  mla_problem problem;
  int32_t num_streams;      /* row sets: B * Q (one per request and query token), or
                               B * ceil(Q / G) when G draft tokens of a request share one
                               (dense bf16 or FP4 cache, Q >= 2, G = min(Q, 48 / H) >= 2) */
  int32_t num_ctas;         /* decode grid size */
  int32_t num_slots;        /* partial-result slots: num_streams + num_ctas - 1 */
  int32_t smem_bytes;       /* dynamic shared memory of the decode kernel */
  int64_t ws_partial_o;     /* byte offset of f32 [num_slots][G * H][512] */
  int64_t ws_partial_lse;   /* byte offset of f32 [num_slots][G * H] */
  int64_t ws_prefix;        /* byte offset of int32 [2][num_streams + 1]: the row sets'
                               tile and cost prefixes of the work split, written by the
                               decode launch when the row sets are too many for the
                               decode kernel's shared memory (else left untouched) */
  int64_t ws_status;        /* byte offset of the uint32 status word */
  int64_t workspace_bytes;  /* total workspace size */
  int64_t planned_tiles;    /* tiles implied by seq_lens_host (0 if not given) */
  int64_t ws_q_hat;         /* byte offset of bf16 [B*Q][H][576]: the absorbed queries
                               mla_decode_run writes when it is given W_UK */
  int32_t split_tokens;     /* as requested from mla_decode_plan (0 = automatic) */
  int32_t sm_count;         /* as given to mla_decode_plan */
  int32_t prefix_pass;      /* 1: each decode launch runs the one-block prefix pre-pass
                               first (row sets too many for the kernel's shared memory) */
  int32_t reserved[3];
} mla_plan;

/*
 * mla_decode_plan -- validate a problem and build the launch plan (host only,
 * no CUDA call).  The plan / run split is the planner + kernel split of the
 * FlashInfer MLA decode ("GLM-4.7-Flash" record, phantomic12
 * inference-research: engine-kernel constraint (1), decode kernels
 * instantiated per page-block size behind a planner).
 *   problem         : the step's shape and options (copied into the plan).
 *   seq_lens_host   : host int32 [batch] context lengths, or NULL.  Used only
 *                     to size the grid: the device kernels re-derive the exact
 *                     work split from the device seq_lens they are given.
 *   sm_count        : streaming multiprocessors to fill (152 on GB300); > 0.
 *   split_tokens    : 0 = automatic: one CTA per SM (at most sm_count CTAs,
 *                     fewer when there are fewer tiles), the row sets' 64-token
 *                     tiles spread evenly over them, so a long row set is split
 *                     over several CTAs and a short one is not.  > 0 (a
 *                     multiple of 64) = split-KV by length: the grid gets
 *                     ceil(total tokens / split_tokens) CTAs (needs
 *                     seq_lens_host), each taking an even share of about
 *                     split_tokens tokens.
 *   plan_out        : written on success.
 *   workspace_bytes : nullable; receives plan_out->workspace_bytes.
 * Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT or MLA_ERR_UNSUPPORTED.
 */
MLA_API int mla_decode_plan(const mla_problem* problem, const int32_t* seq_lens_host,
                    int32_t sm_count, int32_t split_tokens, mla_plan* plan_out,
                    size_t* workspace_bytes);

/*
 * mla_q_absorb -- q_hat[r][h] = [bf16(W_UK[h] q_nope[r][h]) || q_rope[r][h]],
 * the weight absorption of the kv_b_proj key half into the query (the cached
 * latent is shared by all heads and is never decompressed: "GLM-4.7-Flash"
 * record, the serviceability join on the MLA family and the configuration
 * clause on kv_a_proj_with_mqa and kv_b_proj).  fp32 accumulation on the
 * tensor cores, one rounding to bf16.  r = b * Q + j.
 *   q      : bf16 [B*Q][H][256], each head [q_nope (192) || q_rope (64)]
 *            (the 256-wide query head is 192 + 64, same record, head_dim
 *            paragraph)
 *   w_uk   : bf16 [H][512][192]   (k_nope[t] = W_UK[h]^T c_kv[t])
 *   q_hat  : bf16 [B*Q][H][576]   output
 * Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT, MLA_ERR_MISALIGNED or MLA_ERR_CUDA.
 */
MLA_API int mla_q_absorb(const mla_plan* plan, const void* q, const void* w_uk, void* q_hat,
                 mla_stream_t stream);

/*
 * mla_decode_run -- the attention pass over the paged latent cache: scores of
 * every query row against every visible cached row [c_kv || k_rope], online
 * softmax and the weighted sum of latent rows ("GLM-4.7-Flash" record: the
 * MLA decode kernel class; the cache is the shared latent plus the decoupled
 * RoPE key, 576 values = 1,152 bytes per token and layer in bf16).  Each row
 * set (request and query token; or request and a group of G draft tokens,
 * see mla_plan.num_streams, whose G * H rows share every staged tile, each
 * row keeping its own causal window) is cut into contiguous 64-token tiles
 * spread over the plan's CTAs.  A row set handled by one CTA gets its final
 * o_lat and lse here; one split over several CTAs leaves normalised partials
 * (o_i, lse_i) in the workspace, which mla_combine merges.  A row (query
 * token, head) with no visible token gets o_lat = 0 and lse = -inf.
 *   q           : w_uk == NULL: bf16 [B*Q][H][576] absorbed queries q_hat;
 *                 else bf16 [B*Q][H][256] ([q_nope || q_rope]), absorbed here
 *                 through w_uk (as mla_q_absorb) into the workspace first.
 *   w_uk        : NULL, or bf16 [H][512][192].
 *   kv_cache    : MLA_KV_BF16: bf16 [num_pages][P][576];
 *                 MLA_KV_FP8_E4M3_E8M0: uint8 [num_pages][P * 594];
 *                 MLA_KV_FP4_E2M1_E8M0: uint8 [num_pages][P * 324]
 *   block_table : int32 [B][max_pages_per_seq]; entries past a request's
 *                 last page are never read
 *   seq_lens    : device int32 [B], 0 <= T_b <= max_pages_per_seq * P
 *   topk_idx    : NULL for dense; sparse: int32 [B*Q][topk_width] logical
 *                 positions of the request, -1 = masked slot (vllm API docs,
 *                 vllm.models.glm5next.common.model, Glm5NextModel.__init__:
 *                 the top-k buffer is tiled in 128 columns, padded slots
 *                 stay masked)
 *   workspace   : device buffer of workspace_bytes >= plan->workspace_bytes
 *                 (else MLA_ERR_WORKSPACE_TOO_SMALL), zeroed once before its
 *                 first use (its reserved words must stay zero; the status
 *                 word collects MLA_STATUS_* bits until cleared)
 *   o_lat       : f32 [B*Q][H][512] output (latent-space attention output)
 *   lse         : f32 [B*Q][H] output (natural-log LSE of the scaled scores)
 * Calls on one workspace must not overlap on the device.
 * Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT, MLA_ERR_MISALIGNED,
 * MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE_TOO_SMALL or MLA_ERR_CUDA.
 */
MLA_API int mla_decode_run(const mla_plan* plan, const void* q, const void* w_uk,
                   const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                   const int32_t* topk_idx, void* workspace, size_t workspace_bytes,
                   float* o_lat, float* lse, mla_stream_t stream);

/*
 * mla_combine -- completes a step after mla_decode_run (same plan, seq_lens,
 * workspace, o_lat and lse): merges the partials of every row set that was
 * split over several CTAs, lse = ln sum_i exp(lse_i), o_lat = sum_i
 * exp(lse_i - lse) o_i, into o_lat and lse; and, when w_uv is given, applies
 * the kv_b_proj value half to every row in the same call ("GLM-4.7-Flash"
 * record, configuration clause: v_head_dim 256 read back out of the 512-rank
 * latent through kv_b_proj): out[r][h] = bf16(W_UV[h]^T o_lat[r][h]).
 * Without w_uv the merge runs over all SMs (one block per row of each split
 * row set); with it, one kernel per (head, 128 output dims, row block) merges
 * its rows and projects them.  Either is launched as a programmatic
 * dependent of the kernel before it on `stream`, so its set-up (the work
 * split, the W_UV loads) overlaps that kernel's tail.  Both merges give the
 * same bits.
 *   w_uv  : NULL, or bf16 [H][512][256]
 *   out   : bf16 [B*Q][H][256] when w_uv is given, else ignored (may be NULL)
 * After the call o_lat and lse are complete for every row.  Calling it again
 * with the same workspace gives the same result.
 * Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT, MLA_ERR_MISALIGNED,
 * MLA_ERR_WORKSPACE_TOO_SMALL or MLA_ERR_CUDA.
 */
MLA_API int mla_combine(const mla_plan* plan, const int32_t* seq_lens, const void* workspace,
                size_t workspace_bytes, const void* w_uv, float* o_lat, float* lse, void* out,
                mla_stream_t stream);

/*
 * mla_decode_step -- one whole decode step in one call: mla_decode_run, then
 * mla_combine with W_UV (two kernels: the attention pass, then the merge of
 * split row sets inside the W_UV up-projection per head, a programmatic
 * dependent of the first).  Same arguments as mla_decode_run, plus
 *   w_uv : bf16 [H][512][256]
 *   out  : bf16 [B*Q][H][256] output, out[r][h] = bf16(W_UV[h]^T o_lat[r][h])
 * o_lat and lse are complete on return.  ("GLM-4.7-Flash" record: the MLA
 * decode kernel class and the configuration clause's kv_b_proj value half.)
 * Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT, MLA_ERR_MISALIGNED,
 * MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE_TOO_SMALL or MLA_ERR_CUDA.
 */
MLA_API int mla_decode_step(const mla_plan* plan, const void* q, const void* w_uk,
                    const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                    const int32_t* topk_idx, void* workspace, size_t workspace_bytes,
                    const void* w_uv, float* o_lat, float* lse, void* out, mla_stream_t stream);

/*
 * mla_cache_append -- write each request's newest token row into the paged
 * latent cache (the step before decode).  The row is the kv_a projection's
 * output for that token, [c_kv (512) || k_rope (64)] ("vllm.models.glm5next.
 * common.model", load_weights: the kv_a_proj_with_mqa output, fused into
 * fused_qkv_a_proj).  Row b goes to logical position positions[b] of request
 * b: page block_table[b][pos / P], slot pos % P.
 *   problem     : the cache's shape (batch = number of rows, page_size,
 *                 num_pages, max_pages_per_seq, kv_dtype); other fields as
 *                 for mla_decode_plan
 *   new_rows    : bf16 [batch][576], 16-byte aligned
 *   positions   : device int32 [batch]; -1 appends nothing for that request
 *   block_table : device int32 [batch][max_pages_per_seq]
 *   rope_theta  : > 0: k_rope (the last 64 values) is rotated here to the
 *                 token's position before it is stored: pair i = (x[2i],
 *                 x[2i+1]) turns by the angle pos * rope_theta^(-2i/64), in
 *                 fp32, rounded once to bf16 ("GLM-4.7-Flash" record,
 *                 configuration clause: rope_theta 1000000, qk_rope_head_dim
 *                 64).  0: the row's RoPE key is already rotated and is
 *                 stored as given.
 *   kv_cache    : written in place.  MLA_KV_BF16: the row is stored as is.
 *                 MLA_KV_FP8_E4M3_E8M0: each 32-value group is quantised on
 *                 the GPU (GLM-4.7-Flash record, engine-kernel constraint
 *                 (2): FP8 latent, one e8m0 scale per 32 e4m3 values inlined
 *                 per token): scale 2^e, e = ceil(log2(amax / 448)) clamped to
 *                 [-127, 127]; values round-to-nearest-even e4m3 of x / 2^e,
 *                 saturating at 448; an all-zero group gets scale byte 0 and
 *                 zero codes.
 *                 MLA_KV_FP4_E2M1_E8M0: the same per 16-value group with 6
 *                 for 448: e = ceil(log2(amax / 6)), codes the nearest e2m1
 *                 value of x / 2^e, ties to the even code (the sign of a value
 *                 rounding to zero kept), value 2i in the low nibble of byte i.
 *   status      : nullable device uint32; a position past the request's pages
 *                 sets MLA_STATUS_BAD_INDEX, a page id outside [0, num_pages)
 *                 MLA_STATUS_BAD_PAGE, and that row is not written.
 * Rows of one call must go to distinct slots.  Returns MLA_OK,
 * MLA_ERR_INVALID_ARGUMENT, MLA_ERR_MISALIGNED, MLA_ERR_UNSUPPORTED or
 * MLA_ERR_CUDA.
 */
MLA_API int mla_cache_append(const mla_problem* problem, const void* new_rows,
                     const int32_t* positions, const int32_t* block_table, float rope_theta,
                     void* kv_cache, uint32_t* status, mla_stream_t stream);

/*
 * mla_uv_proj -- o[r][h] = bf16(W_UV[h]^T o_lat[r][h]), the kv_b_proj value
 * half applied after attention, in latent space, as a pass of its own
 * ("GLM-4.7-Flash" record, configuration clause: v_head_dim 256 from the
 * 512-rank latent).  mla_combine does the same inside the merge.
 *   o_lat : f32 [rows][num_heads][512];  w_uv : bf16 [num_heads][512][256]
 *   out   : bf16 [rows][num_heads][256]
 * rows >= 0, 1 <= num_heads <= 128.
 */
MLA_API int mla_uv_proj(const float* o_lat, const void* w_uv, void* out, int32_t rows,
                int32_t num_heads, mla_stream_t stream);

/*
 * mla_decode_run_static -- mla_decode_run followed by the merge of
 * mla_combine (without W_UV), for callers that cannot allocate device memory
 * (the pages describe no such call; this library adds it).  Code that runs
 * while a CUDA graph is being captured, or inside a runtime that only hands
 * out the input and output buffers it owns, cannot create the workspace
 * mla_decode_run needs.  This call uses instead one fixed 16 MiB scratch
 * array that the library keeps in device memory (every GPU that loads the
 * library holds it until exit); it calls no allocator.
 *   plan            : from mla_decode_plan; plan->workspace_bytes must be at
 *                     most 16 MiB, else MLA_ERR_WORKSPACE_TOO_SMALL and
 *                     nothing is launched.
 *   q_hat ... lse   : as for mla_decode_run with w_uk == NULL (caller-owned
 *                     inputs, outputs); o_lat and lse are complete on return.
 *   status          : optional device uint32 that receives this call's
 *                     status bits (MLA_STATUS_*), or NULL.
 * Arguments are checked before anything is queued: a rejected call leaves
 * the scratch array untouched.  The scratch array is shared by all calls on
 * a device and keeps the last call's contents; each call clears the parts
 * that must start at zero on `stream` before launching.  Calls that overlap
 * on the GPU race on the array: order them on one stream.  The first call on
 * a device (and the first after that device's context is replaced) looks up
 * the array's address with that device current; make it before any stream
 * capture starts.
 */
MLA_API int mla_decode_run_static(const mla_plan* plan, const void* q_hat, const void* kv_cache,
                          const int32_t* block_table, const int32_t* seq_lens,
                          const int32_t* topk_idx, float* o_lat, float* lse, uint32_t* status,
                          mla_stream_t stream);

/* Synchronous read of the device status word (waits for `stream`). */
MLA_API int mla_get_status(const mla_plan* plan, const void* workspace, uint32_t* bits,
                   mla_stream_t stream);

/* Zero the status word (asynchronous). */
MLA_API int mla_clear_status(const mla_plan* plan, void* workspace, mla_stream_t stream);

/*
 * mla_selftest_bounded_wait -- exercise, without any fault, the bounded
 * waits every kernel of this library uses on its mbarriers.  One block of 64
 * threads waits for an mbarrier phase that nothing completes; every wait gives
 * up after limit_ns nanoseconds, after which MLA_STATUS_TIMEOUT is OR-ed into
 * *status and the time thread 0 waited is written to *waited_ns.
 *   status     : device uint32, 4-byte aligned (e.g. a plan's status word or any
 *                caller word); never read, only OR-ed.
 *   limit_ns   : 1 .. 1e9.
 *   waited_ns  : device uint64, 8-byte aligned, or NULL.
 * Returns MLA_OK once launched (asynchronous on `stream`); a null status or a
 * limit out of range gives MLA_ERR_INVALID_ARGUMENT, a misaligned pointer
 * MLA_ERR_MISALIGNED.
 */
MLA_API int mla_selftest_bounded_wait(uint32_t* status, int64_t limit_ns, uint64_t* waited_ns,
                                      mla_stream_t stream);

/* Static description of an error code; never NULL. */
MLA_API const char* mla_strerror(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
MLA_API int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
