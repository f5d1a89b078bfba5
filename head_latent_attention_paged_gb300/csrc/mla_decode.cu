// Paged MLA latent-cache decode kernel for sm_103a.
//
// One CTA per SM walks a contiguous range of 64-token tiles of the
// concatenated (request, query token) row sets ("streams").  Per tile:
//
//   producer warp : stages the 64 cached rows (576 bf16 each) in shared
//                   memory once -- TMA tiles for dense pages, 16-byte
//                   cp.async gathers for sparse top-k rows -- as nine
//                   [64 rows x 128 B] chunks in the 128-byte swizzle layout,
//                   and the stream's absorbed queries (TMA, double buffered).
//   MMA warp      : S[h, t]   = q_hat[h, :576] . row[t, :576]      (tcgen05,
//                   M = 64 head rows, N = 64 tokens, K = 576, f32 in TMEM);
//                   O^T[d, h] += sum_t row[t, d] P[h, t]            (tcgen05,
//                   M = 128 latent dims x 4, N = padded heads, K = 64 tokens,
//                   A = the same staged tile read MN-major).
//   softmax warps : online softmax in the exp2 domain on S read from TMEM
//                   (one thread per head row), P written to shared memory as
//                   bf16, lazy rescale of O^T in TMEM when the running max
//                   grows by more than 2^8, and at the end of each segment the
//                   normalised partial (o_lat, lse) written to the workspace.
//
// All heads of a request reuse each staged tile, so every cached byte is read
// from HBM once per stream.  Waits are bounded (sm103_ptx.cuh); a timeout
// sets MLA_STATUS_TIMEOUT and the CTA unwinds after draining its own copies
// and MMAs, then releases its tensor memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

namespace {

constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s per wait
constexpr float kRescaleThreshold = 8.0f;           // log2 units: rescale if max grows > 2^8
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxSmem = 232448;                    // 227 KB per CTA

// Control block placed after the data buffers in shared memory.
struct __align__(8) Ctrl {
  uint64_t full[kStages];    // producer -> MMA/softmax: tile staged
  uint64_t empty[kStages];   // MMA -> producer: stage consumed by PV
  uint64_t s_full[kStages];  // MMA -> softmax: S buffer written
  uint64_t s_free[kStages];  // softmax -> MMA: S buffer read
  uint64_t p_full[kStages];  // softmax -> MMA: P written (and O^T rescaled)
  uint64_t q_full[2];        // producer -> MMA: a stream's queries staged
  uint64_t q_empty[2];       // MMA -> producer: last QK on a Q buffer done
  uint64_t o_done;           // MMA -> softmax: one PV completed
  uint64_t o_free;           // softmax -> MMA: epilogue has read O^T
  uint64_t mma_drain;        // MMA warp's final commit
  uint64_t mask[kStages];    // per-stage live-row mask (bit t = row t live)
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t rescale_tile[kStages];
  float alpha[2][kMaxHeads];
  float l_final[kMaxHeads];
};

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  atomicOr(status, bits);
}

// Warp-uniform bounded wait: every lane waits, the warp agrees on the result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort, kWaitLimitNs);
  return __all_sync(0xffffffffu, ok);
}

struct Walker {
  int32_t s, lt, ntiles;
  __device__ __forceinline__ void init(const int32_t* prefix, int32_t S, int32_t g) {
    int32_t lo = 0, hi = S;
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if (prefix[mid] <= g) lo = mid; else hi = mid;
    }
    s = lo;
    lt = g - prefix[s];
    ntiles = prefix[s + 1] - prefix[s];
  }
  __device__ __forceinline__ void next(const int32_t* prefix, int32_t S) {
    if (++lt >= ntiles) {
      lt = 0;
      do { ++s; } while (s < S && prefix[s + 1] == prefix[s]);
      ntiles = (s < S) ? prefix[s + 1] - prefix[s] : 0;
    }
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t tmem_cols(int NP) { return (128 + 4 * NP) <= 256 ? 256u : 512u; }

}  // namespace

DecodeLayout decode_layout(int heads, int heads_pad, int num_streams, int mode) {
  (void)mode;
  DecodeLayout L;
  const int groups = (heads + 7) / 8;
  L.q_group_bytes = groups * 1024;
  L.q_buf_bytes = kChunks * L.q_group_bytes;
  L.off_q = 0;
  const int rest = kStages * kTileBytes + kStages * heads_pad * 128 +
                   static_cast<int>(sizeof(Ctrl)) + (num_streams + 1) * 4 + 1024;
  // Two query buffers when they fit, so the next stream's queries load
  // while the current one computes.  The M=64 QK MMA reads 64 rows from each
  // Q chunk start; rows >= H land in the following memory (later chunks or
  // the stages) and only feed S rows nobody reads.
  L.q_bufs = (2 * L.q_buf_bytes + rest <= kMaxSmem) ? 2 : 1;
  L.off_stage = L.q_bufs * L.q_buf_bytes;
  L.off_p = L.off_stage + kStages * kTileBytes;
  L.off_ctrl = L.off_p + kStages * heads_pad * 128;
  L.total = L.off_ctrl + static_cast<int>(sizeof(Ctrl)) + (num_streams + 1) * 4 + 1024;
  return L;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map,
                      const __grid_constant__ CUtensorMap q_map, const DecodeParams p,
                      const DecodeLayout L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L.off_q;
  uint8_t* sStage = smem + L.off_stage;
  uint8_t* sP = smem + L.off_p;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + L.off_ctrl);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + L.off_ctrl + sizeof(Ctrl));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_streams;
  const int H = p.heads;
  const int NP = p.heads_pad;
  const int QB = L.q_bufs;
  const int max_tokens = p.max_pages * p.page_size;
  volatile int32_t* abort_flag = &ctrl->abort_flag;

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctrl->full[i], kMode == kModeSparseBf16 ? 33 : 1);
      mbar_init(&ctrl->empty[i], 1);
      mbar_init(&ctrl->s_full[i], 1);
      mbar_init(&ctrl->s_free[i], kSoftmaxWarps);
      mbar_init(&ctrl->p_full[i], kSoftmaxWarps);
      ctrl->rescale_tile[i] = -1;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctrl->q_full[i], 1);
      mbar_init(&ctrl->q_empty[i], 1);
    }
    mbar_init(&ctrl->o_done, 1);
    mbar_init(&ctrl->o_free, kSoftmaxWarps);
    mbar_init(&ctrl->mma_drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctrl->tmem_base, tmem_cols(NP));
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    if constexpr (kMode == kModeDenseBf16) prefetch_tmap(&kv_map);
    prefetch_tmap(&q_map);
  }
  // tiles per stream (stream lengths from the device seq_lens)
  for (int s = tid; s < S; s += kThreads) {
    const int b = s / p.q_len, j = s - b * p.q_len;
    const int32_t len = stream_len(p.seq_lens[b], p.q_len, j, p.causal, p.topk_width, max_tokens);
    prefix[s + 1] = (len + kTile - 1) / kTile;
  }
  // P buffers start at zero: rows of padded heads are never written again
  for (int i = tid; i < kStages * NP * 128 / 16; i += kThreads)
    reinterpret_cast<uint4*>(sP)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (warp == 0) {   // exclusive prefix sum of tiles over streams
    int32_t carry = 0;
    if (lane == 0) prefix[0] = 0;
    for (int base = 0; base < S; base += 32) {
      const int s = base + lane;
      int32_t v = (s < S) ? prefix[s + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (s < S) prefix[s + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int32_t total = prefix[S];
  const int32_t c = blockIdx.x;
  const int32_t g0 = static_cast<int32_t>((static_cast<int64_t>(c) * total) / p.num_ctas);
  const int32_t g1 = static_cast<int32_t>((static_cast<int64_t>(c + 1) * total) / p.num_ctas);
  const int32_t ntiles = g1 - g0;
  const uint32_t tmem = ctrl->tmem_base;

  if (ntiles > 0) {
    if (warp == kProducerWarp) {
      // ============================================================ producer
      const uint64_t pol = l2_policy_evict_first();
      Walker wk;
      wk.init(prefix, S, g0);
      int32_t issued = 0, seg = -1;
      bool failed = false;
      for (int32_t i = 0; i < ntiles; ++i) {
        const int stage = i & 1;
        const bool first = (i == 0) || (wk.lt == 0);
        const int b = wk.s / p.q_len, j = wk.s - b * p.q_len;
        if (first) {
          ++seg;
          const int qb = seg % QB;
          if (seg >= QB && !warp_wait(&ctrl->q_empty[qb], ((seg / QB) - 1) & 1, abort_flag)) {
            failed = true;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&ctrl->q_full[qb], static_cast<uint32_t>(kChunks * H * 128));
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
              tma_load_2d(sQ + qb * L.q_buf_bytes + ch * L.q_group_bytes, &q_map, &ctrl->q_full[qb],
                          ch * kChunkElems, wk.s * H, 0ull);
          }
        }
        if (i >= 2 && !warp_wait(&ctrl->empty[stage], ((i >> 1) - 1) & 1, abort_flag)) {
          failed = true;
          break;
        }
        uint8_t* dst = sStage + stage * kTileBytes;
        if constexpr (kMode == kModeDenseBf16) {
          if (lane == 0) {
            const int32_t tok0 = wk.lt * kTile;
            const int32_t len = stream_len(p.seq_lens[b], p.q_len, j, p.causal, 0, max_tokens);
            const int32_t page =
                p.block_table[static_cast<int64_t>(b) * p.max_pages + tok0 / p.page_size];
            const int32_t nvalid = min(kTile, len - tok0);
            uint64_t mask = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
            const bool ok = page >= 0 && page < p.num_pages;
            if (!ok) {
              mask = 0;
              set_status(p.status, MLA_STATUS_BAD_PAGE);
            }
            ctrl->mask[stage] = mask;
            if (ok) {
              mbar_arrive_expect_tx(&ctrl->full[stage], kTileBytes);
              const int32_t row0 = page * p.page_size + (tok0 % p.page_size);
#pragma unroll
              for (int ch = 0; ch < kChunks; ++ch)
                tma_load_2d(dst + ch * kChunkBytes, &kv_map, &ctrl->full[stage], ch * kChunkElems,
                            row0, pol);
            } else {
              mbar_arrive(&ctrl->full[stage]);
            }
          }
        } else if constexpr (kMode == kModeSparseBf16) {
          const int32_t T = min(max(p.seq_lens[b], 0), max_tokens);
          const int32_t window = p.causal ? min(max(T - p.q_len + j + 1, 0), T) : T;
          const int32_t* idx_row =
              p.topk_idx + static_cast<int64_t>(wk.s) * p.topk_width + wk.lt * kTile;
          const uint8_t* src[2];
          bool valid[2];
          uint32_t bad = 0;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int32_t idx = idx_row[lane + 32 * k];
            bool v = idx >= 0 && idx < window;
            if (!v && idx != -1) bad |= MLA_STATUS_BAD_INDEX;
            int32_t page = -1;
            if (v) {
              page = p.block_table[static_cast<int64_t>(b) * p.max_pages + idx / p.page_size];
              if (page < 0 || page >= p.num_pages) {
                v = false;
                bad |= MLA_STATUS_BAD_PAGE;
              }
            }
            valid[k] = v;
            src[k] = v ? p.kv + (static_cast<int64_t>(page) * p.page_size + idx % p.page_size) *
                                    (kDqk * 2)
                       : p.kv;
          }
          if (bad) set_status(p.status, bad);
          const uint32_t lo = __ballot_sync(0xffffffffu, valid[0]);
          const uint32_t hi = __ballot_sync(0xffffffffu, valid[1]);
          for (int r = 0; r < kTile; ++r) {
            const uint8_t* s_row = reinterpret_cast<const uint8_t*>(__shfl_sync(
                0xffffffffu, reinterpret_cast<unsigned long long>(r < 32 ? src[0] : src[1]), r & 31));
            const uint32_t nbytes = (((r < 32 ? lo : hi) >> (r & 31)) & 1u) ? 16u : 0u;
#pragma unroll
            for (int q = 0; q < 3; ++q) {
              const int piece = lane + 32 * q;   // 16-byte piece of the row, 0..71
              if (piece < kDqk * 2 / 16) {
                const int ch = piece >> 3, w16 = piece & 7;
                cp_async_16(dst + ch * kChunkBytes + r * 128 + ((w16 ^ (r & 7)) << 4),
                            s_row + piece * 16, nbytes);
              }
            }
          }
          if (lane == 0) ctrl->mask[stage] = (static_cast<uint64_t>(hi) << 32) | lo;
          cp_async_mbar_arrive(&ctrl->full[stage]);
          if (lane == 0) mbar_arrive(&ctrl->full[stage]);
        }
        __syncwarp();
        ++issued;
        wk.next(prefix, S);
      }
      if (failed && lane == 0) {
        set_status(p.status, MLA_STATUS_TIMEOUT);
        ctrl->abort_flag = 1;
      }
      // drain: everything this warp issued has landed before the CTA exits
      if constexpr (kMode == kModeSparseBf16) asm volatile("cp.async.wait_all;" ::: "memory");
      if (lane == 0) {
        for (int32_t i = max(0, issued - 2); i < issued; ++i)
          (void)mbar_wait(&ctrl->full[i & 1], (i >> 1) & 1, nullptr, kWaitLimitNs);
        for (int32_t k = max(0, seg - QB + 1); k <= seg; ++k)   // last use of each Q buffer
          (void)mbar_wait(&ctrl->q_full[k % QB], (k / QB) & 1, nullptr, kWaitLimitNs);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ================================================================= MMA
      const uint32_t idesc_qk = make_idesc_bf16(64, 64, false, false);
      const uint32_t idesc_pv = make_idesc_bf16(128, static_cast<uint32_t>(NP), true, false);
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t st_base = smem_u32(sStage);
      const uint32_t p_base = smem_u32(sP);
      Walker wk;
      wk.init(prefix, S, g0);
      int32_t seg = -1;
      bool failed = false;
      bool prev_first = false;
      int32_t prev_seg = 0;
      // PV of local tile k; `first`: k opens a segment, `kseg`: its index
      auto issue_pv = [&](int32_t k, bool first, int32_t kseg) -> bool {
        const int st = k & 1;
        if (!warp_wait(&ctrl->p_full[st], (k >> 1) & 1, abort_flag)) return false;
        if (first && kseg > 0 && !warp_wait(&ctrl->o_free, (kseg - 1) & 1, abort_flag)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = st_base + st * kTileBytes;
          const uint32_t b0 = p_base + st * NP * 128;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = make_smem_desc(a0 + (2 * mt) * kChunkBytes + kk * 2048,
                                                 kChunkBytes, 1024, kSmemLayoutSW128);
              const uint64_t bd = make_smem_desc(b0 + kk * 32, 16, 1024, kSmemLayoutSW128);
              mma_bf16_ss(tmem + 128 + mt * NP, ad, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
            }
          }
          mma_commit(&ctrl->empty[st]);
          mma_commit(&ctrl->o_done);
        }
        __syncwarp();
        return true;
      };
      for (int32_t i = 0; i < ntiles; ++i) {
        const int stage = i & 1;
        const bool first = (i == 0) || (wk.lt == 0);
        const bool last = (i == ntiles - 1) || (wk.lt == wk.ntiles - 1);
        if (first) ++seg;
        const int qb = seg % QB;
        if (first && !warp_wait(&ctrl->q_full[qb], (seg / QB) & 1, abort_flag)) { failed = true; break; }
        if (!warp_wait(&ctrl->full[stage], (i >> 1) & 1, abort_flag)) { failed = true; break; }
        if (i >= 2 && !warp_wait(&ctrl->s_free[stage], ((i >> 1) - 1) & 1, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t s_col = tmem + stage * 64;
          const uint32_t a0 = q_base + qb * L.q_buf_bytes;
          const uint32_t b0 = st_base + stage * kTileBytes;
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = make_smem_desc(a0 + ch * L.q_group_bytes + k * 32, 16, 1024, kSmemLayoutSW128);
              const uint64_t bd = make_smem_desc(b0 + ch * kChunkBytes + k * 32, 16, 1024, kSmemLayoutSW128);
              mma_bf16_ss(s_col, ad, bd, idesc_qk, (ch | k) ? 1u : 0u);
            }
          }
          mma_commit(&ctrl->s_full[stage]);
          if (last) mma_commit(&ctrl->q_empty[qb]);
        }
        __syncwarp();
        if (i > 0 && !issue_pv(i - 1, prev_first, prev_seg)) { failed = true; break; }
        prev_first = first;
        prev_seg = seg;
        wk.next(prefix, S);
      }
      if (!failed && !issue_pv(ntiles - 1, prev_first, prev_seg)) failed = true;
      if (failed && lane == 0) {
        set_status(p.status, MLA_STATUS_TIMEOUT);
        ctrl->abort_flag = 1;
      }
      // drain: every issued MMA completes before tensor memory is released
      if (lane == 0) {
        mma_commit(&ctrl->mma_drain);
        (void)mbar_wait(&ctrl->mma_drain, 0, nullptr, kWaitLimitNs);
      }
      __syncwarp();
    } else {
      // ============================================================ softmax
      const int w = warp;                 // 0..3: TMEM lanes [32w, 32w+32)
      const int h = w * 16 + lane;        // head row owned (M=64 accumulator layout)
      const bool owner = lane < 16 && h < H;
      const bool warp_has_heads = w * 16 < H;
      const uint32_t lane_base = static_cast<uint32_t>(w * 32) << 16;
      float m_used = -INFINITY, l_run = 0.f;
      Walker wk;
      wk.init(prefix, S, g0);
      bool failed = false;
      for (int32_t i = 0; i < ntiles; ++i) {
        const int stage = i & 1;
        const bool first = (i == 0) || (wk.lt == 0);
        const bool last = (i == ntiles - 1) || (wk.lt == wk.ntiles - 1);
        bool ok = !failed && warp_wait(&ctrl->full[stage], (i >> 1) & 1, abort_flag);
        const uint64_t mask = ctrl->mask[stage];
        ok = ok && warp_wait(&ctrl->s_full[stage], (i >> 1) & 1, abort_flag);
        float x[64];
        if (ok) {
          tc_fence_after();
          if (warp_has_heads) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + stage * 64, r);
#pragma unroll
            for (int t = 0; t < 32; ++t) x[t] = __uint_as_float(r[t]);
            tmem_ld32(tmem + lane_base + stage * 64 + 32, r);
#pragma unroll
            for (int t = 0; t < 32; ++t) x[32 + t] = __uint_as_float(r[t]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->s_free[stage]);
          if (owner) {
            float mt = -INFINITY;
#pragma unroll
            for (int t = 0; t < 64; ++t) {
              x[t] = ((mask >> t) & 1ull) ? x[t] * p.scale_log2 : -INFINITY;
              mt = fmaxf(mt, x[t]);
            }
            float alpha = 1.f;
            if (first) {
              m_used = mt;
              l_run = 0.f;
            } else if (mt > m_used + kRescaleThreshold) {
              alpha = exp2f(m_used - mt);
              m_used = mt;
              l_run *= alpha;
              ctrl->rescale_tile[stage] = i;
            }
            const float ref = (m_used == -INFINITY) ? 0.f : m_used;
            uint8_t* prow = sP + stage * NP * 128 + h * 128;
            float lsum = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              uint32_t u[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                u[e] = pack_bf16x2(exp2f(x[c8 * 8 + 2 * e] - ref), exp2f(x[c8 * 8 + 2 * e + 1] - ref));
                const __nv_bfloat162 v2 = *reinterpret_cast<__nv_bfloat162*>(&u[e]);
                lsum += __low2float(v2) + __high2float(v2);
              }
              *reinterpret_cast<uint4*>(prow + ((c8 ^ (h & 7)) << 4)) = make_uint4(u[0], u[1], u[2], u[3]);
            }
            l_run += lsum;
            ctrl->alpha[i & 1][h] = alpha;
          }
          if constexpr (kMode != kModeSparseBf16) {
            // Dead rows (tail slots, bad pages): P is 0 there but 0 * NaN
            // would poison the PV sum, so zero their latent values.
            if (mask != ~0ull) {
              uint8_t* tile = sStage + stage * kTileBytes;
              for (int u = tid; u < kTile * 64; u += 128) {
                const int row = u >> 6, piece = u & 63;
                if (!((mask >> row) & 1ull))
                  *reinterpret_cast<uint4*>(tile + (piece >> 3) * kChunkBytes + row * 128 +
                                            ((piece & 7) << 4)) = make_uint4(0, 0, 0, 0);
              }
            }
          }
        }
        if (named_bar_or(1, 128, !ok)) { failed = true; break; }
        if (!first && ctrl->rescale_tile[stage] == i) {
          // every earlier PV has completed before O^T is rescaled in place
          ok = warp_wait(&ctrl->o_done, (i - 1) & 1, abort_flag);
          failed = !ok;
          if (ok) {
            tc_fence_after();
            for (int mt = 0; mt < 4; ++mt) {
              for (int hb = 0; hb < H; hb += 16) {
                uint32_t v[16];
                const uint32_t addr = tmem + lane_base + 128 + mt * NP + hb;
                tmem_ld16(addr, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const int hh = hb + e;
                  const float a = hh < H ? ctrl->alpha[i & 1][hh] : 1.f;
                  v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
                }
                tmem_st16(addr, v);
              }
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->p_full[stage]);
        if (last) {
          // ---- segment epilogue: normalised partial o_lat and its lse
          ok = ok && warp_wait(&ctrl->o_done, i & 1, abort_flag);
          const int32_t slot = wk.s + c;
          if (ok && owner) {
            ctrl->l_final[h] = l_run;
            p.part_lse[static_cast<int64_t>(slot) * H + h] =
                l_run > 0.f ? (m_used + log2f(l_run)) * kLn2 : -INFINITY;
          }
          if (named_bar_or(1, 128, !ok || failed)) { failed = true; break; }
          tc_fence_after();
          float* out = p.part_o + static_cast<int64_t>(slot) * H * kDc;
          for (int mt = 0; mt < 4; ++mt) {
            const int d = mt * 128 + w * 32 + lane;
            for (int hb = 0; hb < H; hb += 16) {
              uint32_t v[16];
              tmem_ld16(tmem + lane_base + 128 + mt * NP + hb, v);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int hh = hb + e;
                if (hh < H) {
                  const float lf = ctrl->l_final[hh];
                  out[static_cast<int64_t>(hh) * kDc + d] = lf > 0.f ? __uint_as_float(v[e]) / lf : 0.f;
                }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->o_free);
        }
        wk.next(prefix, S);
      }
      if (failed && lane == 0) {
        set_status(p.status, MLA_STATUS_TIMEOUT);
        ctrl->abort_flag = 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols(NP));
  }
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap* kv_map,
                          const CUtensorMap* q_map, int mode, cudaStream_t stream) {
  const DecodeLayout L = decode_layout(p.heads, p.heads_pad, p.num_streams, mode);
  dim3 grid(p.num_ctas), block(kThreads);
  cudaError_t err;
  switch (mode) {
    case kModeDenseBf16:
      err = cudaFuncSetAttribute(mla_decode_kernel<kModeDenseBf16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
      if (err != cudaSuccess) return err;
      mla_decode_kernel<kModeDenseBf16><<<grid, block, L.total, stream>>>(*kv_map, *q_map, p, L);
      break;
    case kModeSparseBf16:
      err = cudaFuncSetAttribute(mla_decode_kernel<kModeSparseBf16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
      if (err != cudaSuccess) return err;
      mla_decode_kernel<kModeSparseBf16><<<grid, block, L.total, stream>>>(*kv_map, *q_map, p, L);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int decode_smem_bytes(int heads, int heads_pad, int num_streams, int mode) {
  return decode_layout(heads, heads_pad, num_streams, mode).total;
}

}  // namespace mla
