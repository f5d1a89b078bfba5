// Paged MLA latent-cache decode kernel for sm_103a.
//
// One CTA per SM walks a contiguous range of 64-token tiles of the
// concatenated row sets ("streams"): one per (request, query token), or, in
// the multi-token mode (several draft tokens over a bf16, FP4 or FP8 cache),
// one per group of G draft tokens of a request whose G * H rows share every
// staged tile.  Per tile:
//
//   producer warp : stages the 64 cached rows (576 bf16 each) in shared
//                   memory once -- TMA tiles for dense pages (for sparse
//                   top-k rows, four gather warps issue TMA gather4 loads,
//                   16 rows each) -- as nine [64 rows x 128 B] chunks in the
//                   128-byte swizzle layout, three tiles in flight.  FP8 /
//                   FP4 caches: one bulk copy of the tile's quantised rows
//                   (594 or 324 bytes), FP8 into a ring of two raw slots
//                   beside two bf16 stages, FP4 into the tail of the bf16
//                   stage it becomes, and
//   dequant warps : (FP8 / FP4) turn each row's codes and e8m0 scales into
//                   bf16 values code * 2^(scale - 127), exactly, written as
//                   the swizzled bf16 tile (FP8 in two phases, the first
//                   published early for QK; FP4 in place: first the chunks
//                   below the raw bytes, then, once every dequant warp holds
//                   the rest of its groups in registers, the chunks over
//                   them); rows with no live token become zeros.
//   QK issuers    : S[h, t] = q_hat[h, :576] . row[t, :576]          (tcgen05,
//                   M = 64 rows with q_hat's latent part read from TMEM and
//                   its RoPE part from shared memory, N = 64 tokens from
//                   shared memory, K = 576, f32 in TMEM), split into two
//                   halves of K (two S accumulators) where TMEM allows.
//   softmax warps : online softmax in the exp2 domain on S read from TMEM
//                   (two lanes per row; in the multi-token mode each row
//                   masked past its own draft's causal window), P written to
//                   shared memory as bf16, lazy rescale of O^T in TMEM when
//                   the running max grows by more than 2^8; then four of
//                   their lanes issue O^T[d, h] += sum_t row[t, d] P[h, t]
//                   (tcgen05, M = 128 latent dims x 4, N = padded rows, K =
//                   64 tokens, A = the staged tile read MN-major).  At a
//                   stream change they write the next stream's q_hat into
//                   TMEM, and at the end of each segment the normalised
//                   result (or, for a stream split over several CTAs, a
//                   partial plus its lse, merged by the combine kernel that
//                   follows this one).
//
// All heads of a row set reuse each staged tile, so every cached byte is read
// from HBM once per row set.  Waits are bounded (sm103_ptx.cuh); a timeout
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
constexpr int kDequantWarp0 = 6;    // FP8 / FP4 modes: warps 6..11 dequantise
constexpr int kDequantWarps = 6;
constexpr int kGroupSets = kDequantWarps * 32 / kTile;   // threads per row in the dequant
constexpr int kFp8Items = 36;       // FP8 dequant work items per tile: 18 groups x 2 row halves
// P (bf16 [padded heads][64 tokens], the B operand of PV) lives in the RoPE
// chunk of its own tile's stage: QK(i) is the only reader of that chunk and
// P(i) is written after S(i) is complete, so every stage carries its own P.
constexpr int kPChunkOffset = (kChunks - 1) * kChunkBytes;

constexpr int kPvLanes = 4;         // PV issuers, one per 128-dim block of O^T

constexpr int kGatherWarp0 = 6;     // sparse mode: warps 6..9 gather top-k rows
constexpr int kGatherWarps = 4;
constexpr int kGatherRows = kTile / kGatherWarps;   // 16 rows per gather warp

template <int kMode>
struct ModeTraits {
  static constexpr bool kFp8 = kMode == kModeDenseFp8 || kMode == kModeDenseFp8Multi;
  static constexpr bool kFp4 = kMode == kModeDenseFp4 || kMode == kModeDenseFp4Multi;
  static constexpr bool kQuant = kFp8 || kFp4;   // quantised bytes, dequantised in the CTA
  static constexpr int kRowBytes = kFp4 ? kFp4RowBytes : kFp8RowBytes;    // quantised row
  static constexpr int kRawTileBytes = kTile * kRowBytes;
  static constexpr bool kSparse = kMode == kModeSparseBf16;
  static constexpr bool kMulti =
      kMode == kModeDenseMulti || kMode == kModeDenseFp4Multi || kMode == kModeDenseFp8Multi;
  // dense bf16 staging (TMA tiles, dead rows zeroed by the softmax warps)
  static constexpr bool kDenseBf16 = kMode == kModeDenseBf16 || kMode == kModeDenseMulti;
  // the first softmax warp whose TMEM lanes hold rows: row r of a row set is
  // M-row 16 * kRowWarp0 + r of the QK accumulator
  static constexpr int kRowWarp0 = kMulti ? 1 : 2;
  // Split QK: two issuers each take half of QK's K range into an S
  // accumulator of their own (S = S_a + S_b, summed by the softmax): latent
  // chunks 0-3 and the first half of the RoPE chunk into S_a, chunks 4-7 and
  // the second half into S_b.  A tcgen05.mma costs its issuing thread a
  // fixed time whatever its shape, and MMAs from different threads overlap
  // in the tensor pipe, whether the threads are lanes of one warp or sit in
  // different warps (two warps overlap better).  The dense one-token bf16
  // kernel issues the halves from two warps; the one-token FP8, FP4 and
  // sparse kernels, whose dequant or gather warps take the register file,
  // from two lanes of the MMA warp.  The multi-token kernels keep one QK
  // issuer: their O^T (48 padded rows) leaves no TMEM for a second S.
  static constexpr bool kSplitQK = kMode == kModeDenseBf16;
  static constexpr bool kSplitQKLanes =
      kMode == kModeDenseFp8 || kMode == kModeDenseFp4 || kMode == kModeSparseBf16;
  static constexpr bool kSplitS = kSplitQK || kSplitQKLanes;
  static constexpr int kQkLanes = kSplitQKLanes ? 2 : 1;   // QK issuing lanes of the MMA warp
  // q_hat's RoPE part is a shared-memory A operand (multi-token and split-QK
  // kernels), so that TMEM holds the extra accumulator.
  static constexpr bool kQRopeSmem = kMulti || kSplitS;
  // TMEM columns: q_hat (all 576 values, or the 512 latent ones when the
  // RoPE part is a shared-memory operand), S (64; two of them when QK is
  // split), O^T (4 x heads_pad)
  static constexpr uint32_t kColQ = 0;
  static constexpr uint32_t kColS = kQRopeSmem ? 256 : 288;
  static constexpr uint32_t kColS2 = kColS + 64;
  static constexpr uint32_t kColO = kColS + (kSplitS ? 128 : 64);
  static constexpr int kQTmemChunks = kQRopeSmem ? kChunks - 1 : kChunks;
  static constexpr int kRoleWarps = kQuant ? kDequantWarp0 + kDequantWarps
                                   : kSparse ? kGatherWarp0 + kGatherWarps
                                             : 6;
  static constexpr int kQk2Warp = kRoleWarps;   // second QK issuer (dense one-token kernel)
  // PV issuers, as measured per kernel: lanes 0-1 of softmax warps 0 and 1
  // (which hold no rows) in the one-token FP8 kernel; lanes 0-3 of softmax
  // warp 0 in the multi-token kernels (whose warps 1-3 hold rows); lane 0 of
  // each softmax warp in the one-token bf16, FP4 and sparse kernels
  static constexpr bool kPvTwoWarps = kMode == kModeDenseFp8;
  static constexpr bool kPvOneWarp = (kFp8 || kMulti) && !kPvTwoWarps;
  static constexpr int kThreads = 32 * (kRoleWarps + (kSplitQK ? 1 : 0));
  // FP8: two bf16 stages and a two-slot ring of raw tiles beside them.
  // FP4: three bf16 stages, each raw tile landing in the last
  // kRawTileBytes of the stage it is dequantised into.
  static constexpr bool kRawRing = kFp8;
  static constexpr int kNumStages = kRawRing ? kFp8Stages : kStages;   // bf16 tiles in flight
  // q_hat rows loaded by both lanes of a pair (measured faster in these
  // kernels; the FP8, sparse and quantised multi-token ones keep one lane
  // per row)
  static constexpr bool kQLoadSplit =
      kMode == kModeDenseBf16 || kMode == kModeDenseFp4 || kMode == kModeDenseMulti;
  static constexpr int kQBatch = kThreads > 256 ? (kQRopeSmem ? 2 : 3) : (kQRopeSmem ? 4 : 5);   // q_hat chunks per load batch
  static constexpr int kRawSlots = kRawRing ? kFp8RawSlots : kStages;
  static constexpr int kRawOffset = kTileBytes - kRawTileBytes;
  static_assert(kRawSlots >= 1 && kRawOffset % 16 == 0, "raw tiles need 16-byte aligned slots");
};
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s per wait
constexpr float kRescaleThreshold = 8.0f;           // log2 units: rescale if max grows > 2^8
constexpr float kLn2 = 0.6931471805599453f;

// Tensor memory columns (512 allocated): q_hat as the QK A operand (M=64
// layout, 576 bf16 = 288 columns; 256 in the multi-token mode), S (64 token
// columns), O^T (4 x padded rows).
constexpr uint32_t kTmemCols = 512;
constexpr int kQRopeBytes = 64 * 128;   // RoPE part of q_hat as a shared-memory operand, 64 M-rows x 128 B

// Control block placed after the data buffers in shared memory.
struct __align__(8) Ctrl {
  uint64_t full[kStages];    // producer -> MMA/softmax: tile staged
  uint64_t empty[kStages];   // PV -> producer: stage consumed
  uint64_t s_full;           // MMA -> softmax: S written
  uint64_t s_free;           // softmax -> MMA: S read
  uint64_t q_ready;          // softmax -> MMA: a stream's q_hat is in TMEM
  uint64_t o_done[2];        // PV(j) completed, on o_done[j % 2]
  uint64_t mma_drain[3];     // the issuers' final commits (QK, PV, second QK)
  uint64_t mask[kStages];    // per-stage live-row mask (bit t = row t live)
  uint64_t dq_part[kStages];  // FP8: dequant -> QK, a stage's first phase converted
  uint64_t raw_full[kStages];       // FP8 / FP4: producer -> dequant, bytes landed
  uint64_t raw_empty[kFp8RawSlots]; // FP8: dequant -> producer, raw slot consumed
  uint64_t raw_mask[kFp8RawSlots];  // FP8: live-row mask of the raw tile
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t rescale_tile[2];
  float alpha[2][kMaxRows];
  float l_final[kMaxRows];
};

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  atomicOr(status, bits);
}

// Warp-uniform bounded wait: every lane waits, the warp agrees on the result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort, kWaitLimitNs);
  return __all_sync(0xffffffffu, ok);
}

// First global tile (in stream order) whose cost position is >= u; tile and
// cost prefixes over the S streams, U = cost[S], sc a stream's fixed cost.
__device__ __forceinline__ int32_t first_tile_at(const int32_t* tiles, const int32_t* cost,
                                                 int32_t S, int32_t u, int32_t sc) {
  if (u >= cost[S]) return tiles[S];
  int32_t lo = 0, hi = S;                 // largest s with cost[s] <= u
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (cost[mid] <= u) lo = mid; else hi = mid;
  }
  const int32_t off = u - cost[lo];
  const int32_t k = off <= sc ? 0 : (off - sc + kTileCost - 1) / kTileCost;
  return (k < tiles[lo + 1] - tiles[lo]) ? tiles[lo] + k : tiles[lo + 1];
}

// The pages behind one 64-token tile.  A tile is one piece when pages hold
// 64 or more tokens; with 16- or 32-token pages (the compressed-layer page
// block size: block_size / compress_ratio) it spans 64 / P pages.  Lane k <
// npieces resolves piece k; the result is gathered in every lane.
struct TilePieces {
  int32_t npieces;     // pieces in the tile (1, 2 or 4)
  int32_t rows;        // rows per piece (min(P, 64))
  int32_t nvalid;      // live rows of the tile
  uint32_t ok;         // bit k: piece k holds live rows and a valid page
  int32_t page[4];     // physical page of each piece
  int32_t slot0;       // first slot of the tile within its page (P >= 64)
  uint32_t bad;        // status bits to report
};

__device__ __forceinline__ TilePieces describe_tile(const DecodeParams& p, int b, int j,
                                                    int32_t lt, int lane, int32_t max_tokens) {
  TilePieces t;
  const int32_t tok0 = lt * kTile;
  t.rows = min(p.page_size, kTile);
  t.npieces = kTile / t.rows;
  t.slot0 = tok0 % p.page_size;   // 0 unless P > 64
  // the length and the block-table entry are loaded together (one memory
  // latency); a piece past the request's last page reads an in-bounds entry
  // of its row and ignores it
  const int32_t seq_len = p.seq_lens[b];
  int32_t page = -1;
  if (lane < t.npieces) {
    const int32_t pi = min((tok0 + lane * t.rows) / p.page_size, p.max_pages - 1);
    page = p.block_table[static_cast<int64_t>(b) * p.max_pages + pi];
  }
  const int32_t len = stream_len(seq_len, p.q_len, j, p.causal, 0, max_tokens);
  t.nvalid = min(kTile, len - tok0);
  const bool live = lane < t.npieces && lane * t.rows < t.nvalid;
  const bool good = live && page >= 0 && page < p.num_pages;
  t.ok = __ballot_sync(0xffffffffu, good);
  t.bad = (__ballot_sync(0xffffffffu, live && !good) != 0u) ? MLA_STATUS_BAD_PAGE : 0u;
#pragma unroll
  for (int k = 0; k < 4; ++k) t.page[k] = __shfl_sync(0xffffffffu, page, k);
  return t;
}

// Live-row mask of a tile: rows below nvalid in pieces with a valid page.
__device__ __forceinline__ uint64_t tile_mask(const TilePieces& t) {
  uint64_t m = t.nvalid >= 64 ? ~0ull : ((1ull << t.nvalid) - 1ull);
  uint64_t pm = 0;
  for (int k = 0; k < t.npieces; ++k)
    if ((t.ok >> k) & 1u) pm |= (t.rows >= 64 ? ~0ull : ((1ull << t.rows) - 1ull)) << (k * t.rows);
  return m & pm;
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

// 2^x with the hardware approximation (ex2.approx.ftz: 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// PV into block mt of O^T (latent dims 128 mt .. 128 mt + 127): O^T[mt]
// (+)= V^T[mt] P^T over one staged tile, K = 64 tokens in 4 MMAs.  a0 / b0
// are the descriptors of the tile's chunk 0 (read MN-major) and of its P.
__device__ __forceinline__ void issue_pv_block(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                               uint32_t idesc, int mt, bool first) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_bf16_ss(d_tmem, a0 + ((2 * mt * kChunkBytes + kk * 2048) >> 4), b0 + ((kk * 32) >> 4),
                idesc, (first && kk == 0) ? 0u : 1u);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Write a row set's absorbed queries (q_hat rows q_rows .. q_rows + nrows)
// as the QK A operand.  Row r of the set is M-row 16 * kRowWarp0 + r of the
// M=64 layout, which lives in TMEM lane (m/16)*32 + m%16: lanes 0-15 of
// softmax warp kRowWarp0 + r/16.  Heads of a one-token row set sit in rows
// 32 + h (warps 2 and 3 only, so warps 0 and 1 leave their SM sub-partitions
// to the producer and MMA warps); a multi-token row set (up to 48 rows)
// starts at M-row 16 (warps 1-3).  The 512 latent values go to TMEM, packed
// two per column, and the 64 RoPE values to a shared-memory operand (row m
// at m * 128 bytes, 16-byte units swizzled by m % 8).  Every softmax warp
// calls this; M-rows of warps kRowWarp0.. without a row get zeros, the
// M-rows below are not written (their S rows are never read).  Global loads
// go in batches of kBatch chunks of 64 values to keep many in flight (fewer
// in the kernels whose thread count leaves fewer registers per thread).
// One thread per row (lanes 0-15): the kernels where that measured faster.
template <int kRowWarp0, bool kRopeSmem, int kBatch>
__device__ __forceinline__ void load_q(const uint16_t* q_rows, int nrows, uint32_t taddr_lane,
                                       uint8_t* q_rope, int lane, int w) {
  constexpr int kTmemChunks = kRopeSmem ? kChunks - 1 : kChunks;
  const int r = (w - kRowWarp0) * 16 + (lane & 15);
  const bool live = w >= kRowWarp0 && lane < 16 && r < nrows;
  const uint4* src = reinterpret_cast<const uint4*>(q_rows + static_cast<int64_t>(live ? r : 0) * kDqk);
  if (w >= kRowWarp0) {
#pragma unroll
    for (int cb = 0; cb < kTmemChunks; cb += kBatch) {
      const int n = (kTmemChunks - cb) < kBatch ? (kTmemChunks - cb) : kBatch;
      uint4 v[kBatch][8];
#pragma unroll
      for (int c = 0; c < kBatch; ++c)
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[c][q] = (live && c < n) ? __ldg(src + (cb + c) * 8 + q) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < kBatch; ++c) {
        if (c < n) {
          uint32_t rr[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            rr[4 * q] = v[c][q].x;
            rr[4 * q + 1] = v[c][q].y;
            rr[4 * q + 2] = v[c][q].z;
            rr[4 * q + 3] = v[c][q].w;
          }
          tmem_st32(taddr_lane + (cb + c) * 32, rr);
        }
      }
    }
  }
  if constexpr (kRopeSmem) {
    if (w >= kRowWarp0 && lane < 16) {
      const int m = 16 * w + lane;
      uint8_t* row = q_rope + m * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 v = live ? __ldg(src + (kChunks - 1) * 8 + u) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(row + ((u ^ (m & 7)) << 4)) = v;
      }
    }
  }
}

// Both lanes of a pair per row (l and l + 16).
template <int kRowWarp0, bool kRopeSmem, int kBatch>
__device__ __forceinline__ void load_q_split(const uint16_t* q_rows, int nrows, uint32_t taddr_lane,
                                       uint8_t* q_rope, int lane, int w) {
  static_assert(kRopeSmem && 4 % kBatch == 0, "q_hat's RoPE part is a shared-memory operand");
  if (w < kRowWarp0) return;
  // Lanes l and l + 16 share row l: lane l takes the latent chunks 0-3 and
  // RoPE units 0-3, lane l + 16 chunks 4-7 and units 4-7 (one 16x32bx2
  // store writes both halves of a row)
  const int hf = lane >> 4;
  const int r = (w - kRowWarp0) * 16 + (lane & 15);
  const bool live = r < nrows;
  const uint4* src = reinterpret_cast<const uint4*>(q_rows + static_cast<int64_t>(live ? r : 0) * kDqk);
#pragma unroll
  for (int cb = 0; cb < 4; cb += kBatch) {
    uint4 v[kBatch][8];
#pragma unroll
    for (int c = 0; c < kBatch; ++c)
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[c][q] = live ? __ldg(src + (4 * hf + cb + c) * 8 + q) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < kBatch; ++c) {
      uint32_t rr[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        rr[4 * q] = v[c][q].x;
        rr[4 * q + 1] = v[c][q].y;
        rr[4 * q + 2] = v[c][q].z;
        rr[4 * q + 3] = v[c][q].w;
      }
      tmem_st_rows16_split128(taddr_lane + (cb + c) * 32, rr);
    }
  }
  const int m = 16 * w + (lane & 15);
  uint8_t* row = q_rope + m * 128;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int uu = 4 * hf + u;
    const uint4 v = live ? __ldg(src + (kChunks - 1) * 8 + uu) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(row + ((uu ^ (m & 7)) << 4)) = v;
  }
}

// Ask L2 to fetch a row set's absorbed queries ahead of their load.
__device__ __forceinline__ void prefetch_q(const uint16_t* q_rows, int nrows, int t, int nt) {
  const char* base = reinterpret_cast<const char*>(q_rows);
  const int lines = (nrows * kDqk * 2 + 127) / 128;
  for (int i = t; i < lines; i += nt)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(base + static_cast<int64_t>(i) * 128));
}


__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two e4m3 codes (bytes 0 and 1 of `four` if hi == 0, else bytes 2 and 3)
// as two bf16 holding value * 2^-120, exactly.  An e4m3 code s.eeee.mmm
// placed as the bf16 s.0000eeee.mmm0000 has value 2^(e-127) (1 + m/8) for
// e > 0, which is 2^-120 times the e4m3 value 2^(e-7) (1 + m/8); for e = 0
// both formats are subnormal, (m/8) 2^-126 and (m/8) 2^-6, again a factor
// 2^-120; zeros map to zeros.  The byte permute sign-extends each code to
// 16 bits; the shift and mask then keep the sign bit and the 7 low bits.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_scaled(uint32_t four, int hi) {
  // prmt selector nibbles: bits 0-2 pick a byte, bit 3 replicates its sign
  uint32_t sx;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(sx) : "r"(four), "r"(hi ? 0xB3A2u : 0x9180u));
  return (sx << 4) & 0x87F087F0u;
}

// bf16x2 multiplier that, applied to a code placed as value * 2^-kPlace
// (kPlace = 120 for e4m3 above, 126 for e2m1 below), gives value *
// 2^(b - 127) for an e8m0 byte b: the factor 2^(b - 127 + kPlace) when it is
// a normal bf16 (b + kPlace <= 254), split in two factors (2^127 and the
// rest) beyond; NaN for b = 255.
struct ScaleX2 {
  uint32_t f1, f2;
  bool two;
};
template <uint32_t kPlace>
__device__ __forceinline__ ScaleX2 e8m0_scale_x2(uint32_t b) {
  ScaleX2 sc;
  if (b == 255u) {
    sc.f1 = 0x7FC07FC0u;
    sc.two = false;
  } else if (b + kPlace <= 254u) {
    const uint32_t e = (b + kPlace) << 7;    // bf16 exponent field of 2^(b - 127 + kPlace)
    sc.f1 = e | (e << 16);
    sc.two = false;
  } else {
    sc.f1 = 0x7F007F00u;                     // 2^127
    const uint32_t e = (b + kPlace - 127u) << 7;   // the remaining power, field in [1, 253]
    sc.f2 = e | (e << 16);
    sc.two = true;
  }
  if (!sc.two) sc.f2 = 0x3F803F80u;          // 1.0
  return sc;
}

// One group (32 values) of an FP8 row: its codes as nine aligned words
// (a row starts 2 bytes past a word boundary when `odd`) and its scale byte.
struct Fp8Group {
  uint32_t w[9];
  uint32_t scale;
};

// Load group g of the FP8 row at `row` (2-byte aligned) from shared memory.
__device__ __forceinline__ void load_fp8_group(const uint8_t* row, int g, bool odd, Fp8Group& f) {
  const uint8_t* a = row + 32 * g;
  const uint32_t* a4 = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(3));
#pragma unroll
  for (int k = 0; k < 8; ++k) f.w[k] = a4[k];
  f.w[8] = odd ? a4[8] : 0u;
  f.scale = row[kDqk + g];
}

// The group as 4 x 16 bytes of bf16 (8 values each, in dimension order).
// Exact: every product is an e4m3 value (4 significant bits) times a power
// of two.
__device__ __forceinline__ void convert_fp8_group(const Fp8Group& f, bool odd, uint4 (&o)[4]) {
  const ScaleX2 sc = e8m0_scale_x2<120u>(f.scale);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t r[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int wi = 2 * q + k;
      const uint32_t v = odd ? __funnelshift_r(f.w[wi], f.w[wi + 1], 16) : f.w[wi];
      uint32_t lo = bf16x2_mul(e4m3x2_to_bf16x2_scaled(v, 0), sc.f1);
      uint32_t hi = bf16x2_mul(e4m3x2_to_bf16x2_scaled(v, 1), sc.f1);
      if (sc.two) {
        lo = bf16x2_mul(lo, sc.f2);
        hi = bf16x2_mul(hi, sc.f2);
      }
      r[2 * k] = lo;
      r[2 * k + 1] = hi;
    }
    o[q] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// Eight e2m1 codes (one 32-bit word, value 2i in the low nibble of byte i)
// as four bf16x2 words holding value * 2^-126, exactly.  An e2m1 code
// s.ee.m placed as the bf16 s.000000ee.m000000 (bits 15, 8-7, 6) has value
// 2^(e-127) (1 + m/2) for e > 0, which is 2^-126 times the e2m1 value
// 2^(e-1) (1 + m/2); for e = 0 the bf16 is subnormal, (m/2) 2^-126, against
// the e2m1 subnormal m/2: again a factor 2^-126.  The byte permute puts the
// codes of values 2k and 2k+1 in the low nibbles of the two 16-bit halves
// (selector bit 3 replicates the top bit of a byte that is 0 after the
// mask, giving a zero byte).
__device__ __forceinline__ void e2m1x8_to_bf16x2_scaled(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t even = w & 0x0F0F0F0Fu;          // values 0, 2, 4, 6
  const uint32_t odd = (w >> 4) & 0x0F0F0F0Fu;    // values 1, 3, 5, 7
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t v;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(v) : "r"(even), "r"(odd), "r"(0xC480u + 0x1111u * k));
    r[k] = ((v & 0x00080008u) << 12) | ((v & 0x00070007u) << 6);
  }
}

// One group (16 values) of an FP4 row: two code words and the scale byte.
struct Fp4Group {
  uint32_t w0, w1, scale;
};

// Load group g of the FP4 row at `row` (4-byte aligned) from shared memory.
__device__ __forceinline__ void load_fp4_group(const uint8_t* row, int g, Fp4Group& f) {
  const uint32_t* a4 = reinterpret_cast<const uint32_t*>(row + 8 * g);
  f.w0 = a4[0];
  f.w1 = a4[1];
  f.scale = row[kFp4CodeBytes + g];
}

// The group as 2 x 16 bytes of bf16 in dimension order.  Exact: every
// product is an e2m1 value (2 significant bits) times a power of two.
__device__ __forceinline__ void convert_fp4_group(const Fp4Group& f, uint4 (&o)[2]) {
  const ScaleX2 sc = e8m0_scale_x2<126u>(f.scale);
  uint32_t r[2][4];
  e2m1x8_to_bf16x2_scaled(f.w0, r[0]);
  e2m1x8_to_bf16x2_scaled(f.w1, r[1]);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      r[q][k] = bf16x2_mul(r[q][k], sc.f1);
      if (sc.two) r[q][k] = bf16x2_mul(r[q][k], sc.f2);
    }
    o[q] = make_uint4(r[q][0], r[q][1], r[q][2], r[q][3]);
  }
}

}  // namespace

DecodeLayout decode_layout(int heads, int heads_pad, int num_streams, int mode) {
  (void)heads;
  (void)heads_pad;
  const bool ring = mode == kModeDenseFp8 || mode == kModeDenseFp8Multi;   // bf16 stages + raw ring
  DecodeLayout L;
  L.off_stage = 0;
  L.off_raw = (ring ? kFp8Stages : kStages) * kTileBytes;
  L.off_p = L.off_stage + kPChunkOffset;     // first stage's P; stride kTileBytes
  // q_hat's RoPE part as a shared-memory A operand: 64 M-rows x 128 B from
  // off_qrope, 1024-byte aligned.  Only the M-rows of the row set's softmax
  // warps are written and read back into S; in the FP8 kernels, which have
  // no room for all 8 KB, the M-rows below them (0-31 one-token, 0-15 with
  // draft rows) overlap the end of the raw ring: the MMA reads whatever bytes
  // are there into S rows no one reads.
  const int raw_end = L.off_raw + (ring ? kFp8RawSlots * kFp8TileBytes : 0);
  if (ring) {
    L.off_qrope = ((raw_end + 1023) & ~1023) - (mode == kModeDenseFp8Multi ? 16 : 32) * 128;
    L.off_ctrl = L.off_qrope + kQRopeBytes;
  } else {
    L.off_qrope = raw_end;
    L.off_ctrl = raw_end + kQRopeBytes;
  }
  // the row-set tile and cost prefixes, when they fit; else the pre-pass
  // writes them to the workspace
  const int base = L.off_ctrl + static_cast<int>(sizeof(Ctrl));
  const int with_prefix = base + 2 * (num_streams + 1) * 4;
  L.prefix_in_smem = num_streams <= kSmemStreams && with_prefix <= kMaxSmemBytes;
  L.total = L.prefix_in_smem ? with_prefix : base;
  return L;
}

template <int kMode>
__global__ void __launch_bounds__(ModeTraits<kMode>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p,
                      const DecodeLayout L) {
  using MT = ModeTraits<kMode>;
  constexpr int kThreads = MT::kThreads;
  constexpr int kNumStages = MT::kNumStages;
  // The buffers need 1024-byte alignment (128-byte swizzle atoms); the
  // dynamic shared window starts aligned, which is checked below.
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sStage = smem + L.off_stage;
  uint8_t* sRaw = smem + L.off_raw;   // FP8 raw ring
  uint8_t* sQr = smem + L.off_qrope;  // RoPE part of q_hat (A operand base, M-row 0)
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + L.off_ctrl);
  // the row sets' tile and cost prefixes: computed below into shared memory,
  // or written to the workspace by the pre-pass this launch depends on
  int32_t* prefix = p.prefix_ws != nullptr
                        ? p.prefix_ws
                        : reinterpret_cast<int32_t*>(smem + L.off_ctrl + sizeof(Ctrl));   // tiles
  int32_t* cprefix = prefix + (p.num_streams + 1);                                         // cost

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_streams;
  const int H = p.heads;
  const int NP = p.heads_pad;
  const int G = p.group;
  const int RMAX = p.rows;     // rows of a full row set (partial-slot stride)
  const int max_tokens = p.max_pages * p.page_size;
  volatile int32_t* abort_flag = &ctrl->abort_flag;

  if ((smem_u32(smem) & 1023u) != 0) {   // never expected; refuse rather than corrupt
    if (tid == 0) set_status(p.status, MLA_STATUS_TIMEOUT);
    return;
  }

  // ---------------------------------------------------------------- setup
  // Let a dependent launch (the merge, with or without W_UV) start its
  // prologue as soon as SMs free up; it waits for this grid's completion
  // before reading.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < kNumStages; ++i) {
      // sparse: one byte-count arrival per gather warp
      mbar_init(&ctrl->full[i],
                MT::kQuant ? kDequantWarps : (MT::kSparse ? kGatherWarps : 1));
      mbar_init(&ctrl->empty[i], kPvLanes);   // one commit per PV issuer
    }
    for (int i = 0; i < kStages; ++i) mbar_init(&ctrl->raw_full[i], 1);
    for (int i = 0; i < kStages; ++i) mbar_init(&ctrl->dq_part[i], kDequantWarps);
    for (int i = 0; i < kFp8RawSlots; ++i) mbar_init(&ctrl->raw_empty[i], kDequantWarps);
    for (int i = 0; i < 2; ++i) ctrl->rescale_tile[i] = -1;
    mbar_init(&ctrl->s_full, MT::kSplitS ? 2 : 1);   // one commit per QK issuer
    mbar_init(&ctrl->s_free, kSoftmaxWarps);
    mbar_init(&ctrl->q_ready, kSoftmaxWarps);
    mbar_init(&ctrl->o_done[0], kPvLanes);
    mbar_init(&ctrl->o_done[1], kPvLanes);
    // final commits: the MMA warp's issuing lanes, the PV lanes, the second
    // QK warp
    mbar_init(&ctrl->mma_drain[0], MT::kQkLanes);
    mbar_init(&ctrl->mma_drain[1], kPvLanes);
    mbar_init(&ctrl->mma_drain[2], 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0 && (MT::kDenseBf16 || MT::kSparse)) prefetch_tmap(&kv_map);
  // A launch behind the prefix pre-pass waits for it here (a no-op for a
  // launch that depends on nothing); nothing above reads memory a kernel
  // before this one may write.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // tiles and cost per stream (stream lengths from the device seq_lens)
  if (p.prefix_ws == nullptr) {
    for (int s = tid; s < S; s += kThreads) {
      const StreamGeom gm = stream_geom(s, p.q_len, G);
      const int32_t len = stream_len(p.seq_lens[gm.b], p.q_len, gm.j0 + gm.nq - 1, p.causal,
                                     p.topk_width, max_tokens);
      const int32_t nt = (len + kTile - 1) / kTile;
      prefix[s + 1] = nt;
      cprefix[s + 1] = stream_cost(nt, p.stream_cost);
    }
  }
  __syncthreads();
  if (p.prefix_ws == nullptr && warp < 2) {   // exclusive prefix sums: warp 0 of tiles, warp 1 of cost
    int32_t* arr = warp == 0 ? prefix : cprefix;
    int32_t carry = 0;
    if (lane == 0) arr[0] = 0;
    for (int base = 0; base < S; base += 32) {
      const int s = base + lane;
      int32_t v = (s < S) ? arr[s + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (s < S) arr[s + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int32_t ucost = cprefix[S];
  const int32_t c = blockIdx.x;
  // CTAs that take part in the split (work_ctas): the plan's, but at most
  // one per tile, so that each CTA's cost range spans at least kTileCost
  // units and every CTA between the first and the last owner of a row set's
  // tiles owns some of them (and writes a partial)
  const int32_t nctas = work_ctas(p.num_ctas, prefix[S]);
  const int32_t g0 = c >= nctas ? 0 : first_tile_at(
      prefix, cprefix, S, static_cast<int32_t>((static_cast<int64_t>(c) * ucost) / nctas),
      p.stream_cost);
  const int32_t g1 = c >= nctas ? 0 : first_tile_at(
      prefix, cprefix, S, static_cast<int32_t>((static_cast<int64_t>(c + 1) * ucost) / nctas),
      p.stream_cost);
  const int32_t ntiles = g1 - g0;
  const uint32_t tmem = ctrl->tmem_base;

  if (ntiles > 0) {
    if (warp == kProducerWarp && !MT::kSparse) {
      // ============================================================ producer
      const uint64_t pol = l2_policy_evict_first();
      Walker wk;
      wk.init(prefix, S, g0);
      int32_t issued = 0;
      bool failed = false;
      for (int32_t i = 0; i < ntiles; ++i) {
        const int stage = i % kNumStages;
        const uint32_t reuse_parity = ((i / kNumStages) - 1) & 1;
        // a row set covers query tokens j0 .. j0 + nq - 1: its tiles reach
        // the visible window of the last one
        const StreamGeom gm = stream_geom(wk.s, p.q_len, G);
        const int b = gm.b, j = gm.j0 + gm.nq - 1;
        uint8_t* dst = sStage + stage * kTileBytes;
        // Describe the tile first: its global lookups overlap the stage wait.
        if constexpr (MT::kDenseBf16) {
          if (p.page_size >= kTile) {
            // one page holds the whole tile: one lane describes it
            int32_t row0 = 0;
            uint64_t mask = 0;
            bool ok = false;
            if (lane == 0) {
              const int32_t tok0 = wk.lt * kTile;
              const int32_t len = stream_len(p.seq_lens[b], p.q_len, j, p.causal, 0, max_tokens);
              const int32_t page =
                  p.block_table[static_cast<int64_t>(b) * p.max_pages + tok0 / p.page_size];
              const int32_t nvalid = min(kTile, len - tok0);
              mask = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
              ok = page >= 0 && page < p.num_pages;
              if (!ok) {
                mask = 0;
                set_status(p.status, MLA_STATUS_BAD_PAGE);
              }
              row0 = ok ? page * p.page_size + (tok0 % p.page_size) : 0;
            }
            if (i >= kNumStages && !warp_wait(&ctrl->empty[stage], reuse_parity, abort_flag)) {
              failed = true;
              break;
            }
            if (lane == 0) {
              ctrl->mask[stage] = mask;
              if (ok) {
                mbar_arrive_expect_tx(&ctrl->full[stage], kTileBytes);
#pragma unroll
                for (int ch = 0; ch < kChunks; ++ch)
                  tma_load_2d(dst + ch * kChunkBytes, &kv_map, &ctrl->full[stage], ch * kChunkElems,
                              row0, pol);
              } else {
                mbar_arrive(&ctrl->full[stage]);
              }
            }
          } else {
            // 16- or 32-token pages: the tile spans 64 / P pages
            const TilePieces tp = describe_tile(p, b, j, wk.lt, lane, max_tokens);
            const uint64_t mask = tile_mask(tp);
            if (lane == 0 && tp.bad) set_status(p.status, tp.bad);
            if (i >= kNumStages && !warp_wait(&ctrl->empty[stage], reuse_parity, abort_flag)) {
              failed = true;
              break;
            }
            if (lane == 0) {
              ctrl->mask[stage] = mask;
              if (tp.ok) {
                // the map's box is one piece (P rows) of one 64-dim chunk
                mbar_arrive_expect_tx(&ctrl->full[stage],
                                      __popc(tp.ok) * tp.rows * kChunks * kChunkElems * 2);
                for (int k = 0; k < tp.npieces; ++k) {
                  if (!((tp.ok >> k) & 1u)) continue;
                  const int32_t row0 = tp.page[k] * p.page_size + tp.slot0;
#pragma unroll
                  for (int ch = 0; ch < kChunks; ++ch)
                    tma_load_2d(dst + ch * kChunkBytes + k * tp.rows * 128, &kv_map,
                                &ctrl->full[stage], ch * kChunkElems, row0, pol);
                }
              } else {
                mbar_arrive(&ctrl->full[stage]);
              }
            }
          }
        } else {   // FP8 / FP4 caches: the tile's quantised rows, one bulk copy
          // FP8: ring slot rs, reusable once the dequant warps have read it;
          // FP4: the tail of this tile's stage, reusable once PV has read it
          const int rs = MT::kRawRing ? i % MT::kRawSlots : stage;
          uint8_t* raw_dst = MT::kRawRing ? sRaw + rs * MT::kRawTileBytes : dst + MT::kRawOffset;
          uint64_t* raw_bar = &ctrl->raw_full[rs];
          uint64_t* mask_slot = MT::kRawRing ? &ctrl->raw_mask[rs] : &ctrl->mask[stage];
          uint64_t* reuse_bar = MT::kRawRing ? &ctrl->raw_empty[rs] : &ctrl->empty[stage];
          const uint32_t reuse_par = ((i / MT::kRawSlots) - 1) & 1;
          if (p.page_size >= kTile) {
            // one page holds the whole tile: one lane describes it
            uint64_t mask = 0;
            bool ok = false;
            const uint8_t* src = p.kv;
            uint32_t bytes = 0;
            if (lane == 0) {
              const int32_t tok0 = wk.lt * kTile;
              const int32_t len = stream_len(p.seq_lens[b], p.q_len, j, p.causal, 0, max_tokens);
              const int32_t page =
                  p.block_table[static_cast<int64_t>(b) * p.max_pages + tok0 / p.page_size];
              const int32_t nvalid = min(kTile, len - tok0);
              mask = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
              ok = page >= 0 && page < p.num_pages;
              if (!ok) {
                mask = 0;
                set_status(p.status, MLA_STATUS_BAD_PAGE);
              }
              // rows tok0 .. tok0 + 63 of a page are contiguous; copy the live
              // ones rounded up to 8 rows (8 rows of 594 or 324 bytes are a
              // multiple of 16 B)
              src = p.kv + (static_cast<int64_t>(page) * p.page_size + tok0 % p.page_size) *
                               MT::kRowBytes;
              bytes = static_cast<uint32_t>((nvalid + 7) & ~7) * MT::kRowBytes;
            }
            if (i >= MT::kRawSlots && !warp_wait(reuse_bar, reuse_par, abort_flag)) {
              failed = true;
              break;
            }
            if (lane == 0) {
              *mask_slot = mask;
              if (ok) {
                mbar_arrive_expect_tx(raw_bar, bytes);
                bulk_load(raw_dst, src, bytes, raw_bar, pol);
              } else {
                mbar_arrive(raw_bar);
              }
            }
          } else {
            // 16- or 32-token pages: one bulk copy per page piece
            const TilePieces tp = describe_tile(p, b, j, wk.lt, lane, max_tokens);
            const uint64_t mask = tile_mask(tp);
            if (lane == 0 && tp.bad) set_status(p.status, tp.bad);
            if (i >= MT::kRawSlots && !warp_wait(reuse_bar, reuse_par, abort_flag)) {
              failed = true;
              break;
            }
            if (lane == 0) {
              *mask_slot = mask;
              if (tp.ok) {
                // a piece's rows are contiguous in its page; copy the live ones
                // rounded up to 8 rows (a multiple of 16 B)
                uint32_t total = 0;
                for (int k = 0; k < tp.npieces; ++k)
                  if ((tp.ok >> k) & 1u)
                    total += static_cast<uint32_t>((min(tp.rows, tp.nvalid - k * tp.rows) + 7) & ~7);
                mbar_arrive_expect_tx(raw_bar, total * MT::kRowBytes);
                for (int k = 0; k < tp.npieces; ++k) {
                  if (!((tp.ok >> k) & 1u)) continue;
                  const uint32_t nrows =
                      static_cast<uint32_t>((min(tp.rows, tp.nvalid - k * tp.rows) + 7) & ~7);
                  const uint8_t* src =
                      p.kv + (static_cast<int64_t>(tp.page[k]) * p.page_size + tp.slot0) *
                                 MT::kRowBytes;
                  bulk_load(raw_dst + k * tp.rows * MT::kRowBytes, src, nrows * MT::kRowBytes,
                            raw_bar, pol);
                }
              } else {
                mbar_arrive(raw_bar);
              }
            }
          }
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
      if (lane == 0) {
        if constexpr (MT::kQuant) {
          for (int32_t i = max(0, issued - MT::kRawSlots); i < issued; ++i)
            (void)mbar_wait(&ctrl->raw_full[i % MT::kRawSlots], (i / MT::kRawSlots) & 1, nullptr,
                            kWaitLimitNs);
        } else {
          for (int32_t i = max(0, issued - kNumStages); i < issued; ++i)
            (void)mbar_wait(&ctrl->full[i % kNumStages], (i / kNumStages) & 1, nullptr,
                            kWaitLimitNs);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp || (MT::kSplitQK && warp == MT::kQk2Warp)) {
      // =================================================================== QK
      // Issuer(s) of S = q_hat . rows (or of one half of its K range, each
      // into an S accumulator of its own): lane 0 of this warp, lanes 0 and
      // 1 when QK is split over lanes, or lane 0 of the second QK warp.  QK(t)
      // goes out once tile t is staged, the stream's q_hat is in TMEM and the
      // softmax has read S(t-1).
      const uint32_t idesc_qk = make_idesc_bf16(64, 64, false, false);
      // Descriptors at the buffers' bases; an operand at byte offset x is
      // base + (x >> 4) (the start-address field holds address >> 4 and the
      // whole buffer lies below 256 KB, so the field never carries).
      const uint64_t qk_b0 = make_smem_desc(smem_u32(sStage), 16, 1024, kSmemLayoutSW128);
      // q_hat's RoPE part as QK's A operand (64 M-rows x 64 values, K-major)
      const uint64_t qr_a0 = make_smem_desc(smem_u32(sQr), 16, 1024, kSmemLayoutSW128);
      // QK(j) over chunks [c0, c1) of the staged rows into the S accumulator
      // at column `col` (A = q_hat from TMEM, 4 MMAs per chunk), then the
      // RoPE chunk's K steps [k0, k1) with A = q_hat's RoPE part in shared
      // memory (or from TMEM when it is there).
      auto issue_qk = [&](int st, int c0, int c1, uint32_t col, int k0, int k1) {
        const uint64_t b0 = qk_b0 + static_cast<uint64_t>((st * kTileBytes) >> 4);
        for (int ch = c0; ch < c1; ++ch) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ts(tmem + col, tmem + MT::kColQ + (ch * 4 + k) * 8,
                        b0 + ((ch * kChunkBytes + k * 32) >> 4), idesc_qk,
                        (ch > c0 || k > 0) ? 1u : 0u);
        }
        if constexpr (MT::kQRopeSmem) {
          for (int k = k0; k < k1; ++k)
            mma_bf16_ss(tmem + col, qr_a0 + ((k * 32) >> 4),
                        b0 + (((kChunks - 1) * kChunkBytes + k * 32) >> 4), idesc_qk,
                        (c1 > c0 || k > k0) ? 1u : 0u);
        }
      };
      // An issuer's share of QK: all of it into S, or half of its K range
      // (`second` picks the half: chunks 0-3 and RoPE steps 0-1 into S_a,
      // chunks 4-7 and RoPE steps 2-3 into S_b).
      auto issue_my_qk = [&](int st, bool second) {
        if constexpr (MT::kSplitS) {
          const int c0 = second ? 4 : 0;
          issue_qk(st, c0, c0 + 4, second ? MT::kColS2 : MT::kColS, second ? 2 : 0, second ? 4 : 2);
        } else {
          issue_qk(st, 0, MT::kQTmemChunks, MT::kColS, 0, 4);
        }
      };
      const int role = warp == kMmaWarp ? 0 : 2;    // index of the drain barrier
      const int nl = warp == kMmaWarp ? MT::kQkLanes : 1;
      const uint32_t gmask = (1u << nl) - 1u;
      bool failed = false;
      if (lane < nl) {
        // polled by lane 0 with a short sleep (measured to wake sooner than a
        // suspending mbarrier.try_wait); the other issuing lane follows it
        // (FP8: the tile's first dequant phase, not the whole tile)
        auto ready = [&](int32_t t, int st, bool first, int32_t sg) -> bool {
          bool r = false;
          if (lane == 0)
            r = (!first || mbar_poll(&ctrl->q_ready, sg & 1)) &&
                mbar_poll(MT::kRawRing ? &ctrl->dq_part[st] : &ctrl->full[st],
                          (t / kNumStages) & 1) &&
                (t < 1 || mbar_poll(&ctrl->s_free, (t - 1) & 1));
          return __shfl_sync(gmask, r, 0);
        };
        // bounded wait for one barrier phase, lane 0 polling
        auto wait_phase = [&](uint64_t* bar, uint32_t parity) -> bool {
          bool r = false;
          if (lane == 0) r = mbar_poll(bar, parity);
          if (__shfl_sync(gmask, r, 0)) return true;
          const uint64_t t0 = globaltimer_ns();
          while (true) {
            __nanosleep(20);
            if (lane == 0) r = mbar_poll(bar, parity);
            if (__shfl_sync(gmask, r, 0)) return true;
            if (__shfl_sync(gmask, *abort_flag || globaltimer_ns() - t0 > kWaitLimitNs, 0))
              return false;
          }
        };
        Walker wk;
        wk.init(prefix, S, g0);
        int32_t seg = -1;
        for (int32_t t = 0; t < ntiles; ++t) {
          const int st = t % kNumStages;
          const bool first = (t == 0) || (wk.lt == 0);
          const int32_t sg = first ? seg + 1 : seg;
          if (!ready(t, st, first, sg)) {
            const uint64_t t0 = globaltimer_ns();
            bool ok = false;
            while (true) {
              __nanosleep(20);
              if (ready(t, st, first, sg)) { ok = true; break; }
              if (__shfl_sync(gmask, *abort_flag || globaltimer_ns() - t0 > kWaitLimitNs, 0)) break;
            }
            if (!ok) {
              failed = true;
              break;
            }
          }
          tc_fence_after();
          if constexpr (MT::kRawRing) {
            // FP8: QK follows the dequant's two phases (chunks {0, 1, 4, 5},
            // then {2, 3, 6, 7} and RoPE); each lane of a split QK takes its
            // half: lane L chunks 4L .. 4L + 3 and RoPE steps 2L, 2L + 1
            const uint64_t b0 = qk_b0 + static_cast<uint64_t>((st * kTileBytes) >> 4);
            const int hl = MT::kSplitS ? lane : 0;
            const uint32_t col = hl ? MT::kColS2 : MT::kColS;
            auto chunk = [&](int ch, bool first_mma) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16_ts(tmem + col, tmem + MT::kColQ + (ch * 4 + k) * 8,
                            b0 + ((ch * kChunkBytes + k * 32) >> 4), idesc_qk,
                            (first_mma && k == 0) ? 0u : 1u);
            };
            chunk(4 * hl, true);
            chunk(4 * hl + 1, false);
            if constexpr (!MT::kSplitS) {
              chunk(4, false);
              chunk(5, false);
            }
            bool ok = wait_phase(&ctrl->full[st], (t / kNumStages) & 1);
            if (ok) {
              tc_fence_after();
              chunk(4 * hl + 2, false);
              chunk(4 * hl + 3, false);
              if constexpr (!MT::kSplitS) {
                chunk(6, false);
                chunk(7, false);
              }
              const int k0 = MT::kSplitS ? 2 * hl : 0, k1 = MT::kSplitS ? k0 + 2 : 4;
              for (int k = k0; k < k1; ++k)
                mma_bf16_ss(tmem + col, qr_a0 + ((k * 32) >> 4),
                            b0 + (((kChunks - 1) * kChunkBytes + k * 32) >> 4), idesc_qk, 1u);
            }
            if (!ok) {
              failed = true;
              break;
            }
          } else {
            issue_my_qk(st, warp != kMmaWarp || lane == 1);
          }
          mma_commit(&ctrl->s_full);
          seg = sg;
          wk.next(prefix, S);
        }
      }
      __syncwarp();
      if (failed && lane == 0) {
        set_status(p.status, MLA_STATUS_TIMEOUT);
        ctrl->abort_flag = 1;
      }
      // drain: every issued MMA completes before tensor memory is released
      if (lane < nl) mma_commit(&ctrl->mma_drain[role]);
      if (lane == 0) (void)mbar_wait(&ctrl->mma_drain[role], 0, nullptr, kWaitLimitNs);
      __syncwarp();
    } else if (MT::kQuant && warp >= kDequantWarp0) {
      // ============================================================ dequant
      // Thread t of the 192 owns row t % 64 and groups t / 64 + 3k: a warp
      // covers 32 consecutive rows, so its shared loads (row stride 594 B or
      // 324 B: an odd number of words apart, or 81 words) and its swizzled
      // 16-byte stores spread over the banks.
      const int dt = tid - kDequantWarp0 * 32;
      const int r = dt & 63;
      const int gset = dt >> 6;
      const bool odd = (r & 1) != 0;   // FP8 rows of odd index start 2 bytes past a word
      bool failed = false;
      // store a converted group: FP8 group g fills units 4(g%2).. of chunk g/2,
      // FP4 group g units 2(g%4).. of chunk g/4 (16-byte units, swizzled by row)
      auto store_group = [&](uint8_t* dst, int g, const uint4* o) {
        constexpr int kUnits = MT::kFp4 ? 2 : 4;
        constexpr int kPerChunk = 8 / kUnits;
        const int u0 = (g % kPerChunk) * kUnits;
#pragma unroll
        for (int q = 0; q < kUnits; ++q)
          *reinterpret_cast<uint4*>(dst + (g / kPerChunk) * kChunkBytes +
                                    (((u0 + q) ^ (r & 7)) << 4)) = o[q];
      };
      if constexpr (MT::kRawRing) {
        // FP8: raw slot rs -> bf16 stage bs in two phases, the first
        // published on its own barrier as soon as every dequant warp has
        // finished it, so that QK starts on a tile before the whole tile is
        // converted: chunks {0, 1, 4, 5} (the first two chunks of each QK
        // half), then {2, 3, 6, 7} and the RoPE chunk.  (Each publication
        // costs every warp a proxy fence: five phases measured slower.)  The
        // work is 36 items (one group of 32 values for 32 rows) in that
        // order; warp dw takes items dw + 6k at step k, so the first phase
        // (items 0-15) is complete after step 2 (dq_part) and the second
        // after step 5 (full).
        const int dw = warp - kDequantWarp0;
        for (int32_t i = 0; i < ntiles; ++i) {
          const int rs = i % MT::kRawSlots;
          const int bs = i % kNumStages;
          if (!warp_wait(&ctrl->raw_full[rs], (i / MT::kRawSlots) & 1, abort_flag) ||
              (i >= kNumStages &&
               !warp_wait(&ctrl->empty[bs], ((i / kNumStages) - 1) & 1, abort_flag))) {
            failed = true;
            break;
          }
          const uint64_t mask = ctrl->raw_mask[rs];
          const uint8_t* raw_tile = sRaw + rs * MT::kRawTileBytes;
          uint8_t* tile = sStage + bs * kTileBytes;
#pragma unroll 2
          for (int k = 0; k < kFp8Items / kDequantWarps; ++k) {
            const int item = dw + kDequantWarps * k;
            int g, h;
            if (item >= 32) {                        // the RoPE chunk: groups 16, 17
              g = 16 + ((item - 32) >> 1);
              h = (item - 32) & 1;
            } else {                                 // chunk pair {cp, cp + 4}
              const int cp = item >> 3, within = item & 7, gi = within >> 1;
              h = within & 1;
              g = gi < 2 ? 2 * cp + gi : 2 * cp + 6 + gi;
            }
            const int rr = 32 * h + lane;
            const bool odd_r = (rr & 1) != 0;   // rows of odd index start 2 bytes past a word
            uint4 o[4];
            if ((mask >> rr) & 1ull) {
              Fp8Group f;
              load_fp8_group(raw_tile + rr * MT::kRowBytes, g, odd_r, f);
              convert_fp8_group(f, odd_r, o);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q) o[q] = make_uint4(0, 0, 0, 0);
            }
            uint8_t* dst = tile + (g >> 1) * kChunkBytes + rr * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(dst + ((((g & 1) * 4 + q) ^ (rr & 7)) << 4)) = o[q];
            if (k == 2) {
              fence_proxy_async_smem();   // generic stores -> tensor-core reads
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctrl->dq_part[bs]);
            }
          }
          if (dt == 0) ctrl->mask[bs] = mask;
          fence_proxy_async_smem();   // generic stores -> tensor-core reads
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&ctrl->raw_empty[rs]);
            mbar_arrive(&ctrl->full[bs]);
          }
        }
      } else {
        // FP4: the raw bytes occupy the stage from kRawOffset on (inside
        // chunk 6).  Groups 3k + gset with k < 8 have their bf16 output in
        // chunks 0-5, below them: converted and stored at once.  The other
        // four are loaded into registers and stored after every dequant warp
        // has finished reading raw bytes.
        for (int32_t i = 0; i < ntiles; ++i) {
          const int stage = i % kNumStages;
          const bool ok = warp_wait(&ctrl->raw_full[stage], (i / kNumStages) & 1, abort_flag);
          const uint64_t mask = ctrl->mask[stage];
          const bool live = ok && ((mask >> r) & 1ull);
          uint8_t* tile = sStage + stage * kTileBytes;
          const uint8_t* row_ptr = tile + MT::kRawOffset + r * MT::kRowBytes;
          uint8_t* dst = tile + r * 128;
          constexpr int kDirect = 24 / kGroupSets;            // groups 0-23 lie in chunks 0-5
          constexpr int kKept = kDqk / 16 / kGroupSets - kDirect;
          Fp4Group keep[kKept];
          if (ok) {
#pragma unroll 4
            for (int k = 0; k < kDirect; ++k) {
              const int g = gset + kGroupSets * k;
              uint4 o[2];
              if (live) {
                Fp4Group f;
                load_fp4_group(row_ptr, g, f);
                convert_fp4_group(f, o);
              } else {
                o[0] = o[1] = make_uint4(0, 0, 0, 0);
              }
              store_group(dst, g, o);
            }
            if (live) {
#pragma unroll
              for (int k = 0; k < kKept; ++k)
                load_fp4_group(row_ptr, gset + kGroupSets * (kDirect + k), keep[k]);
            }
          }
          // every dequant warp reaches this barrier once per tile; a failed
          // wait in any of them ends all of them here
          if (named_bar_or(2, kDequantWarps * 32, !ok)) {
            failed = true;
            break;
          }
#pragma unroll
          for (int k = 0; k < kKept; ++k) {
            uint4 o[2];
            if (live) convert_fp4_group(keep[k], o);
            else o[0] = o[1] = make_uint4(0, 0, 0, 0);
            store_group(dst, gset + kGroupSets * (kDirect + k), o);
          }
          fence_proxy_async_smem();   // generic stores -> tensor-core reads
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->full[stage]);
        }
      }
      if (failed && lane == 0) {
        set_status(p.status, MLA_STATUS_TIMEOUT);
        ctrl->abort_flag = 1;
      }
    } else if (MT::kSparse && warp >= kGatherWarp0) {
      // ============================================================= gather
      // Gather warp gw stages tile rows [16 gw, 16 gw + 16): lanes 0..15
      // resolve one top-k slot each (index -> page -> physical cache row, or
      // -1 for a dead slot), then lanes 0..35 issue one TMA gather4 each:
      // rows 16 gw + 4 g .. + 3 of 64-dim chunk c (t = 9 g + c) into the
      // swizzled tile, a dead row reading the map's zero fill.  The warp's
      // 16 bits of the live-row mask go out with its byte count.
      const int gw = warp - kGatherWarp0;
      const uint64_t pol = l2_policy_evict_first();
      Walker wk;
      wk.init(prefix, S, g0);
      bool failed = false;
      int32_t issued = 0;
      for (int32_t i = 0; i < ntiles; ++i) {
        const int stage = i % kNumStages;
        const uint32_t reuse_parity = ((i / kNumStages) - 1) & 1;
        const StreamGeom gm = stream_geom(wk.s, p.q_len, G);   // one query token per row set
        const int b = gm.b, j = gm.j0;
        uint8_t* dst = sStage + stage * kTileBytes;
        const int32_t T = min(max(p.seq_lens[b], 0), max_tokens);
        const int32_t window = p.causal ? min(max(T - p.q_len + j + 1, 0), T) : T;
        const int rl = kGatherRows * gw + (lane & 15);
        const int32_t idx =
            p.topk_idx[static_cast<int64_t>(wk.s) * p.topk_width + wk.lt * kTile + rl];
        bool v = idx >= 0 && idx < window;
        uint32_t bad = (!v && idx != -1) ? MLA_STATUS_BAD_INDEX : 0u;
        int32_t page = -1;
        if (v) {
          page = p.block_table[static_cast<int64_t>(b) * p.max_pages + idx / p.page_size];
          if (page < 0 || page >= p.num_pages) {
            v = false;
            bad |= MLA_STATUS_BAD_PAGE;
          }
        }
        if (bad && lane < 16) set_status(p.status, bad);
        const int32_t prow = v ? page * p.page_size + idx % p.page_size : -1;
        const uint32_t live = __ballot_sync(0xffffffffu, v) & 0xFFFFu;
        if (i >= kNumStages && !warp_wait(&ctrl->empty[stage], reuse_parity, abort_flag)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          reinterpret_cast<volatile uint16_t*>(&ctrl->mask[stage])[gw] = static_cast<uint16_t>(live);
          mbar_arrive_expect_tx(&ctrl->full[stage], kGatherRows * kChunks * 128);
        }
        __syncwarp();
#pragma unroll
        for (int round = 0; round < 2; ++round) {
          const int t = lane + 32 * round;              // 36 gathers: 4 row groups x 9 chunks
          const int tt = t < 4 * kChunks ? t : 0;
          const int g = tt / kChunks, ch = tt - g * kChunks;
          const int32_t y0 = __shfl_sync(0xffffffffu, prow, 4 * g);
          const int32_t y1 = __shfl_sync(0xffffffffu, prow, 4 * g + 1);
          const int32_t y2 = __shfl_sync(0xffffffffu, prow, 4 * g + 2);
          const int32_t y3 = __shfl_sync(0xffffffffu, prow, 4 * g + 3);
          if (t < 4 * kChunks)
            tma_gather4(dst + ch * kChunkBytes + (kGatherRows * gw + 4 * g) * 128, &kv_map,
                        &ctrl->full[stage], ch * kChunkElems, y0, y1, y2, y3, pol);
        }
        ++issued;
        wk.next(prefix, S);
      }
      if (failed && lane == 0) {
        set_status(p.status, MLA_STATUS_TIMEOUT);
        ctrl->abort_flag = 1;
      }
      // every copy this warp issued has landed before the CTA exits
      if (lane == 0)
        for (int32_t i = max(0, issued - kNumStages); i < issued; ++i)
          (void)mbar_wait(&ctrl->full[i % kNumStages], (i / kNumStages) & 1, nullptr, kWaitLimitNs);
      __syncwarp();
    } else if (warp == kProducerWarp) {
      // sparse mode: the gather warps stage the tiles
    } else {
      // ============================================================ softmax
      // Warp w reads TMEM lanes [32w, 32w+32).  Row h of the row set (a head,
      // or (draft token h / H, head h % H) in the multi-token mode) is S row
      // 16 * kRowWarp0 + h: in the M=64 accumulator layout (row r in lane
      // (r/16)*32 + r%16) rows 0..15 are lanes 0..15 of warp kRowWarp0, and
      // so on; lanes 16..31 hold no row, so lane l + 16 takes the upper 32
      // token columns of lane l's row (one shuffle per column) and the pair
      // combines max and sum.  Warps below kRowWarp0 only join the epilogue,
      // the rescale and the dead-row zeroing.
      const int w = warp;
      const int hl = lane & 15;
      const int half = lane >> 4;
      const int h = (w - MT::kRowWarp0) * 16 + hl;
      const uint32_t lane_base = static_cast<uint32_t>(w * 32) << 16;
      const float scale = p.scale_log2;
      // l_run sums the bf16-rounded P the PV uses (it normalises O); l_exp
      // sums the unrounded exponentials (it gives lse).
      float m_used = -INFINITY, l_run = 0.f, l_exp = 0.f;
      Walker wk;
      wk.init(prefix, S, g0);
      bool failed = false;
      // PV(j) has completed: o_done[j % 2] has finished its phase j / 2.  At
      // tile i every PV up to i - kNumStages has completed and been signalled
      // (tile i's stage was released by that PV's commit to empty, issued
      // after its commit to o_done), so each barrier has at most one phase
      // in flight when it is waited on here.
      auto pv_done = [&](int32_t j) -> bool {
        return warp_wait(&ctrl->o_done[j & 1], (j >> 1) & 1, abort_flag);
      };
      // PV operands: A = the staged tile read MN-major (V^T), B = its P
      const uint32_t idesc_pv = make_idesc_bf16(128, static_cast<uint32_t>(NP), true, false);
      const uint64_t pv_a0 = make_smem_desc(smem_u32(sStage), kChunkBytes, 1024, kSmemLayoutSW128);
      const uint64_t pv_b0 = make_smem_desc(smem_u32(sStage + kPChunkOffset), 16, 1024,
                                            kSmemLayoutSW128);
      // q_hat / o_lat rows of row set s and how many there are
      auto first_row = [&](int32_t s) -> int64_t {
        const StreamGeom gm = stream_geom(s, p.q_len, G);
        return (static_cast<int64_t>(gm.b) * p.q_len + gm.j0) * H;
      };
      auto rows_of = [&](int32_t s) -> int { return stream_geom(s, p.q_len, G).nq * H; };
      // a row set's queries into TMEM (and the RoPE part into shared memory)
      auto load_rows = [&](int32_t st_) {
        if constexpr (MT::kQLoadSplit)
          load_q_split<MT::kRowWarp0, MT::kQRopeSmem, MT::kQBatch>(
              p.q_hat + first_row(st_) * kDqk, rows_of(st_), tmem + lane_base, sQr, lane, w);
        else
          load_q<MT::kRowWarp0, MT::kQRopeSmem, MT::kQBatch>(
              p.q_hat + first_row(st_) * kDqk, rows_of(st_), tmem + lane_base, sQr, lane, w);
      };
      // the first stream's queries
      load_rows(wk.s);
      if constexpr (MT::kQRopeSmem) fence_proxy_async_smem();   // RoPE rows -> tensor-core reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->q_ready);
      // rows of the current row set (one per head outside the multi-token mode)
      int nrows = H;
      bool warp_has_heads = w >= MT::kRowWarp0 && (w - MT::kRowWarp0) * 16 < H;
      bool owner = warp_has_heads && h < H;
      int32_t win_end = 0;    // multi-token mode: this thread's row sees positions below this
      for (int32_t i = 0; i < ntiles; ++i) {
        const int stage = i % kNumStages;
        const int pb = i & 1;
        const bool first = (i == 0) || (wk.lt == 0);
        const bool last = (i == ntiles - 1) || (wk.lt == wk.ntiles - 1);
        if (first) {
          if constexpr (MT::kMulti) {
            const StreamGeom gm = stream_geom(wk.s, p.q_len, G);
            nrows = gm.nq * H;
            warp_has_heads = w >= MT::kRowWarp0 && (w - MT::kRowWarp0) * 16 < nrows;
            owner = warp_has_heads && h < nrows;
            // draft token j0 + h / H sees positions up to its own causal
            // limit; the row set's tiles reach the last token's limit
            const int jj = owner ? h / H : gm.nq - 1;
            win_end = stream_len(p.seq_lens[gm.b], p.q_len, gm.j0 + jj, p.causal, 0, max_tokens);
          }
          if (w < MT::kRowWarp0) {
            // warm L2 with the next stream's queries (loaded when this
            // segment ends)
            int32_t sn = wk.s + 1;
            while (sn < S && prefix[sn + 1] == prefix[sn]) ++sn;
            if (sn < S && prefix[sn] < g1)
              prefetch_q(p.q_hat + first_row(sn) * kDqk, rows_of(sn), tid, 32 * MT::kRowWarp0);
          }
        }
        bool ok = !failed && warp_wait(&ctrl->full[stage], (i / kNumStages) & 1, abort_flag);
        const uint64_t mask = ctrl->mask[stage];
        ok = ok && warp_wait(&ctrl->s_full, i & 1, abort_flag);
        if (ok) {
          tc_fence_after();
          float y[32];
          if (warp_has_heads) {
            // lane l < 16 reads columns 0..31 of its row, lane l + 16
            // columns 32..63 of the same row (S = S_a + S_b when split)
            uint32_t r[32];
            tmem_ld_rows16_split32(tmem + lane_base + MT::kColS, r);
#pragma unroll
            for (int t = 0; t < 32; ++t) y[t] = __uint_as_float(r[t]);
            if constexpr (MT::kSplitS) {
              tmem_ld_rows16_split32(tmem + lane_base + MT::kColS2, r);
#pragma unroll
              for (int t = 0; t < 32; ++t) y[t] += __uint_as_float(r[t]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->s_free);
          if (ok && warp_has_heads) {
            // token of y[t] is 32*half + t
            uint32_t hmask = static_cast<uint32_t>(mask >> (32 * half));
            if constexpr (MT::kMulti) {
              // this row's own causal limit inside the tile
              const int32_t lim = win_end - wk.lt * kTile - 32 * half;
              hmask &= lim <= 0 ? 0u : (lim >= 32 ? ~0u : ((1u << lim) - 1u));
            }
            float mt = -INFINITY;
            if (hmask == 0xffffffffu) {
#pragma unroll
              for (int t = 0; t < 32; ++t) mt = fmaxf(mt, y[t]);
            } else {
#pragma unroll
              for (int t = 0; t < 32; ++t) {
                y[t] = ((hmask >> t) & 1u) ? y[t] : -INFINITY;
                mt = fmaxf(mt, y[t]);
              }
            }
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16)) * scale;
            float alpha = 1.f;
            if (first) {
              m_used = mt;
              l_run = 0.f;
              l_exp = 0.f;
            } else if (mt > m_used + kRescaleThreshold) {
              alpha = fast_exp2(m_used - mt);
              m_used = mt;
              l_run *= alpha;
              l_exp *= alpha;
              if (owner && half == 0) ctrl->rescale_tile[pb] = i;
            }
            const float nref = (m_used == -INFINITY) ? 0.f : -m_used;
            uint8_t* prow = sStage + stage * kTileBytes + kPChunkOffset + h * 128;
            float lsum = 0.f, lsum_exp = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint32_t u[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float a = fast_exp2(fmaf(y[c8 * 8 + 2 * e], scale, nref));
                const float b = fast_exp2(fmaf(y[c8 * 8 + 2 * e + 1], scale, nref));
                u[e] = pack_bf16x2(a, b);
                const __nv_bfloat162 v2 = *reinterpret_cast<__nv_bfloat162*>(&u[e]);
                lsum += __low2float(v2) + __high2float(v2);
                lsum_exp += a + b;
              }
              if (owner) {
                const int chunk = 4 * half + c8;
                *reinterpret_cast<uint4*>(prow + ((chunk ^ (h & 7)) << 4)) =
                    make_uint4(u[0], u[1], u[2], u[3]);
              }
            }
            l_run += lsum + __shfl_xor_sync(0xffffffffu, lsum, 16);
            l_exp += lsum_exp + __shfl_xor_sync(0xffffffffu, lsum_exp, 16);
            if (owner && half == 0) ctrl->alpha[pb][h] = alpha;
          }
          if constexpr (MT::kDenseBf16) {
            // Dead rows (tail slots, bad pages): P is 0 there but 0 * NaN
            // would poison the PV sum, so zero their latent values.  (The
            // sparse producer zero-fills them; the FP8 dequant writes zeros.)
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
        // A segment ends at this tile: its epilogue waits for PV(i), which
        // shares o_done[i % 2] with PV(i-2).  A parity wait cannot tell a
        // phase from the one two later, so every warp awaits PV(i-2) before
        // the warps meet and PV(i) is issued (PV(i-4) is complete: the stage
        // tile i fills was released by PV(i-3)).
        if (last && i >= 2 && ok) ok = pv_done(i - 2);
        // P(i) and the zeroed dead rows are generic stores the tensor core
        // reads: fenced by their writers before the warps meet
        fence_proxy_async_smem();
        if (named_bar_or(1, 128, !ok)) { failed = true; break; }
        if (!first && ctrl->rescale_tile[pb] == i) {
          // every earlier PV has completed before O^T is rescaled in place
          ok = (i < 2 || pv_done(i - 2)) && pv_done(i - 1);
          if (ok) {
            tc_fence_after();
            for (int mt = 0; mt < 4; ++mt) {
              for (int hb = 0; hb < nrows; hb += 16) {
                uint32_t v[16];
                const uint32_t addr = tmem + lane_base + MT::kColO + mt * NP + hb;
                tmem_ld16(addr, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const int hh = hb + e;
                  const float a = hh < nrows ? ctrl->alpha[pb][hh] : 1.f;
                  v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
                }
                tmem_st16(addr, v);
              }
            }
          }
          // the rescaled O^T is in place before PV(i) adds to it
          tc_fence_before();
          if (named_bar_or(1, 128, !ok)) { failed = true; break; }
        }
        {
          // PV(i), one 128-dim block b of O^T += V^T P^T over the staged tile
          // per issuer: lane 0 of each softmax warp w (b = w; four warps
          // overlap in the tensor pipe), lanes 0-1 of warps 0-1 (b = 2w +
          // lane; one-token FP8), or lanes 0-3 of warp 0, which holds no rows
          // (b = lane; multi-token).  Each issuer then commits its block to o_done[i % 2] and
          // to the stage's empty barrier (o_done first: a stage seen free
          // implies its PV seen done).
          const bool issuer = MT::kPvTwoWarps ? (w < 2 && lane < 2)
                              : MT::kPvOneWarp ? (w == 0 && lane < kPvLanes) : lane == 0;
          if (issuer) {
            const int b = MT::kPvTwoWarps ? 2 * w + lane : MT::kPvOneWarp ? lane : w;
            tc_fence_after();
            issue_pv_block(tmem + MT::kColO + b * NP,
                           pv_a0 + static_cast<uint64_t>((stage * kTileBytes) >> 4),
                           pv_b0 + static_cast<uint64_t>((stage * kTileBytes) >> 4), idesc_pv, b,
                           first);
            mma_commit(&ctrl->o_done[i & 1]);
            mma_commit(&ctrl->empty[stage]);
          }
          __syncwarp();
        }
        if (last && i + 1 < ntiles) {
          // The next tile opens another stream: its queries replace this
          // stream's in TMEM.  S(i) was this stream's last QK and it has
          // completed, so nothing reads the old queries any more.  Loaded
          // once P(i) is out, so that the load overlaps this segment's
          // epilogue (which first waits for PV(i)) instead of delaying P(i).
          Walker nx = wk;
          nx.next(prefix, S);
          load_rows(nx.s);
          if constexpr (MT::kQRopeSmem) fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->q_ready);
        }
        if (last) {
          // ---- segment epilogue
          ok = !failed && pv_done(i);   // PVs complete in order: all of them
          const int32_t s = wk.s;
          const int32_t c_first =
              tile_owner(tile_cost_pos(cprefix[s], 0, p.stream_cost), ucost, nctas);
          const int32_t c_last = tile_owner(
              tile_cost_pos(cprefix[s], prefix[s + 1] - prefix[s] - 1, p.stream_cost), ucost,
              nctas);
          const bool split = c_first != c_last;
          // an unsplit stream's result is final: straight to the outputs
          // (partial slots hold RMAX rows each)
          float* dst_o = split ? p.part_o + static_cast<int64_t>(s + c) * RMAX * kDc
                               : p.o_lat + first_row(s) * kDc;
          float* dst_lse = split ? p.part_lse + static_cast<int64_t>(s + c) * RMAX
                                 : p.lse + first_row(s);
          if (ok && owner && half == 0) {
            ctrl->l_final[h] = l_run > 0.f ? 1.f / l_run : 0.f;   // o = O / l
            dst_lse[h] = l_run > 0.f ? (m_used + __log2f(l_exp)) * kLn2 : -INFINITY;
          }
          if (named_bar_or(1, 128, !ok || failed)) { failed = true; break; }
          tc_fence_after();
          for (int mt = 0; mt < 4; ++mt) {
            const int d = mt * 128 + w * 32 + lane;
            for (int hb = 0; hb < nrows; hb += 16) {
              uint32_t v[16];
              tmem_ld16(tmem + lane_base + MT::kColO + mt * NP + hb, v);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int hh = hb + e;
                if (hh < nrows) dst_o[static_cast<int64_t>(hh) * kDc + d] = __uint_as_float(v[e]) * ctrl->l_final[hh];
              }
            }
          }
          // O^T is read before the next PV (issued after the warps next
          // meet) overwrites it
          tc_fence_before();
        }
        wk.next(prefix, S);
      }
      if (failed && lane == 0) {
        set_status(p.status, MLA_STATUS_TIMEOUT);
        ctrl->abort_flag = 1;
      }
      // drain: every PV issued here completes before tensor memory is released
      if (MT::kPvTwoWarps ? (w < 2 && lane < 2) : MT::kPvOneWarp ? (w == 0 && lane < kPvLanes) : lane == 0)
        mma_commit(&ctrl->mma_drain[1]);
      if (lane == 0 && (MT::kPvTwoWarps ? w < 2 : (!MT::kPvOneWarp || w == 0)))
        (void)mbar_wait(&ctrl->mma_drain[1], 0, nullptr, kWaitLimitNs);
      __syncwarp();
    }
  }


  // Row sets with no visible token (no tile anywhere): o_lat = 0, lse = -inf.
  for (int s = c; s < S; s += p.num_ctas) {
    if (prefix[s + 1] != prefix[s]) continue;
    const StreamGeom gm = stream_geom(s, p.q_len, G);
    const int64_t row0 = (static_cast<int64_t>(gm.b) * p.q_len + gm.j0) * H;
    const int nr = gm.nq * H;
    float4* o = reinterpret_cast<float4*>(p.o_lat + row0 * kDc);
    for (int e = tid; e < nr * kDc / 4; e += kThreads) o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e = tid; e < nr; e += kThreads) p.lse[row0 + e] = -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

namespace {
template <int kMode>
cudaError_t launch_mode(const CUtensorMap* kv_map, const DecodeParams& p, const DecodeLayout& L,
                        cudaStream_t stream) {
  const cudaError_t err =
      set_smem_attr_once(reinterpret_cast<const void*>(mla_decode_kernel<kMode>), 3 + kMode, L.total);
  if (err != cudaSuccess) return err;
  if (p.prefix_ws == nullptr) {
    mla_decode_kernel<kMode>
        <<<dim3(p.num_ctas), dim3(ModeTraits<kMode>::kThreads), L.total, stream>>>(*kv_map, p, L);
    return cudaGetLastError();
  }
  // behind the prefix pre-pass: a programmatic dependent of it (the kernel
  // waits for it before reading memory)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_ctas);
  cfg.blockDim = dim3(ModeTraits<kMode>::kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(L.total);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<kMode>, *kv_map, p, L);
}
}  // namespace

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap* kv_map, int mode,
                          cudaStream_t stream) {
  const DecodeLayout L = decode_layout(p.heads, p.heads_pad, p.num_streams, mode);
  switch (mode) {
    case kModeDenseBf16: return launch_mode<kModeDenseBf16>(kv_map, p, L, stream);
    case kModeSparseBf16: return launch_mode<kModeSparseBf16>(kv_map, p, L, stream);
    case kModeDenseFp8: return launch_mode<kModeDenseFp8>(kv_map, p, L, stream);
    case kModeDenseFp4: return launch_mode<kModeDenseFp4>(kv_map, p, L, stream);
    case kModeDenseMulti: return launch_mode<kModeDenseMulti>(kv_map, p, L, stream);
    case kModeDenseFp4Multi: return launch_mode<kModeDenseFp4Multi>(kv_map, p, L, stream);
    case kModeDenseFp8Multi: return launch_mode<kModeDenseFp8Multi>(kv_map, p, L, stream);
    default: return cudaErrorInvalidValue;
  }
}

int decode_smem_bytes(int heads, int heads_pad, int num_streams, int mode) {
  return decode_layout(heads, heads_pad, num_streams, mode).total;
}

}  // namespace mla
