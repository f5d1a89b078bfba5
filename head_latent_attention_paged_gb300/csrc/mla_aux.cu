// The smaller kernels of the decode step:
//   * mla_combine_kernel : LSE merge of the split-KV partials of each row set
//                          (one block per row: a head, or a draft token x head);
//   * mla_uv_kernel      : o = W_UV[h]^T o_lat (tcgen05, per head); its
//                          merging variant also does the LSE merge of the
//                          split rows (the decode step's second launch);
//   * mla_absorb_kernel  : q_hat = [W_UK[h] q_nope || q_rope] (query absorption,
//                          tcgen05).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "mla_internal.h"
#include "mla_merge.cuh"
#include "sm103_ptx.cuh"

namespace mla {

namespace {
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}
}  // namespace

// ----------------------------------------------------------------------------
// combine: one block per (row set, row); thread t owns latent dims
// [4t, 4t + 4).  Launched as a programmatic dependent of the decode kernel:
// the work split is derived from seq_lens while the decode runs, then every
// block waits for the decode grid (whose partials it reads) before touching
// its outputs.  Every block waits, even one with nothing to merge, so this
// grid never completes before the decode grid does (the W_UV launch after
// it relies on that for the rows the decode wrote directly).
// ----------------------------------------------------------------------------
namespace {
constexpr int kCombineThreads = 128;   // x 4 dims = 512 latent dims
}  // namespace

__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(const CombineParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int s = blockIdx.x, h = blockIdx.y;   // row h of row set s (a head, or draft x head)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.num_streams;
  const int max_tokens = p.max_pages * p.page_size;
  __shared__ int64_t red64[3][kCombineThreads / 32];
  // cost before stream s, in total, and the total tile count (the decode
  // grid's split): summed here while the decode runs, or read from the
  // pre-pass's prefixes
  int64_t before = 0, tot = 0, tiles = 0;
  if (p.prefix_ws == nullptr) {
    for (int t = tid; t < S; t += kCombineThreads) {
      const StreamGeom gt = stream_geom(t, p.q_len, p.group);
      const int32_t len = stream_len(p.seq_lens[gt.b], p.q_len, gt.j0 + gt.nq - 1, p.causal,
                                     p.topk_width, max_tokens);
      const int32_t nt = (len + kTile - 1) / kTile;
      const int64_t n = stream_cost(nt, p.stream_cost);
      tot += n;
      tiles += nt;
      if (t < s) before += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
    }
    if (lane == 0) { red64[0][warp] = before; red64[1][warp] = tot; red64[2][warp] = tiles; }
    __syncthreads();
    before = tot = tiles = 0;
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) {
      before += red64[0][w];
      tot += red64[1][w];
      tiles += red64[2][w];
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (p.prefix_ws != nullptr) {
    before = p.prefix_ws[S + 1 + s];
    tot = p.prefix_ws[S + 1 + S];
    tiles = p.prefix_ws[S];
  }
  const int32_t nctas = work_ctas(p.num_ctas, static_cast<int32_t>(tiles));
  const StreamGeom gm = stream_geom(s, p.q_len, p.group);
  if (h >= gm.nq * p.heads) return;   // a short last group of draft tokens
  const int32_t len = stream_len(p.seq_lens[gm.b], p.q_len, gm.j0 + gm.nq - 1, p.causal,
                                 p.topk_width, max_tokens);
  const int64_t ntiles = (len + kTile - 1) / kTile;
  if (ntiles == 0) return;   // the decode wrote o_lat = 0, lse = -inf
  const int c0 = tile_owner(tile_cost_pos(before, 0, p.stream_cost), tot, nctas);
  const int c1 = tile_owner(tile_cost_pos(before, static_cast<int32_t>(ntiles - 1), p.stream_cost),
                            tot, nctas);
  if (c0 == c1) return;      // one CTA held the whole row set: its result is final
  const int nseg = c1 - c0 + 1;
  // partial slots hold p.rows rows each
  const float* plse = p.part_lse + static_cast<int64_t>(s + c0) * p.rows + h;
  const float4* po = reinterpret_cast<const float4*>(p.part_o) +
                     (static_cast<int64_t>(s + c0) * p.rows + h) * (kDc / 4) + tid;
  const int64_t ostride = static_cast<int64_t>(p.rows) * (kDc / 4);
  // every warp finds the weights (the same bits), then each thread merges
  // its 4 dims, 8 partials' loads in flight at a time
  const RowWeights rw = merge_weights(plse, nseg, p.rows);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < nseg; k0 += 8) {
    float lv[8];
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = k0 + u < nseg;
      lv[u] = in ? __ldcg(plse + (k0 + u) * static_cast<int64_t>(p.rows)) : -INFINITY;
      v[u] = in ? __ldcg(po + (k0 + u) * ostride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (k0 + u < nseg) merge_fma(acc, merge_weight(lv[u], rw.m), v[u]);
  }
  const int64_t row = (static_cast<int64_t>(gm.b) * p.q_len + gm.j0) * p.heads + h;
  reinterpret_cast<float4*>(p.o_lat + row * kDc)[tid] = merge_scale(acc, rw.inv);
  if (tid == 0) p.lse[row] = rw.lse;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  if (p.num_streams == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_streams, p.rows);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, mla_combine_kernel, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Row-set prefixes for the work split (grids with more row sets than the
// decode kernel keeps in shared memory): tiles[s] and cost[s] = tiles and
// cost units of the row sets before s, for s = 0..S, in p.prefix_ws as
// int32 [2][S + 1].  One block of 1024 threads scans 1024 row sets at a time.
constexpr int kPrefixThreads = 1024;

__global__ void __launch_bounds__(kPrefixThreads) mla_prefix_kernel(const DecodeParams p) {
  __shared__ int32_t wsum[2][kPrefixThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = p.num_streams;
  const int32_t max_tokens = p.max_pages * p.page_size;
  int32_t* tiles = p.prefix_ws;
  int32_t* cost = p.prefix_ws + S + 1;
  if (tid == 0) {
    tiles[0] = 0;
    cost[0] = 0;
  }
  int32_t carry_t = 0, carry_c = 0;
  for (int base = 0; base < S; base += kPrefixThreads) {
    const int s = base + tid;
    int32_t vt = 0, vc = 0;
    if (s < S) {
      const StreamGeom gm = stream_geom(s, p.q_len, p.group);
      const int32_t len = stream_len(p.seq_lens[gm.b], p.q_len, gm.j0 + gm.nq - 1, p.causal,
                                     p.topk_width, max_tokens);
      vt = (len + kTile - 1) / kTile;
      vc = stream_cost(vt, p.stream_cost);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {   // inclusive scan within the warp
      const int32_t nt = __shfl_up_sync(0xffffffffu, vt, o);
      const int32_t nc = __shfl_up_sync(0xffffffffu, vc, o);
      if (lane >= o) {
        vt += nt;
        vc += nc;
      }
    }
    if (lane == 31) {
      wsum[0][warp] = vt;
      wsum[1][warp] = vc;
    }
    __syncthreads();
    if (warp == 0) {   // inclusive scan of the warp totals
      int32_t wt = wsum[0][lane], wc = wsum[1][lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t nt = __shfl_up_sync(0xffffffffu, wt, o);
        const int32_t nc = __shfl_up_sync(0xffffffffu, wc, o);
        if (lane >= o) {
          wt += nt;
          wc += nc;
        }
      }
      wsum[0][lane] = wt;
      wsum[1][lane] = wc;
    }
    __syncthreads();
    if (warp > 0) {
      vt += wsum[0][warp - 1];
      vc += wsum[1][warp - 1];
    }
    if (s < S) {
      tiles[s + 1] = carry_t + vt;
      cost[s + 1] = carry_c + vc;
    }
    carry_t += wsum[0][kPrefixThreads / 32 - 1];
    carry_c += wsum[1][kPrefixThreads / 32 - 1];
    __syncthreads();   // wsum is rewritten by the next round
  }
}

cudaError_t launch_prefix(const DecodeParams& p, cudaStream_t stream) {
  mla_prefix_kernel<<<1, kPrefixThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// UV projection: per (head h, 128 output dims, N rows):
//   D^T[n, r] = sum_k W_UV[h][k][n] * o_lat[r][h][k]
// A = W_UV slice (MN-major, TMA), B = o_lat rows converted to bf16 (K-major,
// written by the threads, all loads issued before any is used), D in TMEM.
// A tcgen05.mma costs its issuing thread a fixed time, so the 32 K-steps go
// out from four threads (warps 0-3, 128 latent dims each) into four
// accumulators that the epilogue sums.  N (16, 32 or 64 rows) is the smallest
// row block whose grid fits the SMs, where one does.
//
// The merging variant (kMerge) is the step's last launch: it builds B from
// the decode's output directly, merging the partials of the rows whose row
// set was split over several CTAs (the same arithmetic as the merge kernel)
// and writing those rows' merged o_lat and lse.  The two CTAs of the output
// halves of one (head, row block) form a cluster: each merges half of the
// rows and stores them, as bf16, into its own B and into the other's
// (distributed shared memory), so every partial is read once.  The 512
// threads keep four partials' loads in flight each; the work split is found
// while the decode still runs.
// ----------------------------------------------------------------------------
namespace {
constexpr int kUvA = 8 * 2 * kChunkBytes;   // 8 K-blocks x 2 n-chunks x 8 KB = 128 KB

struct MergeRow {   // one row of a merging block
  int64_t obase;    // float4 index: the first partial's o (nseg > 0), the o_lat row (nseg == 0)
  int64_t lbase;    // float index of the first partial's lse
  int64_t orow;     // the row of o_lat and lse
  int32_t nseg;     // > 0: partials to merge; 0: the decode's o_lat row is final; -1: no row
  float m, inv;
  int32_t pad;
};

template <int N, bool kMerge>
struct Uv {
  static constexpr int kThreads = kMerge ? 512 : (N == 64 ? 256 : 128);
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kB = 8 * N * 128;                     // 8 K-blocks x N rows x 128 B
  // 16-byte B pieces per thread (a merging CTA builds half of the rows)
  static constexpr int kPieces = (kMerge ? N / 2 : N) * 64 / kThreads;
  // four accumulators of N columns, in an allocation of a power of two >= 32
  static constexpr int kTmemCols = 4 * N <= 32 ? 32 : (4 * N <= 64 ? 64 : (4 * N <= 128 ? 128 : 256));
  // merging blocks: N MergeRow, N + 1 row-set cost prefixes, 2 x kWarps scan sums
  static constexpr int kScratch =
      kMerge ? static_cast<int>(N * sizeof(MergeRow)) + (N + 1 + 2 * kWarps) * 4 : 0;
  static constexpr int kSmem = kUvA + kB + 1024 + 64 + kScratch;
};

// Piece (row r, 8 latent dims 8 piece ..) of B as bf16: K-block piece / 8 of
// the 128-byte-swizzled [kb][N rows][128 B] layout.  Returns its byte offset.
template <int N>
__device__ __forceinline__ uint32_t store_b_piece(uint8_t* sB, int r, int piece, float4 a, float4 b) {
  const int kb = piece >> 3, w16 = piece & 7;
  __nv_bfloat162 x0 = __floats2bfloat162_rn(a.x, a.y), x1 = __floats2bfloat162_rn(a.z, a.w);
  __nv_bfloat162 x2 = __floats2bfloat162_rn(b.x, b.y), x3 = __floats2bfloat162_rn(b.z, b.w);
  const uint32_t off = kb * (N * 128) + r * 128 + ((w16 ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(sB + off) =
      make_uint4(*reinterpret_cast<uint32_t*>(&x0), *reinterpret_cast<uint32_t*>(&x1),
                 *reinterpret_cast<uint32_t*>(&x2), *reinterpret_cast<uint32_t*>(&x3));
  return off;
}
}  // namespace

template <int N, bool kMerge>
__global__ void __launch_bounds__(Uv<N, kMerge>::kThreads, 1)
    mla_uv_kernel(const __grid_constant__ CUtensorMap w_map, const float* o_lat,
                  uint16_t* __restrict__ out, int rows, int heads,
                  const __grid_constant__ CombineParams mp) {
  constexpr int kThreads = Uv<N, kMerge>::kThreads;
  constexpr int kWarps = Uv<N, kMerge>::kWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kUvA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kUvA + Uv<N, kMerge>::kB);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  MergeRow* mrow = reinterpret_cast<MergeRow*>(smem + kUvA + Uv<N, kMerge>::kB + 64);
  int32_t* sbefore = reinterpret_cast<int32_t*>(mrow + N);   // cost before row set s_lo + i
  int32_t* wsum = sbefore + N + 1;                           // [2][kWarps]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int mt = blockIdx.y;          // output dims [128 mt, 128 mt + 128)
  const int r0 = blockIdx.z * N;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 4);           // one commit per issuer
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, Uv<N, kMerge>::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  // merging blocks write into the other CTA of their cluster: it must have
  // started first (this arrive; the matching wait precedes the first store)
  if constexpr (kMerge) cluster_arrive_relaxed();
  if (tid == 0) {
    prefetch_tmap(&w_map);
    mbar_arrive_expect_tx(&bars[0], kUvA);
    for (int kb = 0; kb < 8; ++kb)
      for (int nc = 0; nc < 2; ++nc)
        tma_load_2d(sA + (kb * 2 + nc) * kChunkBytes, &w_map, &bars[0], mt * 128 + nc * 64,
                    h * kDc + kb * 64, 0ull);
  }
  // Merging blocks: row set s of token row R (request b = R / q_len, draft
  // j = R % q_len) is b * ng + j / group.  This block's rows span the row
  // sets s_lo .. s_hi (at most N of them).  The cost before each of them,
  // the total cost and the total tile count give the decode grid's split
  // (the CTAs c0 .. c1 whose partials hold the row set): summed here from
  // seq_lens (an input of the step) before the wait when the decode kernel
  // kept its prefixes in shared memory, else read from the pre-pass's.
  [[maybe_unused]] const int S = mp.num_streams;
  [[maybe_unused]] const int32_t ng = kMerge ? (mp.q_len + mp.group - 1) / mp.group : 1;
  [[maybe_unused]] const int32_t max_tokens = mp.max_pages * mp.page_size;
  // merging blocks run as clusters of the two output halves of one (head,
  // row block): of the block's cnt rows, cluster CTA q merges the q-th half
  // (rows first .. first + mine - 1) and hands them as bf16 to both halves' B
  constexpr int kHalf = N / 2;
  [[maybe_unused]] const uint32_t crank = kMerge ? cluster_ctarank() : 0u;
  [[maybe_unused]] const int cnt = rows - r0 < N ? rows - r0 : N;
  [[maybe_unused]] const int first = static_cast<int>(crank) * ((cnt + 1) / 2);
  [[maybe_unused]] const int mine = crank == 0 ? (cnt + 1) / 2 : cnt / 2;
  [[maybe_unused]] const int my_r = warp * 4 + (lane >> 3);   // a row of the half per 8 lanes
  [[maybe_unused]] int32_t s_lo = 0, s_hi = 0, tot = 0, tiles = 0;
  [[maybe_unused]] int32_t g_nseg = -1;
  [[maybe_unused]] int64_t g_lbase = 0, g_obase = 0, g_orow = 0;
  [[maybe_unused]] auto geometry = [&]() {
    const int R = r0 + first + my_r;
    if (my_r >= mine) return;
    const int b = R / mp.q_len, j = R - b * mp.q_len;
    const int32_t s = b * ng + j / mp.group;
    const StreamGeom gm = stream_geom(s, mp.q_len, mp.group);
    g_orow = static_cast<int64_t>(R) * heads + h;
    g_obase = g_orow * (kDc / 4);
    g_nseg = 0;
    const int32_t len = stream_len(mp.seq_lens[b], mp.q_len, gm.j0 + gm.nq - 1, mp.causal,
                                   mp.topk_width, max_tokens);
    const int32_t nt = (len + kTile - 1) / kTile;
    if (nt == 0) return;   // the decode wrote o_lat = 0, lse = -inf
    const int32_t nctas = work_ctas(mp.num_ctas, tiles);
    const int64_t before = sbefore[s - s_lo];
    const int c0 = tile_owner(tile_cost_pos(before, 0, mp.stream_cost), tot, nctas);
    const int c1 = tile_owner(tile_cost_pos(before, nt - 1, mp.stream_cost), tot, nctas);
    if (c0 == c1) return;  // one CTA held the whole row set: its o_lat row is final
    g_nseg = c1 - c0 + 1;
    // partial slots hold mp.rows rows each; the row's index in its row set
    g_lbase = static_cast<int64_t>(s + c0) * mp.rows + (j - gm.j0) * heads + h;
    g_obase = g_lbase * (kDc / 4);
  };
  if constexpr (kMerge) {
    const int last = (r0 + N < rows ? r0 + N : rows) - 1;
    s_lo = (r0 / mp.q_len) * ng + (r0 % mp.q_len) / mp.group;
    s_hi = (last / mp.q_len) * ng + (last % mp.q_len) / mp.group;
    if (mp.prefix_ws == nullptr) {
      int32_t carry_c = 0, carry_t = 0;
      for (int base = 0; base < S; base += kThreads) {
        const int t = base + tid;
        int32_t vt = 0, vc = 0;
        if (t < S) {
          const StreamGeom gt = stream_geom(t, mp.q_len, mp.group);
          const int32_t len = stream_len(mp.seq_lens[gt.b], mp.q_len, gt.j0 + gt.nq - 1,
                                         mp.causal, mp.topk_width, max_tokens);
          vt = (len + kTile - 1) / kTile;
          vc = stream_cost(vt, mp.stream_cost);
        }
        const int32_t own = vc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {   // inclusive scans within the warp
          const int32_t nt = __shfl_up_sync(0xffffffffu, vt, o);
          const int32_t nc = __shfl_up_sync(0xffffffffu, vc, o);
          if (lane >= o) {
            vt += nt;
            vc += nc;
          }
        }
        if (lane == 31) {
          wsum[warp] = vc;
          wsum[kWarps + warp] = vt;
        }
        __syncthreads();
        if (warp == 0) {   // inclusive scans of the warp totals
          int32_t wc = lane < kWarps ? wsum[lane] : 0, wt = lane < kWarps ? wsum[kWarps + lane] : 0;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int32_t nc = __shfl_up_sync(0xffffffffu, wc, o);
            const int32_t nt = __shfl_up_sync(0xffffffffu, wt, o);
            if (lane >= o) {
              wc += nc;
              wt += nt;
            }
          }
          if (lane < kWarps) {
            wsum[lane] = wc;
            wsum[kWarps + lane] = wt;
          }
        }
        __syncthreads();
        if (t >= s_lo && t <= s_hi)
          sbefore[t - s_lo] = carry_c + (warp > 0 ? wsum[warp - 1] : 0) + vc - own;
        carry_c += wsum[kWarps - 1];
        carry_t += wsum[2 * kWarps - 1];
        __syncthreads();   // sbefore is complete; wsum is rewritten by the next round
      }
      tot = carry_c;
      tiles = carry_t;
      geometry();
    }
  }
  // o_lat and the partials are produced by the launch this one depends on:
  // wait for it (the W_UV loads above already overlap its tail).  o_lat is
  // not a restrict-qualified pointer on purpose: read-only-for-the-kernel
  // loads could be scheduled ahead of this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (kMerge) {
    if (mp.prefix_ws != nullptr) {
      tiles = __ldcg(mp.prefix_ws + S);
      tot = __ldcg(mp.prefix_ws + 2 * S + 1);
      for (int t = s_lo + tid; t <= s_hi; t += kThreads)
        sbefore[t - s_lo] = __ldcg(mp.prefix_ws + S + 1 + t);
      __syncthreads();
      geometry();
    }
    // every warp calls this (each 8-lane group for its own row, or none)
    const RowWeights rw = merge_weights(mp.part_lse + g_lbase, g_nseg > 0 ? g_nseg : 0, mp.rows);
    if (my_r < kHalf && (lane & (kMergeLanes - 1)) == 0) {
      MergeRow& mr = mrow[my_r];
      mr.obase = g_obase;
      mr.lbase = g_lbase;
      mr.orow = g_orow;
      mr.nseg = g_nseg;
      mr.m = rw.m;
      mr.inv = rw.inv;
      if (g_nseg > 0) mp.lse[g_orow] = rw.lse;
    }
    __syncthreads();
    // B: thread t takes piece t % 64 (8 latent dims) of this CTA's rows
    // t / 64 + 8 e (the 32 threads of a warp share their rows), up to four
    // rows at a time, with the loads of 4 / rows partials of each in flight
    const int piece = tid & 63;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* po4 = reinterpret_cast<const float4*>(mp.part_o);
    const float4* ol4 = reinterpret_cast<const float4*>(o_lat);
    float4* ow4 = reinterpret_cast<float4*>(mp.o_lat);
    const int64_t lstride = mp.rows;
    const int64_t ostride = static_cast<int64_t>(mp.rows) * (kDc / 4);
    constexpr int kPieces = Uv<N, kMerge>::kPieces;
    constexpr int kPass = kPieces < 4 ? kPieces : 4;   // rows per pass
    constexpr int kSegU = 4 / kPass;                    // partials per row per load round
    cluster_wait();   // both CTAs of the cluster run
#pragma unroll 1
    for (int p0 = 0; p0 < kPieces; p0 += kPass) {
      float4 va[kPass], vb[kPass];
      int32_t nseg[kPass];
      int64_t ob[kPass], lb[kPass];
      float wm[kPass];
      int32_t maxseg = 0;
#pragma unroll
      for (int e = 0; e < kPass; ++e) {
        const MergeRow& mr = mrow[(tid >> 6) + (kThreads / 64) * (p0 + e)];
        nseg[e] = mr.nseg;
        ob[e] = mr.obase + 2 * piece;
        lb[e] = mr.lbase;
        wm[e] = mr.m;
        const bool direct = mr.nseg == 0;
        va[e] = direct ? __ldcg(ol4 + ob[e]) : zero;
        vb[e] = direct ? __ldcg(ol4 + ob[e] + 1) : zero;
        maxseg = mr.nseg > maxseg ? mr.nseg : maxseg;
      }
      for (int i0 = 0; i0 < maxseg; i0 += kSegU) {
        float lv[kPass][kSegU];
        float4 xa[kPass][kSegU], xb[kPass][kSegU];
#pragma unroll
        for (int e = 0; e < kPass; ++e)
#pragma unroll
          for (int u = 0; u < kSegU; ++u) {
            const int64_t i = i0 + u;
            const bool in = i < nseg[e];
            lv[e][u] = in ? __ldcg(mp.part_lse + lb[e] + i * lstride) : -INFINITY;
            xa[e][u] = in ? __ldcg(po4 + ob[e] + i * ostride) : zero;
            xb[e][u] = in ? __ldcg(po4 + ob[e] + i * ostride + 1) : zero;
          }
#pragma unroll
        for (int e = 0; e < kPass; ++e)
#pragma unroll
          for (int u = 0; u < kSegU; ++u)
            if (i0 + u < nseg[e]) {   // partials in increasing order
              const float w = merge_weight(lv[e][u], wm[e]);
              merge_fma(va[e], w, xa[e][u]);
              merge_fma(vb[e], w, xb[e][u]);
            }
      }
#pragma unroll
      for (int e = 0; e < kPass; ++e) {
        const int rr = (tid >> 6) + (kThreads / 64) * (p0 + e);   // row of the half
        if (rr >= mine) continue;   // the other CTA's row, or past the block's last
        const int r = first + rr;
        if (nseg[e] > 0) {
          const MergeRow& mr = mrow[rr];
          va[e] = merge_scale(va[e], mr.inv);
          vb[e] = merge_scale(vb[e], mr.inv);
          ow4[mr.orow * (kDc / 4) + 2 * piece] = va[e];
          ow4[mr.orow * (kDc / 4) + 2 * piece + 1] = vb[e];
        }
        const uint32_t off = store_b_piece<N>(sB, r, piece, va[e], vb[e]);
        st_cluster_v4(mapa_shared(smem_u32(sB) + off, crank ^ 1u),
                      *reinterpret_cast<const uint4*>(sB + off));
      }
    }
  } else {
    // B: o_lat[r0 + r][h][k] -> bf16, [kb][r][128 B] swizzled.  Item e of
    // this thread is piece (tid + kThreads e): row (tid + kThreads e) / 64,
    // 8 consecutive k.
    float4 va[Uv<N, kMerge>::kPieces], vb[Uv<N, kMerge>::kPieces];
#pragma unroll
    for (int e = 0; e < Uv<N, kMerge>::kPieces; ++e) {
      const int idx = tid + kThreads * e;
      const int r = idx >> 6, piece = idx & 63;
      if (r0 + r < rows) {
        const float4* src = reinterpret_cast<const float4*>(
            o_lat + (static_cast<int64_t>(r0 + r) * heads + h) * kDc + piece * 8);
        va[e] = src[0];
        vb[e] = src[1];
      } else {
        va[e] = vb[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int e = 0; e < Uv<N, kMerge>::kPieces; ++e) {
      const int idx = tid + kThreads * e;
      store_b_piece<N>(sB, idx >> 6, idx & 63, va[e], vb[e]);
    }
  }
  fence_proxy_async_smem();
  if constexpr (kMerge) {
    fence_proxy_async_all();   // this thread's stores into the other CTA's B, too
    cluster_sync_all();        // both halves of B are in both CTAs
    fence_proxy_async_all();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (warp < 4) {
    // issuer w: K-blocks 2w, 2w + 1 (latent dims [128 w, 128 w + 128)) into
    // the accumulator at column N w
    if (lane == 0) {
      const bool ok = mbar_wait(&bars[0], 0, nullptr, kWaitLimitNs);
      tc_fence_after();
      if (ok) {
        const uint32_t idesc = make_idesc_bf16(128, N, true, false);
        const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
        for (int kb = 2 * warp; kb < 2 * warp + 2; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = make_smem_desc(a_base + kb * 2 * kChunkBytes + kk * 2048,
                                               kChunkBytes, 1024, kSmemLayoutSW128);
            const uint64_t bd = make_smem_desc(b_base + kb * (N * 128) + kk * 32, 16, 1024,
                                               kSmemLayoutSW128);
            mma_bf16_ss(tmem + N * warp, ad, bd, idesc, (kb > 2 * warp || kk > 0) ? 1u : 0u);
          }
        }
      }
      mma_commit(&bars[1]);
    }
    __syncwarp();
    if (mbar_wait(&bars[1], 0, nullptr, kWaitLimitNs)) {
      tc_fence_after();
      // warp w reads TMEM lanes 32 w .. (output dims), every column (row)
      const int n = mt * 128 + warp * 32 + lane;
      const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
      for (int cb = 0; cb < N; cb += 16) {
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t v[16];
          tmem_ld16(tmem + lb + N * q + cb, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] += __uint_as_float(v[e]);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = r0 + cb + e;
          if (r < rows) out[(static_cast<int64_t>(r) * heads + h) * kDv + n] = float_to_bf16_bits(acc[e]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Uv<N, kMerge>::kTmemCols);
  }
}

namespace {
template <int N, bool kMerge>
cudaError_t launch_uv(const CUtensorMap* w_map, const float* o_lat, uint16_t* out, int rows,
                      int heads, const CombineParams& mp, cudaStream_t stream) {
  // attribute slots: 1, 2, 10 (projection), 11, 12, 14, 13 (merging projection)
  const int slot = kMerge ? (N == 16 ? 11 : (N == 32 ? 12 : (N == 48 ? 14 : 13)))
                          : (N == 16 ? 1 : (N == 32 ? 2 : 10));
  cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(mla_uv_kernel<N, kMerge>),
                                       slot, Uv<N, kMerge>::kSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(heads, kDv / 128, (rows + N - 1) / N);
  cfg.blockDim = dim3(Uv<N, kMerge>::kThreads);
  cfg.dynamicSmemBytes = Uv<N, kMerge>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;   // the two output halves
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = kDv / 128;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kMerge ? 2 : 1;
  err = cudaLaunchKernelEx(&cfg, mla_uv_kernel<N, kMerge>, *w_map, o_lat, out, rows, heads, mp);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// The row block: 16 rows for at most 16, else the smallest of 32, 48
// (merging blocks only) and 64 whose grid fits the SMs (64 when none does).
template <bool kMerge>
cudaError_t launch_uv_rows(const CUtensorMap* w_map, const float* o_lat, uint16_t* out, int rows,
                           int heads, int sm_count, const CombineParams& mp, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  auto blocks = [&](int n) { return heads * (kDv / 128) * ((rows + n - 1) / n); };
  if (rows <= 16) return launch_uv<16, kMerge>(w_map, o_lat, out, rows, heads, mp, stream);
  if (blocks(32) <= sm_count) return launch_uv<32, kMerge>(w_map, o_lat, out, rows, heads, mp, stream);
  if (kMerge && blocks(48) <= sm_count)
    return launch_uv<48, kMerge>(w_map, o_lat, out, rows, heads, mp, stream);
  return launch_uv<64, kMerge>(w_map, o_lat, out, rows, heads, mp, stream);
}
}  // namespace

cudaError_t launch_uv_proj_tma(const CUtensorMap* w_map, const float* o_lat, uint16_t* out,
                               int rows, int heads, int sm_count, cudaStream_t stream) {
  const CombineParams none = {};
  return launch_uv_rows<false>(w_map, o_lat, out, rows, heads, sm_count, none, stream);
}

cudaError_t launch_merge_uv(const CUtensorMap* w_map, const CombineParams& p, uint16_t* out,
                            int sm_count, cudaStream_t stream) {
  if (p.num_streams == 0) return cudaSuccess;
  return launch_uv_rows<true>(w_map, p.o_lat, out, p.batch * p.q_len, p.heads, sm_count, p, stream);
}

// ----------------------------------------------------------------------------
// bounded-wait self-test: every thread waits for a phase of an mbarrier that
// nothing arrives on; mbar_wait gives up after limit_ns, and the block
// reports MLA_STATUS_TIMEOUT like a kernel whose pipeline stalled.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(64) mla_wait_selftest_kernel(uint32_t* status, uint64_t limit_ns,
                                                               uint64_t* waited_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = globaltimer_ns();
  const bool ok = mbar_wait(&bar, 0, nullptr, limit_ns);
  const uint64_t dt = globaltimer_ns() - t0;
  const bool any_gave_up = __syncthreads_or(!ok);
  if (threadIdx.x == 0) {
    if (any_gave_up) atomicOr(status, MLA_STATUS_TIMEOUT);
    if (waited_ns != nullptr) *waited_ns = dt;
  }
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, uint64_t* waited_ns,
                                 cudaStream_t stream) {
  mla_wait_selftest_kernel<<<1, 64, 0, stream>>>(status, limit_ns, waited_ns);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// query absorption on the tensor cores, per (head h, 128 latent dims, 64 rows):
//   D[d, r] = sum_k W_UK[h][d][k] q[r][h][k]      (k < 192)
// A = the W_UK[h] slice (K-major, three 64-wide TMA boxes of 128 rows), B =
// the rows' q_nope (K-major, written by the threads), D in TMEM (128 lanes x
// N columns); the blocks of the first latent dims also copy q_rope.
// ----------------------------------------------------------------------------
namespace {
constexpr int kAbsRows = 64;                     // rows per block (N <= 64)
constexpr int kAbsA = 3 * 128 * 128;             // 3 K-chunks x 128 rows x 128 B = 48 KB
constexpr int kAbsB = 3 * kAbsRows * 128;        // 3 K-chunks x 64 rows x 128 B = 24 KB
constexpr int kAbsSmem = kAbsA + kAbsB + 1024 + 64;
constexpr int kQIn = kDnope + kDr;               // 256: one head of the un-absorbed query
}  // namespace

__global__ void __launch_bounds__(128, 1)
    mla_absorb_kernel(const __grid_constant__ CUtensorMap w_map, const uint16_t* __restrict__ q,
                      uint16_t* __restrict__ q_hat, int rows, int heads) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kAbsA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kAbsA + kAbsB);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int mb = blockIdx.y;                      // latent dims [128 mb, 128 mb + 128)
  const int r0 = blockIdx.z * kAbsRows;
  const int nrows = min(kAbsRows, rows - r0);
  const int nmma = (nrows + 15) / 16 * 16;        // N of the MMA
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 64);
    tmem_relinquish();
  }
  __syncthreads();
  if (tid == 0) {
    prefetch_tmap(&w_map);
    mbar_arrive_expect_tx(&bars[0], kAbsA);
    for (int kc = 0; kc < 3; ++kc)
      tma_load_2d(sA + kc * (128 * 128), &w_map, &bars[0], kc * 64, h * kDc + mb * 128, 0ull);
  }
  // B: q_nope of the block's rows, [kc][row][128 B] swizzled; rows past the
  // end are zeros
  for (int idx = tid; idx < nmma * 24; idx += 128) {
    const int r = idx / 24, piece = idx - r * 24;
    const int kc = piece >> 3, w16 = piece & 7;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < nrows)
      v = *reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(r0 + r) * heads + h) * kQIn +
                                          piece * 8);
    *reinterpret_cast<uint4*>(sB + kc * (kAbsRows * 128) + r * 128 + ((w16 ^ (r & 7)) << 4)) = v;
  }
  if (mb == 0) {   // the RoPE part is copied unchanged
    for (int idx = tid; idx < nrows * (kDr / 8); idx += 128) {
      const int r = idx / (kDr / 8), piece = idx - r * (kDr / 8);
      const int64_t row = static_cast<int64_t>(r0 + r) * heads + h;
      *reinterpret_cast<uint4*>(q_hat + row * kDqk + kDc + piece * 8) =
          *reinterpret_cast<const uint4*>(q + row * kQIn + kDnope + piece * 8);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (warp == 0) {
    bool ok = mbar_wait(&bars[0], 0, nullptr, kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (lane == 0) {
      if (ok) {
        const uint32_t idesc = make_idesc_bf16(128, static_cast<uint32_t>(nmma), false, false);
        const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
        for (int kc = 0; kc < 3; ++kc) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad =
                make_smem_desc(a_base + kc * (128 * 128) + kk * 32, 16, 1024, kSmemLayoutSW128);
            const uint64_t bd =
                make_smem_desc(b_base + kc * (kAbsRows * 128) + kk * 32, 16, 1024, kSmemLayoutSW128);
            mma_bf16_ss(tmem, ad, bd, idesc, (kc | kk) ? 1u : 0u);
          }
        }
      }
      mma_commit(&bars[1]);   // also when nothing was issued: the waiters below must not stall
    }
    __syncwarp();
  }
  __syncthreads();
  if (mbar_wait(&bars[1], 0, nullptr, kWaitLimitNs)) {
    tc_fence_after();
    const int d = mb * 128 + warp * 32 + lane;
    for (int cb = 0; cb < nmma; cb += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cb, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int r = cb + e;
        if (r < nrows)
          q_hat[(static_cast<int64_t>(r0 + r) * heads + h) * kDqk + d] =
              float_to_bf16_bits(__uint_as_float(v[e]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

cudaError_t launch_q_absorb(const CUtensorMap* w_map, const uint16_t* q, uint16_t* q_hat, int rows,
                            int heads, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(mla_absorb_kernel), 0, kAbsSmem);
  if (err != cudaSuccess) return err;
  dim3 grid(heads, kDc / 128, (rows + kAbsRows - 1) / kAbsRows);
  mla_absorb_kernel<<<grid, 128, kAbsSmem, stream>>>(*w_map, q, q_hat, rows, heads);
  return cudaGetLastError();
}

}  // namespace mla
