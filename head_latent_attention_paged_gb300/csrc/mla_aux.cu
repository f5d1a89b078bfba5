// The smaller kernels of the decode step:
//   * mla_combine_kernel : LSE merge of the split-KV partials of each row set;
//   * mla_uv_kernel      : o = W_UV[h]^T o_lat (tcgen05, per head);
//   * mla_absorb_kernel  : q_hat = [W_UK[h] q_nope || q_rope] (query absorption).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

namespace {
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}
}  // namespace

// ----------------------------------------------------------------------------
// combine: one block per (row set, 4 heads); one warp per head, 16 dims/lane
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(128) mla_combine_kernel(const CombineParams p) {
  const int s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + warp;
  const int S = p.num_streams;
  const int max_tokens = p.max_pages * p.page_size;
  // tiles before stream s, tiles of s, tiles in total (same split as the decode grid)
  int64_t before = 0, tot = 0;
  for (int t = threadIdx.x; t < S; t += blockDim.x) {
    const int b = t / p.q_len, j = t - b * p.q_len;
    const int32_t len = stream_len(p.seq_lens[b], p.q_len, j, p.causal, p.topk_width, max_tokens);
    const int64_t n = (len + kTile - 1) / kTile;
    tot += n;
    if (t < s) before += n;
  }
  __shared__ int64_t red[2][4];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
  }
  if (lane == 0) { red[0][warp] = before; red[1][warp] = tot; }
  __syncthreads();
  before = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  tot = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  if (h >= p.heads) return;
  const int b = s / p.q_len, j = s - b * p.q_len;
  const int32_t len = stream_len(p.seq_lens[b], p.q_len, j, p.causal, p.topk_width, max_tokens);
  const int64_t ntiles = (len + kTile - 1) / kTile;
  float4* out = reinterpret_cast<float4*>(p.o_lat + (static_cast<int64_t>(s) * p.heads + h) * kDc);
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse = -INFINITY;
  if (ntiles > 0) {
    const int c0 = tile_owner(before, tot, p.num_ctas);
    const int c1 = tile_owner(before + ntiles - 1, tot, p.num_ctas);
    if (c0 == c1) return;   // one CTA held the whole row set: its result is final
    float m = -INFINITY;
    for (int c = c0; c <= c1; ++c) m = fmaxf(m, p.part_lse[static_cast<int64_t>(s + c) * p.heads + h]);
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int c = c0; c <= c1; ++c) sum += __expf(p.part_lse[static_cast<int64_t>(s + c) * p.heads + h] - m);
      lse = m + __logf(sum);
      for (int c = c0; c <= c1; ++c) {
        const int64_t slot = s + c;
        const float wgt = __expf(p.part_lse[slot * p.heads + h] - lse);
        if (wgt == 0.f) continue;
        const float4* src = reinterpret_cast<const float4*>(p.part_o + (slot * p.heads + h) * kDc);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 v = src[lane + 32 * k];
          acc[k].x += wgt * v.x; acc[k].y += wgt * v.y;
          acc[k].z += wgt * v.z; acc[k].w += wgt * v.w;
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) out[lane + 32 * k] = acc[k];
  if (lane == 0) p.lse[static_cast<int64_t>(s) * p.heads + h] = lse;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  if (p.num_streams == 0) return cudaSuccess;
  dim3 grid(p.num_streams, (p.heads + 3) / 4);
  mla_combine_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// UV projection: per (head h, 128 output dims, 64 rows):
//   D^T[n, r] = sum_k W_UV[h][k][n] * o_lat[r][h][k]
// A = W_UV[h] slice (MN-major, TMA), B = o_lat rows converted to bf16
// (K-major, written by the threads), D in TMEM (128 lanes x 64 columns).
// ----------------------------------------------------------------------------
namespace {
constexpr int kUvRows = 64;                 // N of the MMA
constexpr int kUvA = 8 * 2 * kChunkBytes;   // 8 K-blocks x 2 n-chunks x 8 KB = 128 KB
constexpr int kUvB = 8 * kUvRows * 128;     // 8 K-blocks x 64 rows x 128 B = 64 KB
constexpr int kUvSmem = kUvA + kUvB + 1024 + 64;
}  // namespace

__global__ void __launch_bounds__(128, 1)
    mla_uv_kernel(const __grid_constant__ CUtensorMap w_map, const float* __restrict__ o_lat,
                  uint16_t* __restrict__ out, int rows, int heads) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kUvA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kUvA + kUvB);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int mt = blockIdx.y;          // output dims [128 mt, 128 mt + 128)
  const int r0 = blockIdx.z * kUvRows;
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
    mbar_arrive_expect_tx(&bars[0], kUvA);
    for (int kb = 0; kb < 8; ++kb)
      for (int nc = 0; nc < 2; ++nc)
        tma_load_2d(sA + (kb * 2 + nc) * kChunkBytes, &w_map, &bars[0], mt * 128 + nc * 64,
                    h * kDc + kb * 64, 0ull);
  }
  // o_lat is produced by the preceding decode launch: wait for it (the W_UV
  // loads above already overlap its tail when launched as a dependent).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // B: o_lat[r0 + r][h][k] -> bf16, [kb][r][128 B] swizzled
  for (int e = tid; e < kUvRows * 64; e += 128) {
    const int r = e >> 6, piece = e & 63;        // piece: 8 consecutive k
    const int kb = piece >> 3, w16 = piece & 7;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r0 + r < rows) {
      const float4* src = reinterpret_cast<const float4*>(
          o_lat + (static_cast<int64_t>(r0 + r) * heads + h) * kDc + piece * 8);
      const float4 a = src[0], b = src[1];
      __nv_bfloat162 x0 = __floats2bfloat162_rn(a.x, a.y), x1 = __floats2bfloat162_rn(a.z, a.w);
      __nv_bfloat162 x2 = __floats2bfloat162_rn(b.x, b.y), x3 = __floats2bfloat162_rn(b.z, b.w);
      v = make_uint4(*reinterpret_cast<uint32_t*>(&x0), *reinterpret_cast<uint32_t*>(&x1),
                     *reinterpret_cast<uint32_t*>(&x2), *reinterpret_cast<uint32_t*>(&x3));
    }
    *reinterpret_cast<uint4*>(sB + kb * (kUvRows * 128) + r * 128 + ((w16 ^ (r & 7)) << 4)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;
  if (warp == 0) {
    ok = mbar_wait(&bars[0], 0, nullptr, kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok && lane == 0) {
      const uint32_t idesc = make_idesc_bf16(128, kUvRows, true, false);
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = make_smem_desc(a_base + kb * 2 * kChunkBytes + kk * 2048, kChunkBytes,
                                             1024, kSmemLayoutSW128);
          const uint64_t bd = make_smem_desc(b_base + kb * (kUvRows * 128) + kk * 32, 16, 1024,
                                             kSmemLayoutSW128);
          mma_bf16_ss(tmem, ad, bd, idesc, (kb | kk) ? 1u : 0u);
        }
      }
      mma_commit(&bars[1]);
    }
    __syncwarp();
  }
  __syncthreads();
  if (mbar_wait(&bars[1], 0, nullptr, kWaitLimitNs)) {
    tc_fence_after();
    const int n = mt * 128 + warp * 32 + lane;
    for (int cb = 0; cb < kUvRows; cb += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cb, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int r = r0 + cb + e;
        if (r < rows) out[(static_cast<int64_t>(r) * heads + h) * kDv + n] = float_to_bf16_bits(__uint_as_float(v[e]));
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

cudaError_t launch_uv_proj_tma(const CUtensorMap* w_map, const float* o_lat, uint16_t* out,
                               int rows, int heads, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(mla_uv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUvSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(heads, kDv / 128, (rows + kUvRows - 1) / kUvRows);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kUvSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, mla_uv_kernel, *w_map, o_lat, out, rows, heads);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// query absorption: q_hat[r][h] = [bf16(W_UK[h] q_nope[r][h]) || q_rope[r][h]]
// one block per (head, 8 rows); thread c computes latent dim c for the 8 rows
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(512) mla_absorb_kernel(const uint16_t* __restrict__ q_nope,
                                                         const uint16_t* __restrict__ q_rope,
                                                         const uint16_t* __restrict__ w_uk,
                                                         uint16_t* __restrict__ q_hat, int rows,
                                                         int heads) {
  __shared__ float qn[8][kDnope];
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * 8;
  const int c = threadIdx.x;
  for (int e = threadIdx.x; e < 8 * kDnope; e += blockDim.x) {
    const int r = e / kDnope, n = e - r * kDnope;
    qn[r][n] = (r0 + r < rows) ? bf16_bits_to_float(q_nope[(static_cast<int64_t>(r0 + r) * heads + h) * kDnope + n]) : 0.f;
  }
  __syncthreads();
  float acc[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) acc[r] = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(w_uk + (static_cast<int64_t>(h) * kDc + c) * kDnope);
  for (int q = 0; q < kDnope / 8; ++q) {
    const uint4 u = wrow[q];
    const uint16_t* wb = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float w = bf16_bits_to_float(wb[e]);
#pragma unroll
      for (int r = 0; r < 8; ++r) acc[r] = fmaf(w, qn[r][q * 8 + e], acc[r]);
    }
  }
  for (int r = 0; r < 8; ++r) {
    if (r0 + r >= rows) break;
    uint16_t* dst = q_hat + (static_cast<int64_t>(r0 + r) * heads + h) * kDqk;
    dst[c] = float_to_bf16_bits(acc[r]);
    if (c < kDr) dst[kDc + c] = q_rope[(static_cast<int64_t>(r0 + r) * heads + h) * kDr + c];
  }
}

cudaError_t launch_q_absorb(const uint16_t* q_nope, const uint16_t* q_rope, const uint16_t* w_uk,
                            uint16_t* q_hat, int rows, int heads, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  dim3 grid(heads, (rows + 7) / 8);
  mla_absorb_kernel<<<grid, kDc, 0, stream>>>(q_nope, q_rope, w_uk, q_hat, rows, heads);
  return cudaGetLastError();
}

}  // namespace mla
