// Cache append: write each request's newest token row (the shared latent
// c_kv and the RoPE key, 576 values; the key rotated here to the token's
// position when a rope_theta is given) into the paged latent cache, as bf16,
// in the FP8 layout (576 e4m3 || 18 e8m0 per token) or in the FP4 layout
// (288 bytes of packed e2m1 || 36 e8m0 per token) with the quantiser run on
// the GPU.
//
// One warp per row.  FP8: for each 32-value group the warp takes the group's
// absolute maximum, picks the scale 2^e with e = ceil(log2(amax / 448))
// (clamped to [-127, 127]; an all-zero group gets e = -127 and zero codes),
// and converts x / 2^e to e4m3 with round-to-nearest-even and saturation at
// 448.  Every step is exact for bf16 inputs: amax and the choice of e are
// read off the float bits, x / 2^e is a power-of-two scaling, and the only
// rounding is the e4m3 conversion itself.
//
// FP4: the same with 16-value groups, e = ceil(log2(amax / 6)) and the
// nearest e2m1 value (ties to the even code, saturating at 6) of x / 2^e;
// value 2i goes to the low nibble of code byte i.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kAppendWarps = 4;   // rows per block

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// ceil(log2(a / 448)) for a > 0 finite, exactly: a = m 2^E with m in [1, 2),
// 448 = 1.75 2^8, so a / 448 = (m / 1.75) 2^(E - 8) and m / 1.75 lies in
// (0.5, 1] unless m > 1.75.  Subnormal a gives a value below -127.
__device__ __forceinline__ int ceil_log2_over_448(float a) {
  const uint32_t bits = __float_as_uint(a);
  const int ef = static_cast<int>((bits >> 23) & 0xFFu);
  if (ef == 0) return -200;
  const uint32_t man = bits & 0x7FFFFFu;
  return (ef - 127) - 8 + (man > 0x600000u ? 1 : 0);
}

// ceil(log2(a / 6)) for a > 0 finite, exactly: 6 = 1.5 2^2, so a / 6 =
// (m / 1.5) 2^(E - 2) with m / 1.5 in [2/3, 1] unless m > 1.5.
__device__ __forceinline__ int ceil_log2_over_6(float a) {
  const uint32_t bits = __float_as_uint(a);
  const int ef = static_cast<int>((bits >> 23) & 0xFFu);
  if (ef == 0) return -200;
  const uint32_t man = bits & 0x7FFFFFu;
  return (ef - 127) - 2 + (man > 0x400000u ? 1 : 0);
}

// Nearest e2m1 code of v (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), ties to
// the even code, saturating at 6; the sign bit of v becomes bit 3.  Each
// comparison moves past one midpoint of the grid: a midpoint between an
// even and the next odd code counts only when exceeded, one between an odd
// and the next even code already when reached.
__device__ __forceinline__ uint32_t f32_to_e2m1(float v) {
  const float a = fabsf(v);
  const uint32_t mag = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                       (a >= 3.5f) + (a > 5.0f);
  return mag | ((__float_as_uint(v) >> 28) & 8u);
}

// Nearest bf16 (ties to even) of a double, as bits: one rounding.  The
// rotated RoPE values are finite and far inside bf16's normal range.
__device__ __forceinline__ uint32_t f64_to_bf16_bits(double x) {
  const __nv_bfloat16 h = __double2bfloat16(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// 2^-e as a float for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float pow2_neg(int e) {
  return e == 127 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// Round-to-nearest-even conversion to e4m3 with saturation at +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t two;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(two) : "f"(v));
  return two & 0xFFu;
}

__global__ void __launch_bounds__(32 * kAppendWarps) mla_append_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (b >= p.rows) return;
  const int32_t pos = p.positions[b];
  if (pos < 0) return;   // nothing to append for this request
  const int64_t max_tokens = static_cast<int64_t>(p.max_pages) * p.page_size;
  if (pos >= max_tokens) {
    if (lane == 0 && p.status) atomicOr(p.status, MLA_STATUS_BAD_INDEX);
    return;
  }
  const int32_t page = p.block_table[static_cast<int64_t>(b) * p.max_pages + pos / p.page_size];
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0 && p.status) atomicOr(p.status, MLA_STATUS_BAD_PAGE);
    return;
  }
  const int64_t row = static_cast<int64_t>(page) * p.page_size + pos % p.page_size;
  const uint16_t* src = p.new_rows + static_cast<int64_t>(b) * kDqk;
  // The RoPE key (values 512..575): lane i holds pair i = (x[512 + 2i],
  // x[513 + 2i]) as two bf16, rotated to position pos when rope_theta > 0:
  // angle pos * theta^(-2i/64), in double precision (positions reach 2^17
  // radians at pair 0), rounded once to bf16.
  uint32_t rope_pair = *reinterpret_cast<const uint32_t*>(src + kDc + 2 * lane);
  if (p.rope_theta > 0.f) {
    const double x0 = bf16_bits_to_f32(static_cast<uint16_t>(rope_pair & 0xFFFFu));
    const double x1 = bf16_bits_to_f32(static_cast<uint16_t>(rope_pair >> 16));
    const double inv_freq = pow(static_cast<double>(p.rope_theta), -2.0 * lane / kDr);
    double sn, cs;
    sincos(static_cast<double>(pos) * inv_freq, &sn, &cs);
    const uint32_t y0 = f64_to_bf16_bits(x0 * cs - x1 * sn);
    const uint32_t y1 = f64_to_bf16_bits(x0 * sn + x1 * cs);
    rope_pair = y0 | (y1 << 16);
  }
  // value v of the row (as stored: RoPE part rotated), read by lane `lane`
  // of the warp for v = 32 k + lane; every lane calls it with the same k
  auto value32 = [&](int k) -> float {
    if (k < kDc / 32) return bf16_bits_to_f32(src[32 * k + lane]);
    const int e = 32 * (k - kDc / 32) + lane;      // RoPE element
    const uint32_t pr = __shfl_sync(0xffffffffu, rope_pair, e >> 1);
    return bf16_bits_to_f32(static_cast<uint16_t>((e & 1) ? (pr >> 16) : (pr & 0xFFFFu)));
  };
  if (p.kv_dtype == MLA_KV_BF16) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint8_t* d = p.kv + row * (kDqk * 2);
    uint4* d4 = reinterpret_cast<uint4*>(d);
    for (int i = lane; i < kDc * 2 / 16; i += 32) d4[i] = s4[i];
    reinterpret_cast<uint32_t*>(d + kDc * 2)[lane] = rope_pair;
    return;
  }
  if (p.kv_dtype == MLA_KV_FP4_E2M1_E8M0) {
    // each pass covers 32 values: lanes 0-15 one 16-value group, 16-31 the next
    uint8_t* dst = p.kv + row * kFp4RowBytes;
    for (int it = 0; it < kDqk / 32; ++it) {
      const int g = 2 * it + (lane >> 4);
      const float x = value32(it);
      float amax = fabsf(x);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int e = -127;
      uint32_t code = 0;
      if (amax > 0.f) {
        e = max(-127, min(127, ceil_log2_over_6(amax)));
        code = f32_to_e2m1(x * pow2_neg(e));
      }
      const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
      if ((lane & 1) == 0) dst[16 * it + (lane >> 1)] = static_cast<uint8_t>(code | (hi << 4));
      if ((lane & 15) == 0) dst[kFp4CodeBytes + g] = static_cast<uint8_t>(e + 127);
    }
    return;
  }
  uint8_t* dst = p.kv + row * kFp8RowBytes;
  for (int g = 0; g < kDqk / 32; ++g) {
    const float x = value32(g);
    float amax = fabsf(x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = -127;
    uint32_t code = 0;
    if (amax > 0.f) {
      e = max(-127, min(127, ceil_log2_over_448(amax)));
      code = f32_to_e4m3(x * pow2_neg(e));
    }
    dst[32 * g + lane] = static_cast<uint8_t>(code);
    if (lane == 0) dst[kDqk + g] = static_cast<uint8_t>(e + 127);
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const int blocks = (p.rows + kAppendWarps - 1) / kAppendWarps;
  mla_append_kernel<<<blocks, 32 * kAppendWarps, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
