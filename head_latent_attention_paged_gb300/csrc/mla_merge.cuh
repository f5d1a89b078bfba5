// LSE merge of a split row set's partial results, shared by the merge kernel
// behind mla_combine and the merge + W_UV kernel, so that both give the same
// bits for every row.
//
// The partials (o_i, lse_i) are each normalised over their own token range:
// o_i = sum_t exp(s_t - lse_i) c_t and lse_i = ln sum_t exp(s_t) over the
// tokens of segment i.  The merged result over all segments is
//   lse = ln sum_i exp(lse_i),   o = sum_i exp(lse_i - lse) o_i,
// computed as m = max_i lse_i, w_i = exp(lse_i - m), sum = sum_i w_i,
// o = (sum_i w_i o_i) / sum and lse = m + ln sum.  A partial with
// lse_i = -inf (no visible token) weighs nothing; all of them -inf gives
// o = 0, lse = -inf.  The order of every sum is fixed (below), so the result
// does not depend on how a kernel spreads its loads.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

namespace mla {

// Lanes that reduce one row's partial lse values together: an aligned group
// of 8 lanes of a warp.  Lane k of the group takes partials k, k + 8, ...
constexpr int kMergeLanes = 8;

struct RowWeights {
  float m;     // max_i lse_i
  float inv;   // 1 / sum_i exp(lse_i - m)  (0 when every lse_i is -inf)
  float lse;   // m + ln sum_i exp(lse_i - m)
};

__device__ __forceinline__ float merge_weight(float lse_i, float m) {
  return lse_i == -INFINITY ? 0.f : __expf(lse_i - m);
}

// Called by all 32 lanes of a warp; each aligned group of 8 lanes passes the
// arguments of its own row (nseg = 0 for a group without one).  plse points
// at the first partial's lse, consecutive partials lie lstride floats apart.
// The loads bypass L1: the partials were written by other CTAs.
__device__ __forceinline__ RowWeights merge_weights(const float* plse, int nseg, int64_t lstride) {
  const int k = threadIdx.x & (kMergeLanes - 1);
  constexpr int kHeld = 4;   // partials k + 8u, u < 4, stay in registers between the passes
  float lv[kHeld];
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < kHeld; ++u) {
    const int i = k + kMergeLanes * u;
    lv[u] = i < nseg ? __ldcg(plse + i * lstride) : -INFINITY;
    m = fmaxf(m, lv[u]);
  }
  for (int i = k + kMergeLanes * kHeld; i < nseg; i += kMergeLanes)
    m = fmaxf(m, __ldcg(plse + i * lstride));
#pragma unroll
  for (int o = kMergeLanes / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // each lane sums its partials in increasing order, then the fixed
  // butterfly over the group (every lane ends with the same bits)
  float sum = 0.f;
#pragma unroll
  for (int u = 0; u < kHeld; ++u)
    if (k + kMergeLanes * u < nseg) sum += merge_weight(lv[u], m);
  for (int i = k + kMergeLanes * kHeld; i < nseg; i += kMergeLanes)
    sum += merge_weight(__ldcg(plse + i * lstride), m);
#pragma unroll
  for (int o = kMergeLanes / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  RowWeights w;
  w.m = m;
  w.inv = (m == -INFINITY) ? 0.f : 1.f / sum;
  w.lse = (m == -INFINITY) ? -INFINITY : m + __logf(sum);
  return w;
}

// acc += w * v, one fused multiply-add per dim; partials are accumulated in
// increasing order from acc = 0, and the merged value is acc * inv.
__device__ __forceinline__ void merge_fma(float4& acc, float w, float4 v) {
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

__device__ __forceinline__ float4 merge_scale(float4 acc, float inv) {
  return make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

}  // namespace mla
