// LSE merge of a split row set's partial results, shared by the decode
// kernel (the CTA that writes a row set's last partial merges it) and the
// merge kernel behind mla_combine, so that both give the same bits.
//
// The partials (o_i, lse_i) are each normalised over their own token range:
// o_i = sum_t exp(s_t - lse_i) c_t and lse_i = ln sum_t exp(s_t) over the
// tokens of segment i.  The merged result over all segments is
//   lse = ln sum_i exp(lse_i),   o = sum_i exp(lse_i - lse) o_i,
// computed in one pass over the partials, 8 at a time, with a running
// maximum m (sum = sum_i exp(lse_i - m), acc = sum_i exp(lse_i - m) o_i,
// both rescaled when m grows).  A partial with lse_i = -inf (no visible
// token) weighs nothing; all of them -inf gives o = 0, lse = -inf.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

namespace mla {

struct MergedRow {
  float4 o;    // this thread's 4 dims of the merged row
  float lse;
};

// Thread t of the 128 owning a row holds dims 4t .. 4t + 3.  plse points at
// the first partial's lse, po at the first partial's float4 of this thread;
// consecutive partials lie lstride floats and ostride float4s apart.  The
// loads bypass L1: the partials may have been written by other CTAs.
__device__ __forceinline__ MergedRow merge_partials(const float* plse, const float4* po, int nseg,
                                                    int64_t lstride, int64_t ostride) {
  float m = -INFINITY, sum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < nseg; k0 += 8) {
    float lv[8];
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = k0 + u < nseg;
      lv[u] = in ? __ldcg(plse + (k0 + u) * lstride) : -INFINITY;
      v[u] = in ? __ldcg(po + (k0 + u) * ostride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mc = m;
#pragma unroll
    for (int u = 0; u < 8; ++u) mc = fmaxf(mc, lv[u]);
    if (mc == -INFINITY) continue;     // nothing live so far
    const float r = (m == -INFINITY) ? 0.f : __expf(m - mc);
    sum *= r;
    acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float w = (lv[u] == -INFINITY) ? 0.f : __expf(lv[u] - mc);
      sum += w;
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
    m = mc;
  }
  MergedRow out;
  out.lse = (m == -INFINITY) ? -INFINITY : m + __logf(sum);
  const float inv = (m == -INFINITY) ? 0.f : 1.f / sum;
  out.o = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  return out;
}

}  // namespace mla
