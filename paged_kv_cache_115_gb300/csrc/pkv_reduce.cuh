// Split-K reduce of decode-attention partial states.
#pragma once

#include "pkv_attention_common.cuh"

namespace pkv {

// ===========================================================================
// Split-K reduce: one warp per (output row, query head); 8 warps per CTA.
// For a row with P >= 2 partials (m_p, l_p, o_p), in the slots meta[row]
// lists:
//   M = max_p m_p,  l = sum_p l_p 2^(m_p - M),
//   out = sum_p o_p 2^(m_p - M) / l
// (the rescaling identity of the online softmax).  Lane i owns D/32
// contiguous output elements and reads them from every partial with one
// vector load; the partial loop is unrolled so several loads are in flight.
// Sequences with P <= 1 were finished by the partition kernel.
// ===========================================================================
constexpr int kReduceWarps = 8;
constexpr int kReduceFast = 8;   // partial counts merged with all loads issued at once

template <int V>
__device__ __forceinline__ void load_f(const float* p, float (&v)[V]) {
  if constexpr (V == 8) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else if constexpr (V == 4) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else if constexpr (V == 2) {
    const float2 a = *reinterpret_cast<const float2*>(p);
    v[0] = a.x; v[1] = a.y;
  } else {
    v[0] = *p;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kReduceWarps * 32)
attn_reduce_kernel(Workspace ws, int S, int H_q, T* __restrict__ out) {
  constexpr int V = D / 32;
  pdl_wait_primary();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long pair = (long long)blockIdx.x * kReduceWarps + warp;
  if (pair >= (long long)S * H_q) return;
  const int s = (int)(pair / H_q), h = (int)(pair - (long long)s * H_q);
  const int4 mt = ws.meta[s];          // partial slots: mt.x .. + mt.y, mt.z .. + mt.w
  const int np = mt.y + mt.w;
  if (np <= 1) return;
  // partial p of the row -> its (m, l) index; the output index is that * D
  auto idx = [&](int p) -> int64_t {
    return (int64_t)(p < mt.y ? mt.x + p : mt.z + (p - mt.y)) * H_q + h;
  };
  const int lv = lane * V;
  if (np <= kReduceFast) {
    // few partials (the common case): the (m, l) pairs and the partial
    // outputs are all loaded at once, so the merge costs one round trip
    const float2 ml = lane < np ? ws.ml[idx(lane)] : make_float2(-INFINITY, 0.f);
    float v[kReduceFast][V];
#pragma unroll
    for (int u = 0; u < kReduceFast; ++u)
      if (u < np) load_f<V>(ws.o + idx(u) * D + lv, v[u]);
    const float M = warp_max(ml.x);
    const float w = lane < np ? exp2f(ml.x - M) : 0.f;
    const float inv = 1.f / warp_sum(ml.y * w);
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
    for (int u = 0; u < kReduceFast; ++u) {
      const float wu = __shfl_sync(0xffffffffu, w, u) * inv;
      if (u < np) {
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(wu, v[u][e], acc[e]);
      }
    }
    T* dst = out + ((int64_t)s * H_q + h) * D + lv;
#pragma unroll
    for (int e = 0; e < V; ++e) dst[e] = from_f32<T>(acc[e]);
    return;
  }
  float M = -INFINITY;
  for (int p = lane; p < np; p += 32) M = fmaxf(M, ws.ml[idx(p)].x);
  M = warp_max(M);
  float lsum = 0.f;
  for (int p = lane; p < np; p += 32) {
    const float2 ml = ws.ml[idx(p)];
    lsum += ml.y * exp2f(ml.x - M);
  }
  lsum = warp_sum(lsum);
  const float inv = 1.f / lsum;

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  for (int p0 = 0; p0 < np; p0 += 32) {
    const int pl = p0 + lane;
    const float w = pl < np ? exp2f(ws.ml[idx(pl)].x - M) * inv : 0.f;
    const int cnt = min(32, np - p0);
#pragma unroll 4
    for (int u = 0; u < cnt; ++u) {
      const float wu = __shfl_sync(0xffffffffu, w, u);
      float v[V];
      load_f<V>(ws.o + idx(p0 + u) * D + lv, v);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = fmaf(wu, v[e], acc[e]);
    }
  }
  T* dst = out + ((int64_t)s * H_q + h) * D + lv;
#pragma unroll
  for (int e = 0; e < V; ++e) dst[e] = from_f32<T>(acc[e]);
}

}  // namespace pkv
