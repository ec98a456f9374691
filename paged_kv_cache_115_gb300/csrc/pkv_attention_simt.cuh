// CUDA-core decode-attention partition kernel (fp32 / bf16 queries; bf16,
// fp32, FP8 e4m3 or INT8 pools; any block size).
#pragma once

#include "pkv_attention_common.cuh"

namespace pkv {

// ===========================================================================
// CUDA-core partition kernel (fp32 or bf16, any block size, G <= 16).
// grid = (Pmax, H_kv, S), block = 128 threads; CTA (p, j, s) covers tokens
// [p*PS, min((p+1)*PS, L)) of sequence s for the G query heads of KV head j.
// Each warp takes every 4th token; the four warps' states are merged in
// shared memory.
// ===========================================================================
constexpr int kSimtThreads = 128;
constexpr int kSimtMaxPS = 1024;

// K/V row loaders: element e of lane `lane` of the row starting at element
// `row` (= (slot * H_kv + j) * D) of the pool, as float.
template <typename T>
struct KvPlain {          // pool stored in the query dtype
  const T* k;
  const T* v;
  __device__ __forceinline__ float ld_k(int64_t i, int64_t) const { return to_f32(k[i]); }
  __device__ __forceinline__ float ld_v(int64_t i, int64_t) const { return to_f32(v[i]); }
};
struct KvFp8 {            // e4m3 codes, one scale per tensor
  const uint8_t* k;
  const uint8_t* v;
  float k_scale, v_scale;
  __device__ __forceinline__ float ld_k(int64_t i, int64_t) const {
    return e4m3_to_f32(k[i]) * k_scale;
  }
  __device__ __forceinline__ float ld_v(int64_t i, int64_t) const {
    return e4m3_to_f32(v[i]) * v_scale;
  }
};
struct KvBf16Fp8 {        // bf16 K pool, e4m3 V codes with one scale
  const __nv_bfloat16* k;
  const uint8_t* v;
  float v_scale;
  __device__ __forceinline__ float ld_k(int64_t i, int64_t) const { return __bfloat162float(k[i]); }
  __device__ __forceinline__ float ld_v(int64_t i, int64_t) const {
    return e4m3_to_f32(v[i]) * v_scale;
  }
};
struct KvInt8 {           // int8 codes, one scale per token slot
  const int8_t* k;
  const int8_t* v;
  const float* k_ts;
  const float* v_ts;
  __device__ __forceinline__ float ld_k(int64_t i, int64_t slot) const {
    return (float)k[i] * k_ts[slot];
  }
  __device__ __forceinline__ float ld_v(int64_t i, int64_t slot) const {
    return (float)v[i] * v_ts[slot];
  }
};

template <typename T, typename KV, int D, int GMAX>
__global__ void __launch_bounds__(kSimtThreads)
attn_simt_kernel(const T* __restrict__ q, KV kv, const int32_t* __restrict__ block_tables,
                 int max_blocks_per_seq, const int32_t* __restrict__ context_lens, int max_len,
                 int H_q, int H_kv, int G, int K, long long num_blocks, float scale_log2,
                 T* __restrict__ out, Workspace ws, int PS) {
  constexpr int E = D / 32;   // elements of a row per lane
  __shared__ int s_bt[kSimtMaxPS + 2];
  __shared__ float s_m[4][GMAX], s_l[4][GMAX];
  __shared__ float s_o[GMAX][D];

  pdl_wait_primary();
  pdl_launch_dependents();

  const int p = blockIdx.x, j = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = effective_len(context_lens[s], max_len, max_blocks_per_seq * K);
  const int np = (L + PS - 1) / PS;
  if (p == 0 && j == 0 && threadIdx.x == 0) ws.meta[s] = make_int4(s * ws.pmax, np, 0, 0);
  if (L == 0) {
    if (p == 0) {
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        out[((int64_t)s * H_q + j * G) * D + i] = from_f32<T>(0.f);
    }
    return;
  }
  if (p >= np) return;
  const int t0 = p * PS, t1 = min(t0 + PS, L);
  const int lb0 = t0 / K, nlb = (t1 - 1) / K - lb0 + 1;
  for (int i = threadIdx.x; i < nlb; i += blockDim.x) {
    int phys = block_tables[(int64_t)s * max_blocks_per_seq + lb0 + i];
    if (phys < 0 || phys >= num_blocks) {
      record_error(PKV_DEVERR_BLOCK_ID);
      phys = -1;
    }
    s_bt[i] = phys;
  }
  for (int i = threadIdx.x; i < GMAX * D; i += blockDim.x) (&s_o[0][0])[i] = 0.f;

  float qr[GMAX][E];
#pragma unroll
  for (int n = 0; n < GMAX; ++n)
#pragma unroll
    for (int e = 0; e < E; ++e)
      qr[n][e] = n < G ? to_f32(q[((int64_t)s * H_q + j * G + n) * D + lane + 32 * e]) : 0.f;
  __syncthreads();

  float m[GMAX], l[GMAX], o[GMAX][E];
#pragma unroll
  for (int n = 0; n < GMAX; ++n) {
    m[n] = -INFINITY;
    l[n] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[n][e] = 0.f;
  }
  for (int t = t0 + warp; t < t1; t += 4) {
    const int lbi = t / K - lb0;
    const int phys = s_bt[lbi];
    const int off = t - (t / K) * K;
    float kr[E], vr[E];
    if (phys >= 0) {
      const int64_t slot = (int64_t)phys * K + off;
      const int64_t row = (slot * H_kv + j) * D;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        kr[e] = kv.ld_k(row + lane + 32 * e, slot);
        vr[e] = kv.ld_v(row + lane + 32 * e, slot);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) kr[e] = vr[e] = 0.f;
    }
#pragma unroll
    for (int n = 0; n < GMAX; ++n) {
      if (n >= G) break;
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) d = fmaf(qr[n][e], kr[e], d);
      const float x = warp_sum(d) * scale_log2;
      const float mn = fmaxf(m[n], x);
      const float a = exp2f(m[n] - mn);
      const float w = exp2f(x - mn);
      l[n] = l[n] * a + w;
#pragma unroll
      for (int e = 0; e < E; ++e) o[n][e] = fmaf(o[n][e], a, w * vr[e]);
      m[n] = mn;
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int n = 0; n < GMAX; ++n) {
      s_m[warp][n] = m[n];
      s_l[warp][n] = l[n];
    }
  }
  __syncthreads();
  float M[GMAX], Lsum[GMAX], f[GMAX];
#pragma unroll
  for (int n = 0; n < GMAX; ++n) {
    M[n] = fmaxf(fmaxf(s_m[0][n], s_m[1][n]), fmaxf(s_m[2][n], s_m[3][n]));
    Lsum[n] = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w)
      Lsum[n] += s_m[w][n] == -INFINITY ? 0.f : s_l[w][n] * exp2f(s_m[w][n] - M[n]);
    f[n] = m[n] == -INFINITY ? 0.f : exp2f(m[n] - M[n]);
  }
  for (int w = 0; w < 4; ++w) {
    if (warp == w) {
#pragma unroll
      for (int n = 0; n < GMAX; ++n)
#pragma unroll
        for (int e = 0; e < E; ++e) s_o[n][lane + 32 * e] += o[n][e] * f[n];
    }
    __syncthreads();
  }
  if (np == 1) {
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int n = i / D, d = i - n * D;
      out[((int64_t)s * H_q + j * G + n) * D + d] = from_f32<T>(s_o[n][d] / Lsum[n]);
    }
  } else {
    const int64_t base = ((int64_t)s * ws.pmax + p) * H_q + j * G;
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int n = i / D, d = i - n * D;
      ws.o[(base + n) * D + d] = s_o[n][d];
    }
    if (threadIdx.x < G) ws.ml[base + threadIdx.x] = make_float2(M[threadIdx.x], Lsum[threadIdx.x]);
  }
}

}  // namespace pkv
