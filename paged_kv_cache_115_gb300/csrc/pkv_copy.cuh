// Integer and data-movement kernels: slot mapping, slot-mapped KV append and
// the copy-on-write block copy.  All of them are bit-exact byte moves or
// integer arithmetic; every device-side index is range-checked before use.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

// a1: slot of each sequence's new token ("推理与 KV Cache 02", 从一个位置找到
// 缓存块: logical block = t / K, offset = t % K, slot = block * K + offset).
// K need not be a power of two; when it is, the compiler's division by a
// run-time value is replaced by the shift the host passes in (log2_bs >= 0).
__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables,
                                    int32_t max_blocks_per_seq,
                                    const int32_t* __restrict__ positions, int32_t num_seqs,
                                    int32_t block_size, int32_t log2_bs, int64_t num_blocks,
                                    int64_t* __restrict__ slot_mapping) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= num_seqs) return;
  const int t = positions[s];
  int64_t slot = -1;
  if (t >= 0) {
    const int lb = log2_bs >= 0 ? (t >> log2_bs) : (t / block_size);
    const int off = log2_bs >= 0 ? (t & (block_size - 1)) : (t - lb * block_size);
    if (lb >= max_blocks_per_seq) {
      record_error(PKV_DEVERR_POSITION);
    } else {
      const int64_t phys = block_tables[(int64_t)s * max_blocks_per_seq + lb];
      if (phys < 0 || phys >= num_blocks) {
        record_error(PKV_DEVERR_BLOCK_ID);
      } else {
        slot = phys * block_size + off;
      }
    }
  }
  slot_mapping[s] = slot;
}

template <int VW>
struct VecT;
template <> struct VecT<16> { using T = uint4; };
template <> struct VecT<8>  { using T = uint2; };
template <> struct VecT<4>  { using T = uint32_t; };
template <> struct VecT<2>  { using T = uint16_t; };
template <> struct VecT<1>  { using T = uint8_t; };

// a2: k_cache.view(-1, row)[slot[i]] = k[i] (and v).  grid = (tokens,
// vector chunks of a row, 2 for K/V); one thread moves VW bytes.
template <int VW>
__global__ void kv_write_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                const int64_t* __restrict__ slot_mapping,
                                uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                int64_t num_slots, int64_t row_bytes) {
  using V = typename VecT<VW>::T;
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t i = blockIdx.x;
  const int64_t e = (int64_t)blockIdx.y * blockDim.x + threadIdx.x;
  if (e * VW >= row_bytes) return;
  const int64_t slot = slot_mapping[i];
  if (slot < 0 || slot >= num_slots) {
    if (slot != -1 && e == 0 && blockIdx.z == 0) record_error(PKV_DEVERR_SLOT);
    return;
  }
  const uint8_t* src = (blockIdx.z ? v : k) + i * row_bytes + e * VW;
  uint8_t* dst = (blockIdx.z ? v_cache : k_cache) + slot * row_bytes + e * VW;
  *reinterpret_cast<V*>(dst) = __ldg(reinterpret_cast<const V*>(src));
}

// a1 + a2 fused: the slot of token i comes from its sequence's block-table
// row and position (as in slot_mapping_kernel) and the K/V rows are stored
// there (as in kv_write_kernel).  grid = (tokens, vector chunks, 2).  The
// slot is also written to `slots` (when non-null) by one thread per token.
template <int VW>
__global__ void kv_append_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                 const int32_t* __restrict__ block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* __restrict__ positions,
                                 int32_t block_size, int32_t log2_bs, int64_t num_blocks,
                                 uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                 int64_t row_bytes, int64_t* __restrict__ slots) {
  using V = typename VecT<VW>::T;
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t i = blockIdx.x;
  const int64_t e = (int64_t)blockIdx.y * blockDim.x + threadIdx.x;
  const bool leader = e == 0 && blockIdx.z == 0;
  const int t = positions[i];
  int64_t slot = -1;
  if (t >= 0) {
    const int lb = log2_bs >= 0 ? (t >> log2_bs) : (t / block_size);
    const int off = log2_bs >= 0 ? (t & (block_size - 1)) : (t - lb * block_size);
    if (lb >= max_blocks_per_seq) {
      if (leader) record_error(PKV_DEVERR_POSITION);
    } else {
      const int64_t phys = block_tables[i * max_blocks_per_seq + lb];
      if (phys < 0 || phys >= num_blocks) {
        if (leader) record_error(PKV_DEVERR_BLOCK_ID);
      } else {
        slot = phys * block_size + off;
      }
    }
  }
  if (leader && slots != nullptr) slots[i] = slot;
  if (slot < 0 || e * VW >= row_bytes) return;
  const uint8_t* src = (blockIdx.z ? v : k) + i * row_bytes + e * VW;
  uint8_t* dst = (blockIdx.z ? v_cache : k_cache) + slot * row_bytes + e * VW;
  *reinterpret_cast<V*>(dst) = __ldg(reinterpret_cast<const V*>(src));
}

// a1 + a2 for packed new tokens of several sequences (prefill): token i
// belongs to the sequence s with cu_seqlens[s] <= i < cu_seqlens[s + 1] and
// sits at position context_lens[s] - n_s + (i - cu_seqlens[s]); its slot
// comes from that sequence's block-table row.  grid = (tokens, vector chunks,
// 2).  Tokens whose position is out of range are skipped and reported.
template <int VW>
__global__ void kv_append_varlen_kernel(const uint8_t* __restrict__ k,
                                        const uint8_t* __restrict__ v,
                                        const int32_t* __restrict__ cu_seqlens,
                                        const int32_t* __restrict__ context_lens, int32_t num_seqs,
                                        const int32_t* __restrict__ block_tables,
                                        int32_t max_blocks_per_seq, int32_t block_size,
                                        int64_t num_blocks, uint8_t* __restrict__ k_cache,
                                        uint8_t* __restrict__ v_cache, int64_t row_bytes,
                                        int64_t* __restrict__ slots) {
  using V = typename VecT<VW>::T;
  pdl_wait_primary();
  pdl_launch_dependents();
  const int i = blockIdx.x;
  const int64_t e = (int64_t)blockIdx.y * blockDim.x + threadIdx.x;
  const bool leader = e == 0 && blockIdx.z == 0;
  int lo = 0, hi = num_seqs;            // largest s with cu_seqlens[s] <= i
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu_seqlens[mid] <= i) lo = mid; else hi = mid;
  }
  const int c0 = cu_seqlens[lo], c1 = cu_seqlens[lo + 1];
  const int pos = context_lens[lo] - (c1 - c0) + (i - c0);
  int64_t slot = -1;
  if (i < c0 || i >= c1 || pos < 0) {
    if (leader) record_error(PKV_DEVERR_POSITION);
  } else {
    const int lb = pos / block_size;
    if (lb >= max_blocks_per_seq) {
      if (leader) record_error(PKV_DEVERR_POSITION);
    } else {
      const int64_t phys = block_tables[(int64_t)lo * max_blocks_per_seq + lb];
      if (phys < 0 || phys >= num_blocks) {
        if (leader) record_error(PKV_DEVERR_BLOCK_ID);
      } else {
        slot = phys * block_size + (pos - lb * block_size);
      }
    }
  }
  if (leader && slots != nullptr) slots[i] = slot;
  if (slot < 0 || e * VW >= row_bytes) return;
  const uint8_t* src = (blockIdx.z ? v : k) + (int64_t)i * row_bytes + e * VW;
  uint8_t* dst = (blockIdx.z ? v_cache : k_cache) + slot * row_bytes + e * VW;
  *reinterpret_cast<V*>(dst) = __ldg(reinterpret_cast<const V*>(src));
}

// a1 + a2 into a quantized pool.  grid = (tokens, 2 for K/V), 128 threads.
// FMT 1: e4m3(x / scale) per element (per-tensor scale).  FMT 2: the token's
// row (all heads) gets scale = max|x| / 127 and codes rint(x / scale), the
// scale stored at the token's slot.  FMT 3: K rows as bfloat16 (rounded to
// nearest even), V rows as FMT 1.  Divisions are IEEE float32 (__fdiv_rn).
constexpr int kQuantThreads = 128;

template <typename TIN, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
kv_append_quant_kernel(const TIN* __restrict__ k, const TIN* __restrict__ v,
                       const int32_t* __restrict__ block_tables, int32_t max_blocks_per_seq,
                       const int32_t* __restrict__ positions, int32_t block_size,
                       int32_t log2_bs, int64_t num_blocks, uint8_t* __restrict__ k_cache,
                       uint8_t* __restrict__ v_cache, int64_t row_elems, float k_scale,
                       float v_scale, float* __restrict__ k_ts, float* __restrict__ v_ts,
                       int64_t* __restrict__ slots) {
  __shared__ float s_red[kQuantThreads / 32];
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t i = blockIdx.x;
  const int z = blockIdx.y;
  const bool leader = threadIdx.x == 0 && z == 0;
  const int t = positions[i];
  int64_t slot = -1;
  if (t >= 0) {
    const int lb = log2_bs >= 0 ? (t >> log2_bs) : (t / block_size);
    const int off = log2_bs >= 0 ? (t & (block_size - 1)) : (t - lb * block_size);
    if (lb >= max_blocks_per_seq) {
      if (leader) record_error(PKV_DEVERR_POSITION);
    } else {
      const int64_t phys = block_tables[i * max_blocks_per_seq + lb];
      if (phys < 0 || phys >= num_blocks) {
        if (leader) record_error(PKV_DEVERR_BLOCK_ID);
      } else {
        slot = phys * block_size + off;
      }
    }
  }
  if (leader && slots != nullptr) slots[i] = slot;
  if (slot < 0) return;
  const TIN* src = (z ? v : k) + i * row_elems;
  uint8_t* dst = (z ? v_cache : k_cache) + slot * row_elems;
  if (FMT == 3 && z == 0) {
    __nv_bfloat16* kd = reinterpret_cast<__nv_bfloat16*>(k_cache) + slot * row_elems;
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x)
      kd[e] = __float2bfloat16_rn(to_f32(src[e]));
  } else if constexpr (FMT == 1 || FMT == 3) {
    const float sc = z ? v_scale : k_scale;
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x)
      dst[e] = f32_to_e4m3(__fdiv_rn(to_f32(src[e]), sc));
  } else {
    float amax = 0.f;
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x)
      amax = fmaxf(amax, fabsf(to_f32(src[e])));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = s_red[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
    const float sc = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.f);
    int8_t* d8 = reinterpret_cast<int8_t*>(dst);
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x) {
      float c = sc == 0.f ? 0.f : rintf(__fdiv_rn(to_f32(src[e]), sc));
      c = fminf(127.f, fmaxf(-127.f, c));
      d8[e] = (int8_t)c;
    }
    if (threadIdx.x == 0) (z ? v_ts : k_ts)[slot] = sc;
  }
}

// Per-token scales of copied blocks (INT8 pools): ts[dst*K + i] = ts[src*K + i].
__global__ void token_scale_copy_kernel(float* __restrict__ k_ts, float* __restrict__ v_ts,
                                        const int64_t* __restrict__ pairs, int64_t num_blocks,
                                        int32_t block_size) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t p = blockIdx.x;
  const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0) record_error(PKV_DEVERR_COPY_PAIR);
    return;
  }
  for (int i = threadIdx.x; i < block_size; i += blockDim.x) {
    k_ts[dst * block_size + i] = k_ts[src * block_size + i];
    v_ts[dst * block_size + i] = v_ts[src * block_size + i];
  }
}

// Failure-path self test: one CTA waits on an mbarrier that nothing ever
// arrives on; the bounded wait must give up after `limit` cycles and record
// PKV_DEVERR_TIMEOUT, leaving the context usable.
__global__ void selftest_wait_timeout_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(b, 0, limit);
  if (!ok && threadIdx.x == 0) record_error(PKV_DEVERR_TIMEOUT);
}

// a5 and block swap: move whole blocks from a source pool to a destination
// pool (the same pool for copy-on-write, a device pool and a mapped host pool
// for swap).  grid = (pairs, slices of a block, tensors); each thread moves
// UNROLL vectors, all loads before all stores, so a CTA keeps
// blockDim.x * UNROLL * VW bytes in flight (what hides the latency of host
// memory across the chip-to-chip link).  A destination block is never also
// a source block in the same launch (caller contract), so the restrict
// qualifiers hold even when the two pools are one.
template <int VW, int UNROLL>
__global__ void block_move_kernel(const uint8_t* __restrict__ src_k,
                                  const uint8_t* __restrict__ src_v, uint8_t* __restrict__ dst_k,
                                  uint8_t* __restrict__ dst_v, const int64_t* __restrict__ pairs,
                                  int64_t src_num_blocks, int64_t dst_num_blocks,
                                  int64_t block_bytes) {
  using V = typename VecT<VW>::T;
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t p = blockIdx.x;
  const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
  if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_error(PKV_DEVERR_COPY_PAIR);
    return;
  }
  const V* s = reinterpret_cast<const V*>((blockIdx.z ? src_v : src_k) + src * block_bytes);
  V* d = reinterpret_cast<V*>((blockIdx.z ? dst_v : dst_k) + dst * block_bytes);
  const int64_t nvec = block_bytes / VW;
  const int64_t first = (int64_t)blockIdx.y * blockDim.x * UNROLL + threadIdx.x;
  V buf[UNROLL];
#pragma unroll
  for (int u = 0; u < UNROLL; ++u) {
    const int64_t e = first + (int64_t)u * blockDim.x;
    if (e < nvec) buf[u] = s[e];
  }
#pragma unroll
  for (int u = 0; u < UNROLL; ++u) {
    const int64_t e = first + (int64_t)u * blockDim.x;
    if (e < nvec) d[e] = buf[u];
  }
}

}  // namespace pkv
