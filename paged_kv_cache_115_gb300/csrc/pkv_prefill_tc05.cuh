// Multi-query paged attention on the 5th-generation tensor cores (tcgen05).
// Same function as attn_prefill_kernel (new token i of n at position
// len - n + i attends to positions 0 .. itself), for tiles of 128 query rows:
//
//   S  = Q K^T   tcgen05.mma M=128 N=64 K=D, Q and K 128-byte-swizzled K-major
//                tiles in shared memory, S (fp32) in TMEM, double-buffered
//   P  = 2^(S' - m)  by 4 softmax warps, one thread per query row, S read
//                from TMEM; P split hi + lo bf16 and stored K-major
//   O += P V     tcgen05.mma M=128 N=D K=64 (x2 for hi and lo), V the
//                MN-major 128-byte-swizzled tile straight from TMA; O (fp32)
//                stays in TMEM for the whole key loop
//
// Warps 0-3: softmax / epilogue (TMEM lanes 0-127 = query rows).  Warp 4:
// TMA producer of 64-token K and V tiles from the paged pool (3 stages).
// Warp 5: TMEM allocation and, on one lane, MMA issue.  The MMA thread issues
// S(kt) before O += P(kt-1) V, so the softmax of tile kt overlaps the tensor
// work of its neighbours.  The running maximum used for the exponentials is
// raised only when a row's new maximum exceeds it by more than 8 (base 2),
// so O in TMEM is rescaled rarely (P <= 2^8 otherwise; the final division by
// the running sum makes the result the same softmax).  Every wait is bounded
// and records PKV_DEVERR_TIMEOUT when it gives up; TMEM is freed on every
// path.
#pragma once

#include "pkv_prefill.cuh"
#include "pkv_umma.cuh"

namespace pkv {

constexpr int kT5Rows = 128;     // query rows per CTA: one M = 128 MMA
constexpr int kT5Stages = 3;     // K/V ring depth
constexpr float kT5Slack = 8.f;  // raise the exponent base only past this (log2 units)

template <int D>
struct T5Cfg {
  static constexpr int NH = D / 64;                       // 64-column halves of a row
  static constexpr int QHALF = kT5Rows * 128;             // 16 KiB
  static constexpr int QBYTES = NH * QHALF;
  static constexpr int KVHALF = kPfBN * 128;              // 8 KiB: 64 rows x 128 B
  static constexpr int KBYTES = NH * KVHALF;
  static constexpr int STAGE = 2 * KBYTES;                // K tile, then V tile
  static constexpr int NBOX = 2 * NH * (kPfBN / 16);      // 16-row boxes per stage
  static constexpr int PBUF = kT5Rows * 128;              // 128 rows x 64 keys bf16
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = QBYTES;
  static constexpr int P_OFF = KV_OFF + kT5Stages * STAGE;   // [buffer][hi, lo]
  static constexpr int BAR_OFF = P_OFF + 4 * PBUF;
  static constexpr int NBAR = 2 * kT5Stages + 8;
  static constexpr int SLOT_OFF = BAR_OFF + 8 * NBAR;
  static constexpr int SMEM = SLOT_OFF + 16 + 1024;          // + alignment slack
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 256;                 // S0 [0,64) S1 [64,128) O [128,128+D)
  static constexpr uint32_t O_COL = 128;
  static constexpr uint32_t IDESC_QK = umma_idesc_bf16(kT5Rows, kPfBN, 0, 0);
  static constexpr uint32_t IDESC_PV = umma_idesc_bf16(kT5Rows, D, 0, 1);
};

template <int D>
__global__ void __launch_bounds__(T5Cfg<D>::THREADS, 1)
attn_prefill_tc05_kernel(const __grid_constant__ PfParams p) {
  using C = T5Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + C::BAR_OFF;
  const uint32_t kv_full = bars, kv_empty = bars + 8 * kT5Stages;   // + 8 * stage
  const uint32_t s_full = bars + 16 * kT5Stages;                    // + 8 * buffer
  const uint32_t p_full = s_full + 16, o_done = s_full + 32, q_full = s_full + 48;
  const uint32_t mma_idle = s_full + 56;        // every issued MMA has completed
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, j = blockIdx.y;
  const int tile = gridDim.x - 1 - blockIdx.x;             // heaviest tiles first

  if (threadIdx.x == 0) {
    for (int i = 0; i < kT5Stages; ++i) {
      mbar_init(kv_full + 8 * i, 1);
      mbar_init(kv_empty + 8 * i, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + 8 * b, 1);
      mbar_init(p_full + 8 * b, kT5Rows);
      mbar_init(o_done + 8 * b, 1);
    }
    mbar_init(q_full, kT5Rows);
    mbar_init(mma_idle, 1);
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(smem_u32(slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  pdl_wait_primary();
  pdl_launch_dependents();

  const int K = p.block_size;
  const int G = p.G;
  const int q0 = p.cu_seqlens[s], q1 = p.cu_seqlens[s + 1];
  const int L = effective_len(p.context_lens[s], p.max_len, p.max_blocks_per_seq * K);
  const int n = q1 - q0;
  bool active = true;
  if (q0 < 0 || n < 0 || q1 > p.num_tokens || n > L) {
    if (threadIdx.x == 0 && tile == 0) record_error(PKV_DEVERR_CONTEXT_LEN);
    active = false;
  }
  const int R = active ? n * G : 0;
  const int r0 = tile * kT5Rows;
  if (r0 >= R) active = false;
  int pmax = -1, nkt = 0;
  if (active) {
    pmax = L - n + min(R - 1, r0 + kT5Rows - 1) / G;   // last key any row sees
    nkt = pmax / kPfBN + 1;
  }

  if (warp == 4) {
    // =================== TMA producer ===================
    if (active) {
      if (lane == 0) {
        prefetch_tensormap(&p.tmap_k);
        prefetch_tensormap(&p.tmap_v);
      }
      const uint64_t policy = l2_policy_evict_normal();   // re-read by the other row tiles
      const int sbl = K < 16 ? 1 : 0;                     // 8-token blocks: two boxes per 16 rows
      const int ncopy = C::NBOX << sbl;
      int kt = 0;
      bool ok = true;
      for (; kt < nkt; ++kt) {
        const int stage = kt % kT5Stages;
        if (!mbar_wait_bounded(kv_empty + 8 * stage, ((kt / kT5Stages) & 1) ^ 1)) {
          record_error(PKV_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(kv_full + 8 * stage, C::STAGE);
        __syncwarp();
        uint8_t* sb = smem + C::KV_OFF + stage * C::STAGE;
        for (int i = lane; i < ncopy; i += 32) {
          const int bi = i >> sbl, u = i & sbl;
          const int kv = bi / (C::NH * 4);
          const int rem = bi - kv * (C::NH * 4);
          const int half = rem >> 2, rb = rem & 3;
          const int tr = rb * 16 + (u << 3);
          const int tok = kt * kPfBN + tr;
          int row = -32;                                  // wholly out of bounds: zeros
          if (tok <= pmax) {
            const int lb = tok / K;
            const long long phys = p.block_tables[(int64_t)s * p.max_blocks_per_seq + lb];
            if (phys < 0 || phys >= p.num_blocks) {
              record_error(PKV_DEVERR_BLOCK_ID);
            } else {
              row = (int)(phys * K + (tok - lb * K));
            }
          }
          tma_load_3d(smem_u32(sb + kv * C::KBYTES + half * C::KVHALF + tr * 128),
                      kv ? &p.tmap_v : &p.tmap_k, kv_full + 8 * stage, half * 64, j, row,
                      policy);
        }
        __syncwarp();
      }
      if (!ok) {
        for (int kk = max(0, kt - kT5Stages); kk < kt; ++kk)
          mbar_wait_bounded(kv_full + 8 * (kk % kT5Stages), (kk / kT5Stages) & 1);
      }
    }
  } else if (warp == 5) {
    // =================== MMA issue (one thread) ===================
    if (active && lane == 0) {
      bool ok = mbar_wait_bounded(q_full, 0);
      tc_fence_after();
      int issued = 0;                       // O += P V products issued so far
      auto pv = [&](int t) -> bool {
        const int b = t & 1, stage = t % kT5Stages;
        if (!mbar_wait_bounded(p_full + 8 * b, (t >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t vb = sbase + C::KV_OFF + stage * C::STAGE + C::KBYTES;
        const uint32_t ph = sbase + C::P_OFF + (2 * b) * C::PBUF;
#pragma unroll
        for (int k16 = 0; k16 < kPfBN / 16; ++k16) {
          const uint64_t bd = umma_desc_sw128(vb + k16 * 2048, C::KVHALF, 1024);
          umma_ss(tmem + C::O_COL, umma_desc_sw128(ph + k16 * 32, 16, 1024), bd, C::IDESC_PV,
                  (t > 0 || k16 > 0) ? 1u : 0u);
          umma_ss(tmem + C::O_COL, umma_desc_sw128(ph + C::PBUF + k16 * 32, 16, 1024), bd,
                  C::IDESC_PV, 1u);
        }
        umma_commit(o_done + 8 * b);
        umma_commit(kv_empty + 8 * stage);
        ++issued;
        return true;
      };
      for (int kt = 0; kt < nkt && ok; ++kt) {
        const int stage = kt % kT5Stages;
        if (!mbar_wait_bounded(kv_full + 8 * stage, (kt / kT5Stages) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = sbase + C::KV_OFF + stage * C::STAGE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad =
              umma_desc_sw128(sbase + C::Q_OFF + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc_sw128(kb + (kk >> 2) * C::KVHALF + (kk & 3) * 32, 16, 1024);
          umma_ss(tmem + (kt & 1) * kPfBN, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
        }
        umma_commit(s_full + 8 * (kt & 1));
        if (kt >= 1 && !pv(kt - 1)) ok = false;
      }
      if (ok && issued < nkt) ok = pv(nkt - 1);
      if (!ok) record_error(PKV_DEVERR_TIMEOUT);
      // TMEM is freed below: wait (bounded) until no MMA is in flight
      umma_commit(mma_idle);
      mbar_wait_bounded(mma_idle, 0);
    }
  } else {
    // =================== softmax warps (thread = query row) ===================
    const int row = threadIdx.x;                 // 0 .. 127 = TMEM lane
    const int r = r0 + row;
    const bool valid = active && r < R;
    const int i = valid ? r / G : 0;
    const int h = j * G + (valid ? r - i * G : 0);
    const int prow = valid ? L - n + i : -1;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    bool ok = true;
    if (active) {
      // this row of Q into the swizzled K-major Q tile
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((int64_t)(q0 + i) * p.H_q + h) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = valid ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + C::Q_OFF + (c >> 3) * C::QHALF + row * 128 +
                                  (((c & 7) ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    const float sl = p.scale_log2;
    float m_used = 0.f, l = 0.f;
    for (int kt = 0; kt < nkt && ok; ++kt) {
      const int b = kt & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(s_full + 8 * b, (kt >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      float x[kPfBN];
      {
        uint32_t sr[32];
        tmem_ld32(tmem + lane_base + b * kPfBN, sr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(sr[e]);
        tmem_ld32(tmem + lane_base + b * kPfBN + 32, sr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[32 + e] = __uint_as_float(sr[e]);
      }
      const int kbase = kt * kPfBN;
      float mt = -INFINITY;
#pragma unroll
      for (int e = 0; e < kPfBN; ++e) {
        x[e] = kbase + e <= prow ? x[e] * sl : -INFINITY;
        mt = fmaxf(mt, x[e]);
      }
      if (kt == 0) {
        m_used = mt == -INFINITY ? 0.f : mt;
      } else {
        const bool need = mt > m_used + kT5Slack;
        if (__any_sync(0xffffffffu, need)) {
          // O in TMEM is rescaled; O += P(kt-1) V must have landed first
          if (!mbar_wait_bounded(o_done + 8 * ((kt - 1) & 1), ((kt - 1) >> 1) & 1)) ok = false;
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const float mn = need ? mt : m_used;
          const float alpha = exp2f(m_used - mn);
          l *= alpha;
          m_used = mn;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + C::O_COL + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_base + C::O_COL + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < kPfBN; ++e) {
        x[e] = exp2f(x[e] - m_used);
        sum += x[e];
      }
      l += sum;
      // P buffer b is free once O += P(kt-2) V has completed
      if (kt >= 2 && !mbar_wait_bounded(o_done + 8 * b, ((kt - 2) >> 1) & 1)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      uint8_t* phi = smem + C::P_OFF + (2 * b) * C::PBUF + row * 128;
#pragma unroll
      for (int cc = 0; cc < kPfBN / 8; ++cc) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16x2(x[cc * 8 + 2 * e], x[cc * 8 + 2 * e + 1], hi[e], lo[e]);
        const int off = ((cc ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(phi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(phi + C::PBUF + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      if (kt == nkt - 1 && L - kbase < kPfBN) {
        // V rows at or past the context end inside fetched boxes may hold
        // anything (NaN included): zero them before O += P V reads them
        const int stage = kt % kT5Stages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(kv_full + 8 * stage, (kt / kT5Stages) & 1));
        if (!ok) break;
        const int z0 = L - kbase, z1 = min(kPfBN, ((pmax - kbase) / 16 + 1) * 16);
        uint8_t* vs = smem + C::KV_OFF + stage * C::STAGE + C::KBYTES;
        for (int x2 = z0 * 8 + row; x2 < z1 * 8; x2 += kT5Rows) {
#pragma unroll
          for (int hh = 0; hh < C::NH; ++hh)
            *reinterpret_cast<uint4*>(vs + hh * C::KVHALF + x2 * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full + 8 * b);
    }
    // ---- epilogue: O / l from TMEM to the output rows
    if (active && ok) {
      const int last = nkt - 1;
      ok = mbar_wait_bounded(o_done + 8 * (last & 1), (last >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const float inv = valid ? 1.f / l : 0.f;
        uint4* orow = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + i) * p.H_q + h) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + C::O_COL + c * 32, o);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2 * e]) * inv,
                                   __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv);
              orow[c * 4 + q4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
    if (active && !ok) record_error(PKV_DEVERR_TIMEOUT);
  }

  // ---- teardown: every warp, every path
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace pkv
