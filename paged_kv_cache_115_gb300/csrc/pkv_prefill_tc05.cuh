// Multi-query paged attention on the 5th-generation tensor cores (tcgen05).
// Same function as attn_prefill_kernel (new token i of n at position
// len - n + i attends to positions 0 .. itself), for tiles of 128 query rows:
//
//   S  = Q K^T   tcgen05.mma M=128 N=64 K=D, Q and K 128-byte-swizzled K-major
//                tiles in shared memory, S (fp32) in TMEM, three buffers
//   P  = 2^(S' - m)  by 8 softmax warps, two threads per query row, S read
//                from TMEM; P split hi + lo bf16 and stored K-major
//   O += P V     tcgen05.mma M=128 N=D K=64 (x2 for hi and lo), V the
//                MN-major 128-byte-swizzled tile straight from TMA; O (fp32)
//                stays in TMEM for the whole key loop
//
// Warps 0-7: softmax / epilogue, two threads per query row (TMEM lanes 0-127
// = query rows; warps 0-3 and 4-7 take the two halves of each key tile and of
// O).  Warps 8 and 10: TMA producers of 64-token K tiles (4-deep ring) and V
// tiles (3-deep ring) from the paged pool; a K slot frees as soon as its
// S = Q K^T has completed, a V slot once O += P V has.  Warp 9: TMEM
// allocation and, on one lane, the S = Q K^T issue, up to three tiles ahead
// (three S buffers, each free again once the softmax has read it); warp 11,
// one lane: the O += P V issue.  The softmax warps never wait for S and the
// tensor work of neighbouring tiles overlaps the softmax.  The running
// maximum used for the exponentials is raised only when a row's new maximum
// exceeds it by more than 8 (base 2),
// so O in TMEM is rescaled rarely (P <= 2^8 otherwise; the final division by
// the running sum makes the result the same softmax).  Every wait is bounded
// and records PKV_DEVERR_TIMEOUT when it gives up; TMEM is freed on every
// path.
#pragma once

#include "pkv_prefill.cuh"
#include "pkv_umma.cuh"

namespace pkv {

// 2^x on the multi-function unit (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (a, b) -> bf16 pairs hi, lo with a ~ hi + lo, without conversion
// instructions: hi truncates a to its upper 16 bits, the remainder a - hi is
// exact in fp32 and is truncated the same way, so that 0 <= a - (hi + lo)
// < 2^-14 a for the finite non-negative a the softmax produces.  The two
// remainders are formed with one packed fp32x2 FMA.
__device__ __forceinline__ void split_bf16x2_trunc(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const float2 t = make_float2(__uint_as_float(ua & 0xffff0000u), __uint_as_float(ub & 0xffff0000u));
  const float2 r = __ffma2_rn(t, make_float2(-1.f, -1.f), make_float2(a, b));
  hi = __byte_perm(ua, ub, 0x7632);
  lo = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

constexpr int kT5Rows = 128;     // query rows per CTA: one M = 128 MMA
constexpr int kT5KStages = 4;    // K ring depth
constexpr int kT5VStages = 3;    // V ring depth
constexpr int kT5SBufs = 3;      // S buffers in TMEM: S = Q K^T runs this many tiles ahead
constexpr float kT5Slack = 8.f;  // raise the exponent base only past this (log2 units)

template <int D>
struct T5Cfg {
  static constexpr int NH = D / 64;                       // 64-column halves of a row
  static constexpr int QHALF = kT5Rows * 128;             // 16 KiB
  static constexpr int QBYTES = NH * QHALF;
  static constexpr int KVHALF = kPfBN * 128;              // 8 KiB: 64 rows x 128 B
  static constexpr int KBYTES = NH * KVHALF;             // one K (or V) tile
  static constexpr int NBOX = NH * (kPfBN / 16);          // 16-row boxes per tile
  static constexpr int PBUF = kT5Rows * 128;              // 128 rows x 64 keys bf16
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = QBYTES;                    // K ring
  static constexpr int V_OFF = K_OFF + kT5KStages * KBYTES;   // V ring
  static constexpr int P_OFF = V_OFF + kT5VStages * KBYTES;   // [buffer][hi, lo]
  static constexpr int RED_OFF = P_OFF + 4 * PBUF;          // float [2][2][128] row maxima
  static constexpr int LSUM_OFF = RED_OFF + 2 * 2 * kT5Rows * 4;   // float [2][128] row sums
  static constexpr int BAR_OFF = LSUM_OFF + 2 * kT5Rows * 4;
  static constexpr int NBAR = 2 * (kT5KStages + kT5VStages) + 2 * kT5SBufs + 9;
  static constexpr int SLOT_OFF = BAR_OFF + 8 * NBAR;
  static constexpr int SMEM = SLOT_OFF + 16 + 1024;          // + alignment slack
  static constexpr int SOFTMAX_THREADS = 2 * kT5Rows;        // two threads per query row
  static constexpr int THREADS = SOFTMAX_THREADS + 128;  // + K producer, 2 MMA issuers, V producer
  static constexpr uint32_t TMEM_COLS = 512;                 // S0-S2 [0,192), O [256,256+D)
  static constexpr uint32_t O_COL = 256;
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
  const uint32_t k_full = bars, k_empty = k_full + 8 * kT5KStages;   // + 8 * stage
  const uint32_t v_full = k_empty + 8 * kT5KStages, v_empty = v_full + 8 * kT5VStages;
  const uint32_t s_full = v_empty + 8 * kT5VStages;                  // + 8 * S buffer
  const uint32_t s_free = s_full + 8 * kT5SBufs;                     // + 8 * S buffer
  const uint32_t p_full = s_free + 8 * kT5SBufs;                     // + 8 * P buffer
  const uint32_t o_done = p_full + 16, q_full = o_done + 16;
  const uint32_t mma_idle = q_full + 8;         // every issued MMA has completed
  const uint32_t x_full = mma_idle + 8;         // + 8 * buffer: row maxima exchanged
  const uint32_t l_full = x_full + 16;          // row sums exchanged
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, j = blockIdx.y;
  const int tile = gridDim.x - 1 - blockIdx.x;             // heaviest tiles first

  if (threadIdx.x == 0) {
    for (int i = 0; i < kT5KStages; ++i) {
      mbar_init(k_full + 8 * i, 1);
      mbar_init(k_empty + 8 * i, 1);
    }
    for (int i = 0; i < kT5VStages; ++i) {
      mbar_init(v_full + 8 * i, 1);
      mbar_init(v_empty + 8 * i, 1);
    }
    for (int b = 0; b < kT5SBufs; ++b) {
      mbar_init(s_full + 8 * b, 1);
      mbar_init(s_free + 8 * b, C::SOFTMAX_THREADS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(p_full + 8 * b, C::SOFTMAX_THREADS);
      mbar_init(o_done + 8 * b, 1);
      mbar_init(x_full + 8 * b, C::SOFTMAX_THREADS);
    }
    mbar_init(q_full, C::SOFTMAX_THREADS);
    mbar_init(mma_idle, 2);
    mbar_init(l_full, C::SOFTMAX_THREADS);
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(slot), C::TMEM_COLS);
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

  if (warp == 8 || warp == 10) {
    // =================== TMA producers: warp 8 K tiles, warp 10 V tiles ===================
    if (active) {
      const int kv = warp == 10;
      const CUtensorMap* map = kv ? &p.tmap_v : &p.tmap_k;
      const int NS = kv ? kT5VStages : kT5KStages;
      const uint32_t full = kv ? v_full : k_full, empty = kv ? v_empty : k_empty;
      uint8_t* ring = smem + (kv ? C::V_OFF : C::K_OFF);
      if (lane == 0) prefetch_tensormap(map);
      const uint64_t policy = l2_policy_evict_normal();   // re-read by the other row tiles
      const int sbl = K < 16 ? 1 : 0;                     // 8-token blocks: two boxes per 16 rows
      const int ncopy = C::NBOX << sbl;
      int kt = 0;
      bool ok = true;
      for (; kt < nkt; ++kt) {
        const int stage = kt % NS;
        if (!mbar_wait_bounded(empty + 8 * stage, ((kt / NS) & 1) ^ 1)) {
          record_error(PKV_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(full + 8 * stage, C::KBYTES);
        __syncwarp();
        uint8_t* sb = ring + stage * C::KBYTES;
        for (int i = lane; i < ncopy; i += 32) {
          const int bi = i >> sbl, u = i & sbl;
          const int half = bi >> 2, rb = bi & 3;
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
          tma_load_3d(smem_u32(sb + half * C::KVHALF + tr * 128), map, full + 8 * stage,
                      half * 64, j, row, policy);
        }
        __syncwarp();
      }
      if (!ok) {
        for (int kk = max(0, kt - NS); kk < kt; ++kk)
          mbar_wait_bounded(full + 8 * (kk % NS), (kk / NS) & 1);
      }
    }
  } else if (warp == 9 || warp == 11) {
    // =================== MMA issue: warp 9 S = Q K^T, warp 11 O += P V ===================
    // Two issuing threads: one tcgen05.mma takes a thread tens of cycles to
    // issue, about as long as a 128 x 64 x 16 product takes to run.
    if (active && lane == 0) {
      bool ok = true;
      if (warp == 9) {
        ok = mbar_wait_bounded(q_full, 0);
        for (int kt = 0; kt < nkt && ok; ++kt) {
          const int stage = kt % kT5KStages, sb = kt % kT5SBufs;
          // S buffer sb is free once the softmax has read S(kt - kT5SBufs)
          if (kt >= kT5SBufs && !mbar_wait_bounded(s_free + 8 * sb, ((kt / kT5SBufs) - 1) & 1)) {
            ok = false;
            break;
          }
          if (!mbar_wait_bounded(k_full + 8 * stage, (kt / kT5KStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb = sbase + C::K_OFF + stage * C::KBYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad =
                umma_desc_sw128(sbase + C::Q_OFF + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024);
            const uint64_t bd =
                umma_desc_sw128(kb + (kk >> 2) * C::KVHALF + (kk & 3) * 32, 16, 1024);
            umma_ss(tmem + sb * kPfBN, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full + 8 * sb);
          umma_commit(k_empty + 8 * stage);
        }
      } else {
        for (int t = 0; t < nkt && ok; ++t) {
          const int b = t & 1, stage = t % kT5VStages;
          if (!mbar_wait_bounded(p_full + 8 * b, (t >> 1) & 1) ||
              !mbar_wait_bounded(v_full + 8 * stage, (t / kT5VStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = sbase + C::V_OFF + stage * C::KBYTES;
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
          umma_commit(v_empty + 8 * stage);
        }
      }
      if (!ok) record_error(PKV_DEVERR_TIMEOUT);
      // TMEM is freed below: wait (bounded) until none of this thread's
      // MMAs is in flight (both issuing threads arrive on mma_idle)
      umma_commit(mma_idle);
      mbar_wait_bounded(mma_idle, 0);
    }
  } else {
    // =================== softmax warps ===================
    // Two threads per query row: warps 0-3 take keys 0-31 of each tile and
    // O columns [0, D/2), warps 4-7 keys 32-63 and O columns [D/2, D); both
    // reach the row's TMEM lane (warp w reads lanes 32 (w mod 4) ..).  The
    // two halves exchange their tile maxima through shared memory.
    const int hk = warp >> 2;
    const int row = (warp & 3) * 32 + lane;      // 0 .. 127 = TMEM lane
    const int r = r0 + row;
    const bool valid = active && r < R;
    const int i = valid ? r / G : 0;
    const int h = j * G + (valid ? r - i * G : 0);
    const int prow = valid ? L - n + i : -1;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + C::RED_OFF);     // [buffer][half][row]
    float* lsum = reinterpret_cast<float*>(smem + C::LSUM_OFF);   // [half][row]
    int pw_min = valid ? prow : 0x7fffffff;      // smallest position of the warp's valid rows
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pw_min = min(pw_min, __shfl_xor_sync(0xffffffffu, pw_min, o));
    bool ok = true;
    if (active) {
      // this half of the row of Q into the swizzled K-major Q tile
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((int64_t)(q0 + i) * p.H_q + h) * D);
#pragma unroll
      for (int c0 = 0; c0 < D / 16; ++c0) {
        const int c = hk * (D / 16) + c0;
        const uint4 v = valid ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + C::Q_OFF + (c >> 3) * C::QHALF + row * 128 +
                                  (((c & 7) ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    const float sl = p.scale_log2;
    const uint32_t ocol = C::O_COL + hk * (D / 2);
    float m_used = 0.f, l = 0.f;
    for (int kt = 0; kt < nkt && ok; ++kt) {
      const int b = kt & 1, sbuf = kt % kT5SBufs;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(s_full + 8 * sbuf, (kt / kT5SBufs) & 1));
      if (!ok) break;
      tc_fence_after();
      float x[32];
      {
        uint32_t sr[32];
        tmem_ld32(tmem + lane_base + sbuf * kPfBN + hk * 32, sr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(sr[e]);
      }
      tc_fence_before();
      mbar_arrive(s_free + 8 * sbuf);           // S buffer may be overwritten
      const int kbase = kt * kPfBN + hk * 32;    // key of x[0]
      // raw scores; the scale (> 0) is applied inside the exponent below.
      // Key ranges wholly below every row's position of this warp need no mask.
      if (kbase + 31 > pw_min) {
        const int lim = prow - kbase;
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = e <= lim ? x[e] : -INFINITY;
      }
      // four independent chains, then combined
      float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int e = 4; e < 32; ++e) m4[e & 3] = fmaxf(m4[e & 3], x[e]);
      float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      red[(b * 2 + hk) * kT5Rows + row] = mt;
      mbar_arrive(x_full + 8 * b);
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(x_full + 8 * b, (kt >> 1) & 1));
      if (!ok) break;
      mt = fmaxf(red[(b * 2) * kT5Rows + row], red[(b * 2 + 1) * kT5Rows + row]) * sl;
      if (kt == 0) {
        m_used = mt == -INFINITY ? 0.f : mt;
      } else {
        const bool need = mt > m_used + kT5Slack;
        if (__any_sync(0xffffffffu, need)) {
          // O in TMEM is rescaled; O += P(kt-1) V must have landed first
          ok = __all_sync(0xffffffffu,
                          mbar_wait_bounded(o_done + 8 * ((kt - 1) & 1), ((kt - 1) >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const float mn = need ? mt : m_used;
          const float alpha = exp2f(m_used - mn);
          l *= alpha;
          m_used = mn;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + ocol + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_base + ocol + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
      const float nm = -m_used;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        x[e] = ex2_approx(fmaf(x[e], sl, nm));
        s4[e & 3] += x[e];
      }
      l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
      // P buffer b is free once O += P(kt-2) V has completed
      if (kt >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_done + 8 * b, ((kt - 2) >> 1) & 1));
      if (!ok) break;
      uint8_t* phi = smem + C::P_OFF + (2 * b) * C::PBUF + row * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16x2(x[cc * 8 + 2 * e], x[cc * 8 + 2 * e + 1], hi[e], lo[e]);
        const int off = (((hk * 4 + cc) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(phi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(phi + C::PBUF + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      const int tbase = kt * kPfBN;
      if (kt == nkt - 1 && L - tbase < kPfBN) {
        // V rows at or past the context end inside fetched boxes may hold
        // anything (NaN included): zero them before O += P V reads them
        const int stage = kt % kT5VStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(v_full + 8 * stage, (kt / kT5VStages) & 1));
        if (!ok) break;
        const int z0 = L - tbase, z1 = min(kPfBN, ((pmax - tbase) / 16 + 1) * 16);
        uint8_t* vs = smem + C::V_OFF + stage * C::KBYTES;
        for (int x2 = z0 * 8 + hk * kT5Rows + row; x2 < z1 * 8; x2 += C::SOFTMAX_THREADS) {
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
      lsum[hk * kT5Rows + row] = l;
      mbar_arrive(l_full);
      const int last = nkt - 1;
      ok = mbar_wait_bounded(l_full, 0) &&
           mbar_wait_bounded(o_done + 8 * (last & 1), (last >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const float lt = lsum[row] + lsum[kT5Rows + row];
        const float inv = valid ? 1.f / lt : 0.f;
        uint4* orow = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + i) * p.H_q + h) * D +
                                               hk * (D / 2));
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + ocol + c * 32, o);
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
  if (warp == 9) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace pkv
