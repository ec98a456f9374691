// Multi-query paged attention on tcgen05 with two 128-row query tiles per CTA.
// Same function as attn_prefill_kernel (new token i of n at position
// len - n + i attends to positions 0 .. itself), for tiles of 128 query rows.
//
// The two query tiles (A: rows r0 .. r0+127, B: the next 128 rows of the same
// KV head and sequence) share every K and V tile: one TMA load feeds
// S_A = Q_A K^T and S_B = Q_B K^T, and O_A += P_A V, O_B += P_B V.  Each tile
// has its own softmax warpgroup, its own two S buffers and its own O in TMEM
// (4 x 128 = 512 columns), so the softmax of one tile runs while the tensor
// cores work on the other.
//
// Warps 0-3: softmax / epilogue of tile A, warps 4-7: of tile B (one thread
// per query row = TMEM lane, a full 64-key tile per thread).  Warp 8: TMA
// producer of K tiles (5-deep ring); warp 10: of V tiles (5-deep ring).
// Warp 9: TMEM allocation and, on one lane, the S = Q K^T issue for both
// tiles (up to two tiles ahead per query tile); warp 11, one lane: the
// O += P V issue.  P (split hi + lo bf16) is written by the softmax over the
// S buffer it came from and read from TMEM by the O += P V product (A operand
// in tensor memory); the S buffer is free again when that product is done.
// K and V rings are 5 deep.  The exponent base of a row is raised only when
// its maximum grows by more than 2^8 (O rescaled in TMEM rarely).  Compiled
// with SOLO (every KV head has at most one tile), tile B is switched off: no
// tile-B products, softmax or barriers.  Every wait is bounded and records
// PKV_DEVERR_TIMEOUT; TMEM is freed on every path after both issuing threads
// have seen their MMAs complete.
#pragma once

#include "pkv_prefill_tc05.cuh"

namespace pkv {

constexpr int kX2KStages = 5;
constexpr int kX2VStages = 5;

template <int D>
struct X2Cfg {
  static constexpr int NH = D / 64;
  static constexpr int QHALF = kT5Rows * 128;             // 16 KiB
  static constexpr int QBYTES = NH * QHALF;               // one query tile
  static constexpr int KVHALF = kPfBN * 128;              // 8 KiB
  static constexpr int KBYTES = NH * KVHALF;              // one K (or V) tile
  static constexpr int NBOX = NH * (kPfBN / 16);
  static constexpr int Q_OFF = 0;                         // [tile][half]
  static constexpr int K_OFF = 2 * QBYTES;
  static constexpr int V_OFF = K_OFF + kX2KStages * KBYTES;
  static constexpr int BAR_OFF = V_OFF + kX2VStages * KBYTES;
  // k_full/k_empty[KS], v_full/v_empty[VS], per tile: s_full[2], p_free[2],
  // p_full[2], o_done, q_full; mma_idle
  static constexpr int NBAR = 2 * (kX2KStages + kX2VStages) + 2 * 8 + 1;
  static constexpr int SLOT_OFF = BAR_OFF + 8 * NBAR;
  static constexpr int SMEM = SLOT_OFF + 16 + 1024;
  static constexpr int THREADS = 384;
  // per tile: S buffers 0, 1 (64 columns each, fp32 S, then P hi | lo as
  // bf16 pairs in the same columns), O (128)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = umma_idesc_bf16(kT5Rows, kPfBN, 0, 0);
  static constexpr uint32_t IDESC_PV = umma_idesc_bf16(kT5Rows, D, 0, 1);
};

// SOLO: every (sequence, KV head) has at most one 128-row query tile; tile B
// is then never used (its warps only stage their empty Q rows).
template <int D, bool SOLO>
__global__ void __launch_bounds__(X2Cfg<D>::THREADS, 1)
attn_prefill_tc05x2_kernel(const __grid_constant__ PfParams p) {
  using C = X2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + C::BAR_OFF;
  const uint32_t k_full = bars, k_empty = k_full + 8 * kX2KStages;
  const uint32_t v_full = k_empty + 8 * kX2KStages, v_empty = v_full + 8 * kX2VStages;
  const uint32_t tb0 = v_empty + 8 * kX2VStages;          // per-tile barriers, 8 each
  // Every barrier of S buffer b (s_full, p_full, p_free) completes once per
  // key tile kt with kt & 1 == b, at phase kt >> 1; a buffer cannot run two
  // phases ahead of its waiter, since S(kt + 2) needs O += P(kt) V done.
  auto s_full = [&](int x, int b) { return tb0 + 64 * x + 8 * b; };
  auto p_free = [&](int x, int b) { return tb0 + 64 * x + 16 + 8 * b; };
  auto p_full = [&](int x, int b) { return tb0 + 64 * x + 32 + 8 * b; };
  auto o_done = [&](int x) { return tb0 + 64 * x + 48; };
  auto q_full = [&](int x) { return tb0 + 64 * x + 56; };
  const uint32_t mma_idle = tb0 + 128;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, j = blockIdx.y;
  const int pair = gridDim.x - 1 - blockIdx.x;             // heaviest tile pairs first

  if (threadIdx.x == 0) {
    for (int i = 0; i < kX2KStages; ++i) {
      mbar_init(k_full + 8 * i, 1);
      mbar_init(k_empty + 8 * i, 2);                      // S_A and S_B both read K
    }
    for (int i = 0; i < kX2VStages; ++i) {
      mbar_init(v_full + 8 * i, 1);
      mbar_init(v_empty + 8 * i, 1);
    }
    for (int x = 0; x < 2; ++x) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(s_full(x, b), 1);
        mbar_init(p_free(x, b), 1);
        mbar_init(p_full(x, b), kT5Rows);
      }
      mbar_init(o_done(x), 1);
      mbar_init(q_full(x), kT5Rows);
    }
    mbar_init(mma_idle, 2);
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
    if (threadIdx.x == 0 && pair == 0) record_error(PKV_DEVERR_CONTEXT_LEN);
    active = false;
  }
  const int R = active ? n * G : 0;
  const int r0 = pair * 2 * kT5Rows;                      // tile A; tile B at r0 + 128
  if (r0 >= R) active = false;
  int pmax = -1, nkt = 0;
  if (active) {
    pmax = L - n + min(R - 1, r0 + 2 * kT5Rows - 1) / G;  // last key any row of the pair sees
    nkt = pmax / kPfBN + 1;
  }
  // tiles per CTA.  With SOLO only tile A; otherwise both, and a tile B
  // without rows (R <= r0 + 128) still runs its masked softmax so that every
  // barrier count stays the same
  constexpr int ntiles = SOLO ? 1 : 2;

  if (warp == 8 || warp == 10) {
    // =================== TMA producers: warp 8 K tiles, warp 10 V tiles ===================
    if (active) {
      const int kv = warp == 10;
      const CUtensorMap* map = kv ? &p.tmap_v : &p.tmap_k;
      const int NS = kv ? kX2VStages : kX2KStages;
      const uint32_t full = kv ? v_full : k_full, empty = kv ? v_empty : k_empty;
      uint8_t* ring = smem + (kv ? C::V_OFF : C::K_OFF);
      if (lane == 0) prefetch_tensormap(map);
      const uint64_t policy = l2_policy_evict_normal();
      const int sbl = K < 16 ? 1 : 0;                     // 8-token blocks: 8-row boxes
      const int ncopy = C::NBOX << sbl;                   // <= 16: one box per lane
      const int bi = lane >> sbl, u = lane & sbl;
      const int half = bi >> 2, rb = bi & 3;
      const int tr = rb * 16 + (u << 3);
      // the block-table entry of this lane's box, loaded one key tile ahead so
      // that its latency hides behind the wait for a free stage
      auto table_entry = [&](int kt) -> long long {
        const int tok = kt * kPfBN + tr;
        if (lane >= ncopy || kt >= nkt || tok > pmax) return -1;
        return p.block_tables[(int64_t)s * p.max_blocks_per_seq + tok / K];
      };
      long long phys_next = table_entry(0);
      int kt = 0;
      bool ok = true;
      for (; kt < nkt; ++kt) {
        const int stage = kt % NS;
        const long long phys = phys_next;
        phys_next = table_entry(kt + 1);
        if (!mbar_wait_bounded(empty + 8 * stage, ((kt / NS) & 1) ^ 1)) {
          record_error(PKV_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(full + 8 * stage, C::KBYTES);
        __syncwarp();
        if (lane < ncopy) {
          const int tok = kt * kPfBN + tr;
          int row = -32;                                  // past the last key: zero fill
          if (tok <= pmax) {
            if (phys < 0 || phys >= p.num_blocks) {
              record_error(PKV_DEVERR_BLOCK_ID);
            } else {
              row = (int)(phys * K + (tok - (tok / K) * K));
            }
          }
          uint8_t* sb = ring + stage * C::KBYTES;
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
    if (active && lane == 0) {
      bool ok = true;
      if (warp == 9) {
        ok = mbar_wait_bounded(q_full(0), 0) && mbar_wait_bounded(q_full(1), 0);
        for (int kt = 0; kt < nkt && ok; ++kt) {
          const int stage = kt % kX2KStages, b = kt & 1;
          if (!mbar_wait_bounded(k_full + 8 * stage, (kt / kX2KStages) & 1)) {
            ok = false;
            break;
          }
          const uint32_t kb = sbase + C::K_OFF + stage * C::KBYTES;
          for (int x = 0; x < ntiles && ok; ++x) {
            // S buffer b of tile x holds P(kt - 2) until O += P(kt - 2) V is done
            if (kt >= 2 && !mbar_wait_bounded(p_free(x, b), ((kt >> 1) - 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t qb = sbase + C::Q_OFF + x * C::QBYTES;
            const uint32_t sd = tmem + x * 256 + b * kPfBN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t ad = umma_desc_sw128(qb + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = umma_desc_sw128(kb + (kk >> 2) * C::KVHALF + (kk & 3) * 32, 16, 1024);
              umma_ss(sd, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full(x, b));
            umma_commit(k_empty + 8 * stage);
          }
          if (SOLO && ok) umma_commit(k_empty + 8 * stage);   // the slot's second arrival
        }
      } else {
        for (int t = 0; t < nkt && ok; ++t) {
          const int stage = t % kX2VStages;
          if (!mbar_wait_bounded(v_full + 8 * stage, (t / kX2VStages) & 1)) {
            ok = false;
            break;
          }
          const uint32_t vb = sbase + C::V_OFF + stage * C::KBYTES;
          for (int x = 0; x < ntiles && ok; ++x) {
            if (!mbar_wait_bounded(p_full(x, t & 1), (t >> 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // P hi in columns 0..31 of the S buffer, P lo in 32..63 (8 per 16 keys)
            const uint32_t pt = tmem + x * 256 + (t & 1) * kPfBN;
            const uint32_t od = tmem + x * 256 + 128;
#pragma unroll
            for (int k16 = 0; k16 < kPfBN / 16; ++k16) {
              const uint64_t bd = umma_desc_sw128(vb + k16 * 2048, C::KVHALF, 1024);
              umma_ts(od, pt + k16 * 8, bd, C::IDESC_PV, (t > 0 || k16 > 0) ? 1u : 0u);
              umma_ts(od, pt + 32 + k16 * 8, bd, C::IDESC_PV, 1u);
            }
            umma_commit(o_done(x));
            umma_commit(p_free(x, t & 1));
          }
          if (ok) umma_commit(v_empty + 8 * stage);
        }
      }
      if (!ok) record_error(PKV_DEVERR_TIMEOUT);
      umma_commit(mma_idle);
      mbar_wait_bounded(mma_idle, 0);
    }
  } else {
    // =================== softmax warps: warps 0-3 tile A, 4-7 tile B ===================
    const int x = warp >> 2;
    const int row = (warp & 3) * 32 + lane;      // TMEM lane = query row of tile x
    const int r = r0 + x * kT5Rows + row;
    const bool valid = active && r < R;
    const int i = valid ? r / G : 0;
    const int h = j * G + (valid ? r - i * G : 0);
    const int prow = valid ? L - n + i : -1;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t scol = x * 256, ocol = x * 256 + 128;
    int pw_min = valid ? prow : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pw_min = min(pw_min, __shfl_xor_sync(0xffffffffu, pw_min, o));
    bool ok = true;
    if (active) {
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((int64_t)(q0 + i) * p.H_q + h) * D);
      uint8_t* qt = smem + C::Q_OFF + x * C::QBYTES;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = valid ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qt + (c >> 3) * C::QHALF + row * 128 +
                                  (((c & 7) ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full(x));
    }
    const float sl = p.scale_log2;
    float m_used = 0.f, l = 0.f;
    const int my_nkt = x < ntiles ? nkt : 0;     // a tile without rows stops here
    for (int kt = 0; kt < my_nkt && ok; ++kt) {
      const int b = kt & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(s_full(x, b), (kt >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      float xs[kPfBN];
      {
        uint32_t sr[32];
        tmem_ld32(tmem + lane_base + scol + b * kPfBN, sr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) xs[e] = __uint_as_float(sr[e]);
        tmem_ld32(tmem + lane_base + scol + b * kPfBN + 32, sr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) xs[32 + e] = __uint_as_float(sr[e]);
      }
      const int kbase = kt * kPfBN;
      if (kbase + kPfBN - 1 > pw_min) {
        const int lim = prow - kbase;
#pragma unroll
        for (int e = 0; e < kPfBN; ++e) xs[e] = e <= lim ? xs[e] : -INFINITY;
      }
      // row maximum: four chains of three-input max over the 64 scores
      float m4[4] = {fmax3(xs[0], xs[1], xs[2]), fmax3(xs[3], xs[4], xs[5]),
                     fmax3(xs[6], xs[7], xs[8]), fmax3(xs[9], xs[10], xs[11])};
#pragma unroll
      for (int e = 12; e + 1 < kPfBN; e += 2) m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], xs[e], xs[e + 1]);
      const float mt = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl;
      if (kt == 0) {
        m_used = mt == -INFINITY ? 0.f : mt;
      } else {
        const bool need = mt > m_used + kT5Slack;
        if (__any_sync(0xffffffffu, need)) {
          // O in TMEM is rescaled; O += P(kt-1) V must have landed first.  S(kt)
          // full implies O += P(kt-2) V done, so o_done is at most one phase behind
          // and its parity names the phase unambiguously
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_done(x), (kt - 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const float mn = need ? mt : m_used;
          const float alpha = exp2f(m_used - mn);
          l *= alpha;
          m_used = mn;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
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
      // p = 2^(s * scale * log2 e - m): the scale and shift as packed fp32x2 FMAs,
      // the row sum as packed adds
      float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(-m_used, -m_used);
#pragma unroll
      for (int c = 0; c < kPfBN / 2; ++c) {
        const float2 y = __ffma2_rn(make_float2(xs[2 * c], xs[2 * c + 1]), sl2, nm2);
        xs[2 * c] = ex2_approx(y.x);
        xs[2 * c + 1] = ex2_approx(y.y);
        s2[c & 1] = __fadd2_rn(s2[c & 1], make_float2(xs[2 * c], xs[2 * c + 1]));
      }
      l += (s2[0].x + s2[0].y) + (s2[1].x + s2[1].y);
      // P hi | lo over the S just read (this thread's row = its TMEM lane)
      {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) split_bf16x2_trunc(xs[2 * c], xs[2 * c + 1], hi[c], lo[c]);
        tmem_st32(tmem + lane_base + scol + b * kPfBN, hi);
        tmem_st32(tmem + lane_base + scol + b * kPfBN + 32, lo);
        tmem_wait_st();
      }
      if (x == 0 && kt == nkt - 1 && L - kbase < kPfBN) {
        // V rows at or past the context end inside fetched boxes may hold
        // anything (NaN included): tile A zeroes them before its O += P V
        // (tile B's product is issued after tile A's)
        const int stage = kt % kX2VStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(v_full + 8 * stage, (kt / kX2VStages) & 1));
        if (!ok) break;
        const int z0 = L - kbase, z1 = min(kPfBN, ((pmax - kbase) / 16 + 1) * 16);
        uint8_t* vs = smem + C::V_OFF + stage * C::KBYTES;
        for (int x2 = z0 * 8 + row; x2 < z1 * 8; x2 += kT5Rows) {
#pragma unroll
          for (int hh = 0; hh < C::NH; ++hh)
            *reinterpret_cast<uint4*>(vs + hh * C::KVHALF + x2 * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full(x, b));
    }
    // ---- epilogue: O / l from TMEM to the output rows
    if (active && ok && my_nkt > 0) {
      // o_done may still be two phases behind here; the last buffer's P-free
      // commit follows every O += P V of this tile
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(p_free(x, (nkt - 1) & 1), ((nkt - 1) >> 1) & 1));
      if (ok) {
        tc_fence_after();
        const float inv = valid ? 1.f / l : 0.f;
        uint4* orow = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + i) * p.H_q + h) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
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
