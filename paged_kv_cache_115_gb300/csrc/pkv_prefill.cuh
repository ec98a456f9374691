// Multi-query paged attention: several new tokens of a sequence attend at
// once over the paged cache (chunked prefill and prefix-hit suffix prefill,
// "KV Cache：长上下文为什么吃显存，PagedAttention 怎么救" §06 and
// "推理与 KV Cache 02:分页、共享与回收如何协作", 前缀索引与 Block Table; several
// speculative candidate tokens, "企业官网建设流程全解析" §8.2).  New token i
// of n sits at position len - n + i and attends to positions 0 .. itself.
//
// Work split: one CTA per (tile of BM query rows, KV head, sequence).  The
// rows of KV head j are the pairs (new token i, query head of j's group),
// row = i * G + head-in-group, so one tile serves every head of the group and
// the K/V tile it streams is read once for all of them.  Tiles are launched
// heaviest first (the last tile sees the most keys).
//
// Roles: warp NW is the producer: its lanes issue TMA loads of 64-token K and
// V tiles (16-row boxes out of the pool viewed as [D, H_kv, num_blocks * K],
// 128-byte swizzle, so a tile is 64 rows of 128-byte lines per 64 columns)
// into a 3-stage ring with full / empty mbarriers.  Key boxes wholly past the
// tile's last query position are not read (TMA fills them with zeros).
// Warps 0 .. NW-1 are consumers, 16 query rows each: S = Q K^T with
// mma.sync m16n8k16 bf16 -> fp32 (Q in registers as A fragments, K tiles
// through ldmatrix as B fragments), causal mask per row, online softmax in
// base 2, O += P V with P split into hi + lo bf16 terms (one bf16 rounding of
// P costs 2^-9 per weight, too much for short cancelling rows) and V through
// ldmatrix.trans.  Every wait is bounded (about a second) and records
// PKV_DEVERR_TIMEOUT when it gives up.
#pragma once

#include "pkv_attention_common.cuh"
#include "pkv_device.cuh"

namespace pkv {

constexpr int kPfBN = 64;       // key tokens per tile
constexpr int kPfStages = 3;

struct PfParams {
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  const __nv_bfloat16* q;         // [T, H_q, D]
  __nv_bfloat16* out;             // [T, H_q, D]
  const int32_t* block_tables;    // [S, max_blocks_per_seq]
  const int32_t* cu_seqlens;      // [S + 1]
  const int32_t* context_lens;    // [S]
  long long num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_tokens;
  int max_len;
  int H_q;
  int G;
  int block_size;
  float scale_log2;               // scale * log2(e)
  // key-range split (mma.sync kernel): num_splits CTAs per row tile, CTA sp
  // taking key tiles [sp * split_tiles, (sp + 1) * split_tiles); with
  // num_splits > 1 every CTA writes an (m, l, o) partial per row into ws
  // (rows indexed by packed token, like sequences in the decode workspace)
  // and the split-K reduce merges them
  int num_splits;
  int split_tiles;
  Workspace ws;
};

template <int D, int NW>
struct PfCfg {
  static constexpr int BM = 16 * NW;                  // query rows per CTA
  static constexpr int NH = D / 64;                   // 64-column halves of a row
  static constexpr int HALF = kPfBN * 128;            // one half of a tile: 64 rows x 128 B
  static constexpr int KBYTES = NH * HALF;
  static constexpr int STAGE = 2 * KBYTES;            // K tile, then V tile
  static constexpr int NBOX = 2 * NH * (kPfBN / 16);  // 16-row boxes per stage
  static constexpr int BAR_OFF = kPfStages * STAGE;
  static constexpr int SMEM = BAR_OFF + 2 * kPfStages * 8 + 1024;   // + alignment slack
  static constexpr int THREADS = 32 * (NW + 1);
};

// Byte address of the 16-byte chunk `chunk` of tile row `row` in a swizzled
// half-tile starting at `base` (128-byte lines, chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t pf_addr(uint32_t base, int row, int chunk) {
  return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <int D, int NW>
__global__ void __launch_bounds__(PfCfg<D, NW>::THREADS)
attn_prefill_kernel(const __grid_constant__ PfParams p) {
  using C = PfCfg<D, NW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t bar_full = smem_u32(smem + C::BAR_OFF);   // + 8 * stage
  const uint32_t bar_empty = bar_full + 8 * kPfStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, j = blockIdx.y;
  const int nsp = p.num_splits;
  const int tix = blockIdx.x / nsp, sp = blockIdx.x - tix * nsp;
  const int tile = gridDim.x / nsp - 1 - tix;              // heaviest tiles first

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, NW);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait_primary();
  pdl_launch_dependents();

  const int K = p.block_size;
  const int G = p.G;
  const int q0 = p.cu_seqlens[s], q1 = p.cu_seqlens[s + 1];
  const int L = effective_len(p.context_lens[s], p.max_len, p.max_blocks_per_seq * K);
  const int n = q1 - q0;
  if (q0 < 0 || n < 0 || q1 > p.num_tokens || n > L) {
    if (threadIdx.x == 0 && tile == 0) record_error(PKV_DEVERR_CONTEXT_LEN);
    return;
  }
  const int R = n * G;
  const int r0 = tile * C::BM;
  if (r0 >= R) return;
  const int i_last = min(R - 1, r0 + C::BM - 1) / G;
  const int pmax = L - n + i_last;              // last key any row of the tile sees
  const int nkt = pmax / kPfBN + 1;
  // this CTA's key tiles
  const int kt0 = nsp > 1 ? min(nkt, sp * p.split_tiles) : 0;
  const int kt1 = nsp > 1 ? min(nkt, kt0 + p.split_tiles) : nkt;

  if (warp == NW) {
    // =================== producer ===================
    if (lane == 0) {
      prefetch_tensormap(&p.tmap_k);
      prefetch_tensormap(&p.tmap_v);
    }
    // K/V tiles are read again by the sequence's other query tiles: keep
    // them in L2 at normal priority
    const uint64_t policy = l2_policy_evict_normal();
    const int sbl = K < 16 ? 1 : 0;           // 8-token blocks: two 8-row boxes per 16 rows
    const int ncopy = C::NBOX << sbl;
    int k = 0;                                 // ring position: kt - kt0
    bool ok = true;
    for (int kt = kt0; kt < kt1; ++kt, ++k) {
      const int stage = k % kPfStages;
      const uint32_t parity = ((k / kPfStages) & 1) ^ 1;
      if (!mbar_wait_bounded(bar_empty + 8 * stage, parity)) {
        record_error(PKV_DEVERR_TIMEOUT);
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * stage, C::STAGE);
      __syncwarp();
      uint8_t* sb = smem + stage * C::STAGE;
      for (int i = lane; i < ncopy; i += 32) {
        const int bi = i >> sbl, u = i & sbl;
        const int kv = bi / (C::NH * 4);
        const int rem = bi - kv * (C::NH * 4);
        const int half = rem >> 2, rb = rem & 3;
        const int tr = rb * 16 + (u << 3);                 // first tile row of the box
        const int tok = kt * kPfBN + tr;
        int row = -32;                                     // wholly out of bounds: zeros
        if (tok <= pmax) {
          const int lb = tok / K;
          const long long phys = p.block_tables[(int64_t)s * p.max_blocks_per_seq + lb];
          if (phys < 0 || phys >= p.num_blocks) {
            record_error(PKV_DEVERR_BLOCK_ID);
          } else {
            row = (int)(phys * K + (tok - lb * K));
          }
        }
        tma_load_3d(smem_u32(sb + kv * C::KBYTES + half * C::HALF + tr * 128),
                    kv ? &p.tmap_v : &p.tmap_k, bar_full + 8 * stage, half * 64, j, row, policy);
      }
      __syncwarp();
    }
    if (!ok) {
      // do not leave the CTA while our own copies may still land in smem
      for (int kk = max(0, k - kPfStages); kk < k; ++kk)
        mbar_wait_bounded(bar_full + 8 * (kk % kPfStages), (kk / kPfStages) & 1);
    }
    return;
  }

  // =================== consumers ===================
  const int g = lane >> 2, t4 = lane & 3;
  const int ra = r0 + warp * 16 + g, rb = ra + 8;
  const bool va = ra < R, vb = rb < R;
  const int ia = va ? ra / G : 0, ib = vb ? rb / G : 0;
  const int ha = j * G + (va ? ra - ia * G : 0), hb = j * G + (vb ? rb - ib * G : 0);
  const int pa = va ? L - n + ia : -1, pb = vb ? L - n + ib : -1;
  int pw = max(pa, pb);                         // last key any row of this warp sees
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pw = max(pw, __shfl_xor_sync(0xffffffffu, pw, o));

  // Q rows as A fragments
  uint32_t qf[D / 16][4];
  {
    const uint32_t* qa = reinterpret_cast<const uint32_t*>(
        p.q + ((int64_t)(q0 + ia) * p.H_q + ha) * D);
    const uint32_t* qb = reinterpret_cast<const uint32_t*>(
        p.q + ((int64_t)(q0 + ib) * p.H_q + hb) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[kk][0] = va ? __ldg(qa + kk * 8 + t4) : 0u;
      qf[kk][1] = vb ? __ldg(qb + kk * 8 + t4) : 0u;
      qf[kk][2] = va ? __ldg(qa + kk * 8 + 4 + t4) : 0u;
      qf[kk][3] = vb ? __ldg(qb + kk * 8 + 4 + t4) : 0u;
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
  const float sl = p.scale_log2;
  const int mi = lane >> 3, rr = lane & 7;     // ldmatrix: matrix and row of this lane

  for (int kt = kt0; kt < kt1; ++kt) {
    const int stage = (kt - kt0) % kPfStages;
    if (!mbar_wait_bounded(bar_full + 8 * stage, ((kt - kt0) / kPfStages) & 1)) {
      record_error(PKV_DEVERR_TIMEOUT);
      return;
    }
    const int kbase = kt * kPfBN;
    const uint32_t kb = smem_u32(smem + stage * C::STAGE);
    const uint32_t vbase = kb + C::KBYTES;
    if (kbase <= pw) {
      if (kt == nkt - 1 && L - kbase < kPfBN) {
        // V rows at or past the context end inside fetched boxes may hold
        // anything (NaN included); zero them so that a 0 weight stays 0.
        // Every consumer warp writes the same zeros before its own reads.
        const int z0 = L - kbase, z1 = min(kPfBN, ((pmax - kbase) / 16 + 1) * 16);
        uint8_t* vs = smem + stage * C::STAGE + C::KBYTES;
        for (int x = z0 * 8 + lane; x < z1 * 8; x += 32) {     // 16-byte chunks per row: 8
#pragma unroll
          for (int h = 0; h < C::NH; ++h)
            *reinterpret_cast<uint4*>(vs + h * C::HALF + x * 16) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // ---- S = Q K^T (16 rows x 64 keys)
      float sc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t hb_ = kb + (kk >> 2) * C::HALF;
        const int ch = (kk & 3) * 2 + (mi & 1);
#pragma unroll
        for (int n16 = 0; n16 < 4; ++n16) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(pf_addr(hb_, n16 * 16 + ((mi >> 1) << 3) + rr, ch), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * n16], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
          mma_bf16_16816(sc[2 * n16 + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
      }
      // ---- causal mask, online softmax (base 2)
      float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int key = kbase + nt * 8 + 2 * t4;
        sc[nt][0] = key <= pa ? sc[nt][0] * sl : -INFINITY;
        sc[nt][1] = key + 1 <= pa ? sc[nt][1] * sl : -INFINITY;
        sc[nt][2] = key <= pb ? sc[nt][2] * sl : -INFINITY;
        sc[nt][3] = key + 1 <= pb ? sc[nt][3] * sl : -INFINITY;
        xa = fmaxf(xa, fmaxf(sc[nt][0], sc[nt][1]));
        xb = fmaxf(xb, fmaxf(sc[nt][2], sc[nt][3]));
      }
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
      xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
      xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
      const float na = fmaxf(ma, xa), nb = fmaxf(mb, xb);
      const float ua = na == -INFINITY ? 0.f : na, ub = nb == -INFINITY ? 0.f : nb;
      const float aa = exp2f(ma - ua), ab = exp2f(mb - ub);
      ma = na;
      mb = nb;
      float sa = 0.f, sbs = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - ua);
        sc[nt][1] = exp2f(sc[nt][1] - ua);
        sc[nt][2] = exp2f(sc[nt][2] - ub);
        sc[nt][3] = exp2f(sc[nt][3] - ub);
        sa += sc[nt][0] + sc[nt][1];
        sbs += sc[nt][2] + sc[nt][3];
      }
      la = la * aa + sa;
      lb = lb * ab + sbs;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        o[dt][0] *= aa;
        o[dt][1] *= aa;
        o[dt][2] *= ab;
        o[dt][3] *= ab;
      }
      // ---- O += P V, P as hi + lo bf16
#pragma unroll
      for (int k16 = 0; k16 < 4; ++k16) {
        uint32_t ph[4], pl[4];
        split_bf16x2(sc[2 * k16][0], sc[2 * k16][1], ph[0], pl[0]);
        split_bf16x2(sc[2 * k16][2], sc[2 * k16][3], ph[1], pl[1]);
        split_bf16x2(sc[2 * k16 + 1][0], sc[2 * k16 + 1][1], ph[2], pl[2]);
        split_bf16x2(sc[2 * k16 + 1][2], sc[2 * k16 + 1][3], ph[3], pl[3]);
        const int key = k16 * 16 + ((mi & 1) << 3) + rr;
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t v0, v1, v2, v3;
          ldmatrix_x4_trans(pf_addr(vbase + (dp >> 2) * C::HALF, key, (dp & 3) * 2 + (mi >> 1)),
                            v0, v1, v2, v3);
          mma_bf16_16816(o[2 * dp], ph[0], ph[1], ph[2], ph[3], v0, v1);
          mma_bf16_16816(o[2 * dp], pl[0], pl[1], pl[2], pl[3], v0, v1);
          mma_bf16_16816(o[2 * dp + 1], ph[0], ph[1], ph[2], ph[3], v2, v3);
          mma_bf16_16816(o[2 * dp + 1], pl[0], pl[1], pl[2], pl[3], v2, v3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
  }

  // ---- normalise and store
  la += __shfl_xor_sync(0xffffffffu, la, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  lb += __shfl_xor_sync(0xffffffffu, lb, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  if (nsp > 1) {
    // partial state of this key range: unnormalised o, running max m (base
    // 2), row sum l; an empty range leaves (-inf, 0, 0), which merges as 0
    if (sp == 0 && t4 == 0) {
      if (va) p.ws.meta[q0 + ia] = make_int4((q0 + ia) * p.ws.pmax, nsp, 0, 0);
      if (vb) p.ws.meta[q0 + ib] = make_int4((q0 + ib) * p.ws.pmax, nsp, 0, 0);
    }
    if (va) {
      const int64_t base = ((int64_t)(q0 + ia) * p.ws.pmax + sp) * p.H_q + ha;
      float2* ob = reinterpret_cast<float2*>(p.ws.o + base * D);
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) ob[dt * 4 + t4] = make_float2(o[dt][0], o[dt][1]);
      if (t4 == 0) p.ws.ml[base] = make_float2(ma, la);
    }
    if (vb) {
      const int64_t base = ((int64_t)(q0 + ib) * p.ws.pmax + sp) * p.H_q + hb;
      float2* ob = reinterpret_cast<float2*>(p.ws.o + base * D);
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) ob[dt * 4 + t4] = make_float2(o[dt][2], o[dt][3]);
      if (t4 == 0) p.ws.ml[base] = make_float2(mb, lb);
    }
    return;
  }
  if (va) {
    const float inv = 1.f / la;
    uint32_t* orow = reinterpret_cast<uint32_t*>(p.out + ((int64_t)(q0 + ia) * p.H_q + ha) * D);
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) orow[dt * 4 + t4] = pack_bf16x2(o[dt][0] * inv, o[dt][1] * inv);
  }
  if (vb) {
    const float inv = 1.f / lb;
    uint32_t* orow = reinterpret_cast<uint32_t*>(p.out + ((int64_t)(q0 + ib) * p.H_q + hb) * D);
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) orow[dt * 4 + t4] = pack_bf16x2(o[dt][2] * inv, o[dt][3] * inv);
  }
}

}  // namespace pkv
