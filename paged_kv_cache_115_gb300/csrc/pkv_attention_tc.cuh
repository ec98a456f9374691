// TMA + tensor-core decode-attention partition kernel (bf16 queries; bf16,
// FP8 e4m3 or INT8 pools).
#pragma once

#include "pkv_attention_common.cuh"

namespace pkv {

// ===========================================================================
// TMA + tensor-core partition kernel (bf16 queries, block_size % 16 == 0,
// G <= 8; bf16 pools with D in {64, 128}, one-byte pools with D = 128).
//
// Work decomposition: the token range of the batch is cut into chunks (16
// tokens for bf16 pools, 32 for one-byte pools), numbered sequence-major;
// with T chunks and n CTAs per KV-head group, CTA i owns chunks
// [floor(i T / n), floor((i+1) T / n)) — equal work per CTA whatever the
// length mix.  A run of chunks of one sequence inside a CTA is a split-K
// partition; its (m, l, o) goes to the workspace unless the CTA holds the
// whole sequence, in which case it writes the final output.
//
// Roles: warp HPC is the producer; its lanes issue the TMA loads of a stage
// (one chunk x HPC heads, K and V: one box of 16 token rows x 128 bytes per
// head, 16-row tile and 128-byte column group) completing on the stage's
// "full" mbarrier.  Warps 0..HPC-1 are consumers, warp w owning KV head
// (group * HPC + w): it waits on "full", computes S^T = K_tile Q^T and
// O^T += V^T P^T with mma.m16n8k16 for each 16-row tile (tokens x heads, the
// q-group padded to 8 columns; P as a hi + lo pair), does the online softmax
// over the chunk with warp shuffles, and arrives on the stage's "empty"
// mbarrier.  A 32-token chunk gives each consumer two independent tile
// products per softmax step, halving the per-token cost of the softmax,
// rescaling and barrier handshakes that bound the one-byte pools.
//
// Shared-memory tiles use the 128-byte swizzle, so the 8 rows a warp phase
// reads (8 tokens, same 16-byte column) land in 8 distinct bank groups.
// ===========================================================================
constexpr int kTile = 16;          // token rows per TMA box and per mma tile
constexpr int kTcChunk = kTile;    // chunk of the bf16 kernel
constexpr int kTcMaxSeqs = 2048;
// shared-prefix mode: sequences per launch, so that the units (at most
// 3/2 of them with groups of two or more) fit the kTcMaxSeqs + 1 chunk starts
constexpr int kTcMaxShareSeqs = 1024;
constexpr int kBoxBytes = kTile * 128;

// tokens per stream-K chunk for a pool format (0 bf16, 1 FP8, 2 INT8,
// 3 bf16 K with FP8 V)
constexpr int tc_chunk_tokens(int ct) { return ct == 1 || ct == 2 ? 2 * kTile : kTile; }

struct TcParams {
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  Workspace ws;
  long long num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int max_len;
  int H_q;
  int G;
  int block_size;
  float scale_log2;   // scale * log2(e) (FP8 pools: times the K scale)
  // one-byte pools only
  float v_scale;            // FP8: scale of the V pool
  const float* k_ts;        // INT8: per-slot scales
  const float* v_ts;
  // several query tokens per sequence (bf16 pools): sequence s owns query
  // rows cu_seqlens[s] .. cu_seqlens[s+1]-1; its new token i of n sits at
  // position len - n + i and is score column i * G + (head in group), so
  // n * G <= 8.  Outputs and partials are indexed by query row.  nullptr:
  // one query per sequence, row s (decode).
  const int32_t* cu_seqlens;
  // shared-prefix groups (bf16 decode, kernel instantiated with SH): share_m
  // consecutive sequences form a group; glen[g] = tokens at the start of
  // every member's context that sit in the same physical blocks (a multiple
  // of 16, written by share_prefix_kernel).  share_m = 1 otherwise.
  int share_m;
  const int* glen;
  // decode: slot distance between the member regions of a shared unit (CTAs
  // + units of the launch; 0 without shared-prefix groups)
  int slot_stride;
};

// Pool formats of the kernel: CT 0 = bf16, 1 = FP8 e4m3 (per-tensor scale),
// 2 = INT8 (per-slot scale), 3 = bf16 K pool with an FP8 e4m3 V pool
// (per-tensor V scale).  A head's row is one 128-byte column group in a
// one-byte pool of D = 128, D / 64 groups in a bf16 pool.  One-byte tiles are read straight
// into f16 mma fragments (e4m3 and int8 codes are exact in f16); bf16 tiles
// go through ldmatrix into bf16 mma fragments.
//
// Stage layout: K boxes [tile][head][column group], then V boxes, then (INT8)
// the 16 per-slot scales of each tile: K tiles, then V tiles.  A box holds
// 16 token rows of 128 bytes in the 128-byte swizzle (row r's 16-byte chunk
// c at chunk c ^ (r & 7)).  A row of a pool block holds every KV head
// contiguously, so one 4-D TMA copy (column, row, column group, head) brings
// a tile's rows for all HPC heads and column groups of the CTA at once.
//
// 8-token blocks (B8): a tile spans two blocks, one copy each, laid out
// [tile][block half][head][column group][8 rows x 128 bytes]: rows 8..15 of
// a tile sit UST bytes after rows 0..7 instead of 1024.  Each 8-row group is
// still a whole 1024-byte swizzle atom, so row r keeps the swizzle phase r & 7.

// Two int8 codes of a word whose bytes were already XORed with 0x80, chosen
// by a byte-permute selector that puts them in the low bytes of two f16
// halves with exponent bits 0x64 (selector nibbles: code byte, 4 = 0x64,
// code byte, 5 = 0x64): each half is 1024 + (code + 128), and subtracting
// 1152 leaves the code exactly.
__device__ __forceinline__ uint32_t s8_pair_to_f16x2(uint32_t xored, uint32_t sel) {
  const uint32_t biased = __byte_perm(xored, 0x6464u, sel);
  __half2 h = *reinterpret_cast<const __half2*>(&biased);
  h = __hsub2(h, __floats2half2_rn(1152.f, 1152.f));
  return *reinterpret_cast<uint32_t*>(&h);
}

// Four e4m3 codes of a word -> two f16 pairs (codes 0, 1 and codes 2, 3),
// the word's 16-bit halves handed to the conversion directly.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(w));
}

// One-byte pools: slack of the lazily raised exponent base.  Weights stay
// below 2^4, so an INT8 weight times its token's V scale stays inside f16
// while that scale is below 2^11 (|v| below ~260,000); the FP8 V scale
// multiplies o once per partition instead.
constexpr float kQuantSlack = 4.f;

__device__ __forceinline__ float ex2_approx_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 4-D tiled load global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

template <int D, int HPC, int NS, int CT = 0, bool B8 = false>
struct TcCfg {
  static constexpr bool KB = CT == 0 || CT == 3;          // K tiles in bf16
  static constexpr bool VB = CT == 0;                     // V tiles in bf16
  static constexpr int TL = CT == 1 || CT == 2 ? 2 : 1;   // 16-row tiles per chunk
  static constexpr int CH = kTile * TL;                   // tokens per chunk
  static constexpr int NHK = KB ? D / 64 : 1;             // boxes per head row, K
  static constexpr int NHV = VB ? D / 64 : 1;             // boxes per head row, V
  static constexpr int NH = NHV;                          // (V tile rows, zeroed past the end)
  static constexpr int KPART = HPC * TL * NHK * kBoxBytes;
  static constexpr int VPART = HPC * TL * NHV * kBoxBytes;
  static constexpr int SCALE_OFF = KPART + VPART;
  static constexpr int SCALE_BYTES = CT == 2 ? 2 * TL * kTile * 4 : 0;
  static constexpr int STAGE = ((KPART + VPART + SCALE_BYTES + 1023) / 1024) * 1024;
  static constexpr int THREADS = (HPC + 1) * 32;
  static constexpr int BAR_OFF = NS * STAGE;
  static constexpr int CSTART_OFF = BAR_OFF + 2 * NS * 8 + 16;
  static constexpr int SMEM = CSTART_OFF + (kTcMaxSeqs + 1) * 4 + 1024;  // + alignment slack
  static constexpr uint32_t TX = KPART + VPART + SCALE_BYTES;  // bytes landing per stage
  static_assert(CT == 0 || D == 128, "one-byte pools need head_dim 128");
  static_assert(CT != 3 || !B8, "the bf16-K / FP8-V pair needs 16-token tiles of one block");
  static_assert(tc_chunk_tokens(CT) == CH, "chunk size");
  static constexpr int TBOXK = HPC * NHK * kBoxBytes;  // one tile, all heads of the CTA
  static constexpr int TBOXV = HPC * NHV * kBoxBytes;
  static constexpr int TBOX = TBOXK;                   // (formats with equal K and V tiles)
  static constexpr int UST = HPC * NHK * 1024;         // B8: one block half of a tile, all heads
  static constexpr int RSTEP8 = B8 ? UST : 1024;       // rows 8..15 relative to rows 0..7
  static constexpr int HSTR = B8 ? 1024 : kBoxBytes;   // column group stride
  // smem offset of row 0 of head h's box (tile t, column group half) of K
  // (kv 0) or V; the B8 layout exists for formats whose K and V tiles match
  __host__ __device__ static constexpr int box_off(int kv, int h, int t, int half) {
    return B8 ? kv * KPART + t * 2 * UST + (h * NHK + half) * 1024
              : (kv ? KPART + t * TBOXV + (h * NHV + half) * kBoxBytes
                    : t * TBOXK + (h * NHK + half) * kBoxBytes);
  }
  // offset of row r (0..15) inside a box
  __host__ __device__ static constexpr int row_off(int r) { return (r & 7) * 128 + (r >> 3) * RSTEP8; }
};

// Largest CTA index i whose range starts at or before chunk c.
__host__ __device__ __forceinline__ int cta_of_chunk(long long c, long long T, int n) {
  return (int)(((c + 1) * (long long)n - 1) / T);
}

// Largest s in [0, S) with cstart[s] <= c (c < cstart[S]).
__host__ __device__ __forceinline__ int seq_of_chunk(const int* cstart, int S, int c) {
  int lo = 0, hi = S;   // invariant: cstart[lo] <= c < cstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cstart[mid] <= c) lo = mid; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// Units of a launch: the stream-K chunks run over units, not sequences.
// Plain mode (m = 1): unit u is sequence u.  Shared-prefix mode (m >= 2):
// sequences are taken in aligned groups of m consecutive ones; group g owns
// units g (m + 1) .. g (m + 1) + m: first its shared unit (the first glen[g]
// tokens, which sit in the same physical blocks in every member's table, so
// that one staged tile serves the query columns of all members at once),
// then one private unit per member s (tokens glen[g] .. L_s).  A unit without
// tokens (or past the last sequence) has no chunks.  A sequence's partial
// states are those of its group's shared unit, then those of its private
// unit, one per CTA that holds chunks of the unit.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int tc_num_units(int S, int m) {
  return m == 1 ? S : ((S + m - 1) / m) * (m + 1);
}
__host__ __device__ __forceinline__ int tc_shared_unit(int s, int m) { return (s / m) * (m + 1); }
__host__ __device__ __forceinline__ int tc_private_unit(int s, int m) {
  return m == 1 ? s : (s / m) * (m + 1) + s % m + 1;
}
// CTAs holding chunks of unit u (0 for a unit without chunks)
__host__ __device__ __forceinline__ int tc_unit_parts(const int* cstart, int u, long long T,
                                                      int n) {
  const int a = cstart[u], b = cstart[u + 1];
  return a < b ? cta_of_chunk(b - 1, T, n) - cta_of_chunk(a, T, n) + 1 : 0;
}
// Partial slots of sequence s in decode (CTA i's partition over unit u
// writes member r's partials to slot r * stride + i + u, r being s's index
// among the unit's sequences: 0 but in a shared unit): (base, count) of its
// private unit, then of its group's shared unit (count 0 in plain mode).
__host__ __device__ __forceinline__ int4 tc_seq_meta(const int* cstart, int s, int m,
                                                     long long T, int n, int stride) {
  const int up = tc_private_unit(s, m);
  const int np = tc_unit_parts(cstart, up, T, n);
  int4 r = make_int4(np ? cta_of_chunk(cstart[up], T, n) + up : 0, np, 0, 0);
  if (m > 1) {
    const int us = tc_shared_unit(s, m);
    const int ns = tc_unit_parts(cstart, us, T, n);
    r.z = ns ? (s % m) * stride + cta_of_chunk(cstart[us], T, n) + us : 0;
    r.w = ns;
  }
  return r;
}

template <int D, int HPC, int NS, int CT = 0, bool B8 = false, bool SH = false>
__global__ void __launch_bounds__(TcCfg<D, HPC, NS, CT, B8>::THREADS, 1)
attn_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<D, HPC, NS, CT, B8>;
  constexpr int TL = C::TL, CH = C::CH;
  // 8-column blocks of the score tile: two in shared-prefix mode (the query
  // heads of a group's members side by side), one otherwise
  constexpr int NB = SH ? 2 : 1;
  static_assert(!SH || CT == 0, "shared-prefix groups need bf16 pools");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t bar_full = smem_u32(smem + C::BAR_OFF);   // + 8 * stage
  const uint32_t bar_empty = bar_full + 8 * NS;
  int* cstart = reinterpret_cast<int*>(smem + C::CSTART_OFF);
  __shared__ int s_wsum[32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.num_seqs;
  const int K = p.block_size;
  const int row_tokens = p.max_blocks_per_seq * K;
  const int M = SH ? p.share_m : 1;
  // several query tokens per sequence (never with shared-prefix groups)
  const int32_t* const cu = SH ? nullptr : p.cu_seqlens;
  const int NU = SH ? tc_num_units(S, M) : S;
  auto seq_len = [&](int s) -> int {
    return effective_len(p.context_lens[s], p.max_len, row_tokens);
  };
  // unit u: first sequence s0 (its table row and first query row), sequences
  // it serves (0: none), tokens [t0, end) of the sequence
  auto unit = [&](int u, int& s0, int& rows, int& t0, int& end) {
    if constexpr (!SH) {
      s0 = u;
      rows = 1;
      t0 = 0;
      end = seq_len(u);
    } else {
      const int g = u / (M + 1), k = u - g * (M + 1);
      const int lg = p.glen[g];
      if (k == 0) {
        s0 = g * M;
        rows = min(M, S - s0);
        t0 = 0;
        end = lg;
      } else {
        s0 = g * M + k - 1;
        rows = s0 < S ? 1 : 0;
        t0 = lg;
        end = rows ? max(seq_len(s0), lg) : lg;
      }
    }
  };
  // chunks of unit u (none for a sequence without query rows)
  auto nchunks = [&](int u) -> int {
    int s0, rows, t0, end;
    unit(u, s0, rows, t0, end);
    if (rows == 0) return 0;
    if (cu != nullptr) {
      const int nq = cu[s0 + 1] - cu[s0];
      if (nq < 0 || nq > end) {
        record_error(PKV_DEVERR_CONTEXT_LEN);
        return 0;
      }
      if (nq == 0) return 0;
    }
    return (end - t0 + CH - 1) / CH;
  };

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, HPC);
    }
    fence_barrier_init();
  }
  // The prefix sums read only the lengths (and, with several query tokens,
  // cu_seqlens), which no kernel of this library writes, so they overlap the
  // previous kernel's tail; shared-prefix groups also need the group lengths
  // the previous kernel (share_prefix_kernel) writes.
  if constexpr (SH) pdl_wait_primary();

  // ---- chunk prefix sums over the units: cstart[u] = sum_{u'<u} chunks(u')
  {
    const int per = (NU + C::THREADS - 1) / C::THREADS;
    const int a = min(NU, tid * per), b = min(NU, a + per);
    int local = 0;
    for (int u = a; u < b; ++u) local += nchunks(u);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (C::THREADS / 32) ? s_wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += v;
      }
      s_wsum[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    int run = (warp ? s_wsum[warp - 1] : 0) + incl - local;
    for (int u = a; u < b; ++u) {
      cstart[u] = run;
      run += nchunks(u);
    }
    if (tid == C::THREADS - 1) cstart[NU] = run;
    __syncthreads();
  }
  pdl_launch_dependents();

  const long long T = cstart[NU];
  // Split over at most T CTAs so that every working CTA owns >= 1 chunk and a
  // unit's partial index (CTA - first CTA of the unit) stays below min(n,
  // chunks of the unit).  CTAs past n only do bookkeeping.
  const int n = (int)(T < (long long)gridDim.x ? (T > 0 ? T : 1) : (long long)gridDim.x);
  const int cta = blockIdx.x, group = blockIdx.y;
  const int head0 = group * HPC;
  const int G = p.G, H_q = p.H_q;
  const int cb = cta < n ? (int)((long long)cta * T / n) : 0;
  const int ce = cta < n ? (int)((long long)(cta + 1) * T / n) : 0;

  // pool rows of the tiles of 32 chunks from c0, one chunk per lane; a tile
  // past the unit's end (or of an out-of-range block) gets a row that is
  // wholly out of bounds, which TMA fills with zeros.  With 8-token blocks a
  // tile spans two blocks (uu = 0, 1).
  constexpr int sbl = B8 ? 1 : 0;          // log2 of the blocks per tile
  auto tile_rows = [&](int c0, int (&row)[TL][2]) {
#pragma unroll
    for (int t = 0; t < TL; ++t) row[t][0] = row[t][1] = -2 * kTile;
    const int c = c0 + lane;
    if (c < ce) {
      const int u = seq_of_chunk(cstart, NU, c);
      int s0, rows, t0, end;
      unit(u, s0, rows, t0, end);
      const int L = (TL > 1 || sbl || SH) ? end : 1 << 30;
#pragma unroll
      for (int t = 0; t < TL; ++t) {
#pragma unroll
        for (int uu = 0; uu < 2; ++uu) {
          const int tok = t0 + (c - cstart[u]) * CH + t * kTile + uu * K;
          if (uu <= sbl && tok < L) {
            const int lb = tok / K;
            const long long phys = p.block_tables[(int64_t)s0 * p.max_blocks_per_seq + lb];
            if (phys < 0 || phys >= p.num_blocks) {
              record_error(PKV_DEVERR_BLOCK_ID);
            } else {
              row[t][uu] = (int)(phys * K + (tok - lb * K));
            }
          }
        }
      }
    }
  };
  // the producer reads its first table entries (no kernel of this library
  // writes the tables) before waiting for the previous kernel
  int row[TL][2];
  if (warp == HPC && cb < ce) tile_rows(cb, row);
  if constexpr (!SH) pdl_wait_primary();

  // ---- bookkeeping (sequence s by CTA s mod grid): partial slots of each
  // output row, and zero outputs of empty sequences
  for (int s = cta + tid * (int)gridDim.x; s < S; s += C::THREADS * (int)gridDim.x) {
    const int4 mt = tc_seq_meta(cstart, s, M, T, n, p.slot_stride);
    if (mt.y + mt.w == 0) {
      // empty context: zero output (decode); a sequence without query rows
      // has no output
      if (cu == nullptr) {
        if (group == 0) p.ws.meta[s] = mt;
        __nv_bfloat16* o = p.out + ((int64_t)s * H_q + head0 * G) * D;
        for (int i = 0; i < HPC * G * D; ++i) o[i] = __float2bfloat16_rn(0.f);
      }
    } else if (group == 0) {
      if (cu == nullptr) {
        p.ws.meta[s] = mt;
      } else {
        // several query rows: row r's partial p in slot r * pmax + p
        for (int r = cu[s]; r < cu[s + 1]; ++r) p.ws.meta[r] = make_int4(r * p.ws.pmax, mt.y, 0, 0);
      }
    }
  }
  if (cb >= ce) return;

  if (warp == HPC) {
    // =================== producer ===================
    if (lane == 0) {
      prefetch_tensormap(&p.tmap_k);
      prefetch_tensormap(&p.tmap_v);
    }
    const uint64_t policy = l2_policy_evict_first();
    int k = 0;
    bool ok = true;
    for (int c0 = cb; c0 < ce && ok; c0 += 32) {
      if (c0 != cb) tile_rows(c0, row);
      const int cnt = min(32, ce - c0);
      for (int b = 0; b < cnt; ++b, ++k) {
        int r[TL][2];
#pragma unroll
        for (int t = 0; t < TL; ++t) {
          r[t][0] = __shfl_sync(0xffffffffu, row[t][0], b);
          r[t][1] = __shfl_sync(0xffffffffu, row[t][1], b);
        }
        const int stage = k % NS;
        const uint32_t parity = ((k / NS) & 1) ^ 1;
        if (!mbar_wait_bounded(bar_empty + 8 * stage, parity)) {
          record_error(PKV_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * stage, C::TX);
        __syncwarp();
        uint8_t* sb = smem + stage * C::STAGE;
        if constexpr (B8) {
          // one 4-D box per (K / V, tile, block half): all heads of the CTA,
          // all column groups, 8 rows; then (INT8) the scales of each half
          constexpr int NB = 4 * TL;
          for (int i = lane; i < NB + (CT == 2 ? NB : 0); i += 32) {
            const int j = i < NB ? i : i - NB;
            const int kv = j / (2 * TL), t = (j >> 1) % TL, u = j & 1;
            const int r0 = t ? r[TL - 1][0] : r[0][0];
            const int r1 = t ? r[TL - 1][1] : r[0][1];
            const int rr = u ? r1 : r0;
            if (i < NB) {
              tma_load_4d(smem_u32(sb + kv * C::KPART + (2 * t + u) * C::UST),
                          kv ? &p.tmap_v : &p.tmap_k, bar_full + 8 * stage, 0, rr, 0, head0,
                          policy);
            } else if constexpr (CT == 2) {
              // a half tile with no rows reads slot 0's scales, which meet zero codes
              const float* src = (kv ? p.v_ts : p.k_ts) + (rr >= 0 ? rr : 0);
              bulk_load(smem_u32(sb + C::SCALE_OFF + (kv * TL + t) * 64 + u * 32), src, 32,
                        bar_full + 8 * stage);
            }
          }
        } else {
          // one 4-D box per (K / V, tile): 16 rows of all heads of the CTA and
          // all column groups; then (INT8) each tile's 16 per-slot scales
          constexpr int NB = 2 * TL;
          for (int i = lane; i < NB + (CT == 2 ? NB : 0); i += 32) {
            const int j = i < NB ? i : i - NB;
            const int kv = j / TL, t = j - kv * TL;
            const int rr = t ? r[TL - 1][0] : r[0][0];
            if (i < NB) {
              tma_load_4d(smem_u32(sb + C::box_off(kv, 0, t, 0)), kv ? &p.tmap_v : &p.tmap_k,
                          bar_full + 8 * stage, 0, rr, 0, head0, policy);
            } else if constexpr (CT == 2) {
              // a tile with no rows reads slot 0's scales, which meet zero codes
              const float* src = (kv ? p.v_ts : p.k_ts) + (rr >= 0 ? rr : 0);
              bulk_load(smem_u32(sb + C::SCALE_OFF + (kv * TL + t) * 64), src, 64,
                        bar_full + 8 * stage);
            }
          }
        }
        __syncwarp();
      }
    }
    if (!ok) {
      // do not leave the CTA while our own copies may still land in smem
      for (int kk = max(0, k - NS); kk < k; ++kk)
        mbar_wait_bounded(bar_full + 8 * (kk % NS), (kk / NS) & 1);
    }
    return;
  }

  // =================== consumers ===================
  const int w = warp;                 // KV head head0 + w
  const int j = head0 + w;
  const int g = lane >> 2, tq = lane & 3;
  const float sl = p.scale_log2;

  uint32_t qf[NB][D / 16][2];
  float o[NB][D / 16][4];
  float slc0 = sl, slc1 = sl;   // per score column (one-byte pools: q's 2^e folded in)
  float m0[NB], m1[NB], l0[NB], l1[NB];
  // INT8 pools: V enters the tensor core as 1152 + code (the exact f16 the
  // byte permute makes, without the subtraction); vw = sum of weight x V
  // scale per column, so that 1152 vw is taken off o at the partition end
  float vw0 = 0.f, vw1 = 0.f;
  int u = seq_of_chunk(cstart, NU, cb);
  int ut0 = 0, uend = 0, ulim = 0;   // the unit's tokens [ut0, uend); min column limit
  int qr0 = 0, nq = 0, ncol = 0;     // first query row, query rows, valid score columns
  int nbv = 1;                       // column blocks holding valid columns
  // score column c (query row qr0 + c / G, head j G + c % G; c >= ncol is
  // padding) sees keys up to its limit: len - n + i for new token i of n
  // (several query tokens per sequence), else the unit's last key
  auto col_lim = [&](int cc) -> int {
    return cc < ncol && cu ? uend - nq + cc / G : uend - 1;
  };
  int k = 0;
  for (int c = cb; c < ce; ++c, ++k) {
    while (c >= cstart[u + 1]) ++u;
    const int a = cstart[u], b = cstart[u + 1];
    if (c == cb || c == a) {
      // ---- new partition: load the q-group(s) as the B fragments of Q^T
      int s0, rows;
      unit(u, s0, rows, ut0, uend);
      qr0 = cu ? cu[s0] : s0;
      nq = cu ? cu[s0 + 1] - qr0 : rows;
      ncol = nq * G;
      nbv = ncol > 8 ? NB : 1;
      ulim = uend - 1;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        ulim = min(ulim, min(col_lim(8 * nb + 2 * tq), col_lim(8 * nb + 2 * tq + 1)));
      if constexpr (C::KB) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          // this lane's B-fragment column 8 nb + g
          const int cq = 8 * nb + g;
          const __nv_bfloat16* qrow =
              p.q + ((int64_t)(qr0 + (cq < ncol ? cq / G : 0)) * H_q + j * G + cq % G) * D;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            if (cq < ncol) {
              qf[nb][ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tq));
              qf[nb][ks][1] =
                  __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tq));
            } else {
              qf[nb][ks][0] = qf[nb][ks][1] = 0u;
            }
          }
        }
      } else {
        // f16 fragments.  The mma k order inside each 16-column step is
        // permuted (k 2tq, 2tq+1 -> d 4tq, 4tq+1; k 2tq+8, 2tq+9 -> d 4tq+2,
        // 4tq+3) to match the K fragments read straight from the byte tile.
        // Each head is scaled by a power of two 2^-e that puts its largest
        // |q| in [2^14, 2^15): exact, and far inside the f16 range; the
        // scores are multiplied back by 2^e.
        const __nv_bfloat16* qrow =
            p.q + ((int64_t)(qr0 + (g < ncol ? g / G : 0)) * H_q + j * G + g % G) * D;
        float qv[D / 16][4];
        float amax = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          if (g < G) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(qrow + ks * 16 + 4 * tq));
            const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
            const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
            qv[ks][0] = lo.x; qv[ks][1] = lo.y; qv[ks][2] = hi.x; qv[ks][3] = hi.y;
          } else {
            qv[ks][0] = qv[ks][1] = qv[ks][2] = qv[ks][3] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qv[ks][e]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));   // head g's max
        const int eg = amax > 0.f ? ilogbf(amax) - 14 : 0;
        const float down = ldexpf(1.f, -eg);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          qf[0][ks][0] = pack_f16x2(qv[ks][0] * down, qv[ks][1] * down);
          qf[0][ks][1] = pack_f16x2(qv[ks][2] * down, qv[ks][3] * down);
        }
        // score columns of this thread are heads 2tq, 2tq+1 (held by lanes 8tq, 8tq+4)
        const int e0 = __shfl_sync(0xffffffffu, eg, 8 * tq);
        const int e1 = __shfl_sync(0xffffffffu, eg, 8 * tq + 4);
        slc0 = ldexpf(sl, e0);
        slc1 = ldexpf(sl, e1);
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
          o[nb][mt][0] = o[nb][mt][1] = o[nb][mt][2] = o[nb][mt][3] = 0.f;
        m0[nb] = m1[nb] = -INFINITY;
        l0[nb] = l1[nb] = 0.f;
      }
      vw0 = vw1 = 0.f;
    }
    const int cpos = ut0 + (c - a) * CH;                 // key position of chunk row 0
    const int valid = min(CH, uend - cpos);             // tokens of this chunk
    const int stage = k % NS;
    if (!mbar_wait_bounded(bar_full + 8 * stage, (k / NS) & 1)) {
      record_error(PKV_DEVERR_TIMEOUT);
      return;
    }
    uint8_t* sb = smem + stage * C::STAGE;
    // per-token-row K scales and V scales (folded into P) of rows g, g+8 of
    // each tile: INT8 per slot, FP8 per tensor (K's folded into sl)
    float ksr[TL][2], vsr[TL][2];
#pragma unroll
    for (int t = 0; t < TL; ++t) {
      if constexpr (CT == 2) {
        const float* kscl = reinterpret_cast<const float*>(sb + C::SCALE_OFF + t * 64);
        const float* vscl = reinterpret_cast<const float*>(sb + C::SCALE_OFF + (TL + t) * 64);
        // slots past the sequence end may hold anything; their weight is 0
        const float k0 = kscl[g], k8 = kscl[g + 8], v0 = vscl[g], v8 = vscl[g + 8];
        ksr[t][0] = isfinite(k0) ? k0 : 0.f;
        ksr[t][1] = isfinite(k8) ? k8 : 0.f;
        vsr[t][0] = isfinite(v0) ? v0 : 0.f;
        vsr[t][1] = isfinite(v8) ? v8 : 0.f;
      } else {
        ksr[t][0] = ksr[t][1] = 1.f;
        vsr[t][0] = vsr[t][1] = 1.f;      // FP8: the V scale multiplies o at the end
      }
    }
    if (valid < CH) {
      // rows past the sequence end may hold anything (stale slots, NaN
      // codes): give them zero V so that 0-weight x V stays 0 in the tensor core
      const int nvec = (CH - valid) * C::NH * 8;
      for (int i = lane; i < nvec; i += 32) {
        const int r = valid + i / (C::NH * 8);          // chunk row: tile r / 16
        const int rem = i % (C::NH * 8);
        const int half = rem >> 3, ch = rem & 7;
        *reinterpret_cast<uint4*>(sb + C::box_off(1, w, r / kTile, half) + C::row_off(r % kTile) +
                                  ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    // ---- S^T[16 tok x 8 columns] = K_tile[16 x D] . Q^T[D x 8], per tile and
    // column block (one K fragment feeds every column block)
    float sacc[NB][TL][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int t = 0; t < TL; ++t) sacc[nb][t][0] = sacc[nb][t][1] = sacc[nb][t][2] = sacc[nb][t][3] = 0.f;
    if constexpr (C::KB) {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int chs = lane >> 4;
      const uint8_t* kt = sb + C::box_off(0, w, 0, 0);
      // one column block: odd k steps accumulate apart and are added at the
      // end, two independent mma chains instead of one (two column blocks
      // are two chains already)
      float sodd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int half = ks >> 2;
        const int ch = ((ks & 3) << 1) + chs;
        const uint32_t addr = smem_u32(kt + half * C::HSTR) + C::row_off(r) + ((ch ^ (r & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(addr, a0, a1, a2, a3);
        if (NB == 1 && (ks & 1)) {
          mma_bf16_16816(sodd, a0, a1, a2, a3, qf[0][ks][0], qf[0][ks][1]);
        } else {
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            if (nb < nbv) mma_bf16_16816(sacc[nb][0], a0, a1, a2, a3, qf[nb][ks][0], qf[nb][ks][1]);
        }
      }
      if (NB == 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[0][0][e] += sodd[e];
      }
    } else {
      // byte tiles: rows g and g+8 share a swizzle phase; the 16-code chunk
      // ks holds d = 16 ks .. 16 ks + 15, this thread's 4 codes at byte 4 tq
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int off = g * 128 + ((ks ^ (g & 7)) << 4) + 4 * tq;
#pragma unroll
        for (int t = 0; t < TL; ++t) {
          const uint8_t* kt = sb + C::box_off(0, w, t, 0);
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(kt + off);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(kt + off + C::RSTEP8);
          uint32_t a0, a1, a2, a3;
          if constexpr (CT == 1) {
            e4m3x4_to_f16x2x2(w0, a0, a2);
            e4m3x4_to_f16x2x2(w1, a1, a3);
          } else {
            const uint32_t x0 = w0 ^ 0x80808080u, x1 = w1 ^ 0x80808080u;
            a0 = s8_pair_to_f16x2(x0, 0x5140);
            a2 = s8_pair_to_f16x2(x0, 0x5342);
            a1 = s8_pair_to_f16x2(x1, 0x5140);
            a3 = s8_pair_to_f16x2(x1, 0x5342);
          }
          mma_f16_16816(sacc[0][t], a0, a1, a2, a3, qf[0][ks][0], qf[0][ks][1]);
        }
      }
    }
    // ---- online softmax on (tok 16t+g / 16t+g+8) x (column 8nb+2tq / 8nb+2tq+1)
    const bool cmask = cpos + CH - 1 > ulim;
    uint32_t pb[NB][TL][2], pc[NB][TL][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      if (nb >= nbv) continue;
      float x[TL][4];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int t = 0; t < TL; ++t) {
        x[t][0] = sacc[nb][t][0] * slc0 * ksr[t][0];
        x[t][1] = sacc[nb][t][1] * slc1 * ksr[t][0];
        x[t][2] = sacc[nb][t][2] * slc0 * ksr[t][1];
        x[t][3] = sacc[nb][t][3] * slc1 * ksr[t][1];
        // causal limit of each score column (decode: the unit's end); a
        // chunk wholly below every column's limit needs no mask
        if (cmask) {
          const int kp = cpos + t * kTile + g;   // key position of row g
          const int limA = col_lim(8 * nb + 2 * tq), limB = col_lim(8 * nb + 2 * tq + 1);
          if (kp > limA) x[t][0] = -INFINITY;
          if (kp > limB) x[t][1] = -INFINITY;
          if (kp + 8 > limA) x[t][2] = -INFINITY;
          if (kp + 8 > limB) x[t][3] = -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(x[t][0], x[t][2]));
        mx1 = fmaxf(mx1, fmaxf(x[t][1], x[t][3]));
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      float pr[TL][4];
      float ps0 = 0.f, ps1 = 0.f;
      if constexpr (CT == 0 || CT == 3) {
        const float mn0 = fmaxf(m0[nb], mx0), mn1 = fmaxf(m1[nb], mx1);
        // a column may have seen no visible key yet (several query rows): keep
        // its state (-inf, 0, 0) instead of forming -inf - -inf
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(m0[nb] - mu0), al1 = exp2f(m1[nb] - mu1);
#pragma unroll
        for (int t = 0; t < TL; ++t) {
          pr[t][0] = exp2f(x[t][0] - mu0);
          pr[t][1] = exp2f(x[t][1] - mu1);
          pr[t][2] = exp2f(x[t][2] - mu0);
          pr[t][3] = exp2f(x[t][3] - mu1);
          ps0 += pr[t][0] + pr[t][2];
          ps1 += pr[t][1] + pr[t][3];
        }
        l0[nb] = l0[nb] * al0 + ps0;
        l1[nb] = l1[nb] * al1 + ps1;
        m0[nb] = mn0;
        m1[nb] = mn1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          o[nb][mt][0] *= al0;
          o[nb][mt][1] *= al1;
          o[nb][mt][2] *= al0;
          o[nb][mt][3] *= al1;
        }
      } else {
        // one-byte pools (consumer-bound): the exponent base m of a column is
        // raised only when a score exceeds it by more than 2^kQuantSlack, so
        // o and l are rescaled rarely; the weights stay below 2^kQuantSlack and
        // the final o / l is the same softmax.  A column that has seen no
        // visible key keeps (-inf, 0, 0).
        const bool need = mx0 > m0[0] + kQuantSlack || mx1 > m1[0] + kQuantSlack;
        if (__any_sync(0xffffffffu, need)) {
          const float mn0 = fmaxf(m0[0], mx0), mn1 = fmaxf(m1[0], mx1);
          const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = exp2f(m0[0] - mu0), al1 = exp2f(m1[0] - mu1);
          l0[0] *= al0;
          l1[0] *= al1;
          vw0 *= al0;
          vw1 *= al1;
          m0[0] = mn0;
          m1[0] = mn1;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            o[0][mt][0] *= al0;
            o[0][mt][1] *= al1;
            o[0][mt][2] *= al0;
            o[0][mt][3] *= al1;
          }
        }
        const float mu0 = m0[0] == -INFINITY ? 0.f : m0[0];
        const float mu1 = m1[0] == -INFINITY ? 0.f : m1[0];
#pragma unroll
        for (int t = 0; t < TL; ++t) {
          pr[t][0] = ex2_approx_ftz(x[t][0] - mu0);
          pr[t][1] = ex2_approx_ftz(x[t][1] - mu1);
          pr[t][2] = ex2_approx_ftz(x[t][2] - mu0);
          pr[t][3] = ex2_approx_ftz(x[t][3] - mu1);
          ps0 += pr[t][0] + pr[t][2];
          ps1 += pr[t][1] + pr[t][3];
        }
        l0[0] += ps0;
        l1[0] += ps1;
      }
      // P enters the tensor core as a hi + lo pair of 16-bit terms so that the
      // product carries ~16 significant bits of each weight (one bf16 rounding
      // of P costs up to 2^-9 relative per weight); one-byte pools: f16 terms
      // of P times the V scale of its token
#pragma unroll
      for (int t = 0; t < TL; ++t) {
        uint32_t ph01, pl01, ph23, pl23;
        if constexpr (C::VB) {
          split_bf16x2(pr[t][0], pr[t][1], ph01, pl01);
          split_bf16x2(pr[t][2], pr[t][3], ph23, pl23);
        } else {
          const float w0 = pr[t][0] * vsr[t][0], w1 = pr[t][1] * vsr[t][0];
          const float w2 = pr[t][2] * vsr[t][1], w3 = pr[t][3] * vsr[t][1];
          if constexpr (CT == 2) {
            vw0 += w0 + w2;
            vw1 += w1 + w3;
          }
          split_f16x2(w0, w1, ph01, pl01);
          split_f16x2(w2, w3, ph23, pl23);
        }
        pb[nb][t][0] = movmatrix_trans(ph01);
        pb[nb][t][1] = movmatrix_trans(ph23);
        pc[nb][t][0] = movmatrix_trans(pl01);
        pc[nb][t][1] = movmatrix_trans(pl23);
      }
    }
    // ---- O^T[D x 8] += V^T[D x 16 tok] . P^T[16 tok x 8], per tile and
    // column block (one V fragment feeds every column block)
    if constexpr (!C::VB) {
      // byte tiles; the rows of each 16-row m tile are permuted: row g -> d =
      // 16 mt + 2g, row g + 8 -> d = 16 mt + 2g + 1.  ldmatrix.trans over 8
      // token rows x 16 bytes (byte pairs as 16-bit elements) hands this
      // thread bytes 2g, 2g+1 of tokens 2tq and 2tq+1; one byte permute pairs
      // the two tokens of each d.  Rows past the end were zeroed above.
      const int lm = lane >> 3, lr = lane & 7;       // matrix and row this lane addresses
      const int tok = (lm & 1) * 8 + lr;
#pragma unroll
      for (int t = 0; t < TL; ++t) {
        const uint32_t vt = smem_u32(sb + C::box_off(1, w, t, 0)) + C::row_off(tok);
#pragma unroll
        for (int mt = 0; mt < D / 16; mt += 2) {
          uint32_t r[4];
          ldmatrix_x4_trans(vt + (((mt + (lm >> 1)) ^ (tok & 7)) << 4), r[0], r[1], r[2], r[3]);
          uint32_t af[2][4];
#pragma unroll
          for (int uu = 0; uu < 2; ++uu) {
            // r[2uu]: tokens 2tq, 2tq+1 of m tile mt + uu; r[2uu+1]: tokens + 8
            if constexpr (CT == 1 || CT == 3) {
              // one permute makes both pairs: bytes (0, 2) low, (1, 3) high
              e4m3x4_to_f16x2x2(__byte_perm(r[2 * uu], 0u, 0x3120), af[uu][0], af[uu][1]);
              e4m3x4_to_f16x2x2(__byte_perm(r[2 * uu + 1], 0u, 0x3120), af[uu][2], af[uu][3]);
            } else {
              // 1152 + code, exact in f16 (the 1152 comes off at the partition end)
              const uint32_t x0 = r[2 * uu] ^ 0x80808080u, x1 = r[2 * uu + 1] ^ 0x80808080u;
              af[uu][0] = __byte_perm(x0, 0x6464u, 0x5240);
              af[uu][1] = __byte_perm(x0, 0x6464u, 0x5341);
              af[uu][2] = __byte_perm(x1, 0x6464u, 0x5240);
              af[uu][3] = __byte_perm(x1, 0x6464u, 0x5341);
            }
          }
          // the hi products of both m tiles before the lo ones (consecutive
          // mma instructions accumulate into different tiles)
#pragma unroll
          for (int lo = 0; lo < 2; ++lo)
#pragma unroll
            for (int uu = 0; uu < 2; ++uu) {
              const uint32_t* pp = lo ? pc[0][t] : pb[0][t];
              mma_f16_16816(o[0][mt + uu], af[uu][0], af[uu][1], af[uu][2], af[uu][3], pp[0],
                            pp[1]);
            }
        }
      }
    } else {
      // two m tiles at a time, the hi products of both before the lo ones, so
      // that consecutive mma instructions accumulate into different tiles
      const int r = (lane & 7) + (lane >> 4) * 8;
      const int chs = (lane >> 3) & 1;
      const uint8_t* vt = sb + C::box_off(1, w, 0, 0);
#pragma unroll
      for (int mt = 0; mt < D / 16; mt += 2) {
        uint32_t a[2][4];
#pragma unroll
        for (int uu = 0; uu < 2; ++uu) {
          const int half = (mt + uu) >> 2;
          const int ch = (((mt + uu) & 3) << 1) + chs;
          const uint32_t addr =
              smem_u32(vt + half * C::HSTR) + C::row_off(r) + ((ch ^ (r & 7)) << 4);
          ldmatrix_x4_trans(addr, a[uu][0], a[uu][1], a[uu][2], a[uu][3]);
        }
#pragma unroll
        for (int lo = 0; lo < 2; ++lo)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int uu = 0; uu < 2; ++uu)
              if (nb < nbv) {
                const uint32_t* pp = lo ? pc[nb][0] : pb[nb][0];
                mma_bf16_16816(o[nb][mt + uu], a[uu][0], a[uu][1], a[uu][2], a[uu][3], pp[0],
                               pp[1]);
              }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);

    if (c == ce - 1 || c == b - 1) {
      // ---- end of partition: write the final output or a partial state of
      // each valid column
      if constexpr (CT == 1 || CT == 3) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[0][mt][e] *= p.v_scale;
      } else if constexpr (CT == 2) {
        float vt0 = vw0, vt1 = vw1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          vt0 += __shfl_xor_sync(0xffffffffu, vt0, off);
          vt1 += __shfl_xor_sync(0xffffffffu, vt1, off);
        }
        const float c0 = 1152.f * vt0, c1 = 1152.f * vt1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          o[0][mt][0] -= c0;
          o[0][mt][1] -= c1;
          o[0][mt][2] -= c0;
          o[0][mt][3] -= c1;
        }
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        if (nb >= nbv) continue;
        float lt0 = l0[nb], lt1 = l1[nb];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
          lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
        }
#pragma unroll
        for (int col = 0; col < 2; ++col) {
          const int cc = 8 * nb + 2 * tq + col;
          if (cc >= ncol) continue;              // padding column
          const int row = (qr0 + cc / G) * H_q + j * G + cc % G;
          // the column's sequence: its query row in decode; the unit's
          // sequence for several query tokens per sequence
          // its partial slot: member * stride + CTA + unit in decode; query
          // row * Pmax + the partition's index within the sequence for several
          // query tokens
          int np, slot;
          if (cu == nullptr) {
            const int4 mt = tc_seq_meta(cstart, row / H_q, M, T, n, p.slot_stride);
            np = mt.y + mt.w;
            slot = (row / H_q - qr0) * p.slot_stride + cta + u;
          } else {
            np = tc_unit_parts(cstart, u, T, n);
            const int part = cta - cta_of_chunk(a, T, n);
            slot = part < p.ws.pmax ? (row / H_q) * p.ws.pmax + part : -1;
          }
          const float lt = col ? lt1 : lt0;
          const float mm = col ? m1[nb] : m0[nb];
          if (np == 1) {
            const float inv = 1.f / lt;
            __nv_bfloat16* orow = p.out + (int64_t)row * D;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              // O^T rows g and g+8 of tile mt are d0 and d1 (see the PV product)
              const int d0 = C::VB ? mt * 16 + g : mt * 16 + 2 * g;
              const int d1 = C::VB ? d0 + 8 : d0 + 1;
              orow[d0] = __float2bfloat16_rn(o[nb][mt][col] * inv);
              orow[d1] = __float2bfloat16_rn(o[nb][mt][2 + col] * inv);
            }
          } else if (slot >= 0) {
            // partial of (slot, head) at slot * H_q + head
            const int64_t pa = (int64_t)slot * H_q + row % H_q;
            float* orow = p.ws.o + pa * D;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              const int d0 = C::VB ? mt * 16 + g : mt * 16 + 2 * g;
              const int d1 = C::VB ? d0 + 8 : d0 + 1;
              orow[d0] = o[nb][mt][col];
              orow[d1] = o[nb][mt][2 + col];
            }
            if (g == 0) p.ws.ml[pa] = make_float2(mm, lt);
          }
        }
      }
    }
  }
}

// ===========================================================================
// Shared-prefix groups: for group g (sequences g m .. g m + m - 1 below S),
// glen[g] = the number of leading tokens that every member reads from the
// same physical blocks: the leading run of block-table entries equal in all
// members' rows, times the block size, capped at the shortest member's length
// and rounded down to whole 16-token chunks (0 for a group of one).  One warp
// per group compares 32 entries at a time and stops at the first difference;
// only entries inside every member's length are read.  Lengths are clamped as
// the attention kernel clamps them (which also reports them).
// ===========================================================================
constexpr int kShareWarps = 8;

__global__ void __launch_bounds__(kShareWarps * 32)
share_prefix_kernel(const int32_t* __restrict__ block_tables, int max_blocks_per_seq,
                    const int32_t* __restrict__ context_lens, int max_len, int S, int K, int m,
                    int* __restrict__ glen) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kShareWarps + warp;
  const int ngroups = (S + m - 1) / m;
  const int cap = min(max_len, max_blocks_per_seq * K);
  int lg = 0;
  if (g < ngroups) {
    const int s0 = g * m, cnt = min(m, S - s0);
    if (cnt >= 2) {
      int lmin = cap;
      for (int i = 0; i < cnt; ++i) {
        const int L = context_lens[s0 + i];
        lmin = min(lmin, L < 0 ? 0 : min(L, cap));
      }
      const int nblk = (lmin + K - 1) / K;
      int run = nblk;
      for (int b0 = 0; b0 < nblk; b0 += 32) {
        const int b = b0 + lane;
        bool same = true;
        if (b < nblk) {
          const int e0 = block_tables[(int64_t)s0 * max_blocks_per_seq + b];
          for (int i = 1; i < cnt; ++i)
            same = same && block_tables[(int64_t)(s0 + i) * max_blocks_per_seq + b] == e0;
        }
        const unsigned diff = __ballot_sync(0xffffffffu, !same);
        if (diff) {
          run = b0 + __ffs(diff) - 1;
          break;
        }
      }
      lg = min(run * K, lmin) / kTile * kTile;
    }
  }
  // the tables and lengths are inputs no kernel of this library writes; the
  // workspace may still be read by the previous launch
  pdl_wait_primary();
  pdl_launch_dependents();
  if (g < ngroups && lane == 0) glen[g] = lg;
}

}  // namespace pkv
