// Host-side checks of the decode kernel (attn_tc_kernel): its shared-memory
// stage layout for every template configuration the library instantiates, and
// its stream-K bookkeeping.
//
// Layout. The producer fills a stage with 4-D TMA boxes. A box lands densely as
// [head][column group][row][128 bytes], at the destination the producer gives
// it: kv * KPART + t * TBOX for 16-row tiles, or kv * KPART + (2t + u) * UST
// for the two 8-row block halves of a B8 tile. The consumers address row r of
// head h, tile t and column group hf at TcCfg::box_off(kv, h, t, hf) +
// TcCfg::row_off(r). This program checks, row by row:
//   * the two addresses agree;
//   * the row keeps the 128-byte swizzle phase r & 7, inside a 1024-byte
//     aligned atom;
//   * no byte is written twice, and the bytes a stage expects (TcCfg::TX)
//     equal the bytes its copies deliver (boxes, then INT8 scales).
//
// Stream-K. With T chunks over n <= T CTAs, CTA i owns chunks
// [floor(iT/n), floor((i+1)T/n)). Checked by brute force: cta_of_chunk(c)
// is the CTA whose range holds chunk c, every CTA owns at least one chunk,
// seq_of_chunk(c) is the sequence whose chunk range holds c (empty sequences
// included), and a sequence never spans more CTAs than the partial slots
// the host plan reserves (min(CTAs per group, ceil(max_len / 16))).
//
// It makes no CUDA call, so it runs without a GPU. tests/test_tc_host.py
// builds and runs it.
#include <algorithm>
#include <cstdio>
#include <random>
#include <vector>

#include "pkv_attention_tc.cuh"

template <int D, int HPC, int CT, bool B8>
int check_layout() {
  using C = pkv::TcCfg<D, HPC, 2, CT, B8>;
  constexpr int TL = C::TL;
  constexpr int box_rows = B8 ? 8 : 16;
  constexpr int parts = B8 ? 2 : 1;   // copies per (tensor, tile)
  int errors = 0;
  std::vector<int> used(C::STAGE, 0);
  long landed = 0;
  auto mark = [&](int at, int bytes) {
    for (int b = 0; b < bytes; ++b) {
      if (at + b >= C::STAGE || used[at + b]++) ++errors;
    }
    landed += bytes;
  };
  for (int kv = 0; kv < 2; ++kv)
    for (int t = 0; t < TL; ++t)
      for (int u = 0; u < parts; ++u) {
        // K boxes, then V boxes (a V tile is smaller than a K tile when V is
        // one-byte and K bf16)
        const int NH = kv ? C::NHV : C::NHK;
        const int dst = B8 ? kv * C::KPART + (2 * t + u) * C::UST
                           : (kv ? C::KPART + t * C::TBOXV : t * C::TBOXK);
        for (int h = 0; h < HPC; ++h)
          for (int hf = 0; hf < NH; ++hf)
            for (int rr = 0; rr < box_rows; ++rr) {
              const int at = dst + ((h * NH + hf) * box_rows + rr) * 128;
              const int r = u * 8 + rr;
              const int want = C::box_off(kv, h, t, hf) + C::row_off(r);
              if (at != want) {
                if (errors < 5)
                  std::printf("D=%d HPC=%d CT=%d B8=%d kv=%d t=%d h=%d hf=%d r=%d: box %d, read %d\n",
                              D, HPC, CT, (int)B8, kv, t, h, hf, r, at, want);
                ++errors;
              }
              if (((at >> 7) & 7) != (r & 7)) ++errors;
              if ((at - (r & 7) * 128) % 1024 != 0) ++errors;
              mark(at, 128);
            }
      }
  if (CT == 2) {
    // each tile's 16 per-slot scales of K, then V (two 32-byte halves in B8)
    for (int kv = 0; kv < 2; ++kv)
      for (int t = 0; t < TL; ++t) mark(C::SCALE_OFF + (kv * TL + t) * 64, 64);
  }
  if (landed != (long)C::TX) {
    std::printf("D=%d HPC=%d CT=%d B8=%d: %ld bytes land, %u expected\n", D, HPC, CT, (int)B8,
                landed, C::TX);
    ++errors;
  }
  return errors;
}

template <int D, int CT, bool B8>
int check_hpc() {
  return check_layout<D, 1, CT, B8>() + check_layout<D, 2, CT, B8>() +
         check_layout<D, 4, CT, B8>() + check_layout<D, 8, CT, B8>();
}

int check_stream_k() {
  int errors = 0;
  for (long long T = 1; T <= 400; ++T)
    for (int n = 1; n <= T && n <= 160; ++n) {
      for (int i = 0; i < n; ++i)
        if ((long long)(i + 1) * T / n <= (long long)i * T / n) ++errors;   // empty CTA
      for (long long c = 0; c < T; ++c) {
        const long long i = pkv::cta_of_chunk(c, T, n);
        if (i < 0 || i >= n || i * T / n > c || c >= (i + 1) * T / n) ++errors;
      }
    }
  std::mt19937 rng(7);
  for (int trial = 0; trial < 4000; ++trial) {
    const int S = 1 + (int)(rng() % 48);
    const int CH = trial & 1 ? 32 : 16;          // bf16 / one-byte chunk sizes
    const int max_len = 1 + (int)(rng() % 3000);
    std::vector<int> cstart(S + 1, 0);
    for (int s = 0; s < S; ++s) {
      const int len = rng() % 5 == 0 ? 0 : (int)(rng() % (max_len + 1));
      cstart[s + 1] = cstart[s] + (len + CH - 1) / CH;
    }
    const long long T = cstart[S];
    if (T == 0) continue;
    for (int c = 0; c < T; ++c) {
      const int s = pkv::seq_of_chunk(cstart.data(), S, c);
      if (s < 0 || s >= S || cstart[s] > c || c >= cstart[s + 1]) ++errors;
    }
    const int grid = 1 + (int)(rng() % 160);     // CTAs per KV-head group
    const int n = (int)(T < grid ? T : grid);
    const int pmax = std::max(1, std::min(grid, (max_len + 15) / 16));
    for (int s = 0; s < S; ++s) {
      if (cstart[s] == cstart[s + 1]) continue;
      const int np = pkv::cta_of_chunk(cstart[s + 1] - 1, T, n) - pkv::cta_of_chunk(cstart[s], T, n) + 1;
      if (np < 1 || np > pmax) ++errors;
    }
  }
  if (errors) std::printf("stream-K errors: %d\n", errors);
  return errors;
}

// Partial slots: for random batches (plain, or groups of m = 16 / G
// sequences with shared lengths glen[g] that are multiples of 16 and at most
// the shortest member's length, 0 for a group of one) and random grids, every
// run of one unit inside a CTA's chunk range is a partition, which gives each
// member of the unit the slot `slot(cta, unit, member, stride)`.  Checked: the
// slots of all partitions are distinct; a sequence's slots are exactly the
// ranges tc_seq_meta lists; slots stay below the plan's bound ((items +
// units) per member region); the tokens a sequence's partitions cover add up
// to its length.  `slot` is member * stride + CTA + unit, or a planted
// variant that must fail.
template <typename Slot>
int check_partial_slots(Slot slot, int trials) {
  int errors = 0;
  std::mt19937 rng(11);
  for (int trial = 0; trial < trials; ++trial) {
    const int G = 1 << (rng() % 4);
    const int m = trial % 3 == 0 ? 1 : 16 / G;
    const int S = 1 + (int)(rng() % 40);
    const int max_len = 1 + (int)(rng() % 2000);
    std::vector<int> len(S), glen((S + m - 1) / m, 0);
    for (int s = 0; s < S; ++s) len[s] = rng() % 7 == 0 ? 0 : (int)(rng() % (max_len + 1));
    if (m > 1) {
      for (int g = 0; g * m < S; ++g) {
        const int cnt = std::min(m, S - g * m);
        int lmin = max_len;
        for (int i = 0; i < cnt; ++i) lmin = std::min(lmin, len[g * m + i]);
        glen[g] = cnt >= 2 && rng() % 4 ? (int)(rng() % (lmin + 1)) / 16 * 16 : 0;
      }
    }
    const int NU = pkv::tc_num_units(S, m);
    std::vector<int> cstart(NU + 1, 0), ut0(NU), uend(NU), us0(NU), urows(NU);
    for (int u = 0; u < NU; ++u) {
      int s0 = u, rows = 1, t0 = 0, end = m == 1 ? len[u] : 0;
      if (m > 1) {
        const int g = u / (m + 1), k = u % (m + 1);
        if (k == 0) {
          s0 = g * m; rows = std::min(m, S - s0); t0 = 0; end = glen[g];
        } else {
          s0 = g * m + k - 1; rows = s0 < S; t0 = glen[g];
          end = rows ? std::max(len[s0], t0) : t0;
        }
      }
      us0[u] = s0; urows[u] = rows; ut0[u] = t0; uend[u] = end;
      cstart[u + 1] = cstart[u] + (rows ? (end - t0 + 15) / 16 : 0);
    }
    const long long T = cstart[NU];
    if (T == 0) continue;
    const int grid = 1 + (int)(rng() % 160);
    const int n = (int)(T < grid ? T : grid);
    const int stride = grid + NU;   // slots per member region
    const long long bound = (long long)stride * m;
    std::vector<std::vector<int>> slots(S);
    std::vector<long long> covered(S, 0);
    std::vector<int> seen;
    for (int i = 0; i < n; ++i) {
      const int cb = (int)((long long)i * T / n), ce = (int)((long long)(i + 1) * T / n);
      for (int c = cb; c < ce; ++c) {
        const int u = pkv::seq_of_chunk(cstart.data(), NU, c);
        if (c != cb && c != cstart[u]) continue;            // not a partition start
        const int last = std::min(ce, cstart[u + 1]);       // partition: chunks c .. last - 1
        const long long tok = std::min<long long>(uend[u], ut0[u] + (long long)(last - cstart[u]) * 16) -
                              (ut0[u] + (long long)(c - cstart[u]) * 16);
        for (int r = 0; r < urows[u]; ++r) {
          const int x = slot(i, u, r, m > 1 ? stride : 0);
          seen.push_back(x);
          if (x < 0 || x >= bound) ++errors;
          slots[us0[u] + r].push_back(x);
          covered[us0[u] + r] += tok;
        }
      }
    }
    std::sort(seen.begin(), seen.end());
    if (std::adjacent_find(seen.begin(), seen.end()) != seen.end()) ++errors;   // shared slot
    for (int s = 0; s < S; ++s) {
      const int4 mt = pkv::tc_seq_meta(cstart.data(), s, m, T, n, m > 1 ? stride : 0);
      std::vector<int> want;
      for (int q = 0; q < mt.y; ++q) want.push_back(mt.x + q);
      for (int q = 0; q < mt.w; ++q) want.push_back(mt.z + q);
      std::vector<int> got = slots[s];
      std::sort(got.begin(), got.end());
      std::sort(want.begin(), want.end());
      if (got != want || covered[s] != len[s]) ++errors;
    }
  }
  return errors;
}

int main() {
  int errors = check_stream_k();
  {
    const int e = check_partial_slots(
        [](int cta, int unit, int member, int stride) { return member * stride + cta + unit; },
        6000);
    // planted mistakes: the members of a shared unit in one slot; the CTA
    // alone as the slot (units of one CTA collide)
    const int planted1 = check_partial_slots(
        [](int cta, int unit, int, int) { return cta + unit; }, 600);
    const int planted2 = check_partial_slots(
        [](int cta, int, int member, int stride) { return member * stride + cta; }, 600);
    const int planted = planted1 && planted2;
    if (e) std::printf("partial slot errors: %d\n", e);
    if (planted == 0) std::printf("planted slot mistake not caught\n");
    errors += e + (planted == 0);
  }
  errors += check_hpc<64, 0, false>() + check_hpc<64, 0, true>();
  errors += check_hpc<128, 0, false>() + check_hpc<128, 0, true>();
  errors += check_hpc<128, 1, false>() + check_hpc<128, 1, true>();
  errors += check_hpc<128, 2, false>() + check_hpc<128, 2, true>();
  errors += check_hpc<128, 3, false>();
  if (errors) {
    std::printf("errors: %d\n", errors);
    return 1;
  }
  std::printf("layout ok: 36 configurations; stream-K ok; partial slots ok\n");
  return 0;
}
