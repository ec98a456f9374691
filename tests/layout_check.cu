// Host-side check of the decode kernel's shared-memory stage layout, for every
// template configuration the library instantiates.
//
// The producer fills a stage with 4-D TMA boxes. A box lands densely as
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
// It makes no CUDA call, so it runs without a GPU. tests/test_layout_host.py
// builds and runs it.
#include <cstdio>
#include <vector>

#include "pkv_attention_tc.cuh"

template <int D, int HPC, int CT, bool B8>
int check_layout() {
  using C = pkv::TcCfg<D, HPC, 2, CT, B8>;
  constexpr int TL = C::TL, NH = C::NH;
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
        const int dst = B8 ? kv * C::KPART + (2 * t + u) * C::UST : kv * C::KPART + t * C::TBOX;
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

int main() {
  int errors = 0;
  errors += check_hpc<64, 0, false>() + check_hpc<64, 0, true>();
  errors += check_hpc<128, 0, false>() + check_hpc<128, 0, true>();
  errors += check_hpc<128, 1, false>() + check_hpc<128, 1, true>();
  errors += check_hpc<128, 2, false>() + check_hpc<128, 2, true>();
  if (errors) {
    std::printf("layout errors: %d\n", errors);
    return 1;
  }
  std::printf("layout ok: 32 configurations\n");
  return 0;
}
