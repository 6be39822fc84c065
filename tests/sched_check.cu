// Host-side check of the Stream-K partition of the GEMM kernels (Sched, for_each_piece) and of the slot choice of the
// split-K reduction, over many (tiles, K blocks, grid) combinations.  Built with nvcc and run on the CPU by
// tests/test_sched.py; prints "OK" or the first violation.
#include <stdio.h>
#include <stdlib.h>

#include <vector>

#include "../quantized_gemm_dequant_gb300/csrc/hq_gemm_kernel.cuh"

using hq::Piece;
using hq::Sched;

static int check(int tiles, int kst, int grid, int sk) {
  std::vector<int> cover((size_t)tiles * kst, 0);
  std::vector<int> slot_of((size_t)tiles * kst, -1);  // partial slot that holds (tile, block), -1 = stored directly
  Sched s0;
  s0.init(tiles, kst, grid, 0, sk);
  // 32-bit fast path against 64-bit arithmetic
  if (s0.narrow) {
    Sched w = s0;
    w.narrow = false;
    for (int c = 0; c <= s0.P; ++c)
      if (w.start(c) != s0.start(c)) return printf("start mismatch tiles=%d kst=%d grid=%d c=%d\n", tiles, kst, grid, c), 1;
    for (int64_t it = 0; it < (int64_t)tiles * kst; it += 1 + it / 7)
      if (w.cta_of(it) != s0.cta_of(it)) return printf("cta_of mismatch it=%lld\n", (long long)it), 1;
  }
  for (int cta = 0; cta < grid; ++cta) {
    Sched s;
    s.init(tiles, kst, grid, cta, sk);
    if (cta >= s.P) continue;  // inactive CTA
    int npieces = 0, npartial_later = 0;
    for_each_piece(s, [&](const Piece& pc) {
      ++npieces;
      if (pc.tile < 0 || pc.tile >= tiles || pc.g0 < 0 || pc.g1 > kst || pc.g0 >= pc.g1) {
        printf("bad piece tiles=%d kst=%d grid=%d cta=%d\n", tiles, kst, grid, cta);
        exit(1);
      }
      if (pc.full != (pc.g0 == 0 && pc.g1 == kst)) exit((printf("full flag\n"), 1));
      if (!pc.full) {
        if (pc.slot != 2 * cta && pc.slot != 2 * cta + 1) exit((printf("slot range\n"), 1));
        if (pc.slot == 2 * cta + 1) ++npartial_later;
      }
      for (int g = pc.g0; g < pc.g1; ++g) {
        ++cover[(size_t)pc.tile * kst + g];
        slot_of[(size_t)pc.tile * kst + g] = pc.full ? -1 : pc.slot;
      }
    });
    if (npartial_later > 1) return printf("two later partial pieces cta=%d\n", cta), 1;
    if (!sk && npieces == 0 && cta < tiles) return printf("idle cta\n"), 1;
  }
  for (size_t i = 0; i < cover.size(); ++i)
    if (cover[i] != 1) return printf("coverage %d at %zu tiles=%d kst=%d grid=%d sk=%d\n", cover[i], i, tiles, kst, grid, sk), 1;
  if (!sk) return 0;
  // the reduction: for a tile cut between CTAs, CTA c's contribution is in slot (c == c_first && start(c) < first_it)
  // ? 2c + 1 : 2c; that must be the slot the GEMM wrote
  for (int t = 0; t < tiles; ++t) {
    const int64_t first_it = (int64_t)t * s0.kst;
    const int c_first = s0.cta_of(first_it), c_last = s0.cta_of(first_it + kst - 1);
    if (c_first == c_last) {
      for (int g = 0; g < kst; ++g)
        if (slot_of[(size_t)t * kst + g] != -1) return printf("uncut tile left partials t=%d\n", t), 1;
      continue;
    }
    for (int c = c_first; c <= c_last; ++c) {
      const int slot = (c == c_first && s0.start(c) < first_it) ? 2 * c + 1 : 2 * c;
      const int64_t lo = s0.start(c) > first_it ? s0.start(c) : first_it;
      const int64_t hi = s0.start(c + 1) < first_it + kst ? s0.start(c + 1) : first_it + kst;
      for (int64_t it = lo; it < hi; ++it)
        if (slot_of[(size_t)it] != slot)
          return printf("slot %d expected %d tiles=%d kst=%d grid=%d t=%d c=%d\n", slot_of[(size_t)it], slot, tiles, kst,
                        grid, t, c), 1;
    }
  }
  return 0;
}

int main() {
  long n = 0;
  const int kst_list[] = {1, 2, 3, 6, 16, 28, 32, 56};
  for (int tiles = 1; tiles <= 260; tiles += (tiles < 40 ? 1 : 7))
    for (int kst : kst_list)
      for (int grid = 1; grid <= 320; grid += (grid < 20 ? 1 : 13))
        for (int sk = 0; sk < 2; ++sk) {
          if (check(tiles, kst, grid, sk)) return 1;
          ++n;
        }
  // the sizes of the workloads: 112 tiles x 32 blocks over 304 and 152 CTAs, 32 x 28 over 152
  if (check(112, 32, 304, 1) || check(112, 32, 152, 1) || check(32, 28, 152, 1) || check(1024, 28, 152, 0)) return 1;
  printf("OK %ld cases\n", n + 4);
  return 0;
}
