// Kernel-layout geometry of packed weights and the launch plan, shared by the
// host API and the device code.
//
// Packed weights are a sequence of fixed-size "stage blocks", one per
// (expert, 128-row N tile, K stage), each holding exactly the bytes one
// pipeline stage of the GEMM kernel copies into shared memory with one bulk
// copy:
//
//  INT4_SYM / UINT4_ZP, K stage = 128 (one quantization group):
//    [0, 8192)      codes, 4 chunks x 128 rows x 16 bytes; chunk j of row r holds
//                   k in [32j, 32j+32) as 4 words; nibble slot i of word w holds
//                   k = 32j + 8w + {0,2,4,6,1,3,5,7}[i], so one mask extracts the
//                   (even k, odd k) pair of a bf16x2.  INT4_SYM stores q + 8.
//    [8192, 8448)   bf16 scale of each row for this group
//    [8448, 8576)   UINT4_ZP only: zero point of each row (one byte)
//  NVFP4, K stage = 256:
//    [0, 16384)     e2m1 codes as the shared-memory image of a 128-row x 128-byte
//                   K-major tile with the 128-byte swizzle (16-byte chunk c of row r
//                   at (r/8)*1024 + (r%8)*128 + ((c ^ r%8) * 16)), low nibble = even k
//    [16384, 18432) ue4m3 block-16 scales as tensor-memory words: word
//                   (l*16 + t*4 + c) holds the 4 scales of MMA step t (64 K) of
//                   row 32c + l (the 16 words of lane l are contiguous)
//    global scales: fp32 [E] after the last expert's blocks
//  MXFP4, K stage = 128:
//    [0, 8192)      e2m1 codes, 8 bytes (16 K) per piece, piece p = r*8 + c lands in
//                   the low half of swizzled 16-byte chunk c of row r
//    [8192, 8704)   e8m0 block-32 scales as tensor-memory words: word (c*32 + l)
//                   holds the 4 scales of row 32c + l
#pragma once
#include <stdint.h>

namespace hq {

enum WeightKind { WK_INT4_SYM = 1, WK_UINT4_ZP = 2, WK_NVFP4 = 3, WK_MXFP4 = 4 };
enum KernelPath { PATH_INT4 = 0, PATH_NVFP4 = 1, PATH_MXFP4 = 2 };

constexpr int TILE_N = 128;  // weight rows per tile (the UMMA M dimension)

struct PackGeom {
  int path;
  int kstage;          // K elements per stage block
  int blk_bytes;       // bytes per stage block
  int64_t n_tiles;     // 128-row tiles along N
  int64_t k_stages;    // stage blocks along K
  int64_t expert_bytes;
  int64_t total_bytes;  // all experts (+ NVFP4 global scales)
  int64_t gscale_off;   // NVFP4: byte offset of the fp32 [E] global scales, else -1
};

inline PackGeom pack_geom(int weight_type, int64_t N, int64_t K, int64_t E) {
  PackGeom g{};
  g.n_tiles = (N + TILE_N - 1) / TILE_N;
  if (weight_type == WK_INT4_SYM || weight_type == WK_UINT4_ZP) {
    g.path = PATH_INT4;
    g.kstage = 128;
    g.blk_bytes = 8192 + 256 + (weight_type == WK_UINT4_ZP ? 128 : 0);
  } else if (weight_type == WK_NVFP4) {
    g.path = PATH_NVFP4;
    g.kstage = 256;
    g.blk_bytes = 16384 + 2048;
  } else {
    g.path = PATH_MXFP4;
    g.kstage = 128;
    g.blk_bytes = 8192 + 512;
  }
  g.k_stages = K / g.kstage;
  g.expert_bytes = g.n_tiles * g.k_stages * (int64_t)g.blk_bytes;
  g.total_bytes = g.expert_bytes * E;
  g.gscale_off = -1;
  if (weight_type == WK_NVFP4) {
    g.gscale_off = g.total_bytes;
    g.total_bytes += ((E * 4 + 255) / 256) * 256;
  }
  return g;
}

}  // namespace hq
