// Kernel-layout geometry of packed weights and the launch plan, shared by the
// host API and the device code.  PATH_INT4 is the integer-decode family: every
// format decoded to bf16 in registers or tensor memory (the 4-bit integer
// formats also by the tcgen05 kernel, the others by the register-decode
// kernel only).
//
// Packed weights are a sequence of fixed-size "stage blocks", one per
// (expert, 128-row N tile, K stage), each holding exactly the bytes one
// pipeline stage of the GEMM kernel copies into shared memory with one bulk
// copy:
//
//  INT4_SYM / UINT4_ZP, K stage = 128 (one quantization group):
//    [0, 8192)      codes, 4 chunks x 128 rows x 16 bytes; chunk j of row r holds
//                   k in [32j, 32j+32) as 4 words; nibble slot i of word w holds
//                   k = 32j + 8(i % 4) + 2w + i / 4, so slots p and p + 4 hold the
//                   (even k, odd k) pair 32j + 8p + 2w (+1): one shift by 4p and one
//                   mask extract it as a bf16x2.  Word w of a row chunk is exactly
//                   what lane (g, t = w) of an ldmatrix of 8x8 b16 matrices receives,
//                   and its four pairs are that lane's pairs of the m16n8k16 A
//                   fragments of the chunk's two 16-K steps (p = 0, 1: first step,
//                   k 2t and 2t + 8; p = 2, 3: second step).  INT4_SYM stores q + 8.
//    [8192, 8448)   bf16 scale of each row for this group
//    [8448, 8576)   UINT4_ZP only: zero point of each row (one byte)
//  MXINT4, K stage = 128: codes as INT4_SYM (q + 8), then
//    [8192, 8704)   e8m0 block-32 scales, 4 bytes per row (the stage's four 32-K
//                   blocks in K order) at 8192 + 4r
//  INT8_SYM / E4M3, K stage = 128:
//    [0, 16384)     codes, 8 chunks x 128 rows x 16 bytes; chunk j of row r holds
//                   k in [16j, 16j+16).  Word w holds the (even, odd) pairs
//                   16j + 2w (+1) and 16j + 2w + 8 (+1): INT8 in byte order
//                   (2w, 2w+8, 2w+1, 2w+9), so each pair sits in bits 0-7 and
//                   16-23 after a shift by 0 or 8; E4M3 in byte order (2w, 2w+1,
//                   2w+8, 2w+9), one pair per 16-bit half.  INT8 codes are two's
//                   complement bytes as given.
//    [16384, 16640) bf16 scale of each row for this group
//  UINT2_ZP, K stage = 128:
//    [0, 4096)      codes, 2 chunks x 128 rows x 16 bytes; chunk j of row r holds
//                   k in [64j, 64j+64); 2-bit slot i of word w holds
//                   k = 64j + 16(p / 2) + 8(p % 2) + 2w + i / 8 with p = i % 8: the
//                   pair p of the word is slots (p, p + 8)
//    [4096, 4352)   bf16 scale of each row for this group
//    [4352, 4480)   zero point of each row (one byte)
//  UINT1_ZP, K stage = 128:
//    [0, 2048)      codes, 1 chunk x 128 rows x 16 bytes; bit b of word w of row r
//                   holds k = 64(p / 8) + 16((p % 8) / 2) + 8(p % 2) + 2w + b / 16 with
//                   p = b % 16: pair p of the word is bits (p, p + 16), and after a
//                   shift by 8 kh the pairs of K half kh sit at bits 2s (k 2w + 16s)
//                   and 2s + 1 (k 2w + 16s + 8) of MMA step s
//    [2048, 2304)   bf16 scale of each row for this group
//    [2304, 2432)   zero point of each row (one byte)
//  UINT3_ZP, K stage = 128:
//    [0, 4096)      bits 0-1 of the codes in the UINT2 layout
//    [4096, 6144)   bit 2 of the codes in the UINT1 layout
//    [6144, 6400)   bf16 scale of each row for this group
//    [6400, 6528)   zero point of each row (one byte)
//  NVFP4, K stage = 256:
//    [0, 16384)     e2m1 codes as the shared-memory image of a 128-row x 128-byte
//                   K-major tile with the 128-byte swizzle (16-byte chunk c of row r
//                   at (r/8)*1024 + (r%8)*128 + ((c ^ r%8) * 16)), low nibble = even k
//    [16384, 18432) ue4m3 block-16 scales as tensor-memory words: word
//                   (l*16 + t*4 + c) holds the 4 scales of MMA step t (64 K) of
//                   row 32c + l (the 16 words of lane l are contiguous)
//    global scales: fp32 [E] after the last expert's blocks
//  MXFP4 with MXFP4 activations (WK_MXFP4_X), K stage = 256: codes as NVFP4, then
//    [16384, 18432) e8m0 block-32 scales as tensor-memory words in the NVFP4 word
//                   order: word (l*16 + t*4 + c) holds the two scales of MMA step t
//                   (64 K) of row 32c + l as bytes (s0, s1, s0, s1)
//  MXFP4, K stage = 128:
//    [0, 8192)      e2m1 codes, 8 bytes (16 K) per piece, piece p = r*8 + c lands in
//                   the low half of swizzled 16-byte chunk c of row r
//    [8192, 8704)   e8m0 block-32 scales as tensor-memory words: word (c*32 + l)
//                   holds the 4 scales of row 32c + l
#pragma once
#include <stdint.h>

namespace hq {

enum WeightKind {
  WK_INT4_SYM = 1,
  WK_UINT4_ZP = 2,
  WK_NVFP4 = 3,
  WK_MXFP4 = 4,
  WK_INT8_SYM = 5,
  WK_UINT2_ZP = 6,
  WK_MXINT4 = 7,
  WK_E4M3 = 8,
  WK_UINT1_ZP = 9,
  WK_UINT3_ZP = 10,
  WK_MXFP4_X = 11  // MXFP4 weights packed for MXFP4 activations (not an API format: chosen by the activation type)
};
// Decode variants of the register-decode kernel, one per integer / e4m3 weight layout
enum DecodeKind { DEC_INT4 = 0, DEC_MXINT4 = 1, DEC_INT8 = 2, DEC_E4M3 = 3, DEC_UINT2 = 4, DEC_UINT1 = 5, DEC_UINT3 = 6 };
inline int decode_kind(int weight_type) {
  switch (weight_type) {
    case WK_MXINT4: return DEC_MXINT4;
    case WK_INT8_SYM: return DEC_INT8;
    case WK_E4M3: return DEC_E4M3;
    case WK_UINT2_ZP: return DEC_UINT2;
    case WK_UINT1_ZP: return DEC_UINT1;
    case WK_UINT3_ZP: return DEC_UINT3;
    default: return DEC_INT4;
  }
}
// Formats only the register-decode kernel reads (any token count)
inline bool register_decode_only(int weight_type) { return weight_type >= WK_INT8_SYM; }
// tcgen05 kernel variants; PATH_MXFP4A: MXFP4 weights with MXFP8 activations (e8m0 block scales on both operands)
// PATH_MXFP4X: MXFP4 weights with MXFP4 activations (e8m0 block scales on both operands, packed e2m1 in the MMA)
enum KernelPath { PATH_INT4 = 0, PATH_NVFP4 = 1, PATH_MXFP4 = 2, PATH_MXFP4A = 3, PATH_MXFP4X = 4 };

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
  } else if (weight_type == WK_MXINT4) {
    g.path = PATH_INT4;
    g.kstage = 128;
    g.blk_bytes = 8192 + 512;
  } else if (weight_type == WK_INT8_SYM || weight_type == WK_E4M3) {
    g.path = PATH_INT4;
    g.kstage = 128;
    g.blk_bytes = 16384 + 256;
  } else if (weight_type == WK_UINT2_ZP) {
    g.path = PATH_INT4;
    g.kstage = 128;
    g.blk_bytes = 4096 + 256 + 128;
  } else if (weight_type == WK_UINT1_ZP) {
    g.path = PATH_INT4;
    g.kstage = 128;
    g.blk_bytes = 2048 + 256 + 128;
  } else if (weight_type == WK_UINT3_ZP) {
    g.path = PATH_INT4;
    g.kstage = 128;
    g.blk_bytes = 6144 + 256 + 128;
  } else if (weight_type == WK_MXFP4_X) {
    g.path = PATH_MXFP4X;
    g.kstage = 256;
    g.blk_bytes = 16384 + 2048;
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
