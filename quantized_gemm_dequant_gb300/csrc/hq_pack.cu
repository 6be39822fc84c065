// Repack (and its inverse) between the standard format and the kernel layout.
// One thread per (expert, N tile, K stage, row); see hq_layout.h for the layout.
#include <cuda_runtime.h>
#include <stdint.h>

#include "hq_layout.h"

namespace hq {

// 4-bit integer layout: K offset, within a 32-K row chunk, of nibble slot i of 32-bit word w (see hq_layout.h).
__device__ __forceinline__ int int4_chunk_k(int w, int i) { return 8 * (i & 3) + 2 * w + (i >> 2); }

struct PackArgs {
  int wt;
  int64_t N, K, E;
  int64_t n_tiles, k_stages;
  int blk_bytes;
  int64_t gscale_off;
};

// INT8 / E4M3 layout: K offset, within a 16-K row chunk, of byte b of word w (see hq_layout.h).
__device__ __forceinline__ int int8_chunk_k(int w, int b) { return 2 * w + ((b & 1) ? 8 : 0) + (b >> 1); }
__device__ __forceinline__ int e4m3_chunk_k(int w, int b) { return 2 * w + ((b & 2) ? 8 : 0) + (b & 1); }
// UINT2 layout: K offset, within a 64-K row chunk, of 2-bit slot i of word w.
__device__ __forceinline__ int uint2_chunk_k(int w, int i) {
  const int p = i & 7;
  return 16 * (p >> 1) + 8 * (p & 1) + 2 * w + (i >> 3);
}

// UINT1 layout (also bit 2 of UINT3 codes): K offset, within a 128-K row, of bit b of word w.
__device__ __forceinline__ int uint1_chunk_k(int w, int b) {
  const int p = b & 15;
  return 64 * (p >> 3) + 16 * ((p & 7) >> 1) + 8 * (p & 1) + 2 * w + (b >> 4);
}

// Bits [pos, pos + n) of a little-endian bit string (n <= 3: at most two bytes).
__device__ __forceinline__ uint32_t get_bits(const uint8_t* row, int64_t pos, int n) {
  uint32_t two = row[pos >> 3];
  if ((int)(pos & 7) + n > 8) two |= (uint32_t)row[(pos >> 3) + 1] << 8;
  return (two >> (pos & 7)) & ((1u << n) - 1u);
}
__device__ __forceinline__ void put_bits(uint8_t* row, int64_t pos, int n, uint32_t v) {
  for (int j = 0; j < n; ++j, ++pos) {
    uint8_t* b = row + (pos >> 3);
    const int sh = (int)(pos & 7);
    *b = (uint8_t)((*b & ~(1u << sh)) | (((v >> j) & 1u) << sh));
  }
}

__device__ __forceinline__ uint32_t get_nibble(const uint8_t* row, int64_t k) {
  uint8_t b = row[k >> 1];
  return (k & 1) ? (b >> 4) : (b & 0xF);
}

// dir = 0: pack (standard -> kernel layout); dir = 1: unpack.
template <int DIR>
__global__ void pack_kernel(PackArgs p, uint8_t* codes, uint8_t* scales, uint8_t* zeros, float* gscale,
                            uint8_t* packed) {
  const int64_t total = p.E * p.n_tiles * p.k_stages * TILE_N;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx % TILE_N);
    int64_t t = idx / TILE_N;
    const int64_t ks = t % p.k_stages;
    t /= p.k_stages;
    const int64_t nt = t % p.n_tiles;
    const int64_t e = t / p.n_tiles;
    const int64_t n = nt * TILE_N + r;
    const bool valid = n < p.N;
    uint8_t* blk = packed + ((e * p.n_tiles + nt) * p.k_stages + ks) * (int64_t)p.blk_bytes;
    const int64_t rowc = (e * p.N + n) * (p.K / 2);  // byte offset of the row in codes (4-bit formats)
    if (p.wt == WK_UINT1_ZP || p.wt == WK_UINT3_ZP) {
      // bit-string codes: UINT3 low two bits as the UINT2 planes, bit 2 (UINT1: the code) as the 1-bit plane
      const int bits = p.wt == WK_UINT1_ZP ? 1 : 3;
      const int64_t ng = p.K / 128;
      uint8_t* row = codes + (e * p.N + n) * (p.K * bits / 8);
      const int lo_bytes = bits == 3 ? 4096 : 0;
      if (bits == 3)
        for (int j = 0; j < 2; ++j) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(blk + (j * 128 + r) * 16);
          for (int w = 0; w < 4; ++w) {
            uint32_t word = DIR == 0 ? 0u : dst[w];
            for (int i = 0; i < 16; ++i) {
              const int64_t k = ks * 128 + 64 * j + uint2_chunk_k(w, i);
              if (DIR == 0) {
                if (valid) word |= get_bits(row, 3 * k, 2) << (2 * i);
              } else if (valid) {
                put_bits(row, 3 * k, 2, word >> (2 * i));
              }
            }
            if (DIR == 0) dst[w] = word;
          }
        }
      {
        uint32_t* dst = reinterpret_cast<uint32_t*>(blk + lo_bytes + r * 16);
        for (int w = 0; w < 4; ++w) {
          uint32_t word = DIR == 0 ? 0u : dst[w];
          for (int b = 0; b < 32; ++b) {
            const int64_t k = ks * 128 + uint1_chunk_k(w, b);
            const int64_t pos = k * bits + bits - 1;  // the code's top bit
            if (DIR == 0) {
              if (valid) word |= get_bits(row, pos, 1) << b;
            } else if (valid) {
              put_bits(row, pos, 1, word >> b);
            }
          }
          if (DIR == 0) dst[w] = word;
        }
      }
      const int soff = lo_bytes + 2048;
      uint16_t* sdst = reinterpret_cast<uint16_t*>(blk + soff) + r;
      uint16_t* ssrc = reinterpret_cast<uint16_t*>(scales) + (e * p.N + n) * ng + ks;
      if (DIR == 0) *sdst = valid ? *ssrc : (uint16_t)0;
      else if (valid) *ssrc = *sdst;
      uint8_t* zdst = blk + soff + 256 + r;
      uint8_t* zsrc = zeros + (e * p.N + n) * ng + ks;
      if (DIR == 0) *zdst = valid ? (uint8_t)(*zsrc & ((1u << bits) - 1u)) : (uint8_t)0;
      else if (valid) *zsrc = *zdst;
    } else if (p.wt == WK_INT8_SYM || p.wt == WK_E4M3 || p.wt == WK_UINT2_ZP) {
      const int64_t ng = p.K / 128;
      const bool two = p.wt == WK_UINT2_ZP;
      if (!two) {
        const int64_t rowb = (e * p.N + n) * p.K;
        for (int j = 0; j < 8; ++j) {
          uint8_t* dst = blk + (j * 128 + r) * 16;
          for (int w = 0; w < 4; ++w)
            for (int b = 0; b < 4; ++b) {
              const int64_t k = ks * 128 + 16 * j + (p.wt == WK_INT8_SYM ? int8_chunk_k(w, b) : e4m3_chunk_k(w, b));
              if (DIR == 0) dst[4 * w + b] = valid ? codes[rowb + k] : (uint8_t)0;
              else if (valid) codes[rowb + k] = dst[4 * w + b];
            }
        }
      } else {
        const int64_t rowq = (e * p.N + n) * (p.K / 4);
        for (int j = 0; j < 2; ++j) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(blk + (j * 128 + r) * 16);
          for (int w = 0; w < 4; ++w) {
            if (DIR == 0) {
              uint32_t word = 0;
              if (valid)
                for (int i = 0; i < 16; ++i) {
                  const int64_t k = ks * 128 + 64 * j + uint2_chunk_k(w, i);
                  word |= (uint32_t)((codes[rowq + (k >> 2)] >> (2 * (k & 3))) & 3u) << (2 * i);
                }
              dst[w] = word;
            } else if (valid) {
              const uint32_t word = dst[w];
              for (int i = 0; i < 16; ++i) {
                const int64_t k = ks * 128 + 64 * j + uint2_chunk_k(w, i);
                uint8_t* bp = codes + rowq + (k >> 2);
                const int sh = 2 * (int)(k & 3);
                *bp = (uint8_t)((*bp & ~(3u << sh)) | (((word >> (2 * i)) & 3u) << sh));
              }
            }
          }
        }
      }
      const int soff = two ? 4096 : 16384;
      uint16_t* sdst = reinterpret_cast<uint16_t*>(blk + soff) + r;
      uint16_t* ssrc = reinterpret_cast<uint16_t*>(scales) + (e * p.N + n) * ng + ks;
      if (DIR == 0) *sdst = valid ? *ssrc : (uint16_t)0;
      else if (valid) *ssrc = *sdst;
      if (two) {
        uint8_t* zdst = blk + 4352 + r;
        uint8_t* zsrc = zeros + (e * p.N + n) * ng + ks;
        if (DIR == 0) *zdst = valid ? (uint8_t)(*zsrc & 0x3) : (uint8_t)0;
        else if (valid) *zsrc = *zdst;
      }
    } else if (p.wt == WK_INT4_SYM || p.wt == WK_UINT4_ZP || p.wt == WK_MXINT4) {
      const int G = 128;
      const int64_t ng = p.K / G;
      const uint32_t xr = (p.wt != WK_UINT4_ZP) ? 8u : 0u;
      for (int j = 0; j < 4; ++j) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(blk + (j * 128 + r) * 16);
        for (int w = 0; w < 4; ++w) {
          const int64_t k0 = ks * 128 + 32 * j;
          if (DIR == 0) {
            uint32_t word = 0;
            if (valid)
              for (int i = 0; i < 8; ++i)
                word |= ((get_nibble(codes + rowc, k0 + int4_chunk_k(w, i)) ^ xr) & 0xF) << (4 * i);
            dst[w] = word;
          } else if (valid) {
            const uint32_t word = dst[w];
            for (int i = 0; i < 8; ++i) {
              const int64_t k = k0 + int4_chunk_k(w, i);
              const uint32_t v = ((word >> (4 * i)) & 0xF) ^ xr;
              uint8_t* b = codes + rowc + (k >> 1);
              *b = (k & 1) ? (uint8_t)((*b & 0x0F) | (v << 4)) : (uint8_t)((*b & 0xF0) | v);
            }
          }
        }
      }
      if (p.wt == WK_MXINT4) {
        uint8_t* d = blk + 8192 + 4 * r;
        uint8_t* s = scales + (e * p.N + n) * (p.K / 32) + ks * 4;
        for (int b = 0; b < 4; ++b) {
          if (DIR == 0) d[b] = valid ? s[b] : (uint8_t)0;
          else if (valid) s[b] = d[b];
        }
        continue;
      }
      uint16_t* sdst = reinterpret_cast<uint16_t*>(blk + 8192) + r;
      uint16_t* ssrc = reinterpret_cast<uint16_t*>(scales) + (e * p.N + n) * ng + ks;
      if (DIR == 0) *sdst = valid ? *ssrc : (uint16_t)0;
      else if (valid) *ssrc = *sdst;
      if (p.wt == WK_UINT4_ZP) {
        uint8_t* zdst = blk + 8448 + r;
        uint8_t* zsrc = zeros + (e * p.N + n) * ng + ks;
        if (DIR == 0) *zdst = valid ? (uint8_t)(*zsrc & 0xF) : (uint8_t)0;
        else if (valid) *zsrc = *zdst;
      }
    } else if (p.wt == WK_NVFP4 || p.wt == WK_MXFP4_X) {
      for (int kb = 0; kb < 128; ++kb) {
        const int c = kb >> 4;
        uint8_t* d = blk + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4) + (kb & 15);
        uint8_t* s = codes + rowc + ks * 128 + kb;
        if (DIR == 0) *d = valid ? *s : (uint8_t)0;
        else if (valid) *s = *d;
      }
      const int l = r & 31, cq = r >> 5;
      if (p.wt == WK_MXFP4_X) {  // two e8m0 scales per MMA step, written twice in the word
        const int64_t nb = p.K / 32;
        for (int tt = 0; tt < 4; ++tt) {
          uint8_t* d = blk + 16384 + (l * 16 + tt * 4 + cq) * 4;
          uint8_t* s = scales + (e * p.N + n) * nb + ks * 8 + tt * 2;
          for (int b = 0; b < 4; ++b) {
            if (DIR == 0) d[b] = valid ? s[b & 1] : (uint8_t)0;
            else if (valid && b < 2) s[b] = d[b];
          }
        }
        continue;
      }
      const int64_t nb = p.K / 16;
      for (int tt = 0; tt < 4; ++tt) {
        uint8_t* d = blk + 16384 + (l * 16 + tt * 4 + cq) * 4;
        uint8_t* s = scales + (e * p.N + n) * nb + ks * 16 + tt * 4;
        for (int b = 0; b < 4; ++b) {
          if (DIR == 0) d[b] = valid ? s[b] : (uint8_t)0;
          else if (valid) s[b] = d[b];
        }
      }
      if (r == 0 && nt == 0 && ks == 0) {
        float* g = reinterpret_cast<float*>(packed + p.gscale_off) + e;
        if (DIR == 0) *g = gscale[e];
        else if (gscale) gscale[e] = *g;
      }
    } else {  // MXFP4
      for (int c = 0; c < 8; ++c) {
        uint8_t* d = blk + (r * 8 + c) * 8;
        uint8_t* s = codes + rowc + ks * 64 + c * 8;
        for (int b = 0; b < 8; ++b) {
          if (DIR == 0) d[b] = valid ? s[b] : (uint8_t)0;
          else if (valid) s[b] = d[b];
        }
      }
      const int l = r & 31, cq = r >> 5;
      const int64_t nb = p.K / 32;
      uint8_t* d = blk + 8192 + (cq * 32 + l) * 4;
      uint8_t* s = scales + (e * p.N + n) * nb + ks * 4;
      for (int b = 0; b < 4; ++b) {
        if (DIR == 0) d[b] = valid ? s[b] : (uint8_t)0;
        else if (valid) s[b] = d[b];
      }
    }
  }
}

cudaError_t launch_pack(int dir, int wt, int64_t N, int64_t K, int64_t E, const void* codes, const void* scales,
                        const void* zeros, const float* gscale, void* packed, cudaStream_t stream) {
  const PackGeom g = pack_geom(wt, N, K, E);
  PackArgs p{wt, N, K, E, g.n_tiles, g.k_stages, g.blk_bytes, g.gscale_off};
  const int64_t total = E * g.n_tiles * g.k_stages * TILE_N;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 65535 * 16) blocks = 65535 * 16;
  if (dir == 0)
    pack_kernel<0><<<(unsigned)blocks, threads, 0, stream>>>(p, (uint8_t*)codes, (uint8_t*)scales, (uint8_t*)zeros,
                                                           (float*)gscale, (uint8_t*)packed);
  else
    pack_kernel<1><<<(unsigned)blocks, threads, 0, stream>>>(p, (uint8_t*)codes, (uint8_t*)scales, (uint8_t*)zeros,
                                                           (float*)gscale, (uint8_t*)packed);
  return cudaGetLastError();
}

}  // namespace hq
