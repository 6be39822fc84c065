// Small-token weight-streaming path for the 4-bit integer formats (dense and MoE).
//
// With at most 32 tokens per tile the UMMA path is limited by its fixed cost
// per 128 x 16 instruction, not by the bytes it moves, so this kernel decodes
// in registers and feeds the legacy warp-level tensor-core instruction
// (mma.sync m16n8k16, bf16 x bf16 -> fp32), in the spirit of the multistage
// copy + MMA pipeline that the Humming announcement reports to beat TMA + UMMA
// at small batch ("Tuning and JIT compilation per workload").
//
// It reads the same packed weight blocks as the UMMA path (see hq_layout.h).
// Each weight row of a block is one row of a 16-row MMA tile; lane (g, t) of
// a warp extracts the (2t, 2t+1) code pair of rows g and g+8 from the shared
// words, so every nibble is decoded by exactly one thread.  Codes become
// exact integers (q - z) in bf16 and are multiplied by the group scale in
// bf16: the same single rounding of (q - z) * s as in the UMMA path, so the
// MMAs accumulate every block straight into the fp32 accumulators.
//
// Two CTAs per SM for 16-token tiles.  Warps 0-7 compute (warp (rg, kh): rows 32rg..32rg+31 of the 128-row tile,
// K half kh of every block); warp 8 produces: one bulk copy of the weight block plus the TMA load (dense) or
// gather4 (MoE) of the token tile for the same 128 K, all on one barrier.
// Pieces and the Stream-K partial slots are those of the UMMA path.
#include "hq_gemm_kernel.cuh"
#include "hq_launch.h"

namespace hq {

constexpr int SM_THREADS = 288;
constexpr int SM_PROD_WARP = 8;

template <int BT>
struct SmallCfg {
  static constexpr int CTAS_PER_SM = BT <= 16 ? 2 : 1;  // 32-token tiles need more registers than two CTAs allow
  static constexpr int W_REGION = 9216;          // one INT4 block (<= 8576 bytes), 1 KB aligned
  static constexpr int ACT_BYTES = 2 * BT * 128;  // two 64-K swizzled atoms
  static constexpr int STAGE = W_REGION + ACT_BYTES;
  // a ring of about 96 KB, so that two CTAs fit on an SM (no tensor memory here)
  static constexpr int STAGES = (96 * 1024) / STAGE > 16 ? 16 : (96 * 1024) / STAGE;
  static constexpr int NT = BT / 8;  // 8-token MMA tiles
  static constexpr int RED_BYTES = 4 * 32 * 2 * NT * 4 * 4;  // K-half exchange of the compute warps
  static constexpr int SMEM_BYTES = STAGES * STAGE + 1024 + 5120 + RED_BYTES;
  static_assert(CTAS_PER_SM * (SMEM_BYTES + 1024) <= 228 * 1024, "CTAs per SM");
};

struct SmallSmem {
  uint64_t full[16];
  uint64_t empty[16];
  int abort_flag;
  int tile_prefix_total;
  uint64_t epi_bar;  // bounded barrier of the 8 compute warps (K-half exchange)
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int BT>
__global__ void __launch_bounds__(SM_THREADS, SmallCfg<BT>::CTAS_PER_SM) hq_gemm_small_kernel(const __grid_constant__ GemmArgs args) {
  using C = SmallCfg<BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SmallSmem& sh = *reinterpret_cast<SmallSmem*>(smem + C::STAGES * C::STAGE);
  int* prefix = reinterpret_cast<int*>(smem + C::STAGES * C::STAGE + 1024);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Dense calls: the producer thread issues the weight copies of its first ring stages before the grid
  // dependency wait (packed weights are read-only inputs, see hq_launch.h), so that they stream while the
  // previous kernel drains; the activation loads of those stages follow the wait on the same barriers.
  int npre = 0;  // producer thread: stages whose weight copy is in flight
  if (tid == SM_PROD_WARP * 32) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 8);
    }
    mbar_init(&sh.epi_bar, 8);
    sh.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&args.tmap_a);
    if (!args.moe) {
      Sched s0;
      s0.init(args.m_tiles * args.n_tiles, args.kst, (int)gridDim.x, (int)blockIdx.x, args.sk);
      if ((int)blockIdx.x < s0.P && s0.tiles > 0)
        for_each_piece(s0, [&](const Piece& pc) {
          const uint8_t* wblk = args.w + ((int64_t)(pc.tile % args.n_tiles) * args.kst) * args.w_blk;
          for (int g = pc.g0; g < pc.g1 && npre < C::STAGES; ++g, ++npre) {
            mbar_arrive_expect_tx(&sh.full[npre], (uint32_t)args.w_blk + C::ACT_BYTES);
            bulk_g2s(smem + npre * C::STAGE, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk, &sh.full[npre]);
          }
        });
    }
  }
  pdl_trigger();
  pdl_wait();  // no global memory a previous kernel may write is touched before this point (weights aside)
  if (args.moe) moe_tile_prefix(args.counts, args.E, args.region_cap, BT, prefix, &sh.tile_prefix_total);
  __syncthreads();
  const int total_tiles = args.moe ? sh.tile_prefix_total * args.n_tiles : args.m_tiles * args.n_tiles;
  Sched sched;
  sched.init(total_tiles, args.kst, (int)gridDim.x, (int)blockIdx.x, args.sk);
  const bool active = (int)blockIdx.x < sched.P && total_tiles > 0;
  volatile int* abort_flag = &sh.abort_flag;
  auto fail = [&](int code) {
    *abort_flag = 1;
    atomicCAS(args.status, 0, code);
  };
  auto tile_rows = [&](int tile, int& e, int& row0, int& nrows) {
    const int mt = tile / args.n_tiles;
    if (args.moe) {
      int lm;
      moe_locate(prefix, args.E, mt, e, lm);
      int cnt = args.counts[e];
      cnt = cnt > args.region_cap ? args.region_cap : cnt;
      row0 = lm * BT;
      nrows = cnt - row0 < BT ? cnt - row0 : BT;
    } else {
      e = 0;
      row0 = mt * BT;
      nrows = args.M - row0 < BT ? args.M - row0 : BT;
    }
  };

  if (active && warp == SM_PROD_WARP) {
    // ============================================================ producer (one thread: a warp-wide loop
    // would reconverge the warp around every wait)
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      uint32_t armed = 0;  // stages with a copy issued (bit s)
      int blk = 0;         // weight blocks of this CTA so far (the first npre were issued before the wait)
      for_each_piece(sched, [&](const Piece& pc) {
        if (!ok) return;
        int e, row0, nrows;
        tile_rows(pc.tile, e, row0, nrows);
        const int nt = pc.tile % args.n_tiles;
        int rbase = row0;  // first row of the 2-D box (dense, or grouped MoE)
        if (args.moe && args.grouped) rbase += args.row_off[e];
        int rows_tok[BT];  // MoE indexed: token of each row of the tile; rows past the expert's count read zeros
        if (args.moe && !args.grouped)
          for (int i = 0; i < BT; ++i)
            rows_tok[i] = i < nrows ? args.region[(int64_t)e * args.region_cap + row0 + i] / args.topk : args.M;
        const uint8_t* wblk = args.w + e * args.w_expert_bytes + ((int64_t)nt * args.kst) * args.w_blk;
        for (int g = pc.g0; g < pc.g1; ++g, ++blk) {
          uint8_t* base = smem + st * C::STAGE;
          uint8_t* act = base + C::W_REGION;
          if (blk >= npre) {
            if (!mbar_wait(&sh.empty[st], ph ^ 1, abort_flag, args.wait_ns)) {
              fail(ERR_TIMEOUT);
              ok = false;
              return;
            }
            mbar_arrive_expect_tx(&sh.full[st], (uint32_t)args.w_blk + C::ACT_BYTES);
            bulk_g2s(base, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk, &sh.full[st]);
          }
          if (!args.moe || args.grouped) {
            for (int j = 0; j < 2; ++j)
              tma_load_2d(act + j * (BT * 128), &args.tmap_a, g * 128 + j * 64, rbase, &sh.full[st]);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int i = 0; i < BT; i += 4)
                tma_gather4(act + j * (BT * 128) + (i >> 3) * 1024 + (i & 7) * 128, &args.tmap_a, g * 128 + j * 64,
                            rows_tok[i], rows_tok[i + 1], rows_tok[i + 2], rows_tok[i + 3], &sh.full[st]);
          }
          armed |= 1u << st;
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
      });
      // every copy this CTA issued lands before its shared memory is released, also when the compute warps gave
      // up (every armed stage's latest phase completes once its bytes arrive)
      int never = 0;
      for (int s = 0; s < C::STAGES; ++s)
        if (armed & (1u << s)) {
          const uint32_t par = (s < st) ? ph : (ph ^ 1);  // phase of the stage's most recent fill
          mbar_wait(&sh.full[s], par, &never, DRAIN_WAIT_NS);
        }
    }
    __syncwarp();
  } else if (active && warp < 8) {
    // ============================================================ compute warps
    // Warp (rg, kh): rows 32*rg .. 32*rg+31 of the tile as two 16-row MMA tiles, and K half kh (two 32-K
    // chunks) of every weight block.  The two K halves meet in shared memory at the end of each piece.
    const int rg = warp & 3, kh = warp >> 2;
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint32_t sh4 = 4u * (uint32_t)t4;
    int rows[4];  // MMA tile m: rows[2m] (fragment rows 0-7), rows[2m+1] (rows 8-15)
#pragma unroll
    for (int i = 0; i < 4; ++i) rows[i] = 32 * rg + 8 * i + g8;
    // ldmatrix.x4 addresses: lanes 8q..8q+7 give the 8 token rows of matrix q = (token group q/2, K half q%2)
    // of the 128-byte-swizzled activation atom; one x4 covers 16 tokens of a 16-K step
    const int lm_tok = ((lane >> 4) << 3) + (lane & 7);  // token within a 16-token group
    const int lm_khi = (lane >> 3) & 1;
    const uint32_t lm_row = (uint32_t)((lm_tok >> 3) * 1024 + (lm_tok & 7) * 128);
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    float* red = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE + 1024 + 5120);  // [4][32 lanes][2][NT][4]
    // CTA-level sync of the 8 compute warps on an mbarrier (bounded, abort-aware: never a hang)
    uint32_t epi_phase = 0;
    auto epi_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.epi_bar);
      if (!mbar_wait(&sh.epi_bar, epi_phase, abort_flag, args.wait_ns)) {
        fail(ERR_TIMEOUT);
        ok = false;
      }
      epi_phase ^= 1;
      return ok;
    };
    for_each_piece(sched, [&](const Piece& pc) {
      if (!ok) return;
      int e, row0, nrows;
      tile_rows(pc.tile, e, row0, nrows);
      const int nt = pc.tile % args.n_tiles;
      float acc[2][C::NT][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < C::NT; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[m][i][j] = 0.0f;
      // output row and multiplier of this lane's token columns (i*8 + 2t, +1), loaded now so that their
      // latency hides behind the mainloop
      int t_row[C::NT][2];
      float t_mul[C::NT][2];
#pragma unroll
      for (int i = 0; i < C::NT; ++i)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col = i * 8 + 2 * t4 + u;
          int orow = -1;
          float f = 1.0f;
          if (kh == 0 && col < nrows) {
            if (args.moe) {
              orow = args.region[(int64_t)e * args.region_cap + row0 + col];
              if (args.topk_w) f = args.topk_w[orow];
            } else {
              orow = row0 + col;
            }
          }
          t_row[i][u] = orow;
          t_mul[i][u] = f;
        }
      for (int g = pc.g0; g < pc.g1; ++g) {
        if (!mbar_wait(&sh.full[st], ph, abort_flag, args.wait_ns)) {
          fail(ERR_TIMEOUT);
          ok = false;
          return;
        }
        const uint8_t* wb = smem + st * C::STAGE;
        const uint32_t act_s = smem_u32(wb + C::W_REGION);
        // each decoded weight is (q - z) * s rounded to bf16 (as in the tensor-core path), so the MMAs
        // accumulate straight into acc and never wait for a block's sums before the next block
        uint32_t ss[4], zz[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t s16 = reinterpret_cast<const uint16_t*>(wb + 8192)[rows[i]];
          ss[i] = s16 | (s16 << 16);
          const uint32_t z = args.zp ? (uint32_t)wb[8448 + rows[i]] : 8u;
          zz[i] = (0x4300u + z) * 0x00010001u;
        }
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {  // 32-K chunk of this warp's K half
          const int j = 2 * kh + jj;
          uint4 w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint4*>(wb + (j * 128 + rows[i]) * 16);
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {  // 16-K step
            const int kk = j * 32 + s2 * 16;  // K within the 128-K block
            const uint32_t atom_s = act_s + (uint32_t)((kk >> 6) * (BT * 128));
            const uint32_t chunk = (uint32_t)(((kk & 63) >> 3) + lm_khi);
            uint32_t b[C::NT][2];
#pragma unroll
            for (int q = 0; q < C::NT / 2; ++q) {
              const uint32_t addr = atom_s + (uint32_t)(q * 2048) + lm_row + ((chunk ^ (uint32_t)(lm_tok & 7)) << 4);
              ldsm_x4(addr, b[2 * q][0], b[2 * q][1], b[2 * q + 1][0], b[2 * q + 1][1]);
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const uint32_t lo = s2 == 0 ? 0 : 2;  // words 2*s2 (K 0-7 of the step) and 2*s2+1 (K 8-15)
              const uint32_t wlo0 = lo == 0 ? w[2 * m].x : w[2 * m].z, whi0 = lo == 0 ? w[2 * m].y : w[2 * m].w;
              const uint32_t wlo1 = lo == 0 ? w[2 * m + 1].x : w[2 * m + 1].z;
              const uint32_t whi1 = lo == 0 ? w[2 * m + 1].y : w[2 * m + 1].w;
              uint32_t a[4];
              a[0] = bf16x2_mul(bf16x2_sub(lop3_and_or(wlo0 >> sh4, 0x000F000Fu, 0x43004300u), zz[2 * m]), ss[2 * m]);
              a[1] = bf16x2_mul(bf16x2_sub(lop3_and_or(wlo1 >> sh4, 0x000F000Fu, 0x43004300u), zz[2 * m + 1]),
                                ss[2 * m + 1]);
              a[2] = bf16x2_mul(bf16x2_sub(lop3_and_or(whi0 >> sh4, 0x000F000Fu, 0x43004300u), zz[2 * m]), ss[2 * m]);
              a[3] = bf16x2_mul(bf16x2_sub(lop3_and_or(whi1 >> sh4, 0x000F000Fu, 0x43004300u), zz[2 * m + 1]),
                                ss[2 * m + 1]);
#pragma unroll
              for (int n8 = 0; n8 < C::NT; ++n8) mma_bf16_16816(acc[m][n8], a, b[n8][0], b[n8][1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[st]);
        if (++st == C::STAGES) {
          st = 0;
          ph ^= 1;
        }
      }
      // ---------------------------------------------------- K halves meet, epilogue
      float* mine = red + ((rg * 32 + lane) * 2) * (C::NT * 4);
      if (kh == 1) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int i = 0; i < C::NT; ++i)
            *reinterpret_cast<float4*>(mine + (m * C::NT + i) * 4) =
                make_float4(acc[m][i][0], acc[m][i][1], acc[m][i][2], acc[m][i][3]);
      }
      if (!epi_sync()) return;
      if (kh == 0) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int i = 0; i < C::NT; ++i) {
            const float4 o = *reinterpret_cast<const float4*>(mine + (m * C::NT + i) * 4);
            acc[m][i][0] += o.x;
            acc[m][i][1] += o.y;
            acc[m][i][2] += o.z;
            acc[m][i][3] += o.w;
          }
        if (pc.full) {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int n = nt * TILE_N + rows[2 * m + rr];
              if (n >= args.N) continue;
              const float bias = args.bias ? bf16_to_f32(args.bias[n]) : 0.0f;
#pragma unroll
              for (int i = 0; i < C::NT; ++i)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int orow = t_row[i][u];
                  if (orow < 0) continue;
                  const float o = acc[m][i][2 * rr + u] * t_mul[i][u] + bias;
                  if (args.comb)  // MoE combine: add into the token's fp32 row
                    red_add_f32(args.comb + (int64_t)(orow / args.comb_k) * args.N + n, o);
                  else
                    args.c[(int64_t)orow * args.N + n] = f32_to_bf16(o);
                }
            }
          }
        } else {
          float* part = args.partials + ((int64_t)pc.slot * BT) * TILE_N;
#pragma unroll
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
              for (int i = 0; i < C::NT; ++i)
#pragma unroll
                for (int u = 0; u < 2; ++u)
                  part[(i * 8 + 2 * t4 + u) * TILE_N + rows[2 * m + rr]] = acc[m][i][2 * rr + u];
        }
      }
      if (!epi_sync()) return;  // the exchange buffer is reused by the next piece
    });
  }
  __syncthreads();
}

template <int BT>
static cudaError_t launch_small_bt(const GemmArgs& a, int grid, cudaStream_t stream) {
  using C = SmallCfg<BT>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(hq_gemm_small_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  return launch_kernel(hq_gemm_small_kernel<BT>, dim3(grid), dim3(SM_THREADS), C::SMEM_BYTES, stream, a);
}

cudaError_t launch_gemm_small(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  switch (bt) {
    case 16: return launch_small_bt<16>(a, grid, stream);
    case 32: return launch_small_bt<32>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hq
