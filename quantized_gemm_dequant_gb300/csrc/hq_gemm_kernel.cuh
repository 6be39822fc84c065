// Persistent warp-specialised quantized GEMM for sm_103a (dense and MoE).
//
// Orientation: the weight tile is the UMMA "A" operand (M = 128 weight rows)
// and the token tile is "B" (N = BT tokens), so D[n, m] sits in tensor memory
// with one weight row per lane.  Small token counts then still fill the
// 128-row MMA.
//
// Two independent shared-memory rings feed the MMA:
//   weight ring      one stage block per 128 K (256 K for NVFP4), one bulk copy each
//   activation ring  one 128-byte-wide K-major tile per stage (64 K of bf16,
//                    128 K of e4m3, 256 K of e2m1), loaded by TMA: a 2-D box for
//                    dense rows, tile::gather4 of the routed rows for MoE
//
// Warp roles (352 threads):
//   warps 0-7  INT4 path: decode the weight block's 4-bit codes into bf16 A
//              tiles in tensor memory (warp w: lane quarter w%4, K half w/4).
//              NVFP4: warps 0-3 copy block scales into tensor memory.
//              MXFP4: warps 0-3 copy the weight block scales, and all 8
//              expand packed e2m1 into the MMA's 16-byte padded layout.
//              All 8: epilogue (tensor memory -> scales -> bf16 store, or a
//              split-K partial).
//   warp 8     weight producer (one thread): bulk copies (dense calls: the
//              first ring stages before the grid dependency wait).
//   warp 9     activation producer: TMA loads (one thread issues; the warp
//              reads the routed-row table for MoE).
//   warp 10    MMA issuer (one thread): tcgen05.mma kind::f16 with A from
//              tensor memory (INT4), kind::mxf4nvf4 scale_vec::4X (NVFP4),
//              kind::mxf8f6f4 scale_vec::1X with e2m1 x e4m3 (MXFP4).
//
// Work is split into pieces (tile, range of weight blocks along K).  With few
// tiles the K blocks of all tiles are dealt out evenly to the CTAs
// (Stream-K); a piece that is not a whole tile leaves fp32 partial sums in
// its own slot, summed afterwards by the split-K reduction kernel.  No CTA
// waits for another.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "hq_layout.h"
#include "hq_launch.h"
#include "hq_ptx.cuh"

namespace hq {

constexpr int NUM_THREADS = 352;
constexpr int WPROD_WARP = 8;
constexpr int APROD_WARP = 9;
constexpr int MMA_WARP = 10;
constexpr int NUM_EPI_THREADS = 256;
constexpr uint64_t DEFAULT_WAIT_NS = 2000000000ull;  // 2 s per pipeline wait unless the host sets another bound
constexpr uint64_t DRAIN_WAIT_NS = 200000000ull;     // waits for this CTA's own copies and MMAs before it exits
constexpr int ERR_TIMEOUT = 5;
constexpr int ERR_BAD_ROUTING = 6;
#if HQ_DEBUG_BOUNDS
// Debug build (libhq_debug.so) only: device-side index checks before global stores and partial-sum accesses.  An
// index outside its buffer records HQ_ERR_BOUNDS in the status word (the first error of a call wins) and the access
// is skipped; nothing traps, so the context stays usable and the host reads the status.
constexpr int ERR_BOUNDS = 8;
// `row` if it is a skipped row (< 0) or inside [0, rows); otherwise records the error and returns -1 (skip).
__device__ __forceinline__ int dbg_row(int row, int rows, int* status) {
  if (row < rows) return row;
  atomicCAS(status, 0, ERR_BOUNDS);
  return -1;
}
// true if a span ending at element `end` fits a buffer of `cap` elements; otherwise records the error.
__device__ __forceinline__ bool dbg_span(int64_t end, int64_t cap, int* status) {
  if (end <= cap) return true;
  atomicCAS(status, 0, ERR_BOUNDS);
  return false;
}
#endif

struct GemmArgs {
  CUtensorMap tmap_a;   // activation data: dense 2-D box of BT rows, MoE one-row boxes for gather4
  CUtensorMap tmap_sf;  // NVFP4 / MXFP8 activation block scales (same row structure)
  const uint8_t* w;        // packed weights, all experts
  int64_t w_expert_bytes;  // bytes per expert
  int w_blk;               // bytes per packed weight block (<= Cfg::W_BLK)
  const float* w_gscale;   // NVFP4 per-expert global scales, else null
  const float* a_scale;    // E4M3: per-token [rows]; NVFP4: global [1]
  const uint16_t* bias;    // bf16 [N] or null
  uint16_t* c;             // bf16 output
  int M;                   // dense rows / MoE tokens
  int N, K;
  int n_tiles, kst;  // 128-row tiles along N, weight blocks along K
  int zp;            // INT4 path: zero points present
  int moe, E, topk;
  const float* topk_w;  // MoE [T*topk] or null
  const int* counts;    // MoE [E] routed rows per expert
  const int* region;    // MoE [E][region_cap] flat (t*topk + j) rows per expert
  int region_cap;
  int grouped;          // MoE: activations already copied into expert-contiguous rows (2-D boxes, no gather)
  const int* row_off;   // MoE grouped: first row of each expert in those rows [E + 1]
  int m_tiles;  // dense: token tiles
  int sk;       // 1: Stream-K split over K blocks
  int* status;
  float* partials;  // Stream-K: tcgen05 kernel [2 * grid][BT][128] fp32, slot 2*cta + {0 first piece, 1 later
                    // piece}; register-decode kernel [grid][BT][128] 64-bit (fp32 value, epoch) words
  float* comb;      // MoE combine: fp32 [T][N]; the output of routed row r is added into token r / comb_k (else null)
  int comb_k;
  const int32_t* ids;  // register-decode kernel, routing fused: topk ids [rows] (else null: routing tables above)
  int fused_rows;      // that many routed rows (T * topk)
  uint64_t wait_ns;  // bound of every pipeline wait (a wait that runs out records HQ_ERR_TIMEOUT)
  int w_evict_first;  // weight copies marked evict-first in L2 (each block read once per call)
#if HQ_DEBUG_BOUNDS
  int dbg_c_rows;          // output rows a kernel may write: dense M, MoE T * topk routed rows (also for the combine)
  int dbg_comb_rows;       // MoE combine: token rows of the fp32 sums (T)
  int64_t dbg_part_elems;  // Stream-K partial-sum buffer, in fp32 values (tcgen05) or 64-bit words (register decode)
#endif
};

template <int PATH, int BT>
struct Cfg {
  static constexpr bool MX = PATH == PATH_MXFP4 || PATH == PATH_MXFP4A;  // MXFP4 weights
  static constexpr bool AMX = PATH == PATH_MXFP4A;                        // MXFP8 activations
  // packed e2m1 on both operands with scale warps feeding both scale sets: NVFP4, and MXFP4 x MXFP4
  static constexpr bool NVF = PATH == PATH_NVFP4 || PATH == PATH_MXFP4X;
  static constexpr bool XMX = PATH == PATH_MXFP4X;  // the MX variant (e8m0 per 32, two scales per MMA step)
  static constexpr int KSTAGE = NVF ? 256 : 128;  // K per weight block
  static constexpr int W_BLK = PATH == PATH_INT4 ? 8576 : (NVF ? 18432 : 8704);
  static constexpr int W_REGION = ((W_BLK + 1023) / 1024) * 1024;
  static constexpr int X_REGION = MX ? 16384 : 0;  // expanded e2m1 A tile (one slot of the X ring)
  // INT4: activation stages per weight block and 64-K atoms per stage.  Tiles of at most 128 tokens take one stage
  // of two atoms per block (one wait for the MMA thread instead of two); 256-token tiles keep two 32 KB stages, so
  // that the ring still holds five of them.
  static constexpr int SUB = PATH == PATH_INT4 ? (BT <= 128 ? 1 : 2) : 1;
  static constexpr int ATOMS = PATH == PATH_INT4 ? 2 / SUB : 1;
  static constexpr int ACT_BYTES = ATOMS * BT * 128;
  static constexpr int ACT_REGION = ((ACT_BYTES + 1023) / 1024) * 1024;
  static constexpr int SF_ROWS = BT < 32 ? 32 : BT;
  // NVFP4 activation scales: dense rows are 16 bytes apart; MoE rows come in gather4 groups of four,
  // each group in its own 128-byte slot (row j at (j/4)*128 + (j%4)*16).  256-token tiles of these paths are
  // dense only: 16 bytes per row, which leaves room for a fourth activation stage.
  static constexpr int ASF_REGION = (NVF || AMX) ? ((SF_ROWS * (BT == 256 ? 16 : 32) + 1023) / 1024) * 1024 : 0;
  static constexpr int A_STAGE = ACT_REGION + ASF_REGION;
  static constexpr int W_STAGE = W_REGION;
  static constexpr int RING_BUDGET = 216 * 1024;
  // MXFP4 weights: the raw blocks and their expansions live in separate rings, so that a raw stage is refilled as
  // soon as it is expanded and the copies run SW blocks ahead while NX expanded slots wait for the MMA
  static constexpr int NX = MX ? (BT <= 64 ? 3 : 2) : 0;
  static constexpr int SW = PATH == PATH_INT4 ? (BT <= 64 ? 12 : 4)
                                              : (NVF ? (BT <= 64 ? 8 : (BT == 128 ? 5 : 4))
                                                     : (BT <= 64 ? 10 : (AMX ? 4 : 6)));
  static constexpr int XRING_BYTES = NX * X_REGION;
  static constexpr int SA_FIT = (RING_BUDGET - SW * W_STAGE - XRING_BYTES) / A_STAGE;
  static constexpr int SA = SA_FIT > 16 ? 16 : SA_FIT;
  static constexpr int CB = BT < 32 ? 1 : BT / 32;  // scale-factor columns per MMA step for B
  static constexpr int SFB_STEP = CB < 4 ? 4 : CB;  // column stride per MMA step (kept 4-aligned)
  static constexpr int SF_STAGE_COLS = NVF ? 16 + 4 * SFB_STEP : 4;
  static constexpr int NA = 4;  // INT4: tensor-memory A slots of 64 columns
  static constexpr int RING_BYTES = SW * W_STAGE + SA * A_STAGE + XRING_BYTES;
  // INT4 256-token tiles keep the epilogue's per-column rows and multipliers (MoE) in shared memory: two pieces x
  // 8 warps x 128 columns x (row, multiplier); in registers they would spill next to the 128-column accumulator slice
  static constexpr int TAB_BYTES = (PATH == PATH_INT4 && BT == 256) ? 2 * 8 * (BT / 2) * 8 : 0;
  static constexpr int SMEM_RAW = RING_BYTES + 1024 /*align*/ + 8192 /*barriers, tile tables, MoE prefix*/ + TAB_BYTES;
  // at least 120 KB so that one CTA (and one 512-column tensor-memory allocation) owns each SM
  static constexpr int SMEM_BYTES = SMEM_RAW < 120 * 1024 ? 120 * 1024 : SMEM_RAW;
  static_assert(SA >= 2, "activation ring too small");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(!NVF || 256 + SW * SF_STAGE_COLS <= 512, "tensor memory");
  static_assert(!MX || 256 + 4 * NX + (AMX ? NX * SFB_STEP : 8) <= 512, "tensor memory");
};

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
// two floats -> bf16x2 (round to nearest even); lo holds a
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
  return d;
}
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

template <int X>
__device__ __forceinline__ void tmem_st_x(uint32_t taddr, const uint32_t* r);
template <>
__device__ __forceinline__ void tmem_st_x<1>(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r[0]) : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_x<2>(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(r[0]), "r"(r[1])
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_x<4>(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_x<8>(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_x<16>(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// ----------------------------------------------------------------- work pieces
struct Piece {
  int tile;    // tile index (token tile major, N tile minor)
  int g0, g1;  // weight-block range along K
  bool full;   // covers all K blocks of the tile
  int slot;    // Stream-K partial slot (2*cta + {0 first piece, 1 last piece})
};

struct Sched {
  int tiles, kst, P, cta, sk;
  int64_t W;    // total block iterations
  bool narrow;  // W * P < 2^32: every product below fits 32 bits (64-bit division is a long software routine)
  __host__ __device__ void init(int tiles_, int kst_, int grid, int cta_, int sk_) {
    tiles = tiles_;
    kst = kst_;
    W = (int64_t)tiles * kst;
    P = sk_ ? (int)((int64_t)grid < W ? grid : W) : grid;
    cta = cta_;
    sk = sk_;
    narrow = (uint64_t)W * (uint64_t)(P > 0 ? P : 1) < (1ull << 32);
  }
  __host__ __device__ int64_t start(int c) const {
    return narrow ? (int64_t)(((uint32_t)c * (uint32_t)W) / (uint32_t)P) : (int64_t)c * W / P;
  }
  // largest CTA whose range starts at or before iteration it
  __host__ __device__ int cta_of(int64_t it) const {
    return narrow ? (int)(((uint32_t)(it + 1) * (uint32_t)P - 1u) / (uint32_t)W) : (int)(((it + 1) * P - 1) / W);
  }
  __host__ __device__ void split(int64_t it, int& t, int& g) const {  // iteration -> (tile, K block)
    if (narrow) {
      t = (int)((uint32_t)it / (uint32_t)kst);
      g = (int)((uint32_t)it - (uint32_t)t * (uint32_t)kst);
    } else {
      t = (int)(it / kst);
      g = (int)(it - (int64_t)t * kst);
    }
  }
};

// (host-callable as well: tests/sched_check.cu checks the partition on the CPU)
template <typename F>
__host__ __device__ __forceinline__ void for_each_piece(const Sched& s, F&& f) {
  if (!s.sk) {
    for (int t = s.cta; t < s.tiles; t += s.P) f(Piece{t, 0, s.kst, true, 0});
    return;
  }
  const int64_t it0 = s.start(s.cta), it1 = s.start(s.cta + 1);
  int64_t it = it0;
  bool first = true;
  while (it < it1) {
    int t, g0;
    s.split(it, t, g0);
    const int64_t left = it1 - it;
    const int g1 = (int)((int64_t)g0 + left < s.kst ? g0 + left : s.kst);
    f(Piece{t, g0, g1, g0 == 0 && g1 == s.kst, 2 * s.cta + (first ? 0 : 1)});
    it += g1 - g0;
    first = false;
  }
}

// ----------------------------------------------------------------- shared state
template <int PATH, int BT>
struct Smem {
  using C = Cfg<PATH, BT>;
  uint64_t w_full[C::SW];
  uint64_t w_empty[C::SW];
  uint64_t ready[C::MX ? C::NX : C::SW];  // FP4 paths: scales in tensor memory (MXFP4: per X slot, with its A)
  uint64_t x_empty[C::MX ? C::NX : 1];     // MXFP4: X slot released by the MMAs that read it
  uint64_t a_full[C::SA];
  uint64_t a_empty[C::SA];
  uint64_t afull[C::NA];  // INT4: decoded A slot written
  uint64_t aempty[C::NA];
  uint64_t dfull;
  uint64_t dempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_prefix_total;
  int rows_tok[256];  // MoE: token index of each row of the activation producer's current tile
};

// Map a global token-tile index to (expert, local token tile) for MoE via the
// per-expert tile prefix held in shared memory.
__device__ __forceinline__ void moe_locate(const int* prefix, int E, int mt, int& e, int& lm) {
  int lo = 0, hi = E;  // find e with prefix[e] <= mt < prefix[e+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= mt) lo = mid;
    else hi = mid;
  }
  e = lo;
  lm = mt - prefix[lo];
}

// MoE token-tile prefix over experts into shared memory: prefix[e] = token tiles of experts before e (prefix[0] = 0,
// prefix[E] = total, also written to *total).  Expert counts are clamped to [0, region_cap].  Every thread of the
// block calls it (it holds a __syncthreads); the counts are read in parallel and one warp scans them.
__device__ __forceinline__ void moe_tile_prefix(const int* counts, int E, int region_cap, int bt, int* prefix,
                                                int* total) {
  const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += nthreads) {
    int cnt = counts[e];
    cnt = cnt < 0 ? 0 : (cnt > region_cap ? region_cap : cnt);
    prefix[e + 1] = (cnt + bt - 1) / bt;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int b0 = 1 + lane * per;
    int run = 0;
    for (int i = 0; i < per; ++i)
      if (b0 + i <= E) run += prefix[b0 + i];
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int acc = incl - run;
    for (int i = 0; i < per; ++i)
      if (b0 + i <= E) {
        acc += prefix[b0 + i];
        prefix[b0 + i] = acc;
      }
    if (lane == 0) prefix[0] = 0;
    if (lane == 31) *total = incl;
  }
}

// COMB instances carry the MoE combine epilogue (args.comb set: routed rows are added into their tokens' fp32 rows);
// the others are compiled without it, so that their register allocation is not shaped by it.
template <int PATH, int BT, bool COMB>
__global__ void __launch_bounds__(NUM_THREADS, 1) hq_gemm_kernel(const __grid_constant__ GemmArgs args) {
  using C = Cfg<PATH, BT>;
  static_assert(sizeof(Smem<PATH, BT>) <= 4096, "shared state");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = smem;                       // SW x W_STAGE
  uint8_t* aring = smem + C::SW * C::W_STAGE;  // SA x A_STAGE
  uint8_t* xring = aring + C::SA * C::A_STAGE;  // NX x X_REGION (MXFP4)
  Smem<PATH, BT>& sh = *reinterpret_cast<Smem<PATH, BT>*>(smem + C::RING_BYTES);
  int* prefix = reinterpret_cast<int*>(smem + C::RING_BYTES + 4096);  // MoE: E + 1 ints (E <= 512)
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---------------------------------------------------------------- setup
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  // Dense calls: the weight producer issues the copies of its first ring stages before the grid dependency wait
  // (packed weights are read-only inputs, see hq_launch.h), so that they stream while the previous kernel drains.
  int npre = 0;  // weight producer thread: stages whose copy is in flight
  if (tid == WPROD_WARP * 32) {
    for (int s = 0; s < C::SW; ++s) {
      mbar_init(&sh.w_full[s], 1);
      mbar_init(&sh.w_empty[s], PATH == PATH_INT4 ? 8 : (C::NVF ? 4 + 1 : 8));
      if (!C::MX) mbar_init(&sh.ready[s], 4);
    }
    for (int x = 0; x < C::NX; ++x) {
      mbar_init(&sh.ready[x], 8);
      mbar_init(&sh.x_empty[x], 1);
    }
    for (int s = 0; s < C::SA; ++s) {
      mbar_init(&sh.a_full[s], 1);
      mbar_init(&sh.a_empty[s], (C::NVF || C::AMX) ? 4 + 1 : 1);
    }
    for (int a = 0; a < C::NA; ++a) {
      mbar_init(&sh.afull[a], 8);
      mbar_init(&sh.aempty[a], 1);
    }
    mbar_init(&sh.dfull, 1);
    mbar_init(&sh.dempty, 8);
    mbar_init(&sh.drain, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
    if (!args.moe) {
      Sched s0;
      s0.init(args.m_tiles * args.n_tiles, args.kst, (int)gridDim.x, (int)blockIdx.x, args.sk);
      if ((int)blockIdx.x < s0.P && s0.tiles > 0)
        for_each_piece(s0, [&](const Piece& pc) {
          const uint8_t* wblk = args.w + ((int64_t)(pc.tile % args.n_tiles) * args.kst) * args.w_blk;
          for (int g = pc.g0; g < pc.g1 && npre < C::SW; ++g, ++npre) {
            mbar_arrive_expect_tx(&sh.w_full[npre], (uint32_t)args.w_blk);
            if (args.w_evict_first)
              bulk_g2s_hint(wring + npre * C::W_STAGE, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk,
                            &sh.w_full[npre], l2_evict_first_policy());
            else
              bulk_g2s(wring + npre * C::W_STAGE, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk,
                       &sh.w_full[npre]);
          }
        });
    }
  }
  if (tid == APROD_WARP * 32) {
    prefetch_tmap(&args.tmap_a);
    if (C::NVF || C::AMX) prefetch_tmap(&args.tmap_sf);
  }
  pdl_trigger();
  pdl_wait();  // no global memory a previous kernel may write is touched before this point (weights aside)
  // MoE: tile prefix over experts (E <= 512 enforced on the host)
  if (args.moe) moe_tile_prefix(args.counts, args.E, args.region_cap, BT, prefix, &sh.tile_prefix_total);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  const int total_tiles = args.moe ? sh.tile_prefix_total * args.n_tiles : args.m_tiles * args.n_tiles;

  Sched sched;
  sched.init(total_tiles, args.kst, (int)gridDim.x, (int)blockIdx.x, args.sk);
  const bool active = (int)blockIdx.x < sched.P && total_tiles > 0;
  volatile int* abort_flag = &sh.abort_flag;

  auto fail = [&](int code) {
    *abort_flag = 1;
    atomicCAS(args.status, 0, code);
  };

  // Row bookkeeping of a tile: token tile (dense) or (expert, local tile) (MoE).
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

  if (active && warp == WPROD_WARP) {
    // ============================================================ weight producer
    if (lane == 0) {
      int ws = 0;
      uint32_t wph = 0;
      bool ok = true;
      int armed[C::SW];
#pragma unroll
      for (int s = 0; s < C::SW; ++s) armed[s] = 0;
      int blk = 0;  // weight blocks of this CTA so far (the first npre were issued before the wait)
      for_each_piece(sched, [&](const Piece& pc) {
        if (!ok) return;
        int e, row0, nrows;
        tile_rows(pc.tile, e, row0, nrows);
        const int nt = pc.tile % args.n_tiles;
        const uint8_t* wblk = args.w + e * args.w_expert_bytes + ((int64_t)nt * args.kst) * args.w_blk;
        for (int g = pc.g0; g < pc.g1; ++g, ++blk) {
          if (blk >= npre) {
            if (!mbar_wait(&sh.w_empty[ws], wph ^ 1, abort_flag, args.wait_ns)) {
              fail(ERR_TIMEOUT);
              ok = false;
              return;
            }
            mbar_arrive_expect_tx(&sh.w_full[ws], (uint32_t)args.w_blk);
            if (args.w_evict_first)
              bulk_g2s_hint(wring + ws * C::W_STAGE, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk,
                            &sh.w_full[ws], l2_evict_first_policy());
            else
              bulk_g2s(wring + ws * C::W_STAGE, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk, &sh.w_full[ws]);
          }
          ++armed[ws];
          if (++ws == C::SW) {
            ws = 0;
            wph ^= 1;
          }
        }
      });
      // Every bulk copy this CTA issued lands before its shared memory is released, also when the consumers gave
      // up (a timeout or abort elsewhere in the CTA): wait for the latest fill of every stage used.
      int never = 0;
      for (int s = 0; s < C::SW; ++s)
        if (armed[s] > 0) mbar_wait(&sh.w_full[s], (uint32_t)((armed[s] - 1) & 1), &never, DRAIN_WAIT_NS);
    }
    __syncwarp();
  } else if (active && warp == APROD_WARP) {
    // ============================================================ activation producer
    constexpr int A_BOX_BYTES = BT * 128;  // one TMA box: BT rows x 128 bytes
    constexpr int SF_BOX_BYTES = BT * 16;
    if (!args.moe || args.grouped) {
      // 2-D boxes: one thread runs the loop (a warp-wide loop would reconverge around every wait)
      if (lane == 0) {
        int as = 0;
        uint32_t aph = 0;
        bool ok = true;
        uint32_t armed = 0;  // stages with a load issued (bit s)
        for_each_piece(sched, [&](const Piece& pc) {
          if (!ok) return;
          int e, row0, nrows;
          tile_rows(pc.tile, e, row0, nrows);
          const int rbase = row0 + (args.moe ? args.row_off[e] : 0);  // first row of the box
          for (int g = pc.g0; g < pc.g1; ++g) {
            for (int j = 0; j < C::SUB; ++j) {
              if (!mbar_wait(&sh.a_empty[as], aph ^ 1, abort_flag, args.wait_ns)) {
                fail(ERR_TIMEOUT);
                ok = false;
                return;
              }
              uint8_t* dst = aring + as * C::A_STAGE;
              // x offset of this stage in the tensor map's element units (bf16: 64 per atom; bytes: 128)
              const int x = PATH == PATH_INT4 ? g * 128 + j * C::ATOMS * 64 : g * 128;
              mbar_arrive_expect_tx(&sh.a_full[as], C::ATOMS * A_BOX_BYTES + ((C::NVF || C::AMX) ? SF_BOX_BYTES : 0));
#pragma unroll
              for (int t = 0; t < C::ATOMS; ++t)
                tma_load_2d(dst + t * A_BOX_BYTES, &args.tmap_a, x + t * 64, rbase, &sh.a_full[as]);
              // block scales: NVFP4 16 bytes per 256-K stage; MXFP8 the 16-byte group of four 128-K stages
              if (C::NVF || C::AMX)
                tma_load_2d(dst + C::ACT_REGION, &args.tmap_sf, C::AMX ? (g >> 2) * 16 : (C::XMX ? (g >> 1) * 16 : g * 16),
                            rbase, &sh.a_full[as]);
              armed |= 1u << as;
              if (++as == C::SA) {
                as = 0;
                aph ^= 1;
              }
            }
          }
        });
        // every load lands before shared memory is released (the latest fill of each stage used)
        int never = 0;
        for (int s = 0; s < C::SA; ++s)
          if (armed & (1u << s)) mbar_wait(&sh.a_full[s], (s < as) ? aph : (aph ^ 1), &never, DRAIN_WAIT_NS);
      }
      __syncwarp();
    } else {
      // routed rows: the warp's lanes issue the four-row gathers in parallel
      int as = 0;
      uint32_t aph = 0;
      bool ok = true;
      uint32_t armed = 0;
      for_each_piece(sched, [&](const Piece& pc) {
        if (!ok) return;
        int e, row0, nrows;
        tile_rows(pc.tile, e, row0, nrows);
        // token index of every row of the tile; rows past the expert's count read zeros (row M)
        for (int i = lane; i < BT; i += 32)
          sh.rows_tok[i] = i < nrows ? args.region[(int64_t)e * args.region_cap + row0 + i] / args.topk : args.M;
        __syncwarp();
        for (int g = pc.g0; g < pc.g1; ++g) {
          for (int j = 0; j < C::SUB; ++j) {
            if (lane == 0) {
              if (!mbar_wait(&sh.a_empty[as], aph ^ 1, abort_flag, args.wait_ns)) {
                fail(ERR_TIMEOUT);
                ok = false;
              }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) return;
            uint8_t* dst = aring + as * C::A_STAGE;
            const int x = PATH == PATH_INT4 ? g * 128 + j * C::ATOMS * 64 : g * 128;
            if (lane == 0)
              mbar_arrive_expect_tx(&sh.a_full[as], C::ATOMS * A_BOX_BYTES + ((C::NVF || C::AMX) ? SF_BOX_BYTES : 0));
            __syncwarp();
            for (int i = lane * 4; i < BT; i += 128) {
              uint8_t* d = dst + (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
              for (int t = 0; t < C::ATOMS; ++t)
                tma_gather4(d + t * A_BOX_BYTES, &args.tmap_a, x + t * 64, sh.rows_tok[i], sh.rows_tok[i + 1],
                            sh.rows_tok[i + 2], sh.rows_tok[i + 3], &sh.a_full[as]);
              if (C::NVF || C::AMX)
                tma_gather4(dst + C::ACT_REGION + (i >> 2) * 128, &args.tmap_sf,
                            C::AMX ? (g >> 2) * 16 : (C::XMX ? (g >> 1) * 16 : g * 16),
                            sh.rows_tok[i],
                            sh.rows_tok[i + 1], sh.rows_tok[i + 2], sh.rows_tok[i + 3], &sh.a_full[as]);
            }
            armed |= 1u << as;
            if (++as == C::SA) {
              as = 0;
              aph ^= 1;
            }
          }
        }
        __syncwarp();  // rows_tok is rewritten for the next piece
      });
      if (lane == 0) {  // every gather lands before shared memory is released
        int never = 0;
        for (int s = 0; s < C::SA; ++s)
          if (armed & (1u << s)) mbar_wait(&sh.a_full[s], (s < as) ? aph : (aph ^ 1), &never, DRAIN_WAIT_NS);
      }
      __syncwarp();
    }
  } else if (active && warp == MMA_WARP) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      int ws = 0, as = 0, aslot = 0, xs = 0;
      uint32_t wph = 0, aph = 0, aslph = 0, xph = 0;
      int pidx = 0;
      bool ok = true;
      auto waitf = [&](uint64_t* bar, uint32_t par) {
        if (!ok) return false;
        if (!mbar_wait(bar, par, abort_flag, args.wait_ns)) {
          fail(ERR_TIMEOUT);
          ok = false;
        }
        return ok;
      };
      for_each_piece(sched, [&](const Piece& pc) {
        if (!waitf(&sh.dempty, (pidx & 1) ^ 1)) return;
        tc_fence_after();
        for (int g = pc.g0; g < pc.g1; ++g) {
          if (PATH == PATH_INT4) {
            if (!waitf(&sh.afull[aslot], aslph)) return;
          } else if (C::MX) {
            if (!waitf(&sh.ready[xs], xph)) return;  // expanded A and scales of this block (its raw stage is free)
          } else {
            if (!waitf(&sh.w_full[ws], wph) || !waitf(&sh.ready[ws], wph)) return;
          }
          for (int j = 0; j < C::SUB; ++j) {
            if (!waitf(&sh.a_full[as], aph)) return;
            // (the stage was written by TMA and is read by the MMA, both in the async proxy: no proxy fence; the
            // expanded MXFP4 tiles are fenced by the warps that write them)
            tc_fence_after();
            const uint32_t act = smem_u32(aring + as * C::A_STAGE);
            const bool first = (g == pc.g0 && j == 0);
            if (PATH == PATH_INT4) {
              constexpr uint32_t idesc = idesc_bf16(128, BT);
#pragma unroll
              for (int t = 0; t < C::ATOMS; ++t) {
                const uint32_t a_t = tmem + 256 + aslot * 64 + (j * C::ATOMS + t) * 32;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint64_t bd = smem_desc(act + t * (BT * 128) + i * 32, 16, 1024, 2);
                  umma_bf16_ts(tmem, a_t + i * 8, bd, idesc, (first && t == 0 && i == 0) ? 0u : 1u);
                }
              }
            } else if (C::NVF) {
              constexpr uint32_t idesc = idesc_block_scaled(128, BT, 1, 1, C::XMX ? 1 : 0, 0, 0);
              const uint32_t wa = smem_u32(wring + ws * C::W_STAGE);
              const uint32_t sf = tmem + 256 + ws * C::SF_STAGE_COLS;
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const uint64_t ad = smem_desc(wa + t * 32, 16, 1024, 2);
                const uint64_t bd = smem_desc(act + t * 32, 16, 1024, 2);
                if (C::XMX)
                  umma_mxf4_ss(tmem, ad, bd, idesc, sf + 4 * t, sf + 16 + t * C::SFB_STEP, (first && t == 0) ? 0u : 1u);
                else
                  umma_nvf4_ss(tmem, ad, bd, idesc, sf + 4 * t, sf + 16 + t * C::SFB_STEP,
                               (first && t == 0) ? 0u : 1u);
              }
            } else {
              const uint32_t xa = smem_u32(xring + xs * C::X_REGION);
              const uint32_t sfa = tmem + 256 + xs * 4;
              // activation block scales: unit scales written once (per-token FP8), or the stage's MXFP8 scales
              const uint32_t sfb = tmem + 256 + 4 * C::NX + (C::AMX ? xs * C::SFB_STEP : 0);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t idesc = idesc_block_scaled(128, BT, 5, 0, 1, i, C::AMX ? i : 0);
                const uint64_t ad = smem_desc(xa + i * 32, 16, 1024, 2);
                const uint64_t bd = smem_desc(act + i * 32, 16, 1024, 2);
                umma_mxf8_ss(tmem, ad, bd, idesc, sfa, sfb, (first && i == 0) ? 0u : 1u);
              }
            }
            umma_commit(&sh.a_empty[as]);
            if (++as == C::SA) {
              as = 0;
              aph ^= 1;
            }
          }
          if (PATH == PATH_INT4) {
            umma_commit(&sh.aempty[aslot]);
            if (++aslot == C::NA) {
              aslot = 0;
              aslph ^= 1;
            }
          } else if (C::MX) {
            umma_commit(&sh.x_empty[xs]);
            if (++xs == C::NX) {
              xs = 0;
              xph ^= 1;
            }
          } else {
            umma_commit(&sh.w_empty[ws]);
            if (++ws == C::SW) {
              ws = 0;
              wph ^= 1;
            }
          }
        }
        umma_commit(&sh.dfull);
        ++pidx;
      });
      // every issued MMA completes before tensor memory is released (also when the epilogue gave up)
      int never = 0;
      umma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, &never, DRAIN_WAIT_NS);
    }
    __syncwarp();
  } else if (active && warp < 8) {
    // ============================================================ decode / scales / epilogue
    const int q = warp & 3;       // tensor-memory lane quarter
    const int h = warp >> 2;      // K half (INT4) / column half (epilogue)
    const int r = q * 32 + lane;  // weight row within the tile
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int ws = 0, as = 0, aslot = 0, xs = 0;
    uint32_t wph = 0, aph = 0, aslph = 0, xph = 0;
    int pidx = 0;
    bool ok = true;
    auto waitf = [&](uint64_t* bar, uint32_t par) {
      if (!ok) return false;
      if (!mbar_wait(bar, par, abort_flag, args.wait_ns)) {
        fail(ERR_TIMEOUT);
        ok = false;
      }
      return ok;
    };
    if (PATH == PATH_MXFP4 && warp < 4) {
      // unit activation block scales (2^0) for every MMA, written once
      uint32_t ones[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) ones[j] = 0x7F7F7F7Fu;
      tmem_st_x<8>(tmem + lane_base + 256 + 4 * C::NX, ones);
      tmem_wait_st();
    }
    constexpr int HC = BT / 2;
    // Per-column output rows and multipliers: MoE rows and per-token activation scales.  NVFP4 tiles of 256 tokens
    // are dense only (the host tiles NVFP4 MoE rows by at most 128), so they carry no table; INT4 tiles of 256
    // tokens keep theirs in shared memory.
    constexpr bool kSmemTables = C::TAB_BYTES > 0;
    constexpr bool kTables = PATH == PATH_MXFP4 || BT <= 128 || kSmemTables;
    constexpr int TPL = (kTables && !kSmemTables) ? (HC + 31) / 32 : 1;
    int2* tabs = reinterpret_cast<int2*>(smem + C::RING_BYTES + 8192);  // [2][8 warps][HC] when kSmemTables
    const int col0 = h * HC;
    if (!kTables && args.moe) {
      fail(ERR_BAD_ROUTING);
      ok = false;
    }
    // What a piece's epilogue needs, gathered when its mainloop starts.
    struct Pend {
      Piece pc;
      int e, row0, nrows, nt;
      int ts;  // shared-memory table slot (alternates between consecutive pieces)
      // this warp's epilogue columns [col0, col0 + HC): output row and multiplier of each, one per lane
      // slot, loaded early so that their latency hides behind the mainloop (read back with shuffles)
      int t_row[TPL];
      float t_mul[TPL];
    };
    int piece_no = 0;
    int gk = 0;  // K block of the next weight stage the mainloop role takes (MXFP8: which scale word)
    auto open_piece = [&](const Piece& pc, Pend& pd) {
      pd.pc = pc;
      tile_rows(pc.tile, pd.e, pd.row0, pd.nrows);
      pd.nt = pc.tile % args.n_tiles;
      pd.ts = piece_no++ & 1;
      if (kSmemTables) {
        if (args.moe) {
          for (int u = 0; u < HC / 32; ++u) {
            const int i = col0 + u * 32 + lane;
            int orow = -1;
            float f = 1.0f;
            if (i < pd.nrows) {
              orow = args.region[(int64_t)pd.e * args.region_cap + pd.row0 + i];
              if (args.topk_w) f = args.topk_w[orow];
            }
            // combine instances keep the routed row's token (its output row) instead of the routed row
            const int key = (COMB && orow >= 0) ? orow / args.comb_k : orow;
            tabs[(pd.ts * 8 + warp) * HC + u * 32 + lane] = make_int2(key, __float_as_int(f));
          }
        }
        return;
      }
#pragma unroll
      for (int u = 0; u < TPL; ++u) {
        const int i = col0 + u * 32 + lane;
        int orow = -1;
        float f = 1.0f;
        if (kTables && (args.moe || PATH == PATH_MXFP4) && i < col0 + HC && i < pd.nrows) {
          int tok;
          if (args.moe) {
            orow = args.region[(int64_t)pd.e * args.region_cap + pd.row0 + i];
            tok = orow / args.topk;
            if (args.topk_w) f = args.topk_w[orow];
          } else {
            orow = pd.row0 + i;
            tok = orow;
          }
          if (PATH == PATH_MXFP4) f *= args.a_scale[tok];
          if (PATH == PATH_NVFP4) f *= args.a_scale[0] * args.w_gscale[pd.e];
        }
        pd.t_row[u] = (COMB && orow >= 0) ? orow / args.comb_k : orow;  // combine: the token
        pd.t_mul[u] = f;
      }
    };
    // mainloop role for the next nblk weight blocks, in ring order
    auto mainloop = [&](int nblk) -> bool {
      for (int k = 0; !(C::NVF && warp >= 4) && k < nblk; ++k) {  // NVFP4 warps 4-7: epilogue only
        if (!waitf(&sh.w_full[ws], wph)) return false;
        uint8_t* wb = wring + ws * C::W_STAGE;
        if (PATH == PATH_INT4) {
          const uint32_t s16 = reinterpret_cast<const uint16_t*>(wb + 8192)[r];
          const uint32_t ss = s16 | (s16 << 16);
          const uint32_t z = args.zp ? (uint32_t)wb[8448 + r] : 8u;
          const uint32_t zz = (0x4300u + z) * 0x00010001u;
          uint4 raw[2];
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
            raw[jj] = *reinterpret_cast<const uint4*>(wb + ((2 * h + jj) * 128 + r) * 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.w_empty[ws]);
          if (!waitf(&sh.aempty[aslot], aslph ^ 1)) return false;
          tc_fence_after();
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            uint32_t out[16];
            const uint32_t wv[4] = {raw[jj].x, raw[jj].y, raw[jj].z, raw[jj].w};
            // pair p of word w4 holds k = 8p + 2 w4 (+1) of the chunk: tensor-memory column 4p + w4
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const uint32_t x = lop3_and_or(wv[w4] >> (4 * p), 0x000F000Fu, 0x43004300u);
                out[p * 4 + w4] = bf16x2_mul(bf16x2_sub(x, zz), ss);
              }
            }
            tmem_st_x<16>(tmem + lane_base + 256 + aslot * 64 + (2 * h + jj) * 16, out);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.afull[aslot]);
          if (++aslot == C::NA) {
            aslot = 0;
            aslph ^= 1;
          }
        } else {
          if (C::NVF && warp < 4) {
            // scale factors -> tensor memory (replicated in every lane quarter)
            const uint32_t sf = tmem + lane_base + 256 + ws * C::SF_STAGE_COLS;
            // lane l's 16 words (4 MMA steps x 4 row groups) are contiguous: four 16-byte loads
            const uint4* wsf = reinterpret_cast<const uint4*>(wb + 16384) + lane * 4;
            uint32_t v[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 q = wsf[j];
              v[4 * j] = q.x;
              v[4 * j + 1] = q.y;
              v[4 * j + 2] = q.z;
              v[4 * j + 3] = q.w;
            }
            tmem_st_x<16>(sf, v);
            if (!waitf(&sh.a_full[as], aph)) return false;
            const uint8_t* asf = aring + as * C::A_STAGE + C::ACT_REGION;
            // one 16-byte load per activation row holds its scales of all four MMA steps (MXFP4: 8 bytes, two e8m0
            // per step, the half of a 16-byte group of two 256-K stages; each pair goes into both halves of its word)
            uint4 rq[C::CB];
#pragma unroll
            for (int cc = 0; cc < C::CB; ++cc) {
              const int j = cc * 32 + lane;
              const int off = (args.moe && !args.grouped) ? (j >> 2) * 128 + (j & 3) * 16 : j * 16;
              if (C::XMX) {
                const uint2 h = *reinterpret_cast<const uint2*>(asf + off + 8 * (gk & 1));
                rq[cc] = make_uint4((h.x & 0xFFFFu) * 0x10001u, (h.x >> 16) * 0x10001u, (h.y & 0xFFFFu) * 0x10001u,
                                    (h.y >> 16) * 0x10001u);
              } else {
                rq[cc] = *reinterpret_cast<const uint4*>(asf + off);
              }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint32_t b[C::CB];
#pragma unroll
              for (int cc = 0; cc < C::CB; ++cc)
                b[cc] = t == 0 ? rq[cc].x : (t == 1 ? rq[cc].y : (t == 2 ? rq[cc].z : rq[cc].w));
              tmem_st_x<C::CB>(sf + 16 + t * C::SFB_STEP, b);
            }
            tmem_wait_st();
            tc_fence_before();
          } else if (C::MX) {
            // the X slot and its scale columns: free once the MMAs of the block NX blocks back completed
            if (!waitf(&sh.x_empty[xs], xph ^ 1)) return false;
            tc_fence_after();
            if (warp < 4) {
              // weight scale factors -> tensor memory (replicated in every lane quarter)
              const uint32_t* wsf = reinterpret_cast<const uint32_t*>(wb + 8192);
              uint32_t v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) v[j] = wsf[j * 32 + lane];
              tmem_st_x<4>(tmem + lane_base + 256 + xs * 4, v);
              if (C::AMX) {
                // MXFP8 activation scales of this stage: token j's four e8m0 bytes (one per 32 K) are word g % 4 of
                // its 16-byte group; token j goes to lane j % 32 of column j / 32 (every lane quarter)
                if (!waitf(&sh.a_full[as], aph)) return false;
                const uint8_t* asf = aring + as * C::A_STAGE + C::ACT_REGION + 4 * (gk & 3);
                uint32_t b[C::CB];
#pragma unroll
                for (int cc = 0; cc < C::CB; ++cc) {
                  const int j = cc * 32 + lane;
                  const int off = (args.moe && !args.grouped) ? (j >> 2) * 128 + (j & 3) * 16 : j * 16;
                  b[cc] = *reinterpret_cast<const uint32_t*>(asf + off);
                }
                tmem_st_x<C::CB>(tmem + lane_base + 256 + 4 * C::NX + xs * C::SFB_STEP, b);
              }
            }
            // all 8 warps: expand packed e2m1 (8 bytes per 16 K) into the padded 16-byte chunks, two chunks of a
            // row per 16-byte load
            uint8_t* xt = xring + xs * C::X_REGION;
#pragma unroll
            for (int q = tid; q < 512; q += 256) {
              const uint4 v = *reinterpret_cast<const uint4*>(wb + q * 16);
              const int rr = q >> 2, cc = (q & 3) * 2;
              uint8_t* row = xt + (rr >> 3) * 1024 + (rr & 7) * 128;
              *reinterpret_cast<uint4*>(row + ((cc ^ (rr & 7)) << 4)) = make_uint4(v.x, v.y, 0u, 0u);
              *reinterpret_cast<uint4*>(row + (((cc + 1) ^ (rr & 7)) << 4)) = make_uint4(v.z, v.w, 0u, 0u);
            }
            fence_proxy_async_smem();
            if (warp < 4) {
              tmem_wait_st();
              tc_fence_before();
            }
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sh.ready[C::MX ? xs : ws]);
            mbar_arrive(&sh.w_empty[ws]);
            if (C::NVF || (C::AMX && warp < 4)) mbar_arrive(&sh.a_empty[as]);
          }
          if (C::MX && ++xs == C::NX) {
            xs = 0;
            xph ^= 1;
          }
          ++gk;
          if (C::NVF || C::AMX) {
            if (++as == C::SA) {
              as = 0;
              aph ^= 1;
            }
          }
        }
        if (++ws == C::SW) {
          ws = 0;
          wph ^= 1;
        }
      }
      return ok;
    };
    auto epilogue = [&](const Pend& pd) -> bool {
      const Piece& pc = pd.pc;
      const int e = pd.e, row0 = pd.row0, nrows = pd.nrows, nt = pd.nt;
      const int* t_row = pd.t_row;
      const float* t_mul = pd.t_mul;
      // ---------------------------------------------------- epilogue
      if (kSmemTables) __syncwarp();  // the piece's table entries were written by the warp's other lanes
      if (!waitf(&sh.dfull, pidx & 1)) return false;
      tc_fence_after();
      // This warp's whole column range goes to registers first: tensor memory is handed back to the next
      // tile's MMAs before any global store is issued.
      constexpr int CHUNK = HC < 16 ? HC : 16;
      uint32_t v[HC];
      // columns past the tile's last token hold padding: up to 64 columns per warp their chunks are neither read nor
      // stored (a cut tile's partial sums are stored whole); the 128-column slices of 256-token tiles keep the
      // straight-line code, whose registers the guards would spill
      const int live = (HC <= 64 && pc.full) ? nrows - col0 : HC;  // warp-uniform
#pragma unroll
      for (int cb = 0; cb < HC; cb += CHUNK) {
        if (cb < live) {
          if (CHUNK == 16) tmem_ld16(tmem + lane_base + col0 + cb, *reinterpret_cast<uint32_t(*)[16]>(v + cb));
          else tmem_ld8(tmem + lane_base + col0 + cb, *reinterpret_cast<uint32_t(*)[8]>(v + cb));
        }
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.dempty);
      const int n = nt * TILE_N + r;
      const float bias_v = (args.bias && n < args.N) ? bf16_to_f32(args.bias[n]) : 0.0f;
      float* part = args.partials + ((int64_t)pc.slot * BT) * TILE_N;
      // Dense INT4 / NVFP4 rows need no table.  Otherwise col is warp-uniform and the entry comes from
      // lane (col - col0) % 32, slot (col - col0) / 32 (slot chosen by selects, so the table stays in registers).
      const bool use_table = kTables && (args.moe || PATH == PATH_MXFP4);
      const float dense_mul = PATH == PATH_NVFP4 ? args.a_scale[0] * args.w_gscale[e] : 1.0f;
      // output row (-1: padding column) and multiplier of token column col
      auto lookup = [&](int col, int& orow, float& mul) {
        if (kSmemTables && use_table) {
          const int2 t = tabs[(pd.ts * 8 + warp) * HC + (col - col0)];
          orow = t.x;
          mul = __int_as_float(t.y);
        } else if (use_table) {
          const int rel = col - col0;
          const int slot = rel >> 5;
          int tr = t_row[0];
          float tm = t_mul[0];
#pragma unroll
          for (int u = 1; u < TPL; ++u)
            if (slot == u) {
              tr = t_row[u];
              tm = t_mul[u];
            }
          orow = __shfl_sync(0xffffffffu, tr, rel & 31);
          mul = __shfl_sync(0xffffffffu, tm, rel & 31);
        } else {
          orow = col < nrows ? row0 + col : -1;
          mul = dense_mul;
        }
      };
      auto store = [&](int col, float acc) {
        int orow;
        float mul;
        lookup(col, orow, mul);
#if HQ_DEBUG_BOUNDS
        orow = dbg_row(orow, args.dbg_c_rows, args.status);
#endif
        if (orow >= 0 && n < args.N) args.c[(int64_t)orow * args.N + n] = f32_to_bf16(acc * mul + bias_v);
      };
      const bool pair_ok = (args.N & 1) == 0 && (reinterpret_cast<uintptr_t>(args.c) & 3) == 0;
#if HQ_DEBUG_BOUNDS
      if (!pc.full && !dbg_span((int64_t)(pc.slot + 1) * BT * TILE_N, args.dbg_part_elems, args.status)) {
        ++pidx;
        return ok;
      }
#endif
      if (!pc.full) {
#pragma unroll
        for (int j = 0; j < HC; ++j) part[(col0 + j) * TILE_N + r] = __uint_as_float(v[j]);
      } else if (COMB) {
        // MoE combine: the routed row's values (x top-k weight) are added into its token's fp32 row; the table holds
        // the token of each column.  N % 4 == 0: a quad of lanes (4 adjacent output features) transposes its 4 x 4
        // accumulators of 4 token columns in two shuffle rounds; then lane b0 + 2 b1 of the quad holds the 4
        // features of column j + b0 + 2 b1, looks up that column's token and top-k weight itself, and adds the 4
        // outputs with one 16-byte reduction.
        const bool quad = (args.N & 3) == 0;
        const int b0 = lane & 1, b1 = (lane >> 1) & 1, tc = b0 + 2 * b1;
        const int n4 = n & ~3;
        float bq[4];  // bias of the quad's 4 features
#pragma unroll
        for (int i = 0; i < 4; ++i) bq[i] = __shfl_sync(0xffffffffu, bias_v, (lane & ~3) + i);
#pragma unroll
        for (int j = 0; j < HC; j += 4) {
          if (j >= live) continue;
          if (quad) {
            const float o0 = __uint_as_float(v[j]), o1 = __uint_as_float(v[j + 1]), o2 = __uint_as_float(v[j + 2]),
                        o3 = __uint_as_float(v[j + 3]);
            // round 1 (lane ^ 1): tokens b0 and b0 + 2, rows 2 b1 and 2 b1 + 1 of the quad
            const float r1a = __shfl_xor_sync(0xffffffffu, b0 ? o0 : o1, 1);
            const float r1b = __shfl_xor_sync(0xffffffffu, b0 ? o2 : o3, 1);
            const float ta0 = b0 ? r1a : o0, ta1 = b0 ? o1 : r1a;  // token b0
            const float tb0 = b0 ? r1b : o2, tb1 = b0 ? o3 : r1b;  // token b0 + 2
            // round 2 (lane ^ 2): token b0 + 2 b1, rows 0..3 of the quad
            const float s0 = __shfl_xor_sync(0xffffffffu, b1 ? ta0 : tb0, 2);
            const float s1 = __shfl_xor_sync(0xffffffffu, b1 ? ta1 : tb1, 2);
            const float x0 = b1 ? s0 : ta0, x1 = b1 ? s1 : ta1, x2 = b1 ? tb0 : s0, x3 = b1 ? tb1 : s1;
            int tok;
            float mul;
            lookup(col0 + j + tc, tok, mul);  // j % 4 == 0: the lanes' columns share one 32-column table slot
#if HQ_DEBUG_BOUNDS
            tok = dbg_row(tok, args.dbg_comb_rows, args.status);
#endif
            if (tok >= 0 && n4 < args.N)
              red_add_v4_f32(args.comb + (int64_t)tok * args.N + n4, x0 * mul + bq[0], x1 * mul + bq[1],
                             x2 * mul + bq[2], x3 * mul + bq[3]);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              int tok;
              float mul;
              lookup(col0 + j + c, tok, mul);  // all lanes: the lookup shuffles
#if HQ_DEBUG_BOUNDS
              tok = dbg_row(tok, args.dbg_comb_rows, args.status);
#endif
              if (tok >= 0 && n < args.N)
                red_add_f32(args.comb + (int64_t)tok * args.N + n, __uint_as_float(v[j + c]) * mul + bias_v);
            }
          }
        }
      } else if (use_table && pair_ok) {
        // Table rows (MoE, MXFP4), even N: the pair exchange of the dense case below, each token column with its
        // own output row and multiplier.
        const bool odd = lane & 1;
        const int n_even = n & ~1;
#pragma unroll
        for (int j = 0; j < HC; j += 2) {
          if (j >= live) continue;
          const int col = col0 + j;
          int orow0, orow1;
          float mul0, mul1;
          lookup(col, orow0, mul0);
          lookup(col + 1, orow1, mul1);
#if HQ_DEBUG_BOUNDS
          orow0 = dbg_row(orow0, args.dbg_c_rows, args.status);
          orow1 = dbg_row(orow1, args.dbg_c_rows, args.status);
#endif
          const uint32_t pk = pack_bf16x2(__uint_as_float(v[j]) * mul0 + bias_v,
                                          __uint_as_float(v[j + 1]) * mul1 + bias_v);  // lo: col, hi: col+1
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? (pk & 0xFFFFu) : (pk >> 16), 1);
          const uint32_t out = odd ? (recv | (pk & 0xFFFF0000u)) : ((pk & 0xFFFFu) | (recv << 16));
          const int orow = odd ? orow1 : orow0;
          if (orow >= 0 && n_even < args.N)
            *reinterpret_cast<uint32_t*>(args.c + (int64_t)orow * args.N + n_even) = out;
        }
      } else if (!use_table && pair_ok) {
        // Dense rows, even N: lanes 2i and 2i+1 swap one value per pair of tokens, so that every lane writes
        // two adjacent outputs (n, n+1) of one token with a single 4-byte store: the even lane token col, the
        // odd lane token col + 1.
        const bool odd = lane & 1;
        const int n_even = n & ~1;
#pragma unroll
        for (int j = 0; j < HC; j += 2) {
          if (j >= live) continue;
          const int col = col0 + j;
          const uint32_t pk = pack_bf16x2(__uint_as_float(v[j]) * dense_mul + bias_v,
                                          __uint_as_float(v[j + 1]) * dense_mul + bias_v);  // lo: col, hi: col+1
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? (pk & 0xFFFFu) : (pk >> 16), 1);
          const uint32_t out = odd ? (recv | (pk & 0xFFFF0000u)) : ((pk & 0xFFFFu) | (recv << 16));
          const int tok = col + (odd ? 1 : 0);
#if HQ_DEBUG_BOUNDS
          if (tok < nrows && dbg_row(row0 + tok, args.dbg_c_rows, args.status) < 0) continue;
#endif
          if (tok < nrows && n_even < args.N)
            *reinterpret_cast<uint32_t*>(args.c + (int64_t)(row0 + tok) * args.N + n_even) = out;
        }
      } else {
#pragma unroll
        for (int j = 0; j < HC; ++j) {
          if (j >= live) continue;
          store(col0 + j, __uint_as_float(v[j]));
        }
      }
      ++pidx;
      return ok;
    };
    // A piece's epilogue runs after the first blocks of the next piece are prepared, so that the MMA finds
    // them ready as soon as the accumulator is released.  No more than the slots the previous piece's MMAs free
    // (the next ones free only after the accumulator): A slots but one (INT4), the X ring (MXFP4), weight stages
    // but one (NVFP4).
    constexpr int PREFILL = PATH == PATH_INT4 ? C::NA - 1 : (C::MX ? C::NX : C::SW - 1);
    Pend prev;
    bool has_prev = false;
    for_each_piece(sched, [&](const Piece& pc) {
      if (!ok) return;
      Pend cur;
      open_piece(pc, cur);
      const int nblk = pc.g1 - pc.g0;
      const int pre = nblk < PREFILL ? nblk : PREFILL;
      gk = pc.g0;
      if (!mainloop(pre)) return;
      if (has_prev && !epilogue(prev)) return;
      if (!mainloop(nblk - pre)) return;
      prev = cur;
      has_prev = true;
    });
    if (ok && has_prev) epilogue(prev);
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Launch one instance: token tile BT, combine epilogue or not.
template <int PATH, int BT, bool COMB>
cudaError_t launch_umma_bt(const GemmArgs& a, int grid, cudaStream_t stream) {
  using C = Cfg<PATH, BT>;
  void (*kernel)(GemmArgs) = hq_gemm_kernel<PATH, BT, COMB>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  return launch_kernel(kernel, dim3(grid), dim3(NUM_THREADS), C::SMEM_BYTES, stream, a);
}

template <int PATH, bool COMB>
cudaError_t launch_umma(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  switch (bt) {
    case 16: return launch_umma_bt<PATH, 16, COMB>(a, grid, stream);
    case 32: return launch_umma_bt<PATH, 32, COMB>(a, grid, stream);
    case 64: return launch_umma_bt<PATH, 64, COMB>(a, grid, stream);
    case 128: return launch_umma_bt<PATH, 128, COMB>(a, grid, stream);
    case 256: return launch_umma_bt<PATH, 256, COMB>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hq
