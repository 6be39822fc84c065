// Small-token weight-streaming path for the integer and FP8 weight formats (dense and MoE).
//
// With at most 32 tokens per tile the UMMA path is limited by its fixed cost
// per 128 x 16 instruction, not by the bytes it moves, so this kernel decodes
// in registers and feeds the warp-level tensor-core instruction (mma.sync
// m16n8k16, bf16 x bf16 -> fp32), in the spirit of the multistage copy + MMA
// pipeline that the Humming announcement reports to beat TMA + UMMA at small
// batch ("Tuning and JIT compilation per workload").  It is also the one
// kernel for the formats the tcgen05 kernel does not decode (INT8, UINT1/2/3,
// MXINT4, FP8 E4M3 weights): there it serves every token count, with 32-token
// tiles beyond 16 tokens.
//
// It reads packed weight blocks of 128 rows x 128 K (see hq_layout.h), whose
// code order makes one ldmatrix.x4 deliver a warp's A-fragment words: every
// register holds (even k, odd k) pairs of one row that the lane feeds to MMA
// steps.  A pair becomes bf16x2 exactly:
//   4/2/1-bit ints      one shift, one mask-and-or (the bf16 of 128 + q) and one
//                       bf16x2 subtraction of 128 + z
//   3-bit ints          two mask-and-ors (low two bits, then the top bit from
//                       the 1-bit plane) and one subtraction
//   8-bit ints          two mask-and-ors (128 + low 7 bits; 128, or 256 when the
//                       sign bit is set) and one subtraction
//   e4m3                cvt to f16x2 (exact), the f16 bits moved into bf16 fields
//                       (value 2^-112 times as large), one multiplication by 2^112
// The MMAs of one quantization group accumulate into fp32 temporaries that are
// added to the running sums times the group scale once per group (a 128-K
// block; a 32-K chunk for MXINT4): the weights the MMAs see are exact and the
// scale costs one FMA per accumulator per group.
//
// Warp roles (288 threads; two CTAs per SM up to 16-token tiles):
//   warps 0-7  compute: warp (rg, kh) owns rows 32rg .. 32rg+31 of the 128-row
//              tile as two 16-row MMA tiles and K half kh of every block; the
//              two K halves meet in shared memory at the end of each piece,
//              after which warp (rg, kh) finishes 16-row half kh (fix-up
//              polls and epilogue on all 8 warps).
//              MMAs on 8-token column tiles that hold no token of the tile are
//              predicated off.
//   warp 8     producer (one thread): per block one bulk copy of the weights
//              plus the TMA box (dense, grouped MoE) or gather4 (indexed MoE)
//              of the token tile, all on one barrier.
//
// Stream-K without a second kernel: the (tile, block) iterations are dealt out
// evenly to the CTAs.  A tile cut between CTAs is finished by the CTA that
// holds its first block (its last piece, so it ends last).  The CTAs holding
// the rest leave their partial sums (their first or only piece) in one slot per
// CTA as 64-bit words (fp32 value, epoch), written with relaxed gpu-scope
// stores; the finishing CTA polls its values until every tag equals the call's
// epoch (bounded) and adds them.  An aligned 64-bit access is single-copy
// atomic, so each value carries its own proof of arrival: no flag, no fence.
// The epoch is one more than the previous call's on the same workspace
// (header word 1); the last CTA to exit stores it there, so a value left by an
// earlier call, even one that stopped on an error, never matches.
#pragma once
#include "hq_gemm_kernel.cuh"
#include "hq_launch.h"

namespace hq {

constexpr int SM_THREADS = 288;
constexpr int SM_PROD_WARP = 8;
constexpr int SM_MAX_STAGES = 24;
constexpr int SM_FUSED_ROWS = 512;  // routed rows up to which a MoE call routes inside this kernel

// Per decode variant: bytes of a packed block and where its scales / zero points sit.
template <int DEC>
struct DecCfg {
  static constexpr int BLK = DEC == DEC_INT4     ? 8576
                             : DEC == DEC_MXINT4 ? 8704
                             : DEC == DEC_UINT2  ? 4480
                             : DEC == DEC_UINT1  ? 2432
                             : DEC == DEC_UINT3  ? 6528
                                                 : 16640;
  static constexpr int SOFF = DEC == DEC_INT8 || DEC == DEC_E4M3 ? 16384
                              : DEC == DEC_UINT2                 ? 4096
                              : DEC == DEC_UINT1                 ? 2048
                              : DEC == DEC_UINT3                 ? 6144
                                                                 : 8192;
  static constexpr int ZOFF = SOFF + 256;
  static constexpr bool ZP_ALWAYS = DEC == DEC_UINT2 || DEC == DEC_UINT1 || DEC == DEC_UINT3;
  static constexpr int PLANE1 = DEC == DEC_UINT3 ? 4096 : 0;  // the 1-bit plane (UINT1 codes, UINT3 bit 2)
};

template <int BT, int DEC>
struct SmallCfg {
  static constexpr int CTAS_PER_SM = BT <= 16 ? 2 : 1;  // 32-token tiles need more registers than two CTAs allow
  static constexpr int ACT_BYTES = 2 * BT * 128;         // two 64-K 128-byte-swizzled atoms (1 KB aligned)
  static constexpr int W_OFF = ACT_BYTES;                // then the weight block
  static constexpr int STAGE = ((ACT_BYTES + DecCfg<DEC>::BLK + 1023) / 1024) * 1024;
  static constexpr int RING = CTAS_PER_SM == 2 ? 96 * 1024 : 192 * 1024;
  static constexpr int STAGES = RING / STAGE > SM_MAX_STAGES ? SM_MAX_STAGES : RING / STAGE;
  static constexpr int NT = BT / 8;                          // 8-token MMA column tiles
  static constexpr int FIX_G = BT == 8 ? 6 : 2;  // contributors polled together (Stream-K fix-up)
  static constexpr int RED_BYTES = 4 * 2 * 32 * NT * 4 * 4;  // K-half exchange: [rg][kh][lane][nt][4] floats
  static constexpr int OFF_SH = STAGES * STAGE;
  static constexpr int OFF_PREFIX = OFF_SH + 1024;           // MoE tile prefix: E + 1 ints (E <= 512)
  static constexpr int OFF_ROUTE = OFF_PREFIX + 2112;         // fused routing: row offsets [E + 1], rows [512]
  static constexpr int OFF_RED = OFF_ROUTE + 2112 + 4 * SM_FUSED_ROWS;
  static constexpr int SMEM_BYTES = OFF_RED + RED_BYTES + 1024 /*alignment*/;
  static_assert(CTAS_PER_SM * (SMEM_BYTES + 1024) <= 228 * 1024, "CTAs per SM");
  static_assert(STAGES >= 4, "ring");
  static_assert(RED_BYTES >= 1024 * 4, "fused routing scratch: 512 counts + 512 ids");
};

struct SmallSmem {
  uint64_t full[SM_MAX_STAGES];
  uint64_t empty[SM_MAX_STAGES];
  uint64_t epi_bar;    // the 8 compute warps (K-half exchange), bounded
  uint64_t epoch_bar;  // the producer thread stored this call's epoch
  int abort_flag;
  int tile_prefix_total;
  uint32_t epoch;
};
static_assert(sizeof(SmallSmem) <= 1024, "shared state");

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d = a * b (zero accumulator input)
__device__ __forceinline__ void mma_bf16_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
// The same two under a warp-uniform guard `on` (a predicated instruction, not a branch: no reconvergence point).
__device__ __forceinline__ void mma_bf16_16816_if(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                                  uint32_t on) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %10, 0;\n\t"
      "@p mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n\t}\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(on));
}
__device__ __forceinline__ void mma_bf16_16816_z_if(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                                    uint32_t on) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %10, 0;\n\t"
      "@p mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%11,%11,%11,%11};\n\t}\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(on), "f"(0.0f));
}

// ---------------------------------------------------------------- pair decoders (exact, bf16x2)
// (q - z) of the 4-bit pair at nibble slots (0, 4) of x: the bf16 of 128 + q minus zz = the bf16 of 128 + z
__device__ __forceinline__ uint32_t dec_u4(uint32_t x, uint32_t zz) {
  return bf16x2_sub(lop3_and_or(x, 0x000F000Fu, 0x43004300u), zz);
}
// (q - z) of the 2-bit pair at bits (0-1, 16-17) of x
__device__ __forceinline__ uint32_t dec_u2(uint32_t x, uint32_t zz) {
  return bf16x2_sub(lop3_and_or(x, 0x00030003u, 0x43004300u), zz);
}
// (q - z) of the 1-bit pair at bits (0, 16) of x
__device__ __forceinline__ uint32_t dec_u1(uint32_t x, uint32_t zz) {
  return bf16x2_sub(lop3_and_or(x, 0x00010001u, 0x43004300u), zz);
}
// (q - z) of the 3-bit pair whose low two bits sit at bits (0-1, 16-17) of lo and whose top bit at bits (2, 18) of hi
__device__ __forceinline__ uint32_t dec_u3(uint32_t lo, uint32_t hi, uint32_t zz) {
  return bf16x2_sub(lop3_and_or(hi, 0x00040004u, lop3_and_or(lo, 0x00030003u, 0x43004300u)), zz);
}
// two's complement bytes at bits 0-7 and 16-23 of x: (128 + (b & 127)) - (128 or 256 when b's sign bit is set)
__device__ __forceinline__ uint32_t dec_i8(uint32_t x) {
  return bf16x2_sub(lop3_and_or(x, 0x007F007Fu, 0x43004300u), lop3_and_or(x, 0x00800080u, 0x43004300u));
}
// two e4m3 bytes (low byte = low half): cvt to f16x2 (exact; every e4m3 value is a normal f16 or zero), the f16
// exponent and top mantissa bits moved into the bf16 fields (the bf16 value is the f16 value times 2^-112, a
// normal bf16), then times 2^112 (exact)
__device__ __forceinline__ uint32_t dec_e4m3(uint32_t two_bytes) {
  uint32_t h;
  asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}\n" : "=r"(h) : "r"(two_bytes));
  const uint32_t t = lop3_and_or(h >> 3, 0x0FFF0FFFu, 0u) | (h & 0x80008000u);
  return bf16x2_mul(t, 0x77807780u);
}
// e8m0 byte -> its fp32 value 2^(b - 127) (b = 0: 2^-127, a subnormal; 0xFF: NaN)
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  return __uint_as_float(b == 0u ? 0x00400000u : (b == 255u ? 0x7FC00000u : (b << 23)));
}

// Routing of a small MoE call, built by every CTA in its own shared memory: the routed rows (t * topk + j) grouped
// by expert in increasing row order (a stable counting sort: the same lists in every CTA, which Stream-K needs, as
// the pieces of one tile run on different CTAs).  off[e] .. off[e + 1] index expert e's rows in `rows`; cnt[e]
// receives the counts (cnt: 1024 ints of scratch, the ids are staged in its upper half).  An id outside [0, E) routes
// nothing and records HQ_ERR_BAD_ROUTING.  Every thread calls it.
__device__ __forceinline__ void fused_route(const int32_t* ids, int nrows, int E, int* cnt, int* off, int* rows,
                                            int* status) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  int* ids_s = cnt + 512;  // the ids, read from global memory once
  for (int r = tid; r < nrows; r += blockDim.x) {
    const int e = ids[r];
    ids_s[r] = e;
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else bad = true;
  }
  if (bad) atomicCAS(status, 0, ERR_BAD_ROUTING);
  __syncthreads();
  if (tid < 32) {  // exclusive scan of the counts (one warp), then cnt becomes each expert's insertion cursor
    const int per = (E + 31) / 32;
    int run = 0;
    for (int i = 0; i < per; ++i)
      if (lane * per + i < E) run += cnt[lane * per + i];
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int acc = incl - run;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        off[e] = acc;
        acc += cnt[e];
        cnt[e] = off[e];
      }
    }
    if (lane == 31) off[E] = incl;
    __syncwarp();
    // rows in increasing order, 32 at a time: rank within the chunk among lanes of the same expert
    for (int r0 = 0; r0 < nrows; r0 += 32) {
      const int r = r0 + lane;
      const int e = r < nrows ? ids_s[r] : -1;
      const bool valid = e >= 0 && e < E;
      const unsigned same = __match_any_sync(0xffffffffu, valid ? e : -1);
      const int rank = __popc(same & ((1u << lane) - 1u));
      const int base = valid ? cnt[e] : 0;
      __syncwarp();
      if (valid) rows[base + rank] = r;
      if (valid && rank == __popc(same) - 1) cnt[e] = base + rank + 1;  // the group's last lane moves the cursor
      __syncwarp();
    }
    // restore the counts
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) cnt[e] = off[e + 1] - off[e];
    }
  }
  __syncthreads();
}

// Routing of at most 32 routed rows (decode-size calls) without a histogram: warp 0 reads the ids (one per lane),
// groups equal experts (__match_any_sync), places each row at (routed rows of smaller experts) + (its rank among the
// rows of its expert), the order fused_route produces, and lists the distinct experts with their token tiles; then
// every thread fills the per-expert row offsets off[0..E] and the tile prefix prefix[0..E] from those 32 entries.
// scratch: 96 ints.  Every thread calls it (two __syncthreads).
__device__ __forceinline__ void fused_route_small(const int32_t* ids, int nrows, int E, int bt, int region_cap,
                                                  int* off, int* rows, int* prefix, int* total, int* scratch,
                                                  int* status) {
  const int tid = threadIdx.x, lane = tid & 31;
  int* ids_s = scratch;           // expert of routed row j, or -1
  int* dist_e = scratch + 32;     // distinct expert held by lane j (the lowest lane of its rows), or -1
  int* dist_t = scratch + 64;     // its token tiles
  if (tid < 32) {
    const int e = lane < nrows ? ids[lane] : -1;
    const bool valid = e >= 0 && e < E;
    if (lane < nrows && !valid) atomicCAS(status, 0, ERR_BAD_ROUTING);
    const unsigned same = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);  // invalid rows stay alone
    const int rank = __popc(same & ((1u << lane) - 1u));
    const int ev = valid ? e : 0x7FFFFFFF;
    int below = 0;  // valid routed rows of smaller experts
#pragma unroll 8
    for (int j = 0; j < 32; ++j) below += __shfl_sync(0xffffffffu, ev, j) < ev ? 1 : 0;
    if (valid) rows[below + rank] = lane;
    const bool lead = valid && __ffs(same) - 1 == lane;
    int cnt = __popc(same);
    cnt = cnt > region_cap ? region_cap : cnt;
    const int tiles = lead ? (cnt + bt - 1) / bt : 0;
    ids_s[lane] = valid ? e : -1;
    dist_e[lane] = lead ? e : -1;
    dist_t[lane] = tiles;
    int sum = tiles;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) *total = sum;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) {
    int o = 0, t = 0;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const int ej = ids_s[j], dj = dist_e[j];
      o += (ej >= 0 && ej < e) ? 1 : 0;
      t += (dj >= 0 && dj < e) ? dist_t[j] : 0;
    }
    off[e] = o;
    prefix[e] = t;
  }
  __syncthreads();
}

template <int BT, int DEC>
__global__ void __launch_bounds__(SM_THREADS, SmallCfg<BT, DEC>::CTAS_PER_SM)
    hq_gemm_small_kernel(const __grid_constant__ GemmArgs args) {
  using C = SmallCfg<BT, DEC>;
  using D = DecCfg<DEC>;
  constexpr int NT = C::NT;
  extern __shared__ uint8_t smem_raw[];
  // 1 KB aligned, by pointer arithmetic on the shared array so that accesses stay shared-memory loads
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  SmallSmem& sh = *reinterpret_cast<SmallSmem*>(smem + C::OFF_SH);
  int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = tid == SM_PROD_WARP * 32;

  // Dense calls: the producer thread issues the weight copies of its first ring stages before the grid
  // dependency wait (packed weights are read-only inputs, see hq_launch.h), so that they stream while the
  // previous kernel drains; the activation boxes of those stages follow right after the wait.
  int npre = 0;                            // producer thread: stages whose weight copy is in flight
  int pre_x[C::STAGES], pre_y[C::STAGES];  // their activation box coordinates (K element, first row)
  if (producer) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 8);
    }
    mbar_init(&sh.epi_bar, 8);
    mbar_init(&sh.epoch_bar, 1);
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
            if (args.w_evict_first)
              bulk_g2s_hint(smem + npre * C::STAGE + C::W_OFF, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk,
                            &sh.full[npre], l2_evict_first_policy());
            else
              bulk_g2s(smem + npre * C::STAGE + C::W_OFF, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk,
                       &sh.full[npre]);
            pre_x[npre] = g * 128;
            pre_y[npre] = (pc.tile / args.n_tiles) * BT;
          }
        });
    }
  }
  pdl_trigger();
  // No global memory a previous kernel may write is touched before griddepcontrol.wait (weights aside).  MoE
  // tiles depend on the routing tables, so MoE calls wait here; dense calls set everything up first and wait only
  // where they first touch such memory: the producer before its activation loads, the compute warps before their
  // first epilogue, every thread before the exit count.
  // fused routing: the CTA's own copy of the per-expert row lists (counts in the red area until the prefix is
  // taken: the exchange buffer is not in use yet)
  int* r_off = reinterpret_cast<int*>(smem + C::OFF_ROUTE);
  int* r_rows = r_off + 528;
  const bool fused = args.ids != nullptr;
  uint32_t epoch_prev = 0;  // producer: header word 1 (MoE calls read it before routing, hiding the load)
  if (args.moe) {
    pdl_wait();
    if (producer) epoch_prev = reinterpret_cast<volatile uint32_t*>(args.status)[1];
    const int* counts = args.counts;
    if (fused && args.fused_rows <= 32) {
      fused_route_small(args.ids, args.fused_rows, args.E, BT, args.region_cap, r_off, r_rows, prefix,
                        &sh.tile_prefix_total, reinterpret_cast<int*>(smem + C::OFF_RED), args.status);
    } else {
      if (fused) {
        int* cnt = reinterpret_cast<int*>(smem + C::OFF_RED);
        fused_route(args.ids, args.fused_rows, args.E, cnt, r_off, r_rows, args.status);
        counts = cnt;
      }
      moe_tile_prefix(counts, args.E, args.region_cap, BT, prefix, &sh.tile_prefix_total);
    }
  }
  __syncthreads();
  if (producer) {
    pdl_wait();
    for (int s = 0; s < npre; ++s)
#pragma unroll
      for (int j = 0; j < 2; ++j)
        tma_load_2d(smem + s * C::STAGE + j * (BT * 128), &args.tmap_a, pre_x[s] + j * 64, pre_y[s], &sh.full[s]);
    // the workspace epoch is needed only when a partial sum is published or collected
    sh.epoch = (args.moe ? epoch_prev : reinterpret_cast<volatile uint32_t*>(args.status)[1]) + 1u;
    mbar_arrive(&sh.epoch_bar);
  }
  const int total_tiles = args.moe ? sh.tile_prefix_total * args.n_tiles : args.m_tiles * args.n_tiles;
  Sched sched;
  sched.init(total_tiles, args.kst, (int)gridDim.x, (int)blockIdx.x, args.sk);
  const bool active = (int)blockIdx.x < sched.P && total_tiles > 0;
  volatile int* abort_flag = &sh.abort_flag;
  auto fail = [&](int code) {
    *abort_flag = 1;
    pdl_wait();
    atomicCAS(args.status, 0, code);
  };
  // routed row (t * topk + j) number i of expert e
  auto routed_row = [&](int e, int i) -> int {
    return fused ? r_rows[r_off[e] + i] : args.region[(int64_t)e * args.region_cap + i];
  };
  auto tile_rows = [&](int tile, int& e, int& row0, int& nrows) {
    const int mt = tile / args.n_tiles;
    if (args.moe) {
      int lm;
      moe_locate(prefix, args.E, mt, e, lm);
      int cnt = fused ? r_off[e + 1] - r_off[e] : args.counts[e];
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
      int blk = 0;         // blocks of this CTA so far (the first npre were issued at the start)
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
            rows_tok[i] = i < nrows ? routed_row(e, row0 + i) / args.topk : args.M;
        const uint8_t* wblk = args.w + e * args.w_expert_bytes + ((int64_t)nt * args.kst) * args.w_blk;
        for (int g = pc.g0; g < pc.g1; ++g, ++blk) {
          uint8_t* act = smem + st * C::STAGE;
          if (blk >= npre) {
            if (!mbar_wait(&sh.empty[st], ph ^ 1, abort_flag, args.wait_ns)) {
              fail(ERR_TIMEOUT);
              ok = false;
              return;
            }
            mbar_arrive_expect_tx(&sh.full[st], (uint32_t)args.w_blk + C::ACT_BYTES);
            if (args.w_evict_first)
              bulk_g2s_hint(act + C::W_OFF, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk, &sh.full[st],
                            l2_evict_first_policy());
            else
              bulk_g2s(act + C::W_OFF, wblk + (int64_t)g * args.w_blk, (uint32_t)args.w_blk, &sh.full[st]);
            if (!args.moe || args.grouped) {
#pragma unroll
              for (int j = 0; j < 2; ++j)
                tma_load_2d(act + j * (BT * 128), &args.tmap_a, g * 128 + j * 64, rbase, &sh.full[st]);
            } else {
#pragma unroll
              for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int i = 0; i < BT; i += 4)
                  tma_gather4(act + j * (BT * 128) + (i >> 3) * 1024 + (i & 7) * 128, &args.tmap_a,
                              g * 128 + j * 64, rows_tok[i], rows_tok[i + 1], rows_tok[i + 2], rows_tok[i + 3],
                              &sh.full[st]);
            }
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
    const int rg = warp & 3, kh = warp >> 2;
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint32_t smem_s = smem_u32(smem);
    // ldmatrix row addresses (weights; relative to the stage's weight block).  lane L gives row L % 16 of the
    // 16-row MMA tile (UINT1/2/3: row L of the warp's 32 rows) in the chunk the variant's matrices name.
    uint32_t w_lane;
    if (DEC == DEC_INT4 || DEC == DEC_MXINT4) w_lane = ((2 * kh + (lane >> 4)) * 128 + 32 * rg + (lane & 15)) * 16;
    else if (DEC == DEC_UINT2 || DEC == DEC_UINT3) w_lane = (kh * 128 + 32 * rg + lane) * 16;
    else if (DEC == DEC_UINT1) w_lane = (32 * rg + lane) * 16;
    else w_lane = ((4 * kh + (lane >> 4)) * 128 + 32 * rg + (lane & 15)) * 16;
    // the 1-bit plane: rows 32 rg + lane, both K halves in one 16-byte row (UINT1 codes, UINT3 bit 2)
    const uint32_t w_lane1 = (uint32_t)D::PLANE1 + (uint32_t)(32 * rg + lane) * 16;
    const uint32_t kh_shift = 8u * (uint32_t)kh;  // this warp's pairs of the 1-bit plane start at bit 8 kh
    // this lane's rows g8, g8 + 8 of both 16-row tiles: scale and zero-point offsets in the block
    uint32_t s_off[2][2], z_off[2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = 32 * rg + 16 * m + 8 * rr + g8;
        s_off[m][rr] = C::W_OFF + D::SOFF + (DEC == DEC_MXINT4 ? 4 * row + 2 * kh : 2 * row);
        z_off[m][rr] = C::W_OFF + D::ZOFF + row;
      }
    const bool zp = args.zp != 0;
    // Activations (atom kh of the stage, 128-byte swizzle): lane L gives token row tok of 8x8 matrix L / 8.
    int a_tok, a_chunk;  // token row and 16-byte chunk offset (relative to the step's first chunk)
    if (BT == 8) {
      a_tok = lane & 7;
      a_chunk = lane >> 3;  // matrices: chunks 2s, 2s+1, 2s+2, 2s+3 (two K steps)
    } else {
      a_tok = ((lane >> 4) << 3) + (lane & 7);  // matrices: (tokens 0-7 | 8-15) x (chunk 2s | 2s+1)
      a_chunk = (lane >> 3) & 1;
    }
    // The swizzled chunk (2s + a_chunk) ^ (tok & 7) splits into a per-lane base and a per-step XOR, because the
    // bits of a_chunk (bit 0; bits 0-1 for 8-token tiles) and of 2s (bits 1-2; bit 2) do not overlap.
    constexpr uint32_t LO = BT == 8 ? 3u : 1u;
    const uint32_t a_row = (uint32_t)(kh * (BT * 128) + (a_tok >> 3) * 1024 + (a_tok & 7) * 128) +
                           (((uint32_t)a_chunk ^ ((uint32_t)a_tok & LO)) << 4);
    const uint32_t a_sw = ((uint32_t)a_tok & 7u & ~LO) << 4;
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);  // [rg][lane][m][NT][4]
    uint32_t epi_phase = 0;
    // CTA-level sync of the 8 compute warps on an mbarrier (bounded, abort-aware: never a hang)
    auto epi_sync = [&]() {
      __syncwarp();
      mbar_arrive_if(&sh.epi_bar, lane == 0);
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
      const int nn = (nrows + 7) >> 3;  // 8-token column tiles holding tokens of this tile (warp-uniform)
      float acc[2][NT][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[m][i][j] = 0.0f;
      // output row and multiplier of this lane's token columns (i*8 + 2t, +1), loaded now so that their
      // latency hides behind the mainloop
      int t_row[NT][2];
      float t_mul[NT][2];
#pragma unroll
      for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col = i * 8 + 2 * t4 + u;
          int orow = -1;
          float f = 1.0f;
          if (col < nrows) {
            if (args.moe) {
              orow = routed_row(e, row0 + col);
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
        const uint32_t stage_s = smem_s + (uint32_t)(st * C::STAGE);
        // group scales (fp32) and 128 + zero point (bf16x2) of rows g8 and g8 + 8 of both MMA tiles
        float sc[2][2][2];  // [m][rr][32-K chunk (MXINT4)]
        uint32_t zz[2][2];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            if (DEC == DEC_MXINT4) {
              const uint32_t two = lds_u16(stage_s + s_off[m][rr]);  // e8m0 of chunks 2kh, 2kh + 1
              sc[m][rr][0] = e8m0_to_f32(two & 0xFFu);
              sc[m][rr][1] = e8m0_to_f32(two >> 8);
            } else {
              sc[m][rr][0] = __uint_as_float(lds_u16(stage_s + s_off[m][rr]) << 16);
            }
            uint32_t z = 8u;  // INT4_SYM and MXINT4 store q + 8
            if (D::ZP_ALWAYS || (DEC == DEC_INT4 && zp)) z = lds_u8(stage_s + z_off[m][rr]);
            zz[m][rr] = z * 0x00010001u + 0x43004300u;
          }
        // weight words
        uint32_t wr[2][8];
        uint32_t wb1[2][2];  // 1-bit plane, shifted to this warp's K half (UINT3: top bit moved to bit 2)
        if (DEC == DEC_UINT1 || DEC == DEC_UINT3) {
          ldsm_x4(stage_s + C::W_OFF + w_lane1, wb1[0][0], wb1[0][1], wb1[1][0], wb1[1][1]);
#pragma unroll
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
              wb1[m][rr] = DEC == DEC_UINT3 ? (wb1[m][rr] >> kh_shift) << 2 : wb1[m][rr] >> kh_shift;
        }
        if (DEC == DEC_UINT2 || DEC == DEC_UINT3) {
          ldsm_x4(stage_s + C::W_OFF + w_lane, wr[0][0], wr[0][1], wr[1][0], wr[1][1]);
        } else if (DEC == DEC_UINT1) {
        } else {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            ldsm_x4(stage_s + C::W_OFF + w_lane + m * 256, wr[m][0], wr[m][1], wr[m][2], wr[m][3]);
            if (DEC == DEC_INT8 || DEC == DEC_E4M3)
              ldsm_x4(stage_s + C::W_OFF + w_lane + m * 256 + 4096, wr[m][4], wr[m][5], wr[m][6], wr[m][7]);
          }
        }
        float tacc[2][NT][4];  // column tiles past nn are predicated off and stay zero
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int n8 = 1; n8 < NT; ++n8)
#pragma unroll
            for (int i = 0; i < 4; ++i) tacc[m][n8][i] = 0.0f;
        uint32_t b[NT][2], b_next[2];  // B fragments of the current K step (8-token tiles: the next one too)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if (BT == 8) {
            // one ldmatrix.x4 covers the 8 tokens of two K steps
            if ((s & 1) == 0) {
              ldsm_x4(stage_s + a_row + (((uint32_t)(32 * s)) ^ a_sw), b[0][0], b[0][1], b_next[0], b_next[1]);
            } else {
              b[0][0] = b_next[0];
              b[0][1] = b_next[1];
            }
          } else {
#pragma unroll
            for (int q = 0; q < NT / 2; ++q)
              ldsm_x4(stage_s + a_row + q * 2048 + (((uint32_t)(32 * s)) ^ a_sw), b[2 * q][0], b[2 * q][1],
                      b[2 * q + 1][0], b[2 * q + 1][1]);
          }
          const bool fresh = s == 0 || (DEC == DEC_MXINT4 && s == 2);  // first step of a scale group
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            uint32_t a[4];  // a0, a2: row g8; a1, a3: row g8 + 8; a0, a1: k 2t, 2t+1; a2, a3: k 2t+8, 2t+9
            if (DEC == DEC_INT4 || DEC == DEC_MXINT4) {
              const int j = s >> 1, sh = 8 * (s & 1);
              a[0] = dec_u4(wr[m][2 * j] >> sh, zz[m][0]);
              a[1] = dec_u4(wr[m][2 * j + 1] >> sh, zz[m][1]);
              a[2] = dec_u4(wr[m][2 * j] >> (sh + 4), zz[m][0]);
              a[3] = dec_u4(wr[m][2 * j + 1] >> (sh + 4), zz[m][1]);
            } else if (DEC == DEC_UINT2) {
              a[0] = dec_u2(wr[m][0] >> (4 * s), zz[m][0]);
              a[1] = dec_u2(wr[m][1] >> (4 * s), zz[m][1]);
              a[2] = dec_u2(wr[m][0] >> (4 * s + 2), zz[m][0]);
              a[3] = dec_u2(wr[m][1] >> (4 * s + 2), zz[m][1]);
            } else if (DEC == DEC_UINT1) {
              a[0] = dec_u1(wb1[m][0] >> (2 * s), zz[m][0]);
              a[1] = dec_u1(wb1[m][1] >> (2 * s), zz[m][1]);
              a[2] = dec_u1(wb1[m][0] >> (2 * s + 1), zz[m][0]);
              a[3] = dec_u1(wb1[m][1] >> (2 * s + 1), zz[m][1]);
            } else if (DEC == DEC_UINT3) {
              a[0] = dec_u3(wr[m][0] >> (4 * s), wb1[m][0] >> (2 * s), zz[m][0]);
              a[1] = dec_u3(wr[m][1] >> (4 * s), wb1[m][1] >> (2 * s), zz[m][1]);
              a[2] = dec_u3(wr[m][0] >> (4 * s + 2), wb1[m][0] >> (2 * s + 1), zz[m][0]);
              a[3] = dec_u3(wr[m][1] >> (4 * s + 2), wb1[m][1] >> (2 * s + 1), zz[m][1]);
            } else {
              const uint32_t rg8 = wr[m][4 * (s >> 1) + 2 * (s & 1)], rg88 = wr[m][4 * (s >> 1) + 2 * (s & 1) + 1];
              if (DEC == DEC_INT8) {
                a[0] = dec_i8(rg8);
                a[1] = dec_i8(rg88);
                a[2] = dec_i8(rg8 >> 8);
                a[3] = dec_i8(rg88 >> 8);
              } else {
                a[0] = dec_e4m3(rg8);
                a[1] = dec_e4m3(rg88);
                a[2] = dec_e4m3(rg8 >> 16);
                a[3] = dec_e4m3(rg88 >> 16);
              }
            }
#pragma unroll
            for (int n8 = 0; n8 < NT; ++n8) {
              if (n8 == 0) {  // every tile holds a token in its first 8 columns
                if (fresh) mma_bf16_16816_z(tacc[m][n8], a, b[n8][0], b[n8][1]);
                else mma_bf16_16816(tacc[m][n8], a, b[n8][0], b[n8][1]);
              } else {
                if (fresh) mma_bf16_16816_z_if(tacc[m][n8], a, b[n8][0], b[n8][1], n8 < nn);
                else mma_bf16_16816_if(tacc[m][n8], a, b[n8][0], b[n8][1], n8 < nn);
              }
            }
          }
          // end of a scale group: the running sums take the group's products times its scale
          if (s == 3 || (DEC == DEC_MXINT4 && s == 1)) {
            const int c = (DEC == DEC_MXINT4 && s == 3) ? 1 : 0;
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
              for (int n8 = 0; n8 < NT; ++n8)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[m][n8][i] = fmaf(sc[m][i >> 1][c], tacc[m][n8][i], acc[m][n8][i]);
          }
        }
        __syncwarp();
        mbar_arrive_if(&sh.empty[st], lane == 0);
        st = st + 1 == C::STAGES ? 0 : st + 1;
        ph ^= st == 0 ? 1u : 0u;
      }
      // ---------------------------------------------------- K halves meet
      // Warp (rg, kh) finishes the 16-row half m = kh of its 32 rows: it hands the other half of its K-half sums to
      // its partner (rg, kh ^ 1) and adds the partner's share of its own half, so that the fix-up polls and the
      // epilogue run on all 8 warps.
      pdl_wait();  // (returns at once after the first piece) the epilogue touches global memory
      float own[NT][4];
      {
        float* give = red + (((rg * 2 + kh) * 32 + lane) * NT) * 4;  // [rg][kh][lane][nt][4]
        const float* take = red + (((rg * 2 + (kh ^ 1)) * 32 + lane) * NT) * 4;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
#pragma unroll
          for (int j = 0; j < 4; ++j) own[i][j] = kh ? acc[1][i][j] : acc[0][i][j];
          if (i < nn)
            *reinterpret_cast<float4*>(give + i * 4) = kh ? make_float4(acc[0][i][0], acc[0][i][1], acc[0][i][2], acc[0][i][3])
                                                          : make_float4(acc[1][i][0], acc[1][i][1], acc[1][i][2], acc[1][i][3]);
        }
        if (!epi_sync()) return;
#pragma unroll
        for (int i = 0; i < NT; ++i)
          if (i < nn) {
            const float4 o = *reinterpret_cast<const float4*>(take + i * 4);
            own[i][0] += o.x;
            own[i][1] += o.y;
            own[i][2] += o.z;
            own[i][3] += o.w;
          }
      }
      // this lane's element (i, 2 rr + u) sits at row 32 rg + 16 kh + 8 rr + g8, token column 8 i + 2 t4 + u
      auto slot_at = [&](int i, int rr, int u) {
        return (8 * i + 2 * t4 + u) * TILE_N + 32 * rg + 16 * kh + 8 * rr + g8;
      };
      if (!pc.full) {
        if (!mbar_wait(&sh.epoch_bar, 0, abort_flag, args.wait_ns)) {
          fail(ERR_TIMEOUT);
          ok = false;
        }
      }
      const uint64_t tag = (uint64_t)sh.epoch << 32;
#if HQ_DEBUG_BOUNDS
      if (ok && !pc.full && !dbg_span(((int64_t)blockIdx.x + 1) * BT * TILE_N, args.dbg_part_elems, args.status))
        ok = false;
#endif
      if (ok && !pc.full && pc.g0 > 0) {
        // the tile started in an earlier CTA: leave the partial sum, tagged with the call's epoch, in this CTA's slot
        uint64_t* part = reinterpret_cast<uint64_t*>(args.partials) + (int64_t)blockIdx.x * BT * TILE_N;
#pragma unroll
        for (int i = 0; i < NT; ++i)
          if (i < nn)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
              for (int u = 0; u < 2; ++u)
                st_relaxed_gpu_u64(part + slot_at(i, rr, u), tag | __float_as_uint(own[i][2 * rr + u]));
      } else if (ok) {
        if (!pc.full) {
          // this CTA holds the tile's first block: add the partial sums of the CTAs holding the rest, each value once
          // its tag shows this call's epoch.  Contributors are polled FIX_G at a time with all their loads in flight
          // together (one L2 round trip per group instead of one per contributor).
          const int64_t first_it = (int64_t)pc.tile * sched.kst;
          const int c_last = sched.cta_of(first_it + sched.kst - 1);
          for (int cb = (int)blockIdx.x + 1; ok && cb <= c_last; cb += C::FIX_G) {
            const int ng = c_last - cb + 1 < C::FIX_G ? c_last - cb + 1 : C::FIX_G;
            uint32_t done = 0;  // contributor cb + j added (bit j; warp-uniform)
            long long t0 = 0;
            for (int tries = 0;; ++tries) {
              uint64_t x[C::FIX_G][NT][4];
#pragma unroll
              for (int j = 0; j < C::FIX_G; ++j) {
                const bool want = j < ng && !((done >> j) & 1u);
                const uint64_t* part =
                    reinterpret_cast<const uint64_t*>(args.partials) + (int64_t)(cb + j) * BT * TILE_N;
#pragma unroll
                for (int i = 0; i < NT; ++i)
#pragma unroll
                  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                      x[j][i][2 * rr + u] = (want && i < nn) ? ld_relaxed_gpu_u64(part + slot_at(i, rr, u)) : tag;
              }
#pragma unroll
              for (int j = 0; j < C::FIX_G; ++j) {
                if (j >= ng || ((done >> j) & 1u)) continue;
                bool mine_ok = true;
#pragma unroll
                for (int i = 0; i < NT; ++i)
#pragma unroll
                  for (int q = 0; q < 4; ++q) mine_ok = mine_ok && (x[j][i][q] >> 32) == (tag >> 32);
                if (__all_sync(0xffffffffu, mine_ok)) {
#pragma unroll
                  for (int i = 0; i < NT; ++i)
#pragma unroll
                    for (int q = 0; q < 4; ++q) own[i][q] += __uint_as_float((uint32_t)x[j][i][q]);
                  done |= 1u << j;
                }
              }
              if (done == (1u << ng) - 1u) break;
              if (tries == 0) {
                t0 = clock64();
              } else if (clock64() - t0 >= 3ll * (long long)args.wait_ns || *abort_flag) {
                fail(ERR_TIMEOUT);
                ok = false;
                break;
              }
              __nanosleep(64);
            }
          }
        }
        if (ok) {
          // ---------------------------------------------------- epilogue
          const bool pair_ok = !args.comb && (args.N & 1) == 0 && (reinterpret_cast<uintptr_t>(args.c) & 3) == 0;
          const bool odd = g8 & 1;
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int n = nt * TILE_N + 32 * rg + 16 * kh + 8 * rr + g8;
            const float bias = (args.bias && n < args.N) ? bf16_to_f32(args.bias[n]) : 0.0f;
#pragma unroll
            for (int i = 0; i < NT; ++i) {
              if (i >= nn) continue;
#if HQ_DEBUG_BOUNDS
              t_row[i][0] = dbg_row(t_row[i][0], args.dbg_c_rows, args.status);
              t_row[i][1] = dbg_row(t_row[i][1], args.dbg_c_rows, args.status);
#endif
              const float o0 = own[i][2 * rr] * t_mul[i][0] + bias;
              const float o1 = own[i][2 * rr + 1] * t_mul[i][1] + bias;
              if (pair_ok) {
                // lanes g8 and g8 ^ 1 hold rows n and n ^ 1: the even lane writes token column 2t (rows n, n + 1),
                // the odd lane token column 2t + 1 (rows n - 1, n), one 4-byte store each
                const float send = odd ? o0 : o1;
                const float recv = __shfl_xor_sync(0xffffffffu, send, 4);
                const int orow = odd ? t_row[i][1] : t_row[i][0];
                const int n_even = n & ~1;
                const uint32_t pk = odd ? pack_bf16x2(recv, o1) : pack_bf16x2(o0, recv);
                if (orow >= 0 && n_even < args.N)
                  *reinterpret_cast<uint32_t*>(args.c + (int64_t)orow * args.N + n_even) = pk;
              } else if (n < args.N) {
                const float o[2] = {o0, o1};
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int orow = t_row[i][u];
                  if (orow < 0) continue;
                  if (args.comb)  // MoE combine: add into the token's fp32 row
                    red_add_f32(args.comb + (int64_t)(orow / args.comb_k) * args.N + n, o[u]);
                  else
                    args.c[(int64_t)orow * args.N + n] = f32_to_bf16(o[u]);
                }
              }
            }
          }
        }
      }
      if (!epi_sync()) return;  // the exchange buffer is reused by the next piece
    });
  }

  // ---------------------------------------------------------------- teardown
  pdl_wait();
  __syncthreads();
  if (tid == 0) {
    // the last CTA to exit stores this call's epoch for the next call on the workspace
    uint32_t* hdr = reinterpret_cast<uint32_t*>(args.status);
    const uint32_t prev = atomicAdd(hdr + 2, 1u);
    if (prev == gridDim.x - 1) {
      hdr[2] = 0u;
      reinterpret_cast<volatile uint32_t*>(hdr)[1] = sh.epoch;
    }
  }
}

template <int BT, int DEC>
cudaError_t launch_small_bt(const GemmArgs& a, int grid, cudaStream_t stream) {
  using C = SmallCfg<BT, DEC>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(hq_gemm_small_kernel<BT, DEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  return launch_kernel(hq_gemm_small_kernel<BT, DEC>, dim3(grid), dim3(SM_THREADS), C::SMEM_BYTES, stream, a);
}

template <int DEC>
cudaError_t launch_small_dec(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  switch (bt) {
    case 8: return launch_small_bt<8, DEC>(a, grid, stream);
    case 16: return launch_small_bt<16, DEC>(a, grid, stream);
    case 32: return launch_small_bt<32, DEC>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hq
