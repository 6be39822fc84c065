// Split-K reduction of the Stream-K pieces.
//
// When tiles are few, the GEMM kernels deal the (tile, K block) iterations out
// evenly to their CTAs; a tile whose K blocks land on several CTAs is left as
// fp32 partial sums, one slot per piece, written without any synchronisation.
// This kernel (chained to the GEMM by programmatic dependent launch) sums the
// partials of every such tile in CTA order, applies the epilogue (per-row
// multiplier, bias) and stores bf16.  Tiles held by a single CTA were already
// written by the GEMM.
#include "hq_gemm_kernel.cuh"
#include "hq_launch.h"

namespace hq {

constexpr int RED_THREADS = 256;
constexpr int RED_COLS = 32;  // token columns per work item: 32 x 128 rows = 1024 float4 groups, 4 per thread

template <int PATH>
__global__ void __launch_bounds__(RED_THREADS) splitk_reduce_kernel(const __grid_constant__ GemmArgs args, int bt,
                                                                   int gemm_grid) {
  __shared__ int prefix[513];
  __shared__ int total_sh;
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // partials (and MoE counts) come from the GEMM
  if (args.moe) {
    moe_tile_prefix(args.counts, args.E, args.region_cap, bt, prefix, &total_sh);  // as the GEMM computed it
    __syncthreads();
  }
  const int total_tiles = args.moe ? total_sh * args.n_tiles : args.m_tiles * args.n_tiles;
  if (total_tiles <= 0) return;
  Sched s;
  s.init(total_tiles, args.kst, gemm_grid, 0, 1);
  const int chunks = (bt + RED_COLS - 1) / RED_COLS;
  const bool vec_store = (args.N & 3) == 0 && (reinterpret_cast<uintptr_t>(args.c) & 7) == 0;
  // work item = (tile, chunk of RED_COLS columns); thread = 4 consecutive rows of one column, 4 columns apart
  const int r4 = (tid & 31) * 4;
  const int cq = tid >> 5;  // 0..7
  for (int item = blockIdx.x; item < total_tiles * chunks; item += gridDim.x) {
    const int tile = (int)((uint32_t)item / (uint32_t)chunks);
    const int col0 = (int)((uint32_t)item - (uint32_t)tile * (uint32_t)chunks) * RED_COLS;
    const int64_t first_it = (int64_t)tile * s.kst;
    const int c_first = s.cta_of(first_it);
    const int c_last = s.cta_of(first_it + s.kst - 1);
    if (c_first == c_last) continue;  // written by the GEMM
    const int mt = tile / args.n_tiles;
    const int nt = tile % args.n_tiles;
    int e = 0, row0, nrows;
    if (args.moe) {
      int lm;
      moe_locate(prefix, args.E, mt, e, lm);
      int cnt = args.counts[e];
      cnt = cnt > args.region_cap ? args.region_cap : cnt;
      row0 = lm * bt;
      nrows = cnt - row0 < bt ? cnt - row0 : bt;
    } else {
      row0 = mt * bt;
      nrows = args.M - row0 < bt ? args.M - row0 : bt;
    }
    if (col0 >= nrows) continue;
    const int n0 = nt * TILE_N + r4;
    float4 acc[RED_COLS / 8];
#pragma unroll
    for (int u = 0; u < RED_COLS / 8; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    // partial slots of the tile in CTA order, four slots per round with every load of a round in flight
    // together; sums are taken in slot order
    for (int c4 = c_first; c4 <= c_last; c4 += 4) {
      float4 v[4][RED_COLS / 8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c4 + k;
        const int slot = (c == c_first && s.start(c) < first_it) ? 2 * c + 1 : 2 * c;
        const float* base = args.partials + ((int64_t)slot * bt) * TILE_N + r4;
#if HQ_DEBUG_BOUNDS
        if (c <= c_last && !dbg_span(((int64_t)slot + 1) * bt * TILE_N, args.dbg_part_elems, args.status)) {
          for (int u = 0; u < RED_COLS / 8; ++u) v[k][u] = make_float4(0.f, 0.f, 0.f, 0.f);
          continue;
        }
#endif
#pragma unroll
        for (int u = 0; u < RED_COLS / 8; ++u) {
          const int col = col0 + cq + 8 * u;
          v[k][u] = (c <= c_last && col < nrows) ? __ldcg(reinterpret_cast<const float4*>(base + (int64_t)col * TILE_N))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int u = 0; u < RED_COLS / 8; ++u) {
          acc[u].x += v[k][u].x;
          acc[u].y += v[k][u].y;
          acc[u].z += v[k][u].z;
          acc[u].w += v[k][u].w;
        }
    }
    float bias4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) bias4[i] = (args.bias && n0 + i < args.N) ? bf16_to_f32(args.bias[n0 + i]) : 0.0f;
    const float mul0 = PATH == PATH_NVFP4 ? args.a_scale[0] * args.w_gscale[e] : 1.0f;
#pragma unroll
    for (int u = 0; u < RED_COLS / 8; ++u) {
      const int col = col0 + cq + 8 * u;
      if (col >= nrows) continue;
      int orow;
      float mul = mul0;
      if (args.moe) {
        orow = args.region[(int64_t)e * args.region_cap + row0 + col];
        if (args.topk_w) mul *= args.topk_w[orow];
        if (PATH == PATH_MXFP4) mul *= args.a_scale[orow / args.topk];
      } else {
        orow = row0 + col;
        if (PATH == PATH_MXFP4) mul *= args.a_scale[orow];
      }
#if HQ_DEBUG_BOUNDS
      if (dbg_row(orow, args.dbg_c_rows, args.status) < 0) continue;
#endif
      const float o[4] = {acc[u].x * mul + bias4[0], acc[u].y * mul + bias4[1], acc[u].z * mul + bias4[2],
                          acc[u].w * mul + bias4[3]};
      if (args.comb) {  // MoE combine: add into the token's fp32 row
        float* dst = args.comb + (int64_t)(orow / args.comb_k) * args.N + n0;
        if ((args.N & 3) == 0 && n0 + 3 < args.N) {
          red_add_v4_f32(dst, o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (n0 + i < args.N) red_add_f32(dst + i, o[i]);
        }
        continue;
      }
      uint16_t* dst = args.c + (int64_t)orow * args.N + n0;
      if (vec_store && n0 + 3 < args.N) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n0 + i < args.N) dst[i] = f32_to_bf16(o[i]);
      }
    }
  }
}

cudaError_t launch_splitk_reduce(int path, const GemmArgs& a, int bt, int gemm_grid, int grid, cudaStream_t stream) {
  switch (path) {
    case PATH_INT4:
      return launch_kernel(splitk_reduce_kernel<PATH_INT4>, dim3(grid), dim3(RED_THREADS), 0, stream, a, bt, gemm_grid);
    case PATH_NVFP4:
      return launch_kernel(splitk_reduce_kernel<PATH_NVFP4>, dim3(grid), dim3(RED_THREADS), 0, stream, a, bt, gemm_grid);
    case PATH_MXFP4:
      return launch_kernel(splitk_reduce_kernel<PATH_MXFP4>, dim3(grid), dim3(RED_THREADS), 0, stream, a, bt, gemm_grid);
    case PATH_MXFP4A:
      return launch_kernel(splitk_reduce_kernel<PATH_MXFP4A>, dim3(grid), dim3(RED_THREADS), 0, stream, a, bt, gemm_grid);
    case PATH_MXFP4X:
      return launch_kernel(splitk_reduce_kernel<PATH_MXFP4X>, dim3(grid), dim3(RED_THREADS), 0, stream, a, bt, gemm_grid);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace hq
