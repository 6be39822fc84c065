// C ABI: argument validation, launch planning and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "../../include/hq.h"
#include "hq_act_quant.h"
#include "hq_gemm_kernel.cuh"
#include "hq_layout.h"
#include "hq_tune.h"

namespace hq {
cudaError_t launch_pack(int dir, int wt, int64_t N, int64_t K, int64_t E, const void* codes, const void* scales,
                        const void* zeros, const float* gscale, void* packed, cudaStream_t stream);
cudaError_t launch_route(const int32_t* ids, int64_t rows, int E, int cap, int* counts, int* region, int* status,
                         cudaStream_t stream);
cudaError_t launch_gemm_int4(const GemmArgs& a, int bt, int grid, cudaStream_t stream);
cudaError_t launch_gemm_nvfp4(const GemmArgs& a, int bt, int grid, cudaStream_t stream);
cudaError_t launch_gemm_mxfp4(const GemmArgs& a, int bt, int grid, cudaStream_t stream);
cudaError_t launch_gemm_mxfp4a(const GemmArgs& a, int bt, int grid, cudaStream_t stream);
cudaError_t launch_gemm_mxfp4x(const GemmArgs& a, int bt, int grid, cudaStream_t stream);
cudaError_t launch_gemm_small(const GemmArgs& a, int bt, int grid, cudaStream_t stream);
cudaError_t launch_gemm_small_fmt(int dec, const GemmArgs& a, int bt, int grid, cudaStream_t stream);
cudaError_t launch_splitk_reduce(int path, const GemmArgs& a, int bt, int gemm_grid, int grid, cudaStream_t stream);
cudaError_t launch_combine_round(const float* acc, int64_t n, uint16_t* c, cudaStream_t stream);
cudaError_t launch_swiglu(const void* x, int64_t R, int64_t I, void* out, cudaStream_t stream);
cudaError_t launch_moe_permute(const int* counts, const int* region, int cap, int E, int topk, int64_t rows,
                               const void* src, int row_bytes, void* dst, const void* sf_src, int sf_bytes, void* sf_dst,
                               int* row_off, cudaStream_t stream);

namespace {

// Bound of every in-kernel pipeline wait for calls enqueued from now on (hq_set_wait_limit_ns).
std::atomic<uint64_t> g_wait_ns{DEFAULT_WAIT_NS};

constexpr int64_t kMaxExperts = 512;
constexpr size_t kHeaderBytes = 256;  // [0] device status, [1] epoch of the last register-decode call, [2] exit count
constexpr int64_t kMaxRows = (int64_t)1 << 30;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validate the descriptor against the supported combinations.
hq_status_t check_format(const hq_format_t* f) {
  if (!f) return HQ_ERR_INVALID_ARG;
  if (f->N < 1 || f->K < 1 || f->num_experts < 1 || f->num_experts > kMaxExperts) return HQ_ERR_INVALID_ARG;
  if (f->N > kMaxRows || f->K > kMaxRows) return HQ_ERR_INVALID_ARG;
  switch (f->weight_type) {
    case HQ_W_INT4_SYM:
      if (f->group_size != 128 || f->scale_type != HQ_S_BF16 || f->has_zero || f->has_global_scale ||
          f->act_type != HQ_A_BF16)
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 128) return HQ_ERR_ALIGNMENT;
      break;
    case HQ_W_UINT4_ZP:
      if (f->group_size != 128 || f->scale_type != HQ_S_BF16 || !f->has_zero || f->has_global_scale ||
          f->act_type != HQ_A_BF16)
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 128) return HQ_ERR_ALIGNMENT;
      break;
    case HQ_W_NVFP4:
      if (f->group_size != 16 || f->scale_type != HQ_S_UE4M3 || f->has_zero || !f->has_global_scale ||
          f->act_type != HQ_A_NVFP4)
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 256) return HQ_ERR_ALIGNMENT;
      break;
    case HQ_W_MXFP4:
      if (f->group_size != 32 || f->scale_type != HQ_S_UE8M0 || f->has_zero || f->has_global_scale ||
          (f->act_type != HQ_A_E4M3_TOKEN && f->act_type != HQ_A_MXFP8 && f->act_type != HQ_A_MXFP4))
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 128) return HQ_ERR_ALIGNMENT;
      // MXFP8 / MXFP4 block scales are loaded 16 bytes (512 K) at a time: rows of K/32 bytes must be 16-byte
      // multiples
      if ((f->act_type == HQ_A_MXFP8 || f->act_type == HQ_A_MXFP4) && f->K % 512) return HQ_ERR_ALIGNMENT;
      break;
    case HQ_W_INT8_SYM:
    case HQ_W_E4M3:
      if (f->group_size != 128 || f->scale_type != HQ_S_BF16 || f->has_zero || f->has_global_scale ||
          f->act_type != HQ_A_BF16)
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 128) return HQ_ERR_ALIGNMENT;
      break;
    case HQ_W_UINT2_ZP:
      if (f->group_size != 128 || f->scale_type != HQ_S_BF16 || !f->has_zero || f->has_global_scale ||
          f->act_type != HQ_A_BF16)
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 128) return HQ_ERR_ALIGNMENT;
      break;
    case HQ_W_UINT1_ZP:
    case HQ_W_UINT3_ZP:
      if (f->group_size != 128 || f->scale_type != HQ_S_BF16 || !f->has_zero || f->has_global_scale ||
          f->act_type != HQ_A_BF16)
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 128) return HQ_ERR_ALIGNMENT;
      break;
    case HQ_W_MXINT4:
      if (f->group_size != 32 || f->scale_type != HQ_S_UE8M0 || f->has_zero || f->has_global_scale ||
          f->act_type != HQ_A_BF16)
        return HQ_ERR_UNSUPPORTED;
      if (f->K % 128) return HQ_ERR_ALIGNMENT;
      break;
    default:
      return HQ_ERR_UNSUPPORTED;
  }
  return HQ_OK;
}

// Packed layout of a descriptor: MXFP4 weights meant for MXFP4 activations are packed like NVFP4 (packed e2m1 in
// the MMA, scales as tensor-memory words), every other format by its weight type.
int pack_kind(const hq_format_t* f) {
  return (f->weight_type == HQ_W_MXFP4 && f->act_type == HQ_A_MXFP4) ? (int)WK_MXFP4_X : f->weight_type;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Launch plan of one call; also fixes the workspace layout.
struct Plan {
  int path = 0;
  int small = 0;  // integer / FP8 weights with at most 32 tokens per tile: register-decode mma.sync kernel
  int dec = 0;    // its decode variant
  int grouped = 0;  // MoE: routed rows copied into expert-contiguous order first (2-D TMA boxes)
  int fused = 0;    // MoE: the register-decode kernel routes the rows itself (no routing kernel)
  int bt = 16;
  int sk = 0;
  int grid = 1;
  int64_t n_tiles = 0, kst = 0, m_tiles = 0;
  int64_t max_tiles = 0;   // upper bound of tiles
  int64_t region_cap = 0;  // MoE rows per expert
  size_t off_counts = 0, off_region = 0, off_partials = 0, ws_bytes = 0;
  size_t off_rowoff = 0, off_gact = 0, off_gsf = 0;  // MoE grouped: expert row offsets, rows, NVFP4 scales
};

int pick_bt_dense(int64_t M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}
// MoE token tile by the mean routed rows per expert.  The UMMA step costs nearly the same for any tile up to 256
// tokens, so once experts carry more than a handful of rows the wide tiles win even with the padding of the rarely
// routed experts; 16-token tiles keep the INT4 register-decode kernel for sparse routing.  Dense-only 256-token
// NVFP4 tiles carry no per-row tables, hence at most 128 for NVFP4.
int pick_bt_moe(int path, int64_t rows, int64_t E) {
  if (E == 1) return pick_bt_dense(rows);  // one expert is a dense GEMM over the routed rows
  const int64_t avg = (rows + E - 1) / E;
  if (avg <= 16) return 16;
  if (path != PATH_NVFP4 && path != PATH_MXFP4A && path != PATH_MXFP4X && avg > 128) return 256;
  return 128;
}

// HQ_MOE_PATH=indexed|grouped overrides the choice of MoE activation path (tests compare both).
int forced_moe_path() {
  const char* v = getenv("HQ_MOE_PATH");
  if (!v) return 0;
  if (!strcmp(v, "indexed")) return 1;
  if (!strcmp(v, "grouped")) return 2;
  return 0;
}

// Activation bytes per row and NVFP4 scale bytes per row.
int64_t act_row_bytes(const hq_format_t* f) {
  return f->act_type == HQ_A_BF16 ? 2 * f->K : ((f->act_type == HQ_A_E4M3_TOKEN || f->act_type == HQ_A_MXFP8) ? f->K : f->K / 2);
}
// Activation block-scale bytes per row (NVFP4: ue4m3 per 16; MXFP8: e8m0 per 32), else 0.
int64_t act_scale_row_bytes(const hq_format_t* f) {
  return f->act_type == HQ_A_NVFP4 ? f->K / 16 : ((f->act_type == HQ_A_MXFP8 || f->act_type == HQ_A_MXFP4) ? f->K / 32 : 0);
}

// HQ_FORCE_PATH=small|umma overrides the choice between the two INT4 kernels (tests compare both).
int forced_path() {
  const char* v = getenv("HQ_FORCE_PATH");
  if (!v) return 0;
  if (!strcmp(v, "small")) return 1;
  if (!strcmp(v, "umma")) return 2;
  return 0;
}

int tune_class(const hq_format_t* f, int path) {
  if (path == PATH_NVFP4) return TC_NVFP4;
  if (path == PATH_MXFP4A) return TC_MXFP4A;
  if (path == PATH_MXFP4X) return TC_MXFP4X;
  if (path == PATH_MXFP4) return TC_MXFP4;
  return register_decode_only(f->weight_type) ? TC_REGDEC : TC_INT4;
}

// Tiles of the launch for token tile bt: (upper bound, planning estimate).  MoE: the host does not know the routing,
// so the bound assumes every routed expert's rows end in a partial tile; the estimate is one tile per expert hit.
void plan_tiles(Plan& p, int64_t M_or_T, int32_t topk, bool moe, int64_t E, int64_t* tiles_est) {
  if (!moe) {
    p.m_tiles = (M_or_T + p.bt - 1) / p.bt;
    p.max_tiles = p.m_tiles * p.n_tiles;
    *tiles_est = p.max_tiles;
  } else {
    const int64_t rows = M_or_T * topk;
    const int64_t active = rows < E ? rows : E;
    p.max_tiles = p.n_tiles * (active + (rows + p.bt - 1) / p.bt);
    *tiles_est = p.n_tiles * active;
  }
}

// The built-in rule, then the tuned table's row for (format class, size bucket), then HQ_TUNE; every choice is
// checked against what the kernels support before it is taken.
// kind: 0 dense (hq_gemm), 1 MoE (hq_moe_gemm), 2 MoE with the top-k combine (hq_moe_gemm_combine)
Plan make_plan(const hq_format_t* f, int64_t M_or_T, int32_t topk, int kind, int sms) {
  const bool moe = kind != 0;
  Plan p;
  const PackGeom g = pack_geom(pack_kind(f), f->N, f->K, f->num_experts);
  p.path = (g.path == PATH_MXFP4 && f->act_type == HQ_A_MXFP8) ? PATH_MXFP4A : g.path;
  p.n_tiles = g.n_tiles;
  p.kst = g.k_stages;
  if (sms < 1) sms = 1;
  size_t off = kHeaderBytes;  // status word, epoch, exit count
  const int64_t E = f->num_experts;
  const int64_t rows = M_or_T * (moe ? topk : 1);
  const int64_t key = moe ? (rows + E - 1) / E : M_or_T;  // size bucket key: M, or routed rows per expert
  if (moe) p.region_cap = M_or_T;  // rows per expert list
  // built-in rule: token tile by size; INT4 tiles of at most 32 tokens on the register-decode kernel
  p.bt = moe ? pick_bt_moe(p.path, rows, E) : pick_bt_dense(M_or_T);
  if (p.path == PATH_INT4) {
    p.dec = decode_kind(f->weight_type);
    p.small = (register_decode_only(f->weight_type) || p.bt <= 32) ? 1 : 0;
    if (p.small) p.bt = p.bt > 32 ? 32 : ((!moe && M_or_T <= 8) ? 8 : p.bt);
  }
  // tuned choice
  TuneChoice tc = tune_lookup(tune_class(f, p.path), kind, key);
  tune_env_override(tc);
  const int force = forced_path();
  if (force) tc.kernel = force == 1 ? 1 : 0;
  if (p.path == PATH_INT4 && !register_decode_only(f->weight_type) && tc.kernel >= 0 && tc.kernel != p.small) {
    p.small = tc.kernel;
    if (p.small && p.bt > 32) p.bt = 32;       // re-tile for the register-decode kernel
    if (!p.small && p.bt < 16) p.bt = 16;
  }
  if (tc.bt > 0) {
    const bool ok = p.small ? (tc.bt == 8 || tc.bt == 16 || tc.bt == 32)
                            : (tc.bt == 16 || tc.bt == 32 || tc.bt == 64 || tc.bt == 128 ||
                               (tc.bt == 256 &&
                                !(moe && (p.path == PATH_NVFP4 || p.path == PATH_MXFP4A || p.path == PATH_MXFP4X))));
    if (ok) p.bt = tc.bt;
  }
  int64_t tiles_est = 0;
  plan_tiles(p, M_or_T, topk, moe, E, &tiles_est);
  // persistent grid: the register-decode kernel holds two CTAs per SM up to 16-token tiles (all CTAs of a launch
  // must be resident at once: owners of cut tiles wait for the other CTAs' partial sums)
  const int max_per_sm = p.small && p.bt <= 16 ? 2 : 1;
  const int per_sm = tc.slots >= 1 && tc.slots <= max_per_sm ? tc.slots : max_per_sm;
  const int64_t slots = (int64_t)per_sm * sms;
  if (p.small) {
    // Stream-K when the tiles fill less than two rounds of CTA slots; with fewer blocks than slots in all (tiny
    // weights) at least two blocks per CTA, so that a cut tile has few contributors to collect (measured: 1024 x 1024
    // INT4 at M = 8, 64 blocks: one block per CTA 6.0 us, whole tiles 5.5 us, two blocks per CTA 5.2 us)
    const int64_t blocks = p.max_tiles * p.kst;
    p.sk = (p.max_tiles < 2 * slots && p.kst > 1) ? 1 : 0;
    if (!moe && p.sk && blocks <= slots && tc.cpb <= 0) tc.cpb = 2;
  } else {
    // UMMA kernel: Stream-K when the tiles fill less than half a wave of SMs (the split then pays for its partial
    // sums and their reduction) or more than one wave but less than two (it evens out the second wave); one
    // partial wave runs whole tiles (measured: 112 INT4 tiles of 256 tokens 36 -> 29 us, 128 NVFP4 tiles of 256
    // tokens 33 -> 21 us).
    p.sk = (p.kst > 1 && (2 * tiles_est < sms || (tiles_est > sms && tiles_est < 2 * (int64_t)sms))) ? 1 : 0;
  }
  if (tc.sk >= 0) p.sk = (tc.sk && p.kst > 1) ? 1 : 0;
  const int64_t W = p.max_tiles * (p.sk ? p.kst : 1);
  p.grid = (int)(W < slots ? (W < 1 ? 1 : W) : slots);
  if (p.sk && tc.cpb > 1) {  // fewer CTAs, each with at least cpb K blocks
    const int64_t g = (W + tc.cpb - 1) / tc.cpb;
    if (g >= 1 && g < p.grid) p.grid = (int)g;
  }
  // MoE activations: grouped when tiles are wide (tile::gather4 cannot feed 64+ routed rows per stage fast enough)
  if (moe) {
    const int fm = forced_moe_path();
    p.grouped = fm == 2 ? 1 : (fm == 1 ? 0 : (tc.grouped >= 0 ? (tc.grouped ? 1 : 0) : (p.bt >= 64 ? 1 : 0)));
    // small MoE calls on the register-decode kernel route inside it (at most 512 routed rows: its shared-memory
    // lists)
    p.fused = (p.small && !p.grouped && rows <= 512 && !getenv("HQ_ROUTE_KERNEL")) ? 1 : 0;
  }
  // Stream-K partial sums first, right after the header: the register-decode kernel tags each of its values with
  // the call's epoch, and the fixed place keeps other tables of other calls on the same workspace out of its slots
  if (p.sk) {
    p.off_partials = off;
    off = align256(off + sizeof(float) * (size_t)2 * p.grid * p.bt * TILE_N);
  }
  if (moe) {
    p.off_counts = off;
    off = align256(off + sizeof(int) * (size_t)f->num_experts);
    p.off_region = off;
    off = align256(off + sizeof(int) * (size_t)(f->num_experts * (p.region_cap > 0 ? p.region_cap : 1)));
    if (p.grouped) {
      p.off_rowoff = off;
      off = align256(off + sizeof(int) * (size_t)(f->num_experts + 1));
      p.off_gact = off;
      off = align256(off + (size_t)(rows * act_row_bytes(f)));
      if (act_scale_row_bytes(f) > 0) {
        p.off_gsf = off;
        off = align256(off + (size_t)(rows * act_scale_row_bytes(f)));
      }
    }
  }
  p.ws_bytes = off;
  return p;
}
#if HQ_DEBUG_BOUNDS

// Debug build: the extents the device-side index checks compare against.  HQ_DEBUG_ROW_LIMIT (for tests) lowers the
// output rows a call may write below the rows that exist, so that a check can be made to catch an index without any
// access outside the buffers.
void dbg_extents(GemmArgs& a, const Plan& p, int64_t c_rows, int64_t comb_rows) {
  const char* v = getenv("HQ_DEBUG_ROW_LIMIT");
  const int64_t lim = v ? atoll(v) : c_rows;
  a.dbg_c_rows = (int)(c_rows < lim ? c_rows : lim);
  a.dbg_comb_rows = (int)(comb_rows < lim ? comb_rows : lim);
  a.dbg_part_elems = p.sk ? (int64_t)(p.small ? 1 : 2) * p.grid * p.bt * TILE_N : 0;
}
#endif

cudaError_t launch_path(const Plan& p, const GemmArgs& a, cudaStream_t s) {
  cudaError_t e;
  if (p.path == PATH_INT4)
    e = !p.small ? launch_gemm_int4(a, p.bt, p.grid, s)
                 : (p.dec == DEC_INT4 ? launch_gemm_small(a, p.bt, p.grid, s)
                                      : launch_gemm_small_fmt(p.dec, a, p.bt, p.grid, s));
  else if (p.path == PATH_NVFP4) e = launch_gemm_nvfp4(a, p.bt, p.grid, s);
  else if (p.path == PATH_MXFP4A) e = launch_gemm_mxfp4a(a, p.bt, p.grid, s);
  else if (p.path == PATH_MXFP4X) e = launch_gemm_mxfp4x(a, p.bt, p.grid, s);
  else e = launch_gemm_mxfp4(a, p.bt, p.grid, s);
  if (e != cudaSuccess || !p.sk || p.small) return e;  // the register-decode kernel finishes cut tiles itself
  // tiles cut between CTAs: sum their partial slots, one CTA per 32 token columns of a tile
  const int64_t items = p.max_tiles * ((p.bt + 31) / 32);
  const int64_t cap = 4 * (int64_t)p.grid;
  const int64_t rg = items < cap ? items : cap;
  return launch_splitk_reduce(p.path, a, p.bt, p.grid, (int)(rg < 1 ? 1 : rg), s);
}

hq_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link needed).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D row-major tensor [rows][inner] of bf16 or bytes; box of box_rows x box_inner elements.
bool encode_2d(CUtensorMap* m, const void* base, bool bf16, uint64_t inner, uint64_t rows, uint32_t box_inner,
               uint32_t box_rows, bool swizzle128) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc || !base) return false;
  const uint64_t esize = bf16 ? 2 : 1;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Activation tensor maps: dense rows as one box of BT rows per stage; MoE rows one at a time (gather4).
bool act_maps(GemmArgs& a, const hq_format_t* f, const hq_act_t* A, int64_t rows, int bt, bool moe) {
  const uint32_t box_rows = moe ? 1u : (uint32_t)bt;
  const uint64_t K = (uint64_t)f->K;
  if (f->act_type == HQ_A_BF16) return encode_2d(&a.tmap_a, A->data, true, K, rows, 64, box_rows, true);
  if (f->act_type == HQ_A_E4M3_TOKEN) return encode_2d(&a.tmap_a, A->data, false, K, rows, 128, box_rows, true);
  if (f->act_type == HQ_A_MXFP8)
    return encode_2d(&a.tmap_a, A->data, false, K, rows, 128, box_rows, true) &&
           encode_2d(&a.tmap_sf, A->scale, false, K / 32, rows, 16, box_rows, false);
  if (f->act_type == HQ_A_MXFP4)
    return encode_2d(&a.tmap_a, A->data, false, K / 2, rows, 128, box_rows, true) &&
           encode_2d(&a.tmap_sf, A->scale, false, K / 32, rows, 16, box_rows, false);
  return encode_2d(&a.tmap_a, A->data, false, K / 2, rows, 128, box_rows, true) &&
         encode_2d(&a.tmap_sf, A->scale, false, K / 16, rows, 16, box_rows, false);
}

}  // namespace
}  // namespace hq

using namespace hq;

extern "C" {

size_t hq_packed_bytes(const hq_format_t* fmt) {
  if (check_format(fmt) != HQ_OK) return 0;
  return (size_t)pack_geom(pack_kind(fmt), fmt->N, fmt->K, fmt->num_experts).total_bytes;
}

hq_status_t hq_pack_weights(const hq_format_t* fmt, const uint8_t* codes, const void* scales, const uint8_t* zeros,
                            const float* global_scale, void* packed, hq_stream_t stream) {
  hq_status_t st = check_format(fmt);
  if (st != HQ_OK) return st;
  if (!codes || !scales || !packed) return HQ_ERR_INVALID_ARG;
  if (fmt->has_zero && !zeros) return HQ_ERR_INVALID_ARG;
  if (fmt->has_global_scale && !global_scale) return HQ_ERR_INVALID_ARG;
  if (!aligned16(packed)) return HQ_ERR_ALIGNMENT;
  return cuda_status(launch_pack(0, pack_kind(fmt), fmt->N, fmt->K, fmt->num_experts, codes, scales, zeros,
                                 global_scale, packed, (cudaStream_t)stream));
}

hq_status_t hq_unpack_weights(const hq_format_t* fmt, const void* packed, uint8_t* codes, void* scales,
                              uint8_t* zeros, float* global_scale, hq_stream_t stream) {
  hq_status_t st = check_format(fmt);
  if (st != HQ_OK) return st;
  if (!codes || !scales || !packed) return HQ_ERR_INVALID_ARG;
  if (fmt->has_zero && !zeros) return HQ_ERR_INVALID_ARG;
  if (!aligned16(packed)) return HQ_ERR_ALIGNMENT;
  return cuda_status(launch_pack(1, pack_kind(fmt), fmt->N, fmt->K, fmt->num_experts, codes, scales, zeros,
                                 global_scale, const_cast<void*>(packed), (cudaStream_t)stream));
}

size_t hq_workspace_bytes(const hq_format_t* fmt, int64_t M_or_T, int32_t topk) {
  if (check_format(fmt) != HQ_OK || M_or_T < 0 || topk < 1) return 0;
  const int sms = num_sms();
  if (fmt->num_experts > 1 || topk > 1) return make_plan(fmt, M_or_T, topk, 1, sms).ws_bytes;
  // one expert with top-1 serves both hq_gemm and hq_moe_gemm: cover both plans
  const size_t d = make_plan(fmt, M_or_T, 1, 0, sms).ws_bytes;
  const size_t m = make_plan(fmt, M_or_T, 1, 1, sms).ws_bytes;
  return d > m ? d : m;
}

int32_t hq_kernels_per_call(const hq_format_t* fmt, int64_t M_or_T, int32_t topk, int32_t moe) {
  if (check_format(fmt) != HQ_OK || M_or_T < 1 || topk < 1 || moe < 0 || moe > 2) return 0;
  const Plan p = make_plan(fmt, M_or_T, topk, moe, num_sms());
  int32_t n = 1 + (p.sk && !p.small ? 1 : 0);  // GEMM (+ split-K reduction of the UMMA kernel)
  if (moe) n += (p.fused ? 0 : 1) + (p.grouped ? 1 : 0);  // routing (+ row permutation), unless fused
  if (moe == 2) n += 1;                    // combine: rounding of the summed token rows
  return n;
}

hq_status_t hq_launch_plan(const hq_format_t* fmt, int64_t M_or_T, int32_t topk, int32_t moe, int32_t* plan_out) {
  if (check_format(fmt) != HQ_OK || M_or_T < 1 || topk < 1 || moe < 0 || moe > 2 || !plan_out) return HQ_ERR_INVALID_ARG;
  const Plan p = make_plan(fmt, M_or_T, topk, moe, num_sms());
  plan_out[0] = p.small;
  plan_out[1] = p.small ? p.dec : p.path;
  plan_out[2] = p.bt;
  plan_out[3] = p.sk;
  plan_out[4] = p.grid;
  plan_out[5] = p.grouped;
  return HQ_OK;
}

hq_status_t hq_workspace_init(void* workspace, size_t bytes, hq_stream_t stream) {
  if (!workspace || bytes == 0) return HQ_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream));
}

hq_status_t hq_gemm(const hq_format_t* fmt, const hq_act_t* A, const void* packedW, const void* bias, void* C,
                    int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes, hq_stream_t stream) {
  hq_status_t st = check_format(fmt);
  if (st != HQ_OK) return st;
  if (fmt->num_experts != 1 || N != fmt->N || K != fmt->K || M < 0 || M > kMaxRows) return HQ_ERR_INVALID_ARG;
  if (M == 0) return HQ_OK;
  if (!A || !A->data || !packedW || !C) return HQ_ERR_INVALID_ARG;
  if (fmt->act_type == HQ_A_E4M3_TOKEN && !A->scale) return HQ_ERR_INVALID_ARG;
  if (fmt->act_type == HQ_A_NVFP4 && (!A->scale || !A->global_scale)) return HQ_ERR_INVALID_ARG;
  if ((fmt->act_type == HQ_A_MXFP8 || fmt->act_type == HQ_A_MXFP4) && !A->scale) return HQ_ERR_INVALID_ARG;
  if (!aligned16(A->data) || !aligned16(packedW) || (A->scale && act_scale_row_bytes(fmt) > 0 && !aligned16(A->scale)))
    return HQ_ERR_ALIGNMENT;
  const int sms = num_sms();
  if (sms < 1) return HQ_ERR_CUDA;
  const Plan p = make_plan(fmt, M, 1, 0, sms);
  if (!workspace || ws_bytes < p.ws_bytes) return HQ_ERR_WORKSPACE;
  const PackGeom g = pack_geom(pack_kind(fmt), N, K, 1);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  GemmArgs a{};
  a.w = static_cast<const uint8_t*>(packedW);
  a.w_expert_bytes = g.expert_bytes;
  a.w_blk = g.blk_bytes;
  a.w_gscale = g.gscale_off >= 0 ? reinterpret_cast<const float*>(a.w + g.gscale_off) : nullptr;
  if (!act_maps(a, fmt, A, M, p.bt, false)) return HQ_ERR_INVALID_ARG;
  a.a_scale = fmt->act_type == HQ_A_NVFP4 ? A->global_scale
                                            : (fmt->act_type == HQ_A_E4M3_TOKEN ? static_cast<const float*>(A->scale)
                                                                                 : nullptr);
  a.bias = static_cast<const uint16_t*>(bias);
  a.c = static_cast<uint16_t*>(C);
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.n_tiles = (int)p.n_tiles;
  a.kst = (int)p.kst;
  a.zp = fmt->has_zero;
  a.moe = 0;
  a.E = 1;
  a.topk = 1;
  a.m_tiles = (int)p.m_tiles;
  a.sk = p.sk;
  a.status = reinterpret_cast<int*>(ws);
  a.partials = p.sk ? reinterpret_cast<float*>(ws + p.off_partials) : nullptr;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  // weights read once per call (one token tile): evict-first in L2, so that they do not push out the kernel code,
  // activations and partial sums that the next call needs
  a.w_evict_first = (p.small || p.m_tiles == 1) ? 1 : 0;
#if HQ_DEBUG_BOUNDS
  dbg_extents(a, p, M, 0);
#endif
  return cuda_status(launch_path(p, a, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Workspace offset of the combine's fp32 token rows (after everything the plan places).
size_t comb_offset(const Plan& p) { return align256(p.ws_bytes); }

// hq_moe_gemm (combine = false: A holds T token rows, C the T*topk routed rows) and hq_moe_gemm_combine (A holds the
// T*topk routed rows, C the T token rows summed over their top-k slots).
hq_status_t moe_call(const hq_format_t* fmt, const hq_act_t* A, const void* packedW, const int32_t* topk_ids,
                     const float* topk_weights, int64_t T, int32_t topk, void* C, void* workspace, size_t ws_bytes,
                     hq_stream_t stream, bool combine) {
  hq_status_t st = check_format(fmt);
  if (st != HQ_OK) return st;
  if (T < 0 || topk < 1 || T * topk > kMaxRows) return HQ_ERR_INVALID_ARG;
  if (T == 0) return HQ_OK;
  if (!A || !A->data || !packedW || !C || !topk_ids) return HQ_ERR_INVALID_ARG;
  if (fmt->act_type == HQ_A_E4M3_TOKEN && !A->scale) return HQ_ERR_INVALID_ARG;
  if (fmt->act_type == HQ_A_NVFP4 && (!A->scale || !A->global_scale)) return HQ_ERR_INVALID_ARG;
  if ((fmt->act_type == HQ_A_MXFP8 || fmt->act_type == HQ_A_MXFP4) && !A->scale) return HQ_ERR_INVALID_ARG;
  if (!aligned16(A->data) || !aligned16(packedW) || (act_scale_row_bytes(fmt) > 0 && !aligned16(A->scale)))
    return HQ_ERR_ALIGNMENT;
  const int sms = num_sms();
  if (sms < 1) return HQ_ERR_CUDA;
  const Plan p = make_plan(fmt, T, topk, combine ? 2 : 1, sms);
  if (combine && fmt->N % 4) return HQ_ERR_ALIGNMENT;
  const size_t need = combine ? comb_offset(p) + sizeof(float) * (size_t)(T * fmt->N) : p.ws_bytes;
  if (!workspace || ws_bytes < need) return HQ_ERR_WORKSPACE;
  const int64_t a_rows = combine ? T * topk : T;  // activation rows: tokens, or routed rows for the combine
  const int a_div = combine ? 1 : topk;          // routed row -> activation row
  const int64_t E = fmt->num_experts;
  const PackGeom g = pack_geom(pack_kind(fmt), fmt->N, fmt->K, E);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  int* counts = reinterpret_cast<int*>(ws + p.off_counts);
  int* region = reinterpret_cast<int*>(ws + p.off_region);
  GemmArgs a{};
  if (p.grouped) {
    // the GEMM reads the expert-contiguous copy with BT-row boxes
    hq_act_t G = *A;
    G.data = ws + p.off_gact;
    if (act_scale_row_bytes(fmt) > 0) G.scale = ws + p.off_gsf;
    if (!act_maps(a, fmt, &G, T * topk, p.bt, false)) return HQ_ERR_INVALID_ARG;
  } else if (!act_maps(a, fmt, A, a_rows, p.bt, true)) {
    return HQ_ERR_INVALID_ARG;
  }
  float* comb = combine ? reinterpret_cast<float*>(ws + comb_offset(p)) : nullptr;
  if (combine && cudaMemsetAsync(comb, 0, sizeof(float) * (size_t)(T * fmt->N), (cudaStream_t)stream) != cudaSuccess)
    return HQ_ERR_CUDA;
  cudaError_t err = cudaSuccess;
  if (!p.fused) {
    err = launch_route(topk_ids, T * topk, (int)E, (int)p.region_cap, counts, region, status, (cudaStream_t)stream);
    if (err != cudaSuccess) return HQ_ERR_CUDA;
  }
  if (p.grouped) {
    err = launch_moe_permute(counts, region, (int)p.region_cap, (int)E, a_div, T * topk, A->data,
                             (int)act_row_bytes(fmt), ws + p.off_gact,
                             act_scale_row_bytes(fmt) > 0 ? A->scale : nullptr, (int)act_scale_row_bytes(fmt),
                             act_scale_row_bytes(fmt) > 0 ? ws + p.off_gsf : nullptr,
                             reinterpret_cast<int*>(ws + p.off_rowoff), (cudaStream_t)stream);
    if (err != cudaSuccess) return HQ_ERR_CUDA;
  }
  a.grouped = p.grouped;
  a.row_off = p.grouped ? reinterpret_cast<const int*>(ws + p.off_rowoff) : nullptr;
  a.w = static_cast<const uint8_t*>(packedW);
  a.w_expert_bytes = g.expert_bytes;
  a.w_blk = g.blk_bytes;
  a.w_gscale = g.gscale_off >= 0 ? reinterpret_cast<const float*>(a.w + g.gscale_off) : nullptr;
  a.a_scale = fmt->act_type == HQ_A_NVFP4 ? A->global_scale
                                            : (fmt->act_type == HQ_A_E4M3_TOKEN ? static_cast<const float*>(A->scale)
                                                                                 : nullptr);
  a.bias = nullptr;
  a.c = static_cast<uint16_t*>(C);
  a.M = (int)T;
  a.N = (int)fmt->N;
  a.K = (int)fmt->K;
  a.n_tiles = (int)p.n_tiles;
  a.kst = (int)p.kst;
  a.zp = fmt->has_zero;
  a.moe = 1;
  a.E = (int)E;
  a.topk = a_div;
  a.topk_w = topk_weights;
  a.comb = comb;
  a.comb_k = topk;
  a.counts = counts;
  a.region = region;
  a.ids = p.fused ? topk_ids : nullptr;
  a.fused_rows = p.fused ? (int)(T * topk) : 0;
  a.region_cap = (int)p.region_cap;
  a.m_tiles = 0;
  a.sk = p.sk;
  a.status = status;
  a.partials = p.sk ? reinterpret_cast<float*>(ws + p.off_partials) : nullptr;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  a.w_evict_first = p.small;  // weights streamed once per call (tiles of one expert share them only at small T)
#if HQ_DEBUG_BOUNDS
  dbg_extents(a, p, T * topk, combine ? T : 0);
#endif
  err = launch_path(p, a, (cudaStream_t)stream);
  if (err != cudaSuccess || !combine) return cuda_status(err);
  return cuda_status(launch_combine_round(comb, T * fmt->N, static_cast<uint16_t*>(C), (cudaStream_t)stream));
}

}  // namespace

extern "C" {

hq_status_t hq_moe_gemm(const hq_format_t* fmt, const hq_act_t* A, const void* packedW, const int32_t* topk_ids,
                        const float* topk_weights, int64_t T, int32_t topk, void* C, void* workspace, size_t ws_bytes,
                        hq_stream_t stream) {
  return moe_call(fmt, A, packedW, topk_ids, topk_weights, T, topk, C, workspace, ws_bytes, stream, false);
}

hq_status_t hq_moe_gemm_combine(const hq_format_t* fmt, const hq_act_t* A, const void* packedW,
                                const int32_t* topk_ids, const float* topk_weights, int64_t T, int32_t topk, void* C,
                                void* workspace, size_t ws_bytes, hq_stream_t stream) {
  return moe_call(fmt, A, packedW, topk_ids, topk_weights, T, topk, C, workspace, ws_bytes, stream, true);
}

size_t hq_moe_combine_workspace_bytes(const hq_format_t* fmt, int64_t T, int32_t topk) {
  if (check_format(fmt) != HQ_OK || T < 0 || topk < 1) return 0;
  const Plan p = make_plan(fmt, T, topk, 2, num_sms());
  return comb_offset(p) + sizeof(float) * (size_t)(T * fmt->N);
}

hq_status_t hq_swiglu(const void* x, int64_t R, int64_t I, void* out, hq_stream_t stream) {
  if (R < 0 || R > kMaxRows || I < 8 || I > kMaxRows) return HQ_ERR_INVALID_ARG;
  if (I % 8) return HQ_ERR_ALIGNMENT;
  if (R == 0) return HQ_OK;
  if (!x || !out) return HQ_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return HQ_ERR_ALIGNMENT;
  return cuda_status(launch_swiglu(x, R, I, out, (cudaStream_t)stream));
}


size_t hq_quantize_act_workspace_bytes(int32_t act_type, int64_t M, int64_t K) {
  if (act_type != HQ_A_E4M3_TOKEN && act_type != HQ_A_NVFP4) return 0;
  if (M < 0 || M > kMaxRows || K < 16 || K > kMaxRows || K % 16) return 0;
  return act_type == HQ_A_NVFP4 ? sizeof(float) * (size_t)hq::ACT_AMAX_MAX_PARTS : 0;
}

hq_status_t hq_quantize_act(int32_t act_type, const void* x, int64_t M, int64_t K, const float* global_amax,
                            void* out_data, void* out_scale, float* out_global, void* workspace, size_t ws_bytes,
                            hq_stream_t stream) {
  if (act_type != HQ_A_E4M3_TOKEN && act_type != HQ_A_NVFP4) return HQ_ERR_UNSUPPORTED;
  if (M < 0 || M > kMaxRows || K < 16 || K > kMaxRows) return HQ_ERR_INVALID_ARG;
  if (K % 16) return HQ_ERR_ALIGNMENT;
  const bool fp8 = act_type == HQ_A_E4M3_TOKEN;
  if (!fp8 && !out_global) return HQ_ERR_INVALID_ARG;
  if (M > 0 && (!x || !out_data || !out_scale)) return HQ_ERR_INVALID_ARG;
  if (M > 0 && (!aligned16(x) || !aligned16(out_data) || !aligned16(out_scale))) return HQ_ERR_ALIGNMENT;
  if (!fp8 && !global_amax) {
    if (!workspace || ws_bytes < hq_quantize_act_workspace_bytes(act_type, M, K)) return HQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return HQ_ERR_ALIGNMENT;
  }
  if (fp8 && M == 0) return HQ_OK;
  return cuda_status(hq::launch_act_quant(fp8 ? 1 : 0, x, M, K, global_amax, out_data, out_scale, out_global,
                                          workspace, (cudaStream_t)stream));
}

hq_status_t hq_last_device_status(void* workspace, int32_t* status_out, hq_stream_t stream) {
  if (!workspace || !status_out) return HQ_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(v), (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return HQ_ERR_CUDA;
  *status_out = v;
  return HQ_OK;
}

void hq_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : DEFAULT_WAIT_NS, std::memory_order_relaxed); }

const char* hq_status_string(hq_status_t s) {
  switch (s) {
    case HQ_OK: return "ok";
    case HQ_ERR_INVALID_ARG: return "invalid argument";
    case HQ_ERR_UNSUPPORTED: return "unsupported format combination";
    case HQ_ERR_ALIGNMENT: return "misaligned pointer or K not a multiple of the K tile";
    case HQ_ERR_CUDA: return "CUDA runtime error";
    case HQ_ERR_TIMEOUT: return "device pipeline wait timed out";
    case HQ_ERR_BAD_ROUTING: return "top-k expert id out of range or rows per expert over capacity";
    case HQ_ERR_WORKSPACE: return "workspace missing or too small";
#if HQ_DEBUG_BOUNDS
    case HQ_ERR_BOUNDS: return "device index outside its buffer (debug build: the access was skipped)";
#endif
    default: return "unknown status";
  }
}

}  // extern "C"
