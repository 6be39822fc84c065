/* hq.h -- C ABI of the GB300 (sm_103a) fused-dequantization quantized GEMM library.
 *
 * The operation is the one the Humming announcement describes for its kernel
 * library: low-bit weights in a unified "standard format" ("A unified
 * quantization representation"), repacked into a kernel layout ("Tuning and JIT
 * compilation per workload", preprocessing paragraph), multiplied by BF16, FP8
 * or FP4 activations with dequantization and scaling inside the kernel and the
 * scales, top-k weights and bias applied in the output stage ("Shared CUDA
 * components across formats and architectures"), for dense GEMMs and for MoE
 * GEMMs whose tokens are spread over experts ("Results: kernel
 * microbenchmarks", WnA16 paragraph on the Indexed and Grouped MoE paths).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers, 16-byte aligned, owned by the
 *    caller.  The library never allocates or frees device memory.
 *  - Calls are asynchronous on `stream`; they return after enqueueing work.
 *    Argument errors are detected on the host and returned synchronously
 *    before anything is enqueued.  Errors found by a kernel (a bounded wait
 *    that timed out, a routing id out of range) are recorded in the status
 *    word at the start of the workspace; read it with hq_last_device_status.
 *  - No C++ exception crosses this interface.  Calls on different streams
 *    with different workspaces may run concurrently: the library keeps no
 *    mutable state of its own between calls, with two exceptions, both
 *    described at their declarations: hq_gemm_static_scratch, whose calls on a
 *    device share one scratch array and must be ordered, and the process-wide
 *    wait bound set by hq_set_wait_limit_ns.
 *  - Kernels are launched with programmatic stream serialization: a call's
 *    kernels may start while the previous kernel on the stream finishes, and
 *    wait for it before touching activations, routing tables, workspace or
 *    outputs.  Packed weights are read-only inputs that a dense GEMM starts
 *    copying before that wait, so they must be complete when the preceding
 *    kernel lets its dependents launch: true for hq_pack_weights and for any
 *    kernel that never executes griddepcontrol.launch_dependents.  Setting
 *    HQ_PDL=0 in the environment restores plain stream order.
 *  - Weights W are [N, K] per expert ("out, in", as for a linear layer);
 *    the product is C[m, n] = sum_k A[m, k] * Wdeq[n, k].
 *  - 4-bit codes are stored two per byte, the low nibble holding the even k.
 */
#ifndef HQ_H_
#define HQ_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HQ_API __attribute__((visibility("default")))
#else
#define HQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* hq_stream_t;

typedef enum {
  HQ_OK = 0,
  HQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent descriptor */
  HQ_ERR_UNSUPPORTED = 2, /* a format combination this library does not implement */
  HQ_ERR_ALIGNMENT = 3,   /* a pointer not 16-byte aligned, or K not a multiple of the tile */
  HQ_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch error, no device) */
  HQ_ERR_TIMEOUT = 5,     /* device: a pipeline wait exceeded its time limit; the output is undefined */
  HQ_ERR_BAD_ROUTING = 6, /* device: a top-k expert id outside [0, E) or repeated within a token */
  HQ_ERR_WORKSPACE = 7,   /* workspace missing or smaller than hq_workspace_bytes() */
  HQ_ERR_BOUNDS = 8       /* device, debug build (libhq_debug.so) only: an index outside its buffer was caught
                             before a store or partial-sum access, which was skipped; the output is undefined */
} hq_status_t;

/* Weight numeric formats (the "standard format" parameters). */
enum {
  HQ_W_INT4_SYM = 1, /* q in [-7, 7] two's complement nibbles (the e0m3 value set), bf16 scale per group */
  HQ_W_UINT4_ZP = 2, /* q, z in [0, 15], value (q - z) * s, bf16 scale and uint4 zero per group */
  HQ_W_NVFP4 = 3,    /* e2m1 codes, ue4m3 scale per 16 K, fp32 global scale per expert */
  HQ_W_MXFP4 = 4,    /* e2m1 codes, e8m0 scale per 32 K (OCP Microscaling) */
  HQ_W_INT8_SYM = 5, /* q in [-127, 127] one two's complement byte each (the e0m7 value set), bf16 scale per group */
  HQ_W_UINT2_ZP = 6, /* q, z in [0, 3], value (q - z) * s, four codes per byte, bf16 scale and zero per group */
  HQ_W_MXINT4 = 7,   /* q in [-7, 7] two's complement nibbles, e8m0 scale per 32 K */
  HQ_W_E4M3 = 8,     /* OCP FP8 E4M3 codes, one byte each, bf16 scale per group */
  HQ_W_UINT1_ZP = 9, /* q, z in {0, 1}, value (q - z) * s, eight codes per byte, bf16 scale and zero per group */
  HQ_W_UINT3_ZP = 10 /* q, z in [0, 7], value (q - z) * s, a 3-bit bit string, bf16 scale and zero per group */
};
/* Scale data types. */
enum { HQ_S_BF16 = 1, HQ_S_UE4M3 = 2, HQ_S_UE8M0 = 3 };
/* Activation formats. */
enum {
  HQ_A_BF16 = 1,       /* bf16 [M, K] */
  HQ_A_E4M3_TOKEN = 2, /* e4m3 [M, K] bytes + fp32 scale per row (token) */
  HQ_A_NVFP4 = 3,      /* e2m1 [M, K/2] packed + ue4m3 [M, K/16] + fp32 global scale [1] */
  HQ_A_MXFP8 = 4,      /* e4m3 [M, K] bytes + e8m0 [M, K/32] block scales (OCP Microscaling MXFP8) */
  HQ_A_MXFP4 = 5       /* e2m1 [M, K/2] packed (low nibble = even k) + e8m0 [M, K/32] (OCP Microscaling MXFP4) */
};

/* The unified quantization description ("standard format").  Supported
 * combinations:
 *   INT4_SYM, group 128, BF16 scales,  no zero, no global, act BF16
 *   UINT4_ZP, group 128, BF16 scales,  zero,    no global, act BF16
 *   NVFP4,    group 16,  UE4M3 scales, no zero, global,    act NVFP4
 *   MXFP4,    group 32,  UE8M0 scales, no zero, no global, act E4M3_TOKEN, MXFP8 or MXFP4
 *   INT8_SYM, group 128, BF16 scales,  no zero, no global, act BF16
 *   UINT2_ZP, group 128, BF16 scales,  zero,    no global, act BF16
 *   MXINT4,   group 32,  UE8M0 scales, no zero, no global, act BF16
 *   E4M3,     group 128, BF16 scales,  no zero, no global, act BF16
 *   UINT1_ZP, group 128, BF16 scales,  zero,    no global, act BF16
 *   UINT3_ZP, group 128, BF16 scales,  zero,    no global, act BF16
 * The last six are the other WnA16 widths and formats of "Results: kernel
 * microbenchmarks" (INT1, INT2, INT3 as GPTQ-style unsigned codes with integer
 * zero points, INT8 as the zero-exponent e0m7 of "Results: quantization
 * support", MXINT4, FP8); MXFP8 and MXFP4 activations are the microscaled
 * W4A8 and W4A4 variants of "W8A8 / W4A8 / W4A4" (both need K a multiple
 * of 512).  Anything else returns HQ_ERR_UNSUPPORTED. */
typedef struct {
  int32_t weight_type;      /* HQ_W_* */
  int32_t group_size;       /* K elements per scale */
  int32_t scale_type;       /* HQ_S_* */
  int32_t has_zero;         /* 1 for UINT4_ZP */
  int32_t has_global_scale; /* 1 for NVFP4 */
  int32_t act_type;         /* HQ_A_* */
  int64_t N;                /* output features per expert, >= 1 */
  int64_t K;                /* input features, multiple of 256 */
  int64_t num_experts;      /* 1 for a dense layer */
} hq_format_t;

/* Activation operand.  data: see HQ_A_*; scale: fp32 [M] for E4M3_TOKEN,
 * ue4m3 [M, K/16] for NVFP4, e8m0 [M, K/32] for MXFP8 and MXFP4, NULL for
 * BF16; global_scale: fp32 [1] for NVFP4. */
typedef struct {
  const void* data;
  const void* scale;
  const float* global_scale;
} hq_act_t;

/* Bytes of the packed (kernel-layout) weight buffer for `fmt` (all experts):
 * the size of the preprocessing output ("Tuning and JIT compilation per
 * workload", preprocessing paragraph).  Returns 0 for an invalid or
 * unsupported descriptor. */
HQ_API size_t hq_packed_bytes(const hq_format_t* fmt);

/* Repack standard-format weights into the kernel layout ("Tuning and JIT
 * compilation per workload", preprocessing paragraph: validate the parameters,
 * pad N to the 128-row tile, reorder codes, scales and zeros into tile order).
 *   codes        uint8 [E][N][K/2] (4-bit formats, low nibble = even k), [E][N][K]
 *                (INT8_SYM, E4M3), [E][N][K/4] (UINT2_ZP, bits 2i..2i+1 of a byte
 *                hold its k = 4b + i) or [E][N][K*b/8] (UINT1_ZP b = 1, UINT3_ZP b = 3:
 *                a little-endian bit string, bit j of code k at bit position k*b + j
 *                of the row, position p being bit p % 8 of byte p / 8)
 *   scales       [E][N][K/group] of scale_type (bf16 as 16-bit patterns, ue4m3/e8m0 bytes)
 *   zeros        uint8 [E][N][K/group], values 0..2^b - 1 for the b-bit zero-point formats
 *                (UINT4_ZP, UINT3_ZP, UINT2_ZP, UINT1_ZP), else NULL
 *   global_scale fp32 [E] (NVFP4), else NULL
 *   packed       hq_packed_bytes(fmt) bytes, written entirely (padding zeroed)
 * Runs one kernel on `stream`.  Bit-exact and invertible by hq_unpack_weights. */
HQ_API hq_status_t hq_pack_weights(const hq_format_t* fmt, const uint8_t* codes, const void* scales, const uint8_t* zeros,
                            const float* global_scale, void* packed, hq_stream_t stream);

/* Inverse of hq_pack_weights: writes the standard-format tensors back (same
 * shapes; zeros / global_scale may be NULL when the format has none).  The
 * repack preserves each scheme's semantics ("A unified quantization
 * representation"); this call makes that checkable bit for bit. */
HQ_API hq_status_t hq_unpack_weights(const hq_format_t* fmt, const void* packed, uint8_t* codes, void* scales,
                              uint8_t* zeros, float* global_scale, hq_stream_t stream);

/* Workspace bytes for a call with M rows (dense) or T tokens with `topk`
 * experts each (MoE; pass topk = 1 for dense).  The workspace holds the
 * device status word, split-K partial sums of the Stream-K schedule and the
 * MoE routing tables (task mapping and scheduling, "Shared CUDA components
 * across formats and architectures").  It
 * must be zeroed once with hq_workspace_init before its first use; calls
 * leave it reusable.  One workspace serves one stream at a time. */
HQ_API size_t hq_workspace_bytes(const hq_format_t* fmt, int64_t M_or_T, int32_t topk);

/* Number of kernels one call launches on the current device: hq_gemm (moe = 0), hq_moe_gemm (moe = 1) or
 * hq_moe_gemm_combine (moe = 2) with M rows / T tokens and `topk` experts each (1 for dense).  Counts this library's kernels only
 * (the routing memset of hq_moe_gemm is not a kernel); 0 for an invalid format or size.  Host-only. */
HQ_API int32_t hq_kernels_per_call(const hq_format_t* fmt, int64_t M_or_T, int32_t topk, int32_t moe);

/* The launch plan of such a call on the current device (built-in rule, tuned table, HQ_TUNE): writes
 * plan_out[0] = GEMM kernel (0 tcgen05, 1 register-decode), plan_out[1] = its variant (tcgen05: 0 INT4, 1 NVFP4,
 * 2 MXFP4 x FP8, 3 MXFP4 x MXFP8, 4 MXFP4 x MXFP4; register-decode: the decode kind, 0 INT4 ... 6 UINT3),
 * plan_out[2] = token tile, plan_out[3] = 1 if K is split over CTAs (Stream-K), plan_out[4] = CTAs launched,
 * plan_out[5] = 1 if MoE rows are copied expert-contiguous first.  moe: 0 hq_gemm, 1 hq_moe_gemm, 2
 * hq_moe_gemm_combine (each kind has its own rows in the tuned table).  Returns HQ_ERR_INVALID_ARG for an invalid
 * format, size, kind or null plan_out.  Host-only ("Tuning and JIT compilation per workload": the per-size choice). */
HQ_API hq_status_t hq_launch_plan(const hq_format_t* fmt, int64_t M_or_T, int32_t topk, int32_t moe, int32_t* plan_out);

/* Zero `bytes` of workspace on `stream` (cudaMemsetAsync).  Errors:
 * HQ_ERR_INVALID_ARG for a null pointer or zero size, HQ_ERR_CUDA. */
HQ_API hq_status_t hq_workspace_init(void* workspace, size_t bytes, hq_stream_t stream);

/* Dense quantized GEMM: C[M, N] (bf16, row-major) = A . Wdeq^T (+ bias[n]).
 * Dequantization and scaling run inside the kernel, scales and the bias in the
 * output stage ("Shared CUDA components across formats and architectures");
 * the dense WnA16 / W4A4 GEMMs of "Results: kernel microbenchmarks".
 *   A       activation operand, M rows of K
 *   packedW hq_pack_weights output with num_experts == 1
 *   bias    bf16 [N] or NULL
 * Output scaling: NVFP4 multiplies by A.global_scale * W global scale,
 * E4M3_TOKEN by the row's token scale.  M may be 0 (no work).  Accumulation is
 * fp32; C is rounded to nearest-even bf16. */
HQ_API hq_status_t hq_gemm(const hq_format_t* fmt, const hq_act_t* A, const void* packedW, const void* bias, void* C,
                    int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes, hq_stream_t stream);

/* MoE grouped GEMM over E = fmt->num_experts experts: the tokens of a batch
 * spread over experts with per-expert work that varies with the routing
 * ("Results: kernel microbenchmarks", WnA16 paragraph on the Indexed and
 * Grouped MoE paths); the top-k weight is applied in the output stage.
 *   A            T token rows of K
 *   topk_ids     int32 [T, topk], distinct expert ids per token in [0, E)
 *   topk_weights fp32 [T, topk] or NULL (NULL = weight 1)
 *   C            bf16 [T * topk, N]: row t*topk + j = topk_weights[t, j] * (A[t] . Wdeq[topk_ids[t, j]]^T)
 * A row whose id is out of range is left unwritten and HQ_ERR_BAD_ROUTING is
 * recorded in the workspace status. */
HQ_API hq_status_t hq_moe_gemm(const hq_format_t* fmt, const hq_act_t* A, const void* packedW, const int32_t* topk_ids,
                        const float* topk_weights, int64_t T, int32_t topk, void* C, void* workspace, size_t ws_bytes,
                        hq_stream_t stream);

/* MoE Down GEMM with the top-k combine fused into its epilogue: the k routed
 * rows of a token are multiplied by their experts and summed with their top-k
 * weights into one output row.  A MoE layer's speed-up counts its Gate-up and
 * Down GEMMs ("Results: kernel microbenchmarks"); this is the second.
 *   A            T * topk routed rows of K (row t*topk + j feeds expert
 *                topk_ids[t, j]), in fmt->act_type: bf16, e4m3 + fp32 scale
 *                per routed row, or NVFP4
 *   topk_ids     int32 [T, topk], distinct expert ids per token in [0, E)
 *   topk_weights fp32 [T, topk] or NULL (NULL = weight 1)
 *   C            bf16 [T, N]: C[t] = sum_j topk_weights[t, j] * (A[t*topk + j] . Wdeq[topk_ids[t, j]]^T)
 *   workspace    hq_moe_combine_workspace_bytes(fmt, T, topk) bytes, zeroed
 *                once by hq_workspace_init before its first use (it holds
 *                the routing tables and an fp32 row per token)
 * N must be a multiple of 4 (HQ_ERR_ALIGNMENT).  The routed rows' products are
 * added into the fp32 rows with atomic reductions (the order of the k additions
 * is not fixed, so the last bits may vary between runs), then rounded to
 * nearest-even bf16.  A routed row whose id is out of range adds nothing and
 * records HQ_ERR_BAD_ROUTING in the workspace status. */
HQ_API size_t hq_moe_combine_workspace_bytes(const hq_format_t* fmt, int64_t T, int32_t topk);
HQ_API hq_status_t hq_moe_gemm_combine(const hq_format_t* fmt, const hq_act_t* A, const void* packedW,
                                       const int32_t* topk_ids, const float* topk_weights, int64_t T, int32_t topk,
                                       void* C, void* workspace, size_t ws_bytes, hq_stream_t stream);

/* Gated activation between a MoE layer's Gate-up and Down GEMMs:
 * out[r, c] = silu(x[r, c]) * x[r, I + c], silu(g) = g / (1 + exp(-g)), for
 * R rows of x = [gate | up] (bf16 [R, 2I], the Gate-up GEMM's output), out
 * bf16 [R, I]; fp32 arithmetic, one rounding to nearest-even bf16.  I must be
 * a multiple of 8 (HQ_ERR_ALIGNMENT); pointers 16-byte aligned. One kernel. */
HQ_API hq_status_t hq_swiglu(const void* x, int64_t R, int64_t I, void* out, hq_stream_t stream);

/* Copy the device status word out of `workspace` (synchronizes `stream`) and
 * clear it.  *status_out receives HQ_OK or the first device-detected error
 * (HQ_ERR_TIMEOUT, HQ_ERR_BAD_ROUTING); the return value reports only whether
 * the copy itself worked (HQ_ERR_INVALID_ARG, HQ_ERR_CUDA), so a failed copy is
 * never mistaken for a device error.  The announcement describes no status
 * interface; this is the library's own error channel. */
HQ_API hq_status_t hq_last_device_status(void* workspace, int32_t* status_out, hq_stream_t stream);

/* Diagnostic: bound, in nanoseconds, of every in-kernel pipeline wait of the
 * GEMM calls enqueued after this call, process-wide (default 2 s; 0 restores
 * the default).  A wait that runs out ends its kernel early with
 * HQ_ERR_TIMEOUT in the workspace status and the output undefined; the
 * kernel still lets its own copies and MMAs finish, so the workspace stays
 * reusable.  Meant for tests of that error path.  The announcement has no
 * counterpart. */
HQ_API void hq_set_wait_limit_ns(uint64_t ns);

/* Size of the fixed device scratch used by hq_gemm_static_scratch (16 MiB per GPU). */
#define HQ_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* Dense GEMM, same operands and result as hq_gemm, for callers that cannot
 * allocate device memory: code running inside a host framework that owns all
 * device memory through its own pool and forbids outside allocations, or
 * latency-critical loops where a cudaMalloc (which may synchronise the device)
 * is not acceptable.  The Humming announcement has no counterpart to this call.
 *  - No workspace argument: scratch comes from one file-scope device array of
 *    HQ_STATIC_SCRATCH_BYTES that every GPU loading this library holds until
 *    the process exits.  The call allocates nothing (no cudaMalloc or cudaFree).
 *  - Calls whose hq_workspace_bytes(fmt, M, 1) exceeds HQ_STATIC_SCRATCH_BYTES
 *    return HQ_ERR_WORKSPACE before enqueueing anything; use hq_gemm then.
 *  - The first call on a device looks up the scratch's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture on the device.
 *  - Every call on a device shares the scratch and leaves its contents behind;
 *    each call first clears the part that must start at zero (one
 *    cudaMemsetAsync on `stream`).  Calls whose executions overlap on the GPU
 *    (different streams, no ordering between them) race on the scratch and
 *    give undefined results: order them.
 *  - Device-detected errors of this variant are not readable through
 *    hq_last_device_status; use hq_gemm with a workspace to observe them. */
HQ_API hq_status_t hq_gemm_static_scratch(const hq_format_t* fmt, const hq_act_t* A, const void* packedW,
                                          const void* bias, void* C, int64_t M, int64_t N, int64_t K,
                                          hq_stream_t stream);

/* Activation quantization: bf16 activations -> the E4M3_TOKEN or NVFP4 operand
 * of hq_gemm / hq_moe_gemm.  The deployment picks a layer's activation type
 * ("Selecting activation types"): token-wise FP8 for W4A8 ("End-to-end
 * inference performance"), NVFP4 for W4A4 ("W8A8 / W4A8 / W4A4").  Scales map
 * the largest magnitude of each scaled unit to the format's largest value;
 * every step is one IEEE binary32 operation and conversions round to nearest
 * even, saturating:
 *   E4M3_TOKEN  s[m] = absmax(x[m, :]) / 448, data = e4m3(x / s[m]); a zero
 *               row gets s = 0 and zero codes.  An e4m3 zero keeps its sign.
 *   NVFP4       g = amax / (6 * 448), amax = the tensor's largest magnitude or
 *               the calibrated *global_amax; per 16 elements of a row
 *               sb = e4m3(amax_b / (6 * g)), d = value(sb) * g,
 *               code = e2m1(x / d) (+0 for a zero result; d = 0: zero codes).
 * Arguments (device pointers, 16-byte aligned, caller-owned):
 *   act_type     HQ_A_E4M3_TOKEN or HQ_A_NVFP4 (else HQ_ERR_UNSUPPORTED)
 *   x            bf16 [M, K] row-major; K a multiple of 16 (else HQ_ERR_ALIGNMENT), M >= 0
 *   global_amax  NVFP4: fp32 [1] calibrated largest magnitude, or NULL to take
 *                the tensor's own (one more kernel reads x first); ignored for E4M3_TOKEN
 *   out_data     E4M3_TOKEN: e4m3 [M, K]; NVFP4: e2m1 [M, K/2], low nibble = even k
 *   out_scale    E4M3_TOKEN: fp32 [M]; NVFP4: ue4m3 [M, K/16]
 *   out_global   NVFP4: fp32 [1] receives g; may be NULL for E4M3_TOKEN
 *   workspace    NVFP4 without global_amax: hq_quantize_act_workspace_bytes()
 *                bytes (HQ_ERR_WORKSPACE if smaller), no initialisation
 *                needed; otherwise may be NULL
 * Asynchronous on `stream`: one kernel, two for NVFP4 without global_amax. */
HQ_API size_t hq_quantize_act_workspace_bytes(int32_t act_type, int64_t M, int64_t K);
HQ_API hq_status_t hq_quantize_act(int32_t act_type, const void* x, int64_t M, int64_t K, const float* global_amax,
                                   void* out_data, void* out_scale, float* out_global, void* workspace,
                                   size_t ws_bytes, hq_stream_t stream);

/* Static description of a status code (never NULL). */
HQ_API const char* hq_status_string(hq_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* HQ_H_ */
