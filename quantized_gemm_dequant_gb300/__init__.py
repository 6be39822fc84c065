"""Python binding of libhq (GB300 fused-dequantization quantized GEMM).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  torch provides device memory and the current stream.  Importing
this package fails loudly if libhq.so has not been built (run
`python -c "import __graft_entry__ as g; g.build()"` or
`python quantized_gemm_dequant_gb300/build.py`).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libhq.so not found at {LIB_PATH}: build the CUDA library first "
                      "(quantized_gemm_dequant_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- C types
HQ_OK, HQ_ERR_INVALID_ARG, HQ_ERR_UNSUPPORTED, HQ_ERR_ALIGNMENT, HQ_ERR_CUDA, HQ_ERR_TIMEOUT, \
    HQ_ERR_BAD_ROUTING, HQ_ERR_WORKSPACE = range(8)
HQ_W_INT4_SYM, HQ_W_UINT4_ZP, HQ_W_NVFP4, HQ_W_MXFP4 = 1, 2, 3, 4
HQ_W_INT8_SYM, HQ_W_UINT2_ZP, HQ_W_MXINT4, HQ_W_E4M3, HQ_W_UINT1_ZP, HQ_W_UINT3_ZP = 5, 6, 7, 8, 9, 10
HQ_S_BF16, HQ_S_UE4M3, HQ_S_UE8M0 = 1, 2, 3
HQ_A_BF16, HQ_A_E4M3_TOKEN, HQ_A_NVFP4, HQ_A_MXFP8, HQ_A_MXFP4 = 1, 2, 3, 4, 5

EXPORTS = ["hq_packed_bytes", "hq_pack_weights", "hq_unpack_weights", "hq_workspace_bytes", "hq_workspace_init",
           "hq_gemm", "hq_moe_gemm", "hq_last_device_status", "hq_status_string", "hq_gemm_static_scratch",
           "hq_kernels_per_call", "hq_launch_plan", "hq_quantize_act_workspace_bytes", "hq_quantize_act",
           "hq_moe_combine_workspace_bytes", "hq_moe_gemm_combine", "hq_swiglu", "hq_set_wait_limit_ns"]


class Format(ctypes.Structure):
    _fields_ = [("weight_type", ctypes.c_int32), ("group_size", ctypes.c_int32), ("scale_type", ctypes.c_int32),
                ("has_zero", ctypes.c_int32), ("has_global_scale", ctypes.c_int32), ("act_type", ctypes.c_int32),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("num_experts", ctypes.c_int64)]


class Act(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
_F = ctypes.POINTER(Format)
_A = ctypes.POINTER(Act)
_lib.hq_packed_bytes.argtypes = [_F]
_lib.hq_packed_bytes.restype = _sz
_lib.hq_pack_weights.argtypes = [_F, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.hq_pack_weights.restype = ctypes.c_int
_lib.hq_unpack_weights.argtypes = [_F, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.hq_unpack_weights.restype = ctypes.c_int
_lib.hq_workspace_bytes.argtypes = [_F, _i64, _i32]
_lib.hq_workspace_bytes.restype = _sz
_lib.hq_workspace_init.argtypes = [_vp, _sz, _vp]
_lib.hq_workspace_init.restype = ctypes.c_int
_lib.hq_gemm.argtypes = [_F, _A, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]
_lib.hq_gemm.restype = ctypes.c_int
_lib.hq_moe_gemm.argtypes = [_F, _A, _vp, _vp, _vp, _i64, _i32, _vp, _vp, _sz, _vp]
_lib.hq_moe_gemm.restype = ctypes.c_int
_lib.hq_last_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32), _vp]
_lib.hq_last_device_status.restype = ctypes.c_int
_lib.hq_gemm_static_scratch.argtypes = [_F, _A, _vp, _vp, _vp, _i64, _i64, _i64, _vp]
_lib.hq_gemm_static_scratch.restype = ctypes.c_int
_lib.hq_kernels_per_call.argtypes = [_F, _i64, _i32, _i32]
_lib.hq_kernels_per_call.restype = _i32
_lib.hq_launch_plan.argtypes = [_F, _i64, _i32, _i32, ctypes.POINTER(ctypes.c_int32)]
_lib.hq_launch_plan.restype = ctypes.c_int
_lib.hq_quantize_act_workspace_bytes.argtypes = [_i32, _i64, _i64]
_lib.hq_quantize_act_workspace_bytes.restype = _sz
_lib.hq_quantize_act.argtypes = [_i32, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.hq_quantize_act.restype = ctypes.c_int
_lib.hq_moe_combine_workspace_bytes.argtypes = [_F, _i64, _i32]
_lib.hq_moe_combine_workspace_bytes.restype = _sz
_lib.hq_moe_gemm_combine.argtypes = [_F, _A, _vp, _vp, _vp, _i64, _i32, _vp, _vp, _sz, _vp]
_lib.hq_moe_gemm_combine.restype = ctypes.c_int
_lib.hq_swiglu.argtypes = [_vp, _i64, _i64, _vp, _vp]
_lib.hq_swiglu.restype = ctypes.c_int
_lib.hq_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
_lib.hq_set_wait_limit_ns.restype = None
_lib.hq_status_string.argtypes = [ctypes.c_int]
_lib.hq_status_string.restype = ctypes.c_char_p

_WEIGHT = {"int4_sym": (HQ_W_INT4_SYM, 128, HQ_S_BF16, 0, 0, HQ_A_BF16),
           "uint4_zp": (HQ_W_UINT4_ZP, 128, HQ_S_BF16, 1, 0, HQ_A_BF16),
           "nvfp4": (HQ_W_NVFP4, 16, HQ_S_UE4M3, 0, 1, HQ_A_NVFP4),
           "mxfp4": (HQ_W_MXFP4, 32, HQ_S_UE8M0, 0, 0, HQ_A_E4M3_TOKEN),
           "int8_sym": (HQ_W_INT8_SYM, 128, HQ_S_BF16, 0, 0, HQ_A_BF16),
           "uint2_zp": (HQ_W_UINT2_ZP, 128, HQ_S_BF16, 1, 0, HQ_A_BF16),
           "mxint4": (HQ_W_MXINT4, 32, HQ_S_UE8M0, 0, 0, HQ_A_BF16),
           "e4m3": (HQ_W_E4M3, 128, HQ_S_BF16, 0, 0, HQ_A_BF16),
           "uint1_zp": (HQ_W_UINT1_ZP, 128, HQ_S_BF16, 1, 0, HQ_A_BF16),
           "uint3_zp": (HQ_W_UINT3_ZP, 128, HQ_S_BF16, 1, 0, HQ_A_BF16)}
_ACT_FMT = {"bf16": HQ_A_BF16, "e4m3_tok": HQ_A_E4M3_TOKEN, "nvfp4": HQ_A_NVFP4, "mxfp8": HQ_A_MXFP8,
            "mxfp4": HQ_A_MXFP4}


class HQError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


def status_string(code):
    return _lib.hq_status_string(int(code)).decode()


def _check(code, where):
    if code != HQ_OK:
        raise HQError(code, where)


def make_format(wfmt, N, K, num_experts=1, **override):
    """The standard-format descriptor of one of the supported weight formats."""
    wt, g, st, hz, hg, at = _WEIGHT[wfmt]
    f = Format(wt, g, st, hz, hg, at, int(N), int(K), int(num_experts))
    for k, v in override.items():
        setattr(f, k, v)
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def packed_bytes(fmt):
    return int(_lib.hq_packed_bytes(ctypes.byref(fmt)))


def pack_weights(fmt, codes, scales, zeros=None, global_scale=None, out=None, stream=None):
    """Repack standard-format weight tensors (on the GPU) into the kernel layout; returns a uint8 tensor."""
    nb = packed_bytes(fmt)
    if nb == 0:
        raise HQError(HQ_ERR_UNSUPPORTED, "hq_packed_bytes")
    if out is None:
        out = torch.empty(nb, dtype=torch.uint8, device=codes.device)
    _check(_lib.hq_pack_weights(ctypes.byref(fmt), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(global_scale),
                                _ptr(out), _stream(stream)), "hq_pack_weights")
    return out


def unpack_weights(fmt, packed, codes, scales, zeros=None, global_scale=None, stream=None):
    _check(_lib.hq_unpack_weights(ctypes.byref(fmt), _ptr(packed), _ptr(codes), _ptr(scales), _ptr(zeros),
                                  _ptr(global_scale), _stream(stream)), "hq_unpack_weights")


def workspace_bytes(fmt, rows, topk=1):
    return int(_lib.hq_workspace_bytes(ctypes.byref(fmt), int(rows), int(topk)))


def kernels_per_call(fmt, rows, topk=1, moe=False):
    """Kernels one gemm (moe=False), moe_gemm (moe=True) or moe_gemm_combine (moe="combine") call launches on the
    current device."""
    m = 2 if moe == "combine" else (1 if moe else 0)
    return int(_lib.hq_kernels_per_call(ctypes.byref(fmt), int(rows), int(topk), m))


def launch_plan(fmt, rows, topk=1, moe=False):
    """The planner's choice for such a call on the current device: dict(kernel ('umma' | 'regdec'), variant, bt, sk,
    grid, grouped)."""
    m = 2 if moe == "combine" else (1 if moe else 0)
    out = (ctypes.c_int32 * 6)()
    _check(_lib.hq_launch_plan(ctypes.byref(fmt), int(rows), int(topk), m, out), "hq_launch_plan")
    return dict(kernel="regdec" if out[0] else "umma", variant=int(out[1]), bt=int(out[2]), sk=int(out[3]),
                grid=int(out[4]), grouped=int(out[5]))


def make_workspace(fmt, rows, topk=1, device="cuda", stream=None):
    """Allocate (through torch) and zero a workspace for calls with `rows` rows / tokens."""
    nb = workspace_bytes(fmt, rows, topk)
    if nb == 0:
        raise HQError(HQ_ERR_INVALID_ARG, "hq_workspace_bytes")
    ws = torch.empty(nb, dtype=torch.uint8, device=device)
    _check(_lib.hq_workspace_init(_ptr(ws), nb, _stream(stream)), "hq_workspace_init")
    return ws


def _act(a):
    return Act(a["data"].data_ptr(), a["scale"].data_ptr() if a.get("scale") is not None else None,
               a["gscale"].data_ptr() if a.get("gscale") is not None else None)


def gemm(fmt, act, packed, M, bias=None, out=None, workspace=None, stream=None):
    """C[M, N] bf16 = A . Wdeq^T (+ bias).  `act` is {'data', 'scale'?, 'gscale'?} of device tensors."""
    dev = act["data"].device
    if out is None:
        out = torch.empty((M, fmt.N), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = make_workspace(fmt, M, 1, dev, stream)
    A = _act(act)
    _check(_lib.hq_gemm(ctypes.byref(fmt), ctypes.byref(A), _ptr(packed), _ptr(bias), _ptr(out), int(M), fmt.N,
                        fmt.K, _ptr(workspace), workspace.numel(), _stream(stream)), "hq_gemm")
    return out


def gemm_static_scratch(fmt, act, packed, M, bias=None, out=None, stream=None):
    """hq_gemm without a workspace: scratch comes from the library's fixed per-GPU device array."""
    dev = act["data"].device
    if out is None:
        out = torch.empty((M, fmt.N), dtype=torch.bfloat16, device=dev)
    A = _act(act)
    _check(_lib.hq_gemm_static_scratch(ctypes.byref(fmt), ctypes.byref(A), _ptr(packed), _ptr(bias), _ptr(out),
                                       int(M), fmt.N, fmt.K, _stream(stream)), "hq_gemm_static_scratch")
    return out


def moe_gemm(fmt, act, packed, topk_ids, topk_weights=None, out=None, workspace=None, stream=None):
    """C[T*topk, N] bf16, row t*topk+j = topk_w[t,j] * (A[t] . Wdeq[ids[t,j]]^T)."""
    T, k = topk_ids.shape
    dev = act["data"].device
    if out is None:
        out = torch.empty((T * k, fmt.N), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = make_workspace(fmt, T, k, dev, stream)
    A = _act(act)
    _check(_lib.hq_moe_gemm(ctypes.byref(fmt), ctypes.byref(A), _ptr(packed), _ptr(topk_ids), _ptr(topk_weights),
                            int(T), int(k), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)),
           "hq_moe_gemm")
    return out


def make_combine_workspace(fmt, T, topk, device="cuda", stream=None):
    """Allocate and zero a workspace for `moe_gemm_combine` with T tokens of `topk` routed rows."""
    nb = int(_lib.hq_moe_combine_workspace_bytes(ctypes.byref(fmt), int(T), int(topk)))
    if nb == 0:
        raise HQError(HQ_ERR_INVALID_ARG, "hq_moe_combine_workspace_bytes")
    ws = torch.empty(nb, dtype=torch.uint8, device=device)
    _check(_lib.hq_workspace_init(_ptr(ws), nb, _stream(stream)), "hq_workspace_init")
    return ws


def moe_gemm_combine(fmt, act, packed, topk_ids, topk_weights=None, out=None, workspace=None, stream=None):
    """MoE Down GEMM + top-k combine: act holds the T*topk routed rows (row t*topk+j -> expert ids[t, j]);
    C[T, N] bf16 with C[t] = sum_j topk_w[t, j] * (A[t*topk+j] . Wdeq[ids[t, j]]^T)."""
    T, k = topk_ids.shape
    dev = act["data"].device
    if out is None:
        out = torch.empty((T, fmt.N), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = make_combine_workspace(fmt, T, k, dev, stream)
    A = _act(act)
    _check(_lib.hq_moe_gemm_combine(ctypes.byref(fmt), ctypes.byref(A), _ptr(packed), _ptr(topk_ids),
                                    _ptr(topk_weights), int(T), int(k), _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream(stream)), "hq_moe_gemm_combine")
    return out


def swiglu(x, out=None, stream=None):
    """x bf16 [R, 2I] = [gate | up] -> bf16 [R, I] = silu(gate) * up."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous() and x.shape[1] % 2 == 0
    R, I2 = x.shape
    if out is None:
        out = torch.empty((R, I2 // 2), dtype=torch.bfloat16, device=x.device)
    _check(_lib.hq_swiglu(_ptr(x), int(R), int(I2 // 2), _ptr(out), _stream(stream)), "hq_swiglu")
    return out


def set_wait_limit_ns(ns):
    """Bound (ns) of every in-kernel pipeline wait of the GEMM calls enqueued from now on; 0 restores 2 s."""
    _lib.hq_set_wait_limit_ns(int(ns))


def last_device_status(workspace, stream=None):
    v = ctypes.c_int32(0)
    _check(_lib.hq_last_device_status(_ptr(workspace), ctypes.byref(v), _stream(stream)), "hq_last_device_status")
    return int(v.value)


def pack_inputs(inputs, device="cuda", stream=None):
    """Pack the weights of a workload dict (see the workload package) onto `device`; returns (fmt, packed)."""
    w = inputs["w"]
    E = inputs.get("E", 1)
    fmt = make_format(inputs["wfmt"], inputs["N"], inputs["K"], E)
    if "afmt" in inputs:
        fmt.act_type = _ACT_FMT[inputs["afmt"]]
    t = {k: v.to(device).contiguous() for k, v in w.items()}
    scales = t["scales"].view(torch.uint8) if t["scales"].dtype == torch.bfloat16 else t["scales"]
    packed = pack_weights(fmt, t["codes"], scales, t.get("zeros"), t.get("gscale"), stream=stream)
    return fmt, packed


_ACT_TYPE = {"e4m3_tok": HQ_A_E4M3_TOKEN, "nvfp4": HQ_A_NVFP4}


def quantize_act_workspace_bytes(afmt, M, K):
    return int(_lib.hq_quantize_act_workspace_bytes(_ACT_TYPE[afmt], int(M), int(K)))


def quantize_act(afmt, x, global_amax=None, out=None, workspace=None, stream=None):
    """bf16 activations x [M, K] (cuda) -> the activation operand dict of `gemm` / `moe_gemm`:
    'e4m3_tok': {data e4m3 bytes [M, K], scale fp32 [M]}; 'nvfp4': {data packed e2m1 [M, K/2], scale ue4m3 [M, K/16],
    gscale fp32 [1]}.  `global_amax` (NVFP4): fp32 tensor [1] with a calibrated largest magnitude, else the tensor's
    own.  `out` (same dict layout) receives the result when given."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    M, K = x.shape
    at = _ACT_TYPE[afmt]
    dev = x.device
    if out is None:
        if afmt == "e4m3_tok":
            out = dict(data=torch.empty((M, K), dtype=torch.uint8, device=dev),
                       scale=torch.empty((M,), dtype=torch.float32, device=dev))
        else:
            out = dict(data=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                       scale=torch.empty((M, K // 16), dtype=torch.uint8, device=dev),
                       gscale=torch.empty((1,), dtype=torch.float32, device=dev))
    need = quantize_act_workspace_bytes(afmt, M, K)
    if workspace is None and need > 0 and global_amax is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.hq_quantize_act(at, _ptr(x), M, K, _ptr(global_amax) if global_amax is not None else None,
                                _ptr(out["data"]), _ptr(out["scale"]),
                                _ptr(out["gscale"]) if "gscale" in out else None,
                                _ptr(workspace) if workspace is not None else None, ws_bytes, _stream(stream)),
           "hq_quantize_act")
    return out
