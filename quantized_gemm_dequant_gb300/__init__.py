"""Python binding of libhq (GB300 fused-dequantization quantized GEMM).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  torch provides device memory and the current stream.  Importing
this package fails loudly if libhq.so has not been built (run
`python -c "import __graft_entry__ as g; g.build()"` or
`python quantized_gemm_dequant_gb300/build.py`).  With HQ_LIBRARY=debug in the
environment it loads libhq_debug.so instead: the same kernels with device-side
index checks that report HQ_ERR_BOUNDS through the workspace status.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
DEBUG = os.environ.get("HQ_LIBRARY", "") == "debug"
LIB_PATH = os.path.join(_HERE, "libhq_debug.so" if DEBUG else "libhq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{os.path.basename(LIB_PATH)} not found at {LIB_PATH}: build the CUDA library first "
                      "(quantized_gemm_dequant_gb300/build.py" + (" --debug)" if DEBUG else ")"))

_lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- C types
HQ_OK, HQ_ERR_INVALID_ARG, HQ_ERR_UNSUPPORTED, HQ_ERR_ALIGNMENT, HQ_ERR_CUDA, HQ_ERR_TIMEOUT, \
    HQ_ERR_BAD_ROUTING, HQ_ERR_WORKSPACE, HQ_ERR_BOUNDS = range(9)
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


class HQArgError(HQError, ValueError):
    """A tensor argument refused by the binding before the library is called: of the wrong type, dtype or layout,
    smaller than the call reads or writes, or not in the current CUDA device's memory.  The C ABI takes bare
    pointers and sizes, so such a tensor would otherwise reach the kernels as a wrong or out-of-bounds address."""

    def __init__(self, where, msg):
        self.code = HQ_ERR_INVALID_ARG
        RuntimeError.__init__(self, f"{where}: {msg}")


def status_string(code):
    return _lib.hq_status_string(int(code)).decode()


def _check(code, where):
    if code != HQ_OK:
        raise HQError(code, where)


# bits of one weight code and bytes of one scale, per format code (the layouts of hq_pack_weights' inputs)
_CODE_BITS = {HQ_W_INT4_SYM: 4, HQ_W_UINT4_ZP: 4, HQ_W_NVFP4: 4, HQ_W_MXFP4: 4, HQ_W_INT8_SYM: 8, HQ_W_UINT2_ZP: 2,
              HQ_W_MXINT4: 4, HQ_W_E4M3: 8, HQ_W_UINT1_ZP: 1, HQ_W_UINT3_ZP: 3}
_SCALE_BYTES = {HQ_S_BF16: 2, HQ_S_UE4M3: 1, HQ_S_UE8M0: 1}
_BF16 = (torch.bfloat16,)
_F32 = (torch.float32,)
_I32 = (torch.int32,)


class _Args:
    """The tensor arguments of one call, checked in two passes so that every tensor's type, dtype, layout and size
    are judged before any tensor's device: `add` checks one tensor (None passes: the library checks required
    pointers) and keeps it; `ptrs` then checks that every kept tensor is in the current CUDA device's memory and
    returns their pointers in the order added."""

    def __init__(self, where):
        self.where = where
        self.items = []

    def add(self, t, name, nbytes=0, dtypes=None):
        w = self.where
        if t is not None:
            if not isinstance(t, torch.Tensor):
                raise HQArgError(w, f"{name} must be a torch.Tensor, not {type(t).__name__}")
            if dtypes is not None and t.dtype not in dtypes:
                raise HQArgError(w, f"{name} has dtype {t.dtype}; expected {' or '.join(str(d) for d in dtypes)}")
            if not t.is_contiguous():
                raise HQArgError(w, f"{name} must be contiguous")
            have = t.numel() * t.element_size()
            if have < nbytes:
                raise HQArgError(w, f"{name} holds {have} bytes; the call reads or writes {nbytes}")
        self.items.append((name, t))
        return self

    def act(self, a, fmt, rows):
        """The activation operand of `rows` rows of K in fmt.act_type: data, per-row or block scales, NVFP4 global
        scale, each against the bytes the call reads."""
        K, at = fmt.K, fmt.act_type
        row = {HQ_A_BF16: 2 * K, HQ_A_E4M3_TOKEN: K, HQ_A_MXFP8: K, HQ_A_NVFP4: K // 2, HQ_A_MXFP4: K // 2}.get(at, 0)
        srow = {HQ_A_E4M3_TOKEN: 4, HQ_A_NVFP4: K // 16, HQ_A_MXFP8: K // 32, HQ_A_MXFP4: K // 32}.get(at, 0)
        if not isinstance(a, dict) or "data" not in a:
            raise HQArgError(self.where, "act must be a dict with 'data' (and 'scale', 'gscale' where the format "
                                         "has them)")
        self.add(a["data"], "act['data']", rows * row, _BF16 if at == HQ_A_BF16 else None)
        self.add(a.get("scale"), "act['scale']", rows * srow, _F32 if at == HQ_A_E4M3_TOKEN else None)
        return self.add(a.get("gscale"), "act['gscale']", 4 if at == HQ_A_NVFP4 else 0, _F32)

    def ptrs(self):
        dev = None
        out = []
        for name, t in self.items:
            if t is None:
                out.append(None)
                continue
            if not t.is_cuda:
                raise HQArgError(self.where, f"{name} is on {t.device}; the library takes device memory")
            if dev is None:
                dev = torch.cuda.current_device()
            if t.device.index != dev:
                raise HQArgError(self.where, f"{name} is on {t.device}, not on the current device cuda:{dev}")
            out.append(ctypes.c_void_p(t.data_ptr()))
        return out


def _ptr(t):
    """Pointer of a tensor this binding allocated on the current device (already known to be right)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _nbytes(t):
    return t.numel() * t.element_size()


def make_format(wfmt, N, K, num_experts=1, **override):
    """The standard-format descriptor of one of the supported weight formats."""
    wt, g, st, hz, hg, at = _WEIGHT[wfmt]
    f = Format(wt, g, st, hz, hg, at, int(N), int(K), int(num_experts))
    for k, v in override.items():
        setattr(f, k, v)
    return f


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
    if codes is None or scales is None:
        raise HQArgError("hq_pack_weights", "codes and scales are required")
    args = _standard(fmt, codes, scales, zeros, global_scale, "hq_pack_weights").add(out, "out", nb)
    p = args.ptrs()
    if out is None:
        out = torch.empty(nb, dtype=torch.uint8, device=codes.device)
        p[4] = _ptr(out)
    _check(_lib.hq_pack_weights(ctypes.byref(fmt), *p, _stream(stream)), "hq_pack_weights")
    return out


def unpack_weights(fmt, packed, codes, scales, zeros=None, global_scale=None, stream=None):
    """Inverse of pack_weights: writes the standard-format tensors (same shapes) back."""
    args = _Args("hq_unpack_weights").add(packed, "packed", packed_bytes(fmt))
    p = _standard(fmt, codes, scales, zeros, global_scale, "hq_unpack_weights", args).ptrs()
    _check(_lib.hq_unpack_weights(ctypes.byref(fmt), *p, _stream(stream)), "hq_unpack_weights")


def _standard(fmt, codes, scales, zeros, global_scale, where, args=None):
    """The standard-format weight tensors of `fmt` (codes, scales, zeros, global scale), checked against their
    sizes: codes of b bits per weight, one scale (and zero point) per group of each of E * N rows."""
    args = args or _Args(where)
    rows = fmt.num_experts * fmt.N
    groups = fmt.K // fmt.group_size if fmt.group_size > 0 else 0
    args.add(codes, "codes", rows * (fmt.K * _CODE_BITS.get(fmt.weight_type, 0) // 8))
    args.add(scales, "scales", rows * groups * _SCALE_BYTES.get(fmt.scale_type, 0))
    args.add(zeros, "zeros", rows * groups if fmt.has_zero else 0)
    return args.add(global_scale, "global_scale", 4 * fmt.num_experts if fmt.has_global_scale else 0, _F32)


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


def gemm(fmt, act, packed, M, bias=None, out=None, workspace=None, stream=None):
    """C[M, N] bf16 = A . Wdeq^T (+ bias).  `act` is {'data', 'scale'?, 'gscale'?} of device tensors."""
    w = "hq_gemm"
    args = _Args(w).act(act, fmt, M).add(packed, "packed", packed_bytes(fmt)).add(bias, "bias", 2 * fmt.N, _BF16)
    args.add(out, "out", 2 * M * fmt.N, _BF16).add(workspace, "workspace")
    pd, ps, pg, pw, pb, pc, pws = args.ptrs()
    dev = act["data"].device
    if out is None:
        out = torch.empty((M, fmt.N), dtype=torch.bfloat16, device=dev)
        pc = _ptr(out)
    if workspace is None:
        workspace = make_workspace(fmt, M, 1, dev, stream)
        pws = _ptr(workspace)
    A = Act(pd, ps, pg)
    _check(_lib.hq_gemm(ctypes.byref(fmt), ctypes.byref(A), pw, pb, pc, int(M), fmt.N, fmt.K, pws,
                        _nbytes(workspace), _stream(stream)), w)
    return out


def gemm_static_scratch(fmt, act, packed, M, bias=None, out=None, stream=None):
    """hq_gemm without a workspace: scratch comes from the library's fixed per-GPU device array."""
    w = "hq_gemm_static_scratch"
    args = _Args(w).act(act, fmt, M).add(packed, "packed", packed_bytes(fmt)).add(bias, "bias", 2 * fmt.N, _BF16)
    pd, ps, pg, pw, pb, pc = args.add(out, "out", 2 * M * fmt.N, _BF16).ptrs()
    if out is None:
        out = torch.empty((M, fmt.N), dtype=torch.bfloat16, device=act["data"].device)
        pc = _ptr(out)
    A = Act(pd, ps, pg)
    _check(_lib.hq_gemm_static_scratch(ctypes.byref(fmt), ctypes.byref(A), pw, pb, pc, int(M), fmt.N, fmt.K,
                                       _stream(stream)), w)
    return out


def _moe_args(w, fmt, act, packed, topk_ids, topk_weights, out, workspace, combine):
    """Checked arguments of a MoE call: routing ids int32 [T, topk], top-k weights fp32 [T, topk], the activation
    rows (T, or T * topk routed rows for the combine), packed weights, the bf16 output rows (T * topk, or T for the
    combine) and the workspace.  Returns (T, topk, args)."""
    if not isinstance(topk_ids, torch.Tensor) or topk_ids.dim() != 2:
        raise HQArgError(w, "topk_ids must be a 2-D [T, topk] tensor")
    T, k = int(topk_ids.shape[0]), int(topk_ids.shape[1])
    args = _Args(w).add(topk_ids, "topk_ids", 4 * T * k, _I32).add(topk_weights, "topk_weights", 4 * T * k, _F32)
    args.act(act, fmt, T * k if combine else T).add(packed, "packed", packed_bytes(fmt))
    args.add(out, "out", 2 * (T if combine else T * k) * fmt.N, _BF16).add(workspace, "workspace")
    return T, k, args


def moe_gemm(fmt, act, packed, topk_ids, topk_weights=None, out=None, workspace=None, stream=None):
    """C[T*topk, N] bf16, row t*topk+j = topk_w[t,j] * (A[t] . Wdeq[ids[t,j]]^T)."""
    w = "hq_moe_gemm"
    T, k, args = _moe_args(w, fmt, act, packed, topk_ids, topk_weights, out, workspace, combine=False)
    pid, ptw, pd, ps, pg, pw, pc, pws = args.ptrs()
    dev = act["data"].device
    if out is None:
        out = torch.empty((T * k, fmt.N), dtype=torch.bfloat16, device=dev)
        pc = _ptr(out)
    if workspace is None:
        workspace = make_workspace(fmt, T, k, dev, stream)
        pws = _ptr(workspace)
    A = Act(pd, ps, pg)
    _check(_lib.hq_moe_gemm(ctypes.byref(fmt), ctypes.byref(A), pw, pid, ptw, int(T), int(k), pc, pws,
                            _nbytes(workspace), _stream(stream)), w)
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
    w = "hq_moe_gemm_combine"
    T, k, args = _moe_args(w, fmt, act, packed, topk_ids, topk_weights, out, workspace, combine=True)
    pid, ptw, pd, ps, pg, pw, pc, pws = args.ptrs()
    dev = act["data"].device
    if out is None:
        out = torch.empty((T, fmt.N), dtype=torch.bfloat16, device=dev)
        pc = _ptr(out)
    if workspace is None:
        workspace = make_combine_workspace(fmt, T, k, dev, stream)
        pws = _ptr(workspace)
    A = Act(pd, ps, pg)
    _check(_lib.hq_moe_gemm_combine(ctypes.byref(fmt), ctypes.byref(A), pw, pid, ptw, int(T), int(k), pc, pws,
                                    _nbytes(workspace), _stream(stream)), w)
    return out


def swiglu(x, out=None, stream=None):
    """x bf16 [R, 2I] = [gate | up] -> bf16 [R, I] = silu(gate) * up."""
    w = "hq_swiglu"
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or x.shape[1] % 2:
        raise HQArgError(w, "x must be a 2-D [R, 2I] tensor")
    R, I2 = x.shape
    px, po = _Args(w).add(x, "x", 2 * R * I2, _BF16).add(out, "out", R * I2, _BF16).ptrs()
    if out is None:
        out = torch.empty((R, I2 // 2), dtype=torch.bfloat16, device=x.device)
        po = _ptr(out)
    _check(_lib.hq_swiglu(px, int(R), int(I2 // 2), po, _stream(stream)), w)
    return out


def set_wait_limit_ns(ns):
    """Bound (ns) of every in-kernel pipeline wait of the GEMM calls enqueued from now on; 0 restores 2 s."""
    _lib.hq_set_wait_limit_ns(int(ns))


def last_device_status(workspace, stream=None):
    v = ctypes.c_int32(0)
    pws, = _Args("hq_last_device_status").add(workspace, "workspace", 4).ptrs()
    _check(_lib.hq_last_device_status(pws, ctypes.byref(v), _stream(stream)), "hq_last_device_status")
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
    w = "hq_quantize_act"
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise HQArgError(w, "x must be a 2-D [M, K] tensor")
    M, K = x.shape
    at = _ACT_TYPE[afmt]
    nvfp4 = at == HQ_A_NVFP4
    args = _Args(w).add(x, "x", 2 * M * K, _BF16).add(global_amax, "global_amax", 4, _F32)
    if out is not None:
        args.add(out["data"], "out['data']", M * (K // 2) if nvfp4 else M * K)
        args.add(out["scale"], "out['scale']", M * (K // 16) if nvfp4 else 4 * M, None if nvfp4 else _F32)
        args.add(out.get("gscale"), "out['gscale']", 4 if nvfp4 else 0, _F32)
    args.add(workspace, "workspace")
    p = args.ptrs()
    dev = x.device
    if out is None:
        if afmt == "e4m3_tok":
            out = dict(data=torch.empty((M, K), dtype=torch.uint8, device=dev),
                       scale=torch.empty((M,), dtype=torch.float32, device=dev))
        else:
            out = dict(data=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                       scale=torch.empty((M, K // 16), dtype=torch.uint8, device=dev),
                       gscale=torch.empty((1,), dtype=torch.float32, device=dev))
        pd, ps, pg = _ptr(out["data"]), _ptr(out["scale"]), _ptr(out.get("gscale"))
    else:
        pd, ps, pg = p[2:5]
    pws = p[-1]
    need = quantize_act_workspace_bytes(afmt, M, K)
    if workspace is None and need > 0 and global_amax is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        pws = _ptr(workspace)
    ws_bytes = _nbytes(workspace) if workspace is not None else 0
    _check(_lib.hq_quantize_act(at, p[0], M, K, p[1], pd, ps, pg, pws, ws_bytes, _stream(stream)), w)
    return out
