"""ctypes binding of libmoeq.so: same names as the C ABI in include/moeq.h.

Argument marshalling only.  Each function checks dtypes/shapes/devices of
the torch tensors it is given, allocates missing outputs with torch (the
caller side of the ABI owns memory), and passes raw device pointers plus the
current CUDA stream.  All computation happens in the library's kernels; if
the library is missing, every call raises -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoeq.so")

MQ_OK, MQ_ERR_INVALID_ARG, MQ_ERR_UNSUPPORTED, MQ_ERR_CUDA, MQ_ERR_WORKSPACE = range(5)
MQ_DEV_BAD_EXPERT_ID = 0x1
MQ_DEV_WAIT_TIMEOUT = 0x2
# moe_quant_forward_ex option flags (include/moeq.h)
MQ_FWD_W8_UINT8 = 0x1
MQ_FWD_SCALE_F16 = 0x2
MQ_FWD_SCALE_BF16 = 0x4
MQ_FWD_SCALE_PER_TENSOR = 0x8
MQ_FWD_ACT_F16 = 0x10
MQ_FWD_ROUTER_WEIGHT_ON_INPUT = 0x20
MQ_FWD_PATH_TENSOR_CORE = 0x40
MQ_FWD_PATH_DECODE = 0x80
MQ_FWD_PATH_LAYER = 0x100
_PATH_FLAGS = {"auto": 0, "tc": MQ_FWD_PATH_TENSOR_CORE, "decode": MQ_FWD_PATH_DECODE,
               "layer": MQ_FWD_PATH_LAYER}
# mq_route_opts.scoring_func
MQ_SCORING_SOFTMAX = 0
MQ_SCORING_SIGMOID = 1


class MqRouteOpts(ctypes.Structure):
    """struct mq_route_opts (include/moeq.h)."""
    _fields_ = [("scoring_func", ctypes.c_int), ("renormalize", ctypes.c_int),
                ("num_expert_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("e_score_correction_bias", ctypes.c_void_p),
                ("routed_scaling_factor", ctypes.c_float)]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGNATURES = {
    "mq_status_string": (ctypes.c_char_p, [_i32]),
    "mq_last_error_message": (ctypes.c_char_p, []),
    "mq_device_status": (_i32, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_quantize_int8_per_channel": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "moe_quantize_uint4_group": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp]),
    "moe_topk_route": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_topk_route_ex": (_i32, [_vp, _i32, _i32, _i32, ctypes.POINTER(MqRouteOpts), _vp, _vp,
                                 _vp]),
    "moe_align_capacity": (_i64, [_i32, _i32, _i32, _i32]),
    "moe_align_block": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp]),
    "moe_quant_forward_workspace": (_sz, [_i32] * 7),
    "moe_quant_forward": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                 _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "moe_quant_forward_ex": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                    _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                    ctypes.c_uint, _vp]),
    "moe_quant_forward_logits_workspace": (_sz, [_i32] * 7),
    "moe_quant_forward_logits": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                        _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                        ctypes.c_uint, _vp]),
    "moe_quant_forward_logits_ex": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                           ctypes.POINTER(MqRouteOpts), _i32, _i32, _i32, _vp,
                                           _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, ctypes.c_uint,
                                           _vp]),
    "moe_quant_forward_noalloc": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                         _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mq_kernel_launch_count": (ctypes.c_longlong, []),
    "mq_test_layer_wait_extra": (_i32, [_i32]),
    "mq_profile_enable": (_i32, [_i32]),
    "mq_profile_read": (_i32, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong), _i32]),
}

PROF_SLOTS = ("quant", "route", "align", "gemm1", "gemm2", "combine", "gather", "act_f16",
              "layer")

_lib = None


class MoeqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"moeq status {status}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libmoeq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != MQ_OK:
        msg = lib().mq_last_error_message().decode()
        raise MoeqError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def mq_kernel_launch_count() -> int:
    """Kernels launched by the library in this process so far."""
    return int(lib().mq_kernel_launch_count())


def mq_test_layer_wait_extra(extra: int) -> None:
    """Testing aid (moeq.h): with extra > 0 the one-launch layer's down
    units wait for gate/up completions that never come, and their bounded
    waits run out; 0 restores normal operation."""
    _check(lib().mq_test_layer_wait_extra(int(extra)))


def mq_profile_enable(on: bool) -> None:
    _check(lib().mq_profile_enable(int(bool(on))))


def mq_profile_read() -> dict:
    """{slot name: (total device ms, timed launches)} since the last read."""
    n = len(PROF_SLOTS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_longlong * n)()
    _check(lib().mq_profile_read(ms, cnt, n))
    return {PROF_SLOTS[i]: (float(ms[i]), int(cnt[i])) for i in range(n) if cnt[i]}


def mq_status_string(status: int) -> str:
    return lib().mq_status_string(status).decode()


def mq_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status bits."""
    flags = ctypes.c_uint32(0)
    _check(lib().mq_device_status(_stream(stream), ctypes.byref(flags)))
    return int(flags.value)


def moe_quantize_int8_per_channel(w, q=None, scale=None, stream=None):
    """bf16 [rows, cols] -> (int8 [rows, cols], float32 [rows])."""
    w2d = w.reshape(-1, w.shape[-1])
    _need(w2d, torch.bfloat16, "w", 2)
    rows, cols = w2d.shape
    if q is None:
        q = torch.empty(w.shape, dtype=torch.int8, device=w.device)
    if scale is None:
        scale = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _need(q, torch.int8, "q")
    _need(scale, torch.float32, "scale")
    if q.numel() != w.numel() or scale.numel() != rows:
        raise ValueError("q / scale have the wrong size")
    _check(lib().moe_quantize_int8_per_channel(_ptr(w2d), rows, cols, _ptr(q), _ptr(scale),
                                               _stream(stream)))
    return q, scale


def moe_quantize_uint4_group(w, group_size, stream=None):
    """bf16 [.., N, K] -> (qweight uint8 [.., N, K/2], scales f16 [.., N, K/gs],
    qzeros uint8 [.., N/2, K/gs])."""
    w2d = w.reshape(-1, w.shape[-1])
    _need(w2d, torch.bfloat16, "w", 2)
    rows, cols = w2d.shape
    lead = tuple(w.shape[:-2])
    N = w.shape[-2]
    G = cols // group_size if group_size > 0 else 0
    qw = torch.empty(*w.shape[:-1], cols // 2, dtype=torch.uint8, device=w.device)
    sc = torch.empty(*w.shape[:-1], max(G, 1), dtype=torch.float16, device=w.device)
    qz = torch.empty(*lead, N // 2, max(G, 1), dtype=torch.uint8, device=w.device)
    _check(lib().moe_quantize_uint4_group(_ptr(w2d), rows, cols, group_size, _ptr(qw), _ptr(sc),
                                          _ptr(qz), _stream(stream)))
    return qw, sc, qz


def route_opts(E, renormalize, scoring_func="softmax", num_expert_group=0, topk_group=0,
               e_score_correction_bias=None, routed_scaling_factor=1.0):
    """The router options as an mq_route_opts, and whether they are the plain
    softmax router (moe_topk_route's).  e_score_correction_bias: fp32 [E] on
    the device, or None."""
    if scoring_func not in ("softmax", "sigmoid"):
        raise ValueError("scoring_func must be 'softmax' or 'sigmoid'")
    if e_score_correction_bias is not None:
        _need(e_score_correction_bias, torch.float32, "e_score_correction_bias", 1)
        if e_score_correction_bias.numel() != E:
            raise ValueError(f"e_score_correction_bias must hold E = {E} values")
    o = MqRouteOpts(MQ_SCORING_SIGMOID if scoring_func == "sigmoid" else MQ_SCORING_SOFTMAX,
                    int(bool(renormalize)), int(num_expert_group or 0), int(topk_group or 0),
                    _ptr(e_score_correction_bias), float(routed_scaling_factor))
    plain = (scoring_func == "softmax" and (num_expert_group or 0) <= 1
             and e_score_correction_bias is None and float(routed_scaling_factor) == 1.0)
    return o, plain


def moe_topk_route(logits, k, renormalize, topk_w=None, topk_ids=None, stream=None,
                   scoring_func="softmax", num_expert_group=0, topk_group=0,
                   e_score_correction_bias=None, routed_scaling_factor=1.0):
    """fp32 [T, E] -> (topk_w fp32 [T, k], topk_ids int32 [T, k]).  Router
    options other than the defaults go through moe_topk_route_ex."""
    _need(logits, torch.float32, "logits", 2)
    T, E = logits.shape
    opts, plain = route_opts(E, renormalize, scoring_func, num_expert_group, topk_group,
                             e_score_correction_bias, routed_scaling_factor)
    if topk_w is None:
        topk_w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    if topk_ids is None:
        topk_ids = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    _need(topk_w, torch.float32, "topk_w")
    _need(topk_ids, torch.int32, "topk_ids")
    if topk_w.numel() != T * k or topk_ids.numel() != T * k:
        raise ValueError("topk_w / topk_ids must hold T * k elements")
    if plain:
        _check(lib().moe_topk_route(_ptr(logits), T, E, k, int(bool(renormalize)), _ptr(topk_w),
                                    _ptr(topk_ids), _stream(stream)))
    else:
        _check(lib().moe_topk_route_ex(_ptr(logits), T, E, k, ctypes.byref(opts), _ptr(topk_w),
                                       _ptr(topk_ids), _stream(stream)))
    return topk_w, topk_ids


def moe_align_capacity(T, k, E, block_m) -> int:
    return int(lib().moe_align_capacity(T, k, E, block_m))


def moe_align_block(topk_ids, E, block_m, stream=None):
    """int32 [T, k] -> (sorted_slot_ids [cap], block_expert [cap/bm],
    expert_offsets [E+1], num_padded [1]); all int32 on the device."""
    _need(topk_ids, torch.int32, "topk_ids", 2)
    T, k = topk_ids.shape
    cap = moe_align_capacity(T, k, E, block_m)
    if cap < 0:
        raise ValueError("bad align arguments")
    dev = topk_ids.device
    sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    block_expert = torch.empty(max(cap // block_m, 1), dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    num_padded = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib().moe_align_block(_ptr(topk_ids), T, k, E, block_m, _ptr(sorted_ids),
                                 _ptr(block_expert), _ptr(offsets), _ptr(num_padded), cap,
                                 _stream(stream)))
    return sorted_ids, block_expert, offsets, num_padded


def moe_quant_forward_workspace(T, H, I, E, k, bits=8, group_size=-1) -> int:
    return int(lib().moe_quant_forward_workspace(T, H, I, E, k, bits, group_size))


def forward_flags(x, w13, s13, bits, apply_router_weight_on_input=False, path="auto"):
    """moe_quant_forward_ex flags implied by the tensors' dtypes and shapes:
    uint8 8-bit codes (moe_wna16), float16 / bfloat16 scales, one scale per
    expert (fewer scale elements than experts x output rows), float16
    activations; and the consumers of the expert GEMMs: path "auto" (by
    GEMM and batch size), "tc" (tcgen05 for both, two launches), "decode"
    (warp-level MMAs for both) or "layer" (both GEMMs in one tcgen05
    launch, 8-bit codes)."""
    if path not in _PATH_FLAGS:
        raise ValueError("path must be 'auto', 'tc', 'decode' or 'layer'")
    f = _PATH_FLAGS[path]
    if bits == 8:
        if w13.dtype == torch.uint8:
            f |= MQ_FWD_W8_UINT8
        if s13.dtype == torch.float16:
            f |= MQ_FWD_SCALE_F16
        elif s13.dtype == torch.bfloat16:
            f |= MQ_FWD_SCALE_BF16
        if s13.numel() < w13.shape[0] * w13.shape[1]:
            f |= MQ_FWD_SCALE_PER_TENSOR
    if x.dtype == torch.float16:
        f |= MQ_FWD_ACT_F16
    if apply_router_weight_on_input:
        f |= MQ_FWD_ROUTER_WEIGHT_ON_INPUT
    return f


def check_weights(w13, w2, s13, s2, bits, has_zp, z13=None, z2=None):
    """Dtype, device and contiguity checks of the expert weights, scales and
    zero points, shared by every forward wrapper (the kernels read them
    through raw device pointers and tensor maps)."""
    if bits == 8:
        if w13.dtype not in (torch.int8, torch.uint8) or w2.dtype != w13.dtype:
            raise TypeError("8-bit weights must be int8 (or uint8 codes), both alike")
        _need(w13, w13.dtype, "w13", 3)
        _need(w2, w2.dtype, "w2", 3)
        if s13.dtype not in (torch.float32, torch.float16, torch.bfloat16) or s2.dtype != s13.dtype:
            raise TypeError("8-bit scales must be float32, float16 or bfloat16, both alike")
        _need(s13, s13.dtype, "s13")
        _need(s2, s2.dtype, "s2")
        E = w13.shape[0]
        if (s13.numel() < E * w13.shape[1]) != (s2.numel() < E * w2.shape[1]):
            raise ValueError("per-tensor scales must be given for both w13 and w2")
        if has_zp:
            if w13.dtype != torch.uint8:
                raise ValueError("zero points need uint8 codes")
            _need(z13, torch.uint8, "z13")
            _need(z2, torch.uint8, "z2")
    elif bits == 4:
        _need(w13, torch.uint8, "w13", 3)
        _need(w2, torch.uint8, "w2", 3)
        _need(s13, torch.float16, "s13")
        _need(s2, torch.float16, "s2")
        if has_zp:
            _need(z13, torch.uint8, "z13")
            _need(z2, torch.uint8, "z2")
    else:
        raise ValueError(f"bits must be 8 or 4, got {bits}")


def moe_quant_forward(x, w13, w2, s13, s2, topk_w, topk_ids, bits=8, group_size=-1,
                      has_zp=False, z13=None, z2=None, workspace=None, out=None, stream=None,
                      apply_router_weight_on_input=False, inplace=False, path="auto"):
    """The fused expert MLP (moe_quant_forward / moe_quant_forward_ex in
    include/moeq.h).  x is bf16 or f16 [T, H]; 8-bit weights are int8 with
    float32 scales (experts_int8), or uint8 codes with float32 / float16 /
    bfloat16 scales and optional per-row zeros (moe_wna16 8-bit); a scale of
    one element per expert is a per-tensor scale.  inplace=True writes the
    result into x."""
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"x must be bfloat16 or float16, got {x.dtype}")
    _need(x, x.dtype, "x", 2)
    T, H = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    k = topk_ids.shape[-1] if topk_ids.dim() == 2 else 1
    check_weights(w13, w2, s13, s2, bits, has_zp, z13, z2)
    _need(topk_w, torch.float32, "topk_w")
    _need(topk_ids, torch.int32, "topk_ids")
    flags = forward_flags(x, w13, s13, bits, apply_router_weight_on_input, path)
    ws_need = moe_quant_forward_workspace(T, H, I, E, k, bits, group_size)
    if workspace is None:
        workspace = torch.empty(max(ws_need, 16), dtype=torch.uint8, device=x.device)
    _need(workspace, torch.uint8, "workspace")
    if inplace:
        out = x
    if out is None:
        out = torch.empty(T, H, dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out", 2)
    _check(lib().moe_quant_forward_ex(
        _ptr(x), T, H, I, E, k, bits, group_size, int(bool(has_zp)),
        _ptr(w13), _ptr(w2), _ptr(s13), _ptr(s2), _ptr(z13 if has_zp else None),
        _ptr(z2 if has_zp else None), _ptr(topk_w), _ptr(topk_ids),
        _ptr(workspace), workspace.numel(), _ptr(out), flags, _stream(stream)))
    return out


def moe_quant_forward_logits(x, router_logits, w13, w2, s13, s2, top_k, renormalize=True, bits=8,
                             group_size=-1, has_zp=False, z13=None, z2=None, workspace=None,
                             out=None, stream=None, apply_router_weight_on_input=False,
                             inplace=False, scoring_func="softmax", num_expert_group=0,
                             topk_group=0, e_score_correction_bias=None,
                             routed_scaling_factor=1.0, path="auto"):
    """Routing and the expert MLP in one call (moe_quant_forward_logits, or
    moe_quant_forward_logits_ex with router options, in include/moeq.h): the
    same result as moe_topk_route followed by moe_quant_forward, bitwise."""
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"x must be bfloat16 or float16, got {x.dtype}")
    _need(x, x.dtype, "x", 2)
    _need(router_logits, torch.float32, "router_logits", 2)
    T, H = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    if router_logits.shape != (T, E):
        raise ValueError(f"router_logits must be [{T}, {E}]")
    check_weights(w13, w2, s13, s2, bits, has_zp, z13, z2)
    flags = forward_flags(x, w13, s13, bits, apply_router_weight_on_input, path)
    opts, plain = route_opts(E, renormalize, scoring_func, num_expert_group, topk_group,
                             e_score_correction_bias, routed_scaling_factor)
    ws_need = int(lib().moe_quant_forward_logits_workspace(T, H, I, E, top_k, bits, group_size))
    if workspace is None:
        workspace = torch.empty(max(ws_need, 16), dtype=torch.uint8, device=x.device)
    _need(workspace, torch.uint8, "workspace")
    if inplace:
        out = x
    if out is None:
        out = torch.empty(T, H, dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out", 2)
    tail = (bits, group_size, int(bool(has_zp)), _ptr(w13), _ptr(w2), _ptr(s13), _ptr(s2),
            _ptr(z13 if has_zp else None), _ptr(z2 if has_zp else None),
            _ptr(workspace), workspace.numel(), _ptr(out), flags, _stream(stream))
    if plain:
        _check(lib().moe_quant_forward_logits(_ptr(x), _ptr(router_logits), T, H, I, E, top_k,
                                              int(bool(renormalize)), *tail))
    else:
        _check(lib().moe_quant_forward_logits_ex(_ptr(x), _ptr(router_logits), T, H, I, E, top_k,
                                                 ctypes.byref(opts), *tail))
    return out


def moe_quant_forward_noalloc(x, w13, w2, s13, s2, topk_w, topk_ids, bits=8, group_size=-1,
                              has_zp=False, z13=None, z2=None, out=None, stream=None):
    """moe_quant_forward with the library's fixed scratch instead of a
    workspace (for callers that cannot allocate; see include/moeq.h)."""
    _need(x, torch.bfloat16, "x", 2)
    T, H = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    k = topk_ids.shape[-1] if topk_ids.dim() == 2 else 1
    check_weights(w13, w2, s13, s2, bits, has_zp, z13, z2)
    if bits == 8 and (w13.dtype != torch.int8 or s13.dtype != torch.float32
                      or s13.numel() != E * w13.shape[1]):
        raise TypeError("moe_quant_forward_noalloc takes the experts_int8 format (int8 codes, "
                        "float32 per-channel scales) or uint4")
    _need(topk_w, torch.float32, "topk_w")
    _need(topk_ids, torch.int32, "topk_ids")
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out", 2)
    _check(lib().moe_quant_forward_noalloc(
        _ptr(x), T, H, I, E, k, bits, group_size, int(bool(has_zp)),
        _ptr(w13), _ptr(w2), _ptr(s13), _ptr(s2), _ptr(z13 if has_zp else None),
        _ptr(z2 if has_zp else None), _ptr(topk_w), _ptr(topk_ids), _ptr(out), _stream(stream)))
    return out
