"""Python binding of the C-ABI library ``libmdw.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls and does no arithmetic of
its own: torch tensors supply device memory and the current CUDA stream, and every step of
the decode path runs in the library's kernels. If the library is missing or fails to load
this module raises; there is no CPU fallback.
"""

from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmdw.so")

MDW_MAGIC = 0x3157444D
FMT_BF16, FMT_FP8, FMT_MXFP4 = 1, 2, 3
STATUS = {0: "MDW_OK", 1: "MDW_ERR_INVALID_ARG", 2: "MDW_ERR_UNSUPPORTED_SHAPE",
          3: "MDW_ERR_FORMAT_MISMATCH", 4: "MDW_ERR_WORKSPACE_TOO_SMALL", 5: "MDW_ERR_CUDA",
          6: "MDW_ERR_TIMEOUT", 7: "MDW_ERR_DEVICE_BOUNDS"}
HIDDEN, INTER = 2560, 768
MAX_M, MAX_TOPK, MAX_VOCAB_TOPK, MAX_EXPERTS = 32, 8, 32, 512

# exported symbols declared in include/moe_decode_weight.h
SYMBOLS = ["mdw_status_string", "mdw_version", "mdw_moe_workspace_bytes", "mdw_moe_workspace_layout",
           "moe_decode_layer", "quantize_lm_head_fp8", "mdw_lm_head_bf16_init",
           "mdw_lm_head_workspace_bytes", "lm_head_fp8", "lm_head_bf16", "lm_head_fp8_rmsnorm",
           "mdw_stack_workspace_bytes",
           "moe_decode_stack", "mdw_device_status", "moe_decode_layer_noalloc", "mdw_sample_topk",
           "lm_head_fp8_sample", "moe_decode_stack_routed", "mdw_debug_set_spin_budget"]


class MdwError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class MoeWeightsC(C.Structure):
    _fields_ = [("magic", C.c_uint32), ("fmt", C.c_int32), ("num_experts", C.c_int32),
                ("top_k", C.c_int32), ("hidden", C.c_int32), ("inter", C.c_int32),
                ("router_w", C.c_void_p), ("w13_q", C.c_void_p), ("w13_s", C.c_void_p),
                ("w2_q", C.c_void_p), ("w2_s", C.c_void_p), ("sh_w13_q", C.c_void_p),
                ("sh_w13_s", C.c_void_p), ("sh_w2_q", C.c_void_p), ("sh_w2_s", C.c_void_p)]


class LMHeadC(C.Structure):
    _fields_ = [("magic", C.c_uint32), ("fmt", C.c_int32), ("vocab", C.c_int64),
                ("hidden", C.c_int32), ("reserved", C.c_int32), ("w", C.c_void_p),
                ("row_scale", C.c_void_p)]


class MoeWsLayoutC(C.Structure):
    _fields_ = [(n, C.c_size_t) for n in ("header", "xq", "sx", "logits", "ids", "gates",
                                          "slot_expert", "pair_token", "pair_slot", "pair_gate",
                                          "h", "hq", "sh", "total")]


_lib = None


def lib() -> C.CDLL:
    """Load libmdw.so (once) and declare its signatures. Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with moe_decode_weight_gb300.build.build()")
    L = C.CDLL(LIB_PATH)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    L.mdw_status_string.restype = C.c_char_p
    L.mdw_status_string.argtypes = [C.c_int]
    L.mdw_version.restype = i32
    L.mdw_debug_set_spin_budget.restype = i64
    L.mdw_debug_set_spin_budget.argtypes = [i64]
    L.mdw_moe_workspace_bytes.restype = sz
    L.mdw_moe_workspace_bytes.argtypes = [C.POINTER(MoeWeightsC), i32]
    L.mdw_moe_workspace_layout.restype = C.c_int
    L.mdw_moe_workspace_layout.argtypes = [C.POINTER(MoeWeightsC), i32, C.POINTER(MoeWsLayoutC)]
    L.moe_decode_layer.restype = C.c_int
    L.moe_decode_layer.argtypes = [C.POINTER(MoeWeightsC), i32, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
    L.quantize_lm_head_fp8.restype = C.c_int
    L.quantize_lm_head_fp8.argtypes = [vp, i64, i32, vp, vp, C.POINTER(LMHeadC), vp]
    L.mdw_lm_head_bf16_init.restype = C.c_int
    L.mdw_lm_head_bf16_init.argtypes = [vp, i64, i32, C.POINTER(LMHeadC)]
    L.mdw_lm_head_workspace_bytes.restype = sz
    L.mdw_lm_head_workspace_bytes.argtypes = [C.POINTER(LMHeadC), i32, i32]
    for name in ("lm_head_fp8", "lm_head_bf16", "lm_head_fp8_rmsnorm"):
        f = getattr(L, name)
        f.restype = C.c_int
        f.argtypes = [C.POINTER(LMHeadC), i32, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    L.mdw_stack_workspace_bytes.restype = sz
    L.mdw_stack_workspace_bytes.argtypes = [C.POINTER(MoeWeightsC), i32, C.POINTER(LMHeadC), i32, i32]
    L.moe_decode_stack.restype = C.c_int
    L.moe_decode_stack.argtypes = [C.POINTER(MoeWeightsC), i32, C.POINTER(LMHeadC), i32, vp, vp, vp, vp,
                                   i32, vp, vp, vp, sz, vp]
    L.moe_decode_stack_routed.restype = C.c_int
    L.moe_decode_stack_routed.argtypes = [C.POINTER(MoeWeightsC), i32, C.POINTER(LMHeadC), i32, vp, vp, vp, vp,
                                          i32, vp, vp, vp, vp, sz, vp]
    L.mdw_device_status.restype = C.c_int
    L.mdw_device_status.argtypes = [vp, vp]
    L.moe_decode_layer_noalloc.restype = C.c_int
    L.moe_decode_layer_noalloc.argtypes = [C.POINTER(MoeWeightsC), i32, vp, vp, i32, vp, vp, vp, vp, vp, vp]
    f64 = C.c_double
    L.mdw_sample_topk.restype = C.c_int
    L.mdw_sample_topk.argtypes = [i32, i32, vp, vp, f64, f64, vp, vp, vp]
    L.lm_head_fp8_sample.restype = C.c_int
    L.lm_head_fp8_sample.argtypes = [C.POINTER(LMHeadC), i32, vp, i32, i32, f64, f64, vp, vp, vp, vp, vp, sz, vp]
    _lib = L
    return L


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        raise MdwError(fn, code)


# ----------------------------------------------------------------------------- handles


@dataclass
class MoeWeights:
    """One layer's device tensors and the C descriptor that points at them."""
    router_w: torch.Tensor
    w13_q: torch.Tensor
    w13_s: torch.Tensor
    w2_q: torch.Tensor
    w2_s: torch.Tensor
    shared: tuple | None
    top_k: int = 8
    c: MoeWeightsC = field(init=False)

    def __post_init__(self):
        sh = self.shared if self.shared is not None else (None,) * 4
        self.c = MoeWeightsC(MDW_MAGIC, FMT_MXFP4, self.w13_q.shape[0], self.top_k, HIDDEN, INTER,
                             *(t.data_ptr() if t is not None else None for t in
                               (self.router_w, self.w13_q, self.w13_s, self.w2_q, self.w2_s, *sh)))


@dataclass
class LMHead:
    """A head descriptor plus the tensors it points at (kept alive here)."""
    c: LMHeadC
    tensors: tuple


def mdw_status_string(code: int) -> str:
    return lib().mdw_status_string(code).decode()


def mdw_version() -> int:
    return lib().mdw_version()


def mdw_debug_set_spin_budget(cycles: int) -> int:
    """Test hook: bound of the kernels' inter-block waits in clock64 cycles (<= 0: the
    default); returns the previous bound."""
    return lib().mdw_debug_set_spin_budget(int(cycles))


def mdw_moe_workspace_bytes(w: MoeWeights, m: int) -> int:
    return lib().mdw_moe_workspace_bytes(C.byref(w.c), m)


def mdw_moe_workspace_layout(w: MoeWeights, m: int) -> dict:
    out = MoeWsLayoutC()
    _check("mdw_moe_workspace_layout", lib().mdw_moe_workspace_layout(C.byref(w.c), m, C.byref(out)))
    return {n: getattr(out, n) for n, _ in MoeWsLayoutC._fields_}


def moe_decode_layer(w: MoeWeights, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor,
                     residual=None, topk_override=None, topk_ids_out=None, topk_w_out=None,
                     stream=None) -> None:
    m = x.shape[0]
    code = lib().moe_decode_layer(C.byref(w.c), m, _ptr(x), _ptr(y), int(y.dtype == torch.float32),
                                  _ptr(residual), _ptr(topk_override), _ptr(topk_ids_out),
                                  _ptr(topk_w_out), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream))
    _check("moe_decode_layer", code)


def moe_decode_layer_noalloc(w: MoeWeights, x: torch.Tensor, y: torch.Tensor, residual=None,
                             topk_override=None, topk_ids_out=None, topk_w_out=None,
                             device_status_out=None, stream=None) -> None:
    """moe_decode_layer for callers that cannot allocate device memory: the library's own
    fixed scratch array replaces the workspace (see the C declaration for its limits)."""
    code = lib().moe_decode_layer_noalloc(C.byref(w.c), x.shape[0], _ptr(x), _ptr(y),
                                          int(y.dtype == torch.float32), _ptr(residual),
                                          _ptr(topk_override), _ptr(topk_ids_out), _ptr(topk_w_out),
                                          _ptr(device_status_out), _stream(stream))
    _check("moe_decode_layer_noalloc", code)


def quantize_lm_head_fp8(w_bf16: torch.Tensor, q_out: torch.Tensor, scale_out: torch.Tensor,
                         stream=None) -> LMHead:
    head = LMHeadC()
    code = lib().quantize_lm_head_fp8(_ptr(w_bf16), w_bf16.shape[0], w_bf16.shape[1], _ptr(q_out),
                                      _ptr(scale_out), C.byref(head), _stream(stream))
    _check("quantize_lm_head_fp8", code)
    return LMHead(head, (q_out, scale_out))


def mdw_lm_head_bf16_init(w_bf16: torch.Tensor) -> LMHead:
    head = LMHeadC()
    _check("mdw_lm_head_bf16_init",
           lib().mdw_lm_head_bf16_init(_ptr(w_bf16), w_bf16.shape[0], w_bf16.shape[1], C.byref(head)))
    return LMHead(head, (w_bf16,))


def mdw_lm_head_workspace_bytes(head: LMHead, m: int, topk: int) -> int:
    return lib().mdw_lm_head_workspace_bytes(C.byref(head.c), m, topk)


def _head(fn: str, head: LMHead, h: torch.Tensor, argmax_out, ws, logits=None, topk=1, topk_idx=None,
          topk_val=None, stream=None):
    code = getattr(lib(), fn)(C.byref(head.c), h.shape[0], _ptr(h), _ptr(logits), _ptr(argmax_out), topk,
                              _ptr(topk_idx), _ptr(topk_val), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream))
    _check(fn, code)


def lm_head_fp8(head: LMHead, h: torch.Tensor, argmax_out: torch.Tensor, ws: torch.Tensor, logits=None,
                topk: int = 1, topk_idx=None, topk_val=None, stream=None) -> None:
    _head("lm_head_fp8", head, h, argmax_out, ws, logits, topk, topk_idx, topk_val, stream)


def lm_head_bf16(head: LMHead, h: torch.Tensor, argmax_out: torch.Tensor, ws: torch.Tensor, logits=None,
                 topk: int = 1, topk_idx=None, topk_val=None, stream=None) -> None:
    _head("lm_head_bf16", head, h, argmax_out, ws, logits, topk, topk_idx, topk_val, stream)


def lm_head_fp8_rmsnorm(head: LMHead, r: torch.Tensor, argmax_out: torch.Tensor, ws: torch.Tensor,
                        logits=None, topk: int = 1, topk_idx=None, topk_val=None, stream=None) -> None:
    _head("lm_head_fp8_rmsnorm", head, r, argmax_out, ws, logits, topk, topk_idx, topk_val, stream)


def mdw_sample_topk(topk_val: torch.Tensor, topk_idx: torch.Tensor, temperature: float, top_p: float,
                    u: torch.Tensor, token_out: torch.Tensor, stream=None) -> None:
    """Draw one token per row of the [M, k] candidates (u: float64 [M] uniforms in [0, 1))."""
    m, k = topk_val.shape
    _check("mdw_sample_topk", lib().mdw_sample_topk(m, k, _ptr(topk_val), _ptr(topk_idx), float(temperature),
                                                      float(top_p), _ptr(u), _ptr(token_out), _stream(stream)))


def lm_head_fp8_sample(head: LMHead, h: torch.Tensor, token_out: torch.Tensor, ws: torch.Tensor, u: torch.Tensor,
                       temperature: float, top_p: float, topk: int, norm_input: bool = False, topk_idx=None,
                       topk_val=None, stream=None) -> None:
    """FP8 head (optionally on bf16(RMSNorm(h))) and the draw on its top-k, in one launch per
    16 tokens."""
    _check("lm_head_fp8_sample",
           lib().lm_head_fp8_sample(C.byref(head.c), h.shape[0], _ptr(h), 1 if norm_input else 0, topk,
                                    float(temperature), float(top_p), _ptr(u), _ptr(token_out), _ptr(topk_idx),
                                    _ptr(topk_val), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def _layer_array(layers):
    """ctypes array of layer descriptors (a prebuilt array is passed through unchanged)."""
    if isinstance(layers, C.Array):
        return layers
    arr = (MoeWeightsC * len(layers))()
    for i, w in enumerate(layers):
        arr[i] = w.c
    return arr


def mdw_stack_workspace_bytes(layers, head, m: int, topk: int) -> int:
    hc = C.byref(head.c) if head is not None else None
    return lib().mdw_stack_workspace_bytes(_layer_array(layers), len(layers), hc, m, topk)


def moe_decode_stack(layers, head, r0: torch.Tensor, argmax_out, ws: torch.Tensor,
                     resid_out=None, logits=None, topk: int = 1, topk_idx=None, topk_val=None,
                     stream=None) -> None:
    """head=None runs the layers only (resid_out required); lm_head_fp8_rmsnorm finishes."""
    arr = _layer_array(layers)
    hc = C.byref(head.c) if head is not None else None
    code = lib().moe_decode_stack(arr, len(layers), hc, r0.shape[0], _ptr(r0), _ptr(resid_out),
                                  _ptr(logits), _ptr(argmax_out), topk, _ptr(topk_idx), _ptr(topk_val),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check("moe_decode_stack", code)


def moe_decode_stack_routed(layers, head, r0: torch.Tensor, argmax_out, ws: torch.Tensor, topk_override,
                            resid_out=None, logits=None, topk: int = 1, topk_idx=None, topk_val=None,
                            stream=None) -> None:
    """moe_decode_stack with imposed routing: topk_override int32 [L, M, K] on the device (or None)."""
    arr = _layer_array(layers)
    hc = C.byref(head.c) if head is not None else None
    code = lib().moe_decode_stack_routed(arr, len(layers), hc, r0.shape[0], _ptr(r0), _ptr(resid_out),
                                         _ptr(logits), _ptr(argmax_out), topk, _ptr(topk_idx), _ptr(topk_val),
                                         _ptr(topk_override), _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream))
    _check("moe_decode_stack_routed", code)


def mdw_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the device status word of the workspace."""
    return lib().mdw_device_status(_ptr(ws), _stream(stream))
