"""Python binding of the GB300 MXFP4 MoE expert-FFN library (libmoe_ffn.so).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C names of include/moe_ffn.h and take device
pointers as ints or torch tensors (their data_ptr()).  There is no fallback:
if the library is not built, loading it raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_ffn.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_OOM = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_INTERNAL = 4, 5, 6
MOE_OPT_PATH, MOE_OPT_TIMING, MOE_OPT_SCORING, MOE_OPT_ROUTED_SCALE, MOE_OPT_ACT_FORMAT = 1, 2, 3, 4, 5
MOE_OPT_SHARED_FORMAT, MOE_OPT_WAIT_LIMIT = 6, 7
WAIT_LIMIT_DEFAULT = 1 << 24
MOE_SHARED_MXFP4, MOE_SHARED_FP8_B32 = 0, 1
MOE_SCORING_SOFTMAX, MOE_SCORING_SIGMOID = 0, 1
MOE_ACT_FP8, MOE_ACT_FP4 = 0, 1
PATH_AUTO, PATH_SIMT, PATH_MMA = 0, 1, 2

# every symbol include/moe_ffn.h declares
EXPORTS = ("moe_layer_create", "moe_destroy", "moe_layer_destroy", "moe_route", "moe_forward", "moe_step",
           "moe_forward_host", "moe_quantize_act", "moe_quantize_act4", "moe_segments", "moe_rmsnorm", "moe_sync",
           "moe_set_option", "moe_get_kernel_times", "moe_status_string", "moe_abi_version",
           "moe_route_static", "moe_stack_forward_host", "moe_layer_create_range", "moe_forward_partial",
           "moe_combine_partials")
ROUTE_STATIC_MAX_TOKENS = 64


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class MoeConfig(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("inter", C.c_int32), ("n_experts", C.c_int32),
                ("top_k", C.c_int32), ("n_shared", C.c_int32), ("max_tokens", C.c_int32)]


class MxMat(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p)]


class MoeWeights(C.Structure):
    _fields_ = [("gate", MxMat), ("up", MxMat), ("down", MxMat),
                ("s_gate", MxMat), ("s_up", MxMat), ("s_down", MxMat),
                ("router_w", C.c_void_p), ("router_b", C.c_void_p)]


_lib = None
P = C.c_void_p
I32 = C.c_int32


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        L.moe_layer_create.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights), C.c_int,
                                       C.POINTER(P)]
        L.moe_destroy.argtypes = [P]
        L.moe_layer_destroy.argtypes = [P]
        L.moe_route.argtypes = [P, P, I32, P, P, P, P, P]
        L.moe_forward.argtypes = [P, P, I32, P, P, P, P, P]
        L.moe_step.argtypes = [P, P, I32, P, P, P, P, P, P]
        L.moe_forward_host.argtypes = [P, P, I32, P, P]
        L.moe_quantize_act.argtypes = [P, P, I32, P, P, P]
        L.moe_quantize_act4.argtypes = [P, P, I32, P, P, P]
        L.moe_segments.argtypes = [P, P, I32, P, P, P]
        L.moe_rmsnorm.argtypes = [P, I32, I32, C.c_float, P, P]
        L.moe_sync.argtypes = [P, P]
        L.moe_set_option.argtypes = [P, I32, C.c_int64]
        L.moe_get_kernel_times.argtypes = [P, C.POINTER(C.c_char_p), C.POINTER(C.c_double),
                                           C.POINTER(C.c_int64), I32, C.POINTER(I32)]
        L.moe_route_static.argtypes = [P, I32, I32, I32, I32, P, P, P, P, P]
        L.moe_stack_forward_host.argtypes = [P, I32, P, I32, C.c_float, P, P]
        L.moe_layer_create_range.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights), C.c_int, I32, I32,
                                             C.POINTER(P)]
        L.moe_forward_partial.argtypes = [P, P, I32, P, P, P, P]
        L.moe_combine_partials.argtypes = [P, I32, I32, I32, P, P, P]
        L.moe_status_string.argtypes = [C.c_int]
        L.moe_status_string.restype = C.c_char_p
        L.moe_abi_version.restype = I32
        for name in EXPORTS:
            if name not in ("moe_status_string", "moe_abi_version"):
                getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def ptr(t) -> int | None:
    """Device/host address of a tensor, array or int (None stays NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def stream_handle(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> int:
    if status != MOE_OK:
        raise MoeError(status, where)
    return status


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_layer_create(cfg: MoeConfig, weights: MoeWeights, device: int = 0) -> int:
    h = P()
    _check(lib().moe_layer_create(C.byref(cfg), C.byref(weights), device, C.byref(h)),
           "moe_layer_create")
    return h.value


def moe_destroy(h: int) -> None:
    _check(lib().moe_destroy(h), "moe_destroy")


def moe_layer_create_range(cfg: MoeConfig, weights: MoeWeights, expert_begin: int, expert_end: int,
                           device: int = 0) -> int:
    h = P()
    _check(lib().moe_layer_create_range(C.byref(cfg), C.byref(weights), device, expert_begin, expert_end,
                                        C.byref(h)), "moe_layer_create_range")
    return h.value


def moe_forward_partial(h, x, T, topk_idx, topk_w, y_partial, stream=None) -> None:
    _check(lib().moe_forward_partial(h, ptr(x), T, ptr(topk_idx), ptr(topk_w), ptr(y_partial),
                                     stream_handle(stream)), "moe_forward_partial")


def moe_combine_partials(partials, n_parts, T, H, residual, y, stream=None) -> None:
    _check(lib().moe_combine_partials(ptr(partials), n_parts, T, H, ptr(residual), ptr(y), stream_handle(stream)),
           "moe_combine_partials")


def moe_layer_destroy(h: int) -> None:
    _check(lib().moe_layer_destroy(h), "moe_layer_destroy")


def moe_route(h, x, T, logits_in, logits_out, topk_idx, topk_w, stream=None) -> None:
    _check(lib().moe_route(h, ptr(x), T, ptr(logits_in), ptr(logits_out), ptr(topk_idx),
                           ptr(topk_w), stream_handle(stream)), "moe_route")


def moe_forward(h, x, T, topk_idx, topk_w, residual, y, stream=None) -> None:
    _check(lib().moe_forward(h, ptr(x), T, ptr(topk_idx), ptr(topk_w), ptr(residual), ptr(y),
                             stream_handle(stream)), "moe_forward")


def moe_step(h, x, T, residual, y, topk_idx=None, topk_w=None, logits_out=None,
             stream=None) -> None:
    _check(lib().moe_step(h, ptr(x), T, ptr(residual), ptr(y), ptr(topk_idx), ptr(topk_w),
                          ptr(logits_out), stream_handle(stream)), "moe_step")


def moe_forward_host(h, x_host, T, y_host, stream=None) -> None:
    _check(lib().moe_forward_host(h, ptr(x_host), T, ptr(y_host), stream_handle(stream)),
           "moe_forward_host")


def moe_quantize_act(h, x, T, q, s, stream=None) -> None:
    _check(lib().moe_quantize_act(h, ptr(x), T, ptr(q), ptr(s), stream_handle(stream)),
           "moe_quantize_act")


def moe_quantize_act4(h, x, T, q, s, stream=None) -> None:
    _check(lib().moe_quantize_act4(h, ptr(x), T, ptr(q), ptr(s), stream_handle(stream)),
           "moe_quantize_act4")


def moe_segments(h, topk_idx, T, offsets, perm, stream=None) -> None:
    _check(lib().moe_segments(h, ptr(topk_idx), T, ptr(offsets), ptr(perm), stream_handle(stream)),
           "moe_segments")


def moe_rmsnorm(x, T, H, eps, out, stream=None) -> None:
    _check(lib().moe_rmsnorm(ptr(x), T, H, eps, ptr(out), stream_handle(stream)), "moe_rmsnorm")


def moe_route_static(x, T, H, E, k, router_w, router_b, topk_idx, topk_w, stream=None) -> None:
    """Router that allocates nothing (its scratch is built into the library);
    the same results as moe_route for up to ROUTE_STATIC_MAX_TOKENS tokens."""
    _check(lib().moe_route_static(ptr(x), T, H, E, k, ptr(router_w), ptr(router_b), ptr(topk_idx),
                                  ptr(topk_w), stream_handle(stream)), "moe_route_static")


def moe_stack_forward_host(handles, x_host, T, norm_eps, y_host, stream=None) -> None:
    """A stack of layers (handles, or Layer objects) from host x to host y:
    per layer x = x + step(rmsnorm(x)) (norm_eps >= 0) or x + step(x) (norm_eps < 0)."""
    hs = [h.handle if isinstance(h, Layer) else h for h in handles]
    arr = (P * len(hs))(*hs)
    _check(lib().moe_stack_forward_host(arr, len(hs), ptr(x_host), T, norm_eps, ptr(y_host),
                                        stream_handle(stream)), "moe_stack_forward_host")


def moe_sync(h, stream=None) -> int:
    """Returns the status (does not raise), so callers can test error paths."""
    return lib().moe_sync(h, stream_handle(stream))


def moe_set_option(h, option: int, value: int) -> None:
    _check(lib().moe_set_option(h, option, value), "moe_set_option")


def moe_get_kernel_times(h) -> list[tuple[str, float, int]]:
    cap = 16
    names = (C.c_char_p * cap)()
    ms = (C.c_double * cap)()
    cnt = (C.c_int64 * cap)()
    n = I32()
    _check(lib().moe_get_kernel_times(h, names, ms, cnt, cap, C.byref(n)), "moe_get_kernel_times")
    return [(names[i].decode(), ms[i], cnt[i]) for i in range(min(n.value, cap))]


class Layer:
    """Owns one moe_layer handle and keeps the weight tensors it borrows alive.

    weights: dict with gate/up/down(_codes|_scales) banks, s_gate/s_up/s_down
    (_codes|_scales) shared banks, router_w and optional router_b, all CUDA
    tensors in the canonical layout of include/moe_ffn.h.
    """

    def __init__(self, hidden, inter, n_experts, top_k, n_shared, max_tokens, weights: dict,
                 device: int = 0, expert_range: tuple[int, int] | None = None):
        self.cfg = MoeConfig(hidden, inter, n_experts, top_k, n_shared, max_tokens)
        self.weights = weights
        w = MoeWeights()
        for m in ("gate", "up", "down", "s_gate", "s_up", "s_down"):
            setattr(w, m, MxMat(ptr(weights.get(f"{m}_codes")), ptr(weights.get(f"{m}_scales"))))
        w.router_w = ptr(weights["router_w"])
        w.router_b = ptr(weights.get("router_b"))
        self._w = w
        if expert_range is None:
            self.handle = moe_layer_create(self.cfg, w, device)
        else:  # expert parallelism: the routed banks hold experts expert_range[0] .. [1] - 1
            self.handle = moe_layer_create_range(self.cfg, w, expert_range[0], expert_range[1], device)

    def route(self, x, T, idx, w, logits_in=None, logits_out=None, stream=None):
        moe_route(self.handle, x, T, logits_in, logits_out, idx, w, stream)

    def forward(self, x, T, idx, w, y, residual=None, stream=None):
        moe_forward(self.handle, x, T, idx, w, residual, y, stream)

    def step(self, x, T, y, residual=None, idx=None, w=None, logits_out=None, stream=None):
        moe_step(self.handle, x, T, residual, y, idx, w, logits_out, stream)

    def forward_partial(self, x, T, idx, w, y_partial, stream=None):
        moe_forward_partial(self.handle, x, T, idx, w, y_partial, stream)

    def forward_host(self, x_host, T, y_host, stream=None):
        moe_forward_host(self.handle, x_host, T, y_host, stream)

    def quantize_act(self, x, T, q, s, stream=None):
        moe_quantize_act(self.handle, x, T, q, s, stream)

    def quantize_act4(self, x, T, q, s, stream=None):
        moe_quantize_act4(self.handle, x, T, q, s, stream)

    def set_act_format(self, fmt: int):
        """MOE_ACT_FP8 (the layer's definition) or MOE_ACT_FP4 (the variant)."""
        moe_set_option(self.handle, MOE_OPT_ACT_FORMAT, fmt)

    def set_shared_format(self, fmt: int):
        """MOE_SHARED_MXFP4 (default) or MOE_SHARED_FP8_B32 for the shared experts' weights."""
        moe_set_option(self.handle, MOE_OPT_SHARED_FORMAT, fmt)

    def segments(self, idx, T, offsets, perm, stream=None):
        moe_segments(self.handle, idx, T, offsets, perm, stream)

    def sync(self, stream=None) -> int:
        return moe_sync(self.handle, stream)

    def set_option(self, option, value):
        moe_set_option(self.handle, option, value)

    def set_scoring(self, scoring: int, routed_scale: float = 1.0):
        """Scoring mode (MOE_SCORING_*) and routed scaling factor."""
        import struct
        moe_set_option(self.handle, MOE_OPT_SCORING, scoring)
        moe_set_option(self.handle, MOE_OPT_ROUTED_SCALE,
                       struct.unpack("<I", struct.pack("<f", routed_scale))[0])

    def kernel_times(self):
        return moe_get_kernel_times(self.handle)

    def close(self):
        if self.handle:
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
