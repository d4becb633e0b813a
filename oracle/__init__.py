"""Python access to the fp64 CPU oracle (oracle/oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check in
__graft_entry__.py and by the cpu_baseline / reference leg of bench.py, never
by the product package.  This wrapper only marshals numpy arrays into the C
functions; every step of the arithmetic is in oracle.c.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def compile_library(src: str, out: str) -> None:
    """gcc -O2 (OpenMP, no floating-point contraction, no -march flags) of one C source."""
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp",
                           "-o", out, src, "-lm"])


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so.  ORACLE_LIB names another build of
    the same exports to load instead (the tests' planted-mistake variants)."""
    other = os.environ.get("ORACLE_LIB")
    if other:
        return other
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_library(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


P = C.c_void_p


def _declare(L):
    L.orc_e2m1_value.restype = C.c_double
    L.orc_e2m1_value.argtypes = [C.c_int]
    L.orc_ue8m0_value.restype = C.c_double
    L.orc_ue8m0_value.argtypes = [C.c_int]
    L.orc_e4m3_value.restype = C.c_double
    L.orc_e4m3_value.argtypes = [C.c_int]
    L.orc_e4m3_encode.restype = C.c_int
    L.orc_e4m3_encode.argtypes = [C.c_double]
    L.orc_block_exponent.restype = C.c_int
    L.orc_block_exponent.argtypes = [C.c_double]
    L.orc_quantize_block.argtypes = [P, C.c_int, P, P]
    L.orc_bf16_value.restype = C.c_double
    L.orc_bf16_value.argtypes = [C.c_uint16]
    L.orc_bf16_round.restype = C.c_uint16
    L.orc_bf16_round.argtypes = [C.c_double]
    L.orc_quantize_act.argtypes = [P, C.c_int, C.c_int, P, P]
    L.orc_e2m1_encode.restype = C.c_int
    L.orc_e2m1_encode.argtypes = [C.c_double]
    L.orc_block_exponent4.restype = C.c_int
    L.orc_block_exponent4.argtypes = [C.c_double]
    L.orc_quantize_block4.argtypes = [P, C.c_int, P, P]
    L.orc_quantize_act4.argtypes = [P, C.c_int, C.c_int, P, P]
    L.orc_expert_ffn_fmt.restype = C.c_int
    L.orc_expert_ffn_fmt.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P, P, P, P]
    L.orc_moe_layer_fmt.restype = C.c_int
    L.orc_moe_layer_fmt.argtypes = [C.c_int] * 7 + [P, P, P, P, P, P, P, P, C.c_int]
    L.orc_router_logits.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P, C.c_int]
    L.orc_topk.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
    L.orc_exp_f32.restype = C.c_float
    L.orc_exp_f32.argtypes = [C.c_float]
    L.orc_sigmoid_f32.restype = C.c_float
    L.orc_sigmoid_f32.argtypes = [C.c_float]
    L.orc_topk_sigmoid.argtypes = [P, P, C.c_int, C.c_int, C.c_int, C.c_double, P, P]
    L.orc_segments.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
    L.orc_expert_ffn.restype = C.c_int
    L.orc_expert_ffn.argtypes = [P, C.c_int, C.c_int, P, P, P, P, P, P]
    L.orc_moe_layer.restype = C.c_int
    L.orc_moe_layer.argtypes = [C.c_int] * 6 + [P, P, P, P, P, P, P, P, C.c_int]
    L.orc_rmsnorm.argtypes = [P, C.c_int, C.c_int, C.c_double, P]
    L.orc_max_threads.restype = C.c_int


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return lib().orc_max_threads()


# ---------------------------------------------------------------- formats
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def ue8m0_value(s: int) -> float:
    return lib().orc_ue8m0_value(int(s))


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def block_exponent(amax: float) -> int:
    return lib().orc_block_exponent(float(amax))


def quantize_block(v) -> tuple[np.ndarray, int]:
    v = _c(v, np.float64)
    q = np.zeros(v.size, np.uint8)
    s = np.zeros(1, np.uint8)
    lib().orc_quantize_block(_p(v), v.size, _p(q), _p(s))
    return q, int(s[0])


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def block_exponent4(amax: float) -> int:
    return lib().orc_block_exponent4(float(amax))


def quantize_block4(v) -> tuple[np.ndarray, int]:
    v = _c(v, np.float64)
    q = np.zeros(v.size, np.uint8)
    s = np.zeros(1, np.uint8)
    lib().orc_quantize_block4(_p(v), v.size, _p(q), _p(s))
    return q, int(s[0])


def quantize_act4(x_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """FP4 variant: packed E2M1 codes [T][H/2] (even element in the low nibble)
    and UE8M0 scale bytes [T][H/32]."""
    x = _c(x_bits, np.uint16)
    T, H = x.shape
    q = np.zeros((T, H // 2), np.uint8)
    s = np.zeros((T, H // 32), np.uint8)
    lib().orc_quantize_act4(_p(x), T, H, _p(q), _p(s))
    return q, s


def bf16_value(b: int) -> float:
    return lib().orc_bf16_value(int(b))


def bf16_round(v: float) -> int:
    return lib().orc_bf16_round(float(v))


def quantize_act(x_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    x = _c(x_bits, np.uint16)
    T, H = x.shape
    q = np.zeros((T, H), np.uint8)
    s = np.zeros((T, H // 32), np.uint8)
    lib().orc_quantize_act(_p(x), T, H, _p(q), _p(s))
    return q, s


# ---------------------------------------------------------------- routing
def router_logits(x_bits, W, b=None, threads: int = 0) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    W = _c(W, np.float32)
    T, H = x.shape
    E = W.shape[0]
    out = np.zeros((T, E), np.float32)
    bb = None if b is None else _c(b, np.float32)
    lib().orc_router_logits(_p(x), T, H, E, _p(W), None if bb is None else _p(bb), _p(out),
                            threads or max_threads())
    return out


def topk(logits, k: int) -> tuple[np.ndarray, np.ndarray]:
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    lib().orc_topk(_p(lg), T, E, k, _p(idx), _p(w))
    return idx, w


def sigmoid_f32(logits) -> np.ndarray:
    """The oracle's fp32 sigmoid (fixed sequence of fp32 operations)."""
    lg = _c(logits, np.float32).ravel()
    return np.array([lib().orc_sigmoid_f32(float(v)) for v in lg], np.float32).reshape(np.shape(logits))


def topk_sigmoid(logits, bias, k: int, scale: float = 1.0) -> tuple[np.ndarray, np.ndarray]:
    """Sigmoid scoring: selection on fp32 sigmoid(l) + bias, weights s / sum(s) * scale."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    bb = None if bias is None else _c(bias, np.float32)
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    lib().orc_topk_sigmoid(_p(lg), None if bb is None else _p(bb), T, E, k, C.c_double(scale), _p(idx), _p(w))
    return idx, w


def segments(idx, n_experts: int) -> tuple[np.ndarray, np.ndarray]:
    ix = _c(idx, np.int32)
    T, k = ix.shape
    off = np.zeros(n_experts + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    lib().orc_segments(_p(ix), T, k, n_experts, _p(off), _p(perm))
    return off, perm


# ---------------------------------------------------------------- experts
_MAT_KEYS = ("gate", "up", "down")


class _Mat(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("fmt", C.c_int)]


class _Expert(C.Structure):
    _fields_ = [("gate", _Mat), ("up", _Mat), ("down", _Mat)]


def _expert_struct(ex: dict | None, keep: list) -> _Expert:
    s = _Expert()
    if ex is None:
        return s
    for m in _MAT_KEYS:
        c = _c(ex[f"{m}_codes"], np.uint8)
        sc = _c(ex[f"{m}_scales"], np.uint8)
        keep += [c, sc]
        setattr(s, m, _Mat(c.ctypes.data, sc.ctypes.data, int(ex.get("fmt", 0))))
    return s


def expert_ffn(ex: dict, xq_row, xs_row, act4: bool = False) -> dict:
    """One expert on one quantised token (one code per element: E4M3, or E2M1
    with act4): h (fp64), its codes, o (fp64)."""
    keep: list = []
    st = _expert_struct(ex, keep)
    I, H2 = ex["gate_codes"].shape
    H = H2 if int(ex.get("fmt", 0)) == 1 else 2 * H2  # FP8 codes: one byte per element
    xq = _c(xq_row, np.uint8)
    xs = _c(xs_row, np.uint8)
    h = np.zeros(I, np.float64)
    hq = np.zeros(I, np.uint8)
    hs = np.zeros(I // 32, np.uint8)
    o = np.zeros(H, np.float64)
    rc = lib().orc_expert_ffn_fmt(C.byref(st), H, I, int(act4), _p(xq), _p(xs), _p(h), _p(hq), _p(hs),
                                  _p(o))
    if rc != 0:
        raise ValueError("oracle: expert weights missing")
    return {"h": h, "hq": hq, "hs": hs, "o": o}


def moe_layer(x_bits, idx, w, experts: dict, shared: list, n_experts: int, inter: int,
              residual=None, threads: int = 0, act4: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """The layer on T tokens.  experts maps expert id -> six arrays (only the
    ids that idx uses are needed); act4 selects the FP4-activation variant.
    Returns (y bf16 bits [T][H], y fp64)."""
    x = _c(x_bits, np.uint16)
    T, H = x.shape
    ix = _c(idx, np.int32)
    k = ix.shape[1]
    ww = _c(w, np.float64)
    keep: list = []
    arr = (_Expert * max(n_experts, 1))()
    for e, ex in experts.items():
        arr[e] = _expert_struct(ex, keep)
    sh = (_Expert * max(len(shared), 1))()
    for i, ex in enumerate(shared):
        sh[i] = _expert_struct(ex, keep)
    res = None if residual is None else _c(residual, np.uint16)
    y = np.zeros((T, H), np.uint16)
    y64 = np.zeros((T, H), np.float64)
    rc = lib().orc_moe_layer_fmt(T, H, inter, n_experts, k, len(shared), int(act4), _p(x), _p(ix), _p(ww),
                             C.cast(arr, C.c_void_p), C.cast(sh, C.c_void_p),
                             None if res is None else _p(res), _p(y), _p(y64),
                             threads or max_threads())
    if rc != 0:
        raise ValueError("oracle: a routed expert is missing or out of range")
    return y, y64


def rmsnorm(x_bits, eps: float = 1e-6) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    T, H = x.shape
    out = np.zeros((T, H), np.uint16)
    lib().orc_rmsnorm(_p(x), T, H, float(eps), _p(out))
    return out
