"""Seeded synthetic inputs for the MXFP4 MoE expert-FFN layer.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It holds no arithmetic of the method itself: it only turns seeds
into bytes (packed E2M1 codes, UE8M0 scale bytes), bf16 activations, fp32
router weights and an optional router bias.

Expert banks are produced by a counter-based generator so that any single
expert can be regenerated on the host without producing the whole bank: the
64-bit word j of a stream is ``mix64(key + (j + 1) * GAMMA)``, the SplitMix64
output function of Steele, Lea and Flood ("Fast splittable pseudorandom number
generators", OOPSLA 2014).  ``synth/fill.cu`` implements the same definition
on the GPU to fill multi-GB banks in place; ``tests/test_synth.py`` checks the
two produce identical bytes.

Byte i of a code stream is byte (i mod 8) (little-endian) of word i // 8.
Byte i of a scale stream is ``127 + lo + (b mod (hi - lo + 1))`` where b is
byte i of its own stream, so scales are 2**e with e uniform on [lo, hi].
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

from .workloads import WORKLOADS, Workload  # noqa: F401

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB

# stream ids: 2 * matrix + kind, matrix 0 gate / 1 up / 2 down, kind 0 codes / 1 scales
GATE, UP, DOWN = 0, 1, 2
CODES, SCALES = 0, 1


def mix64(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def fold(k: int, v: int) -> int:
    return mix64(k + (v + 1) * GAMMA)


def stream_key(seed: int, layer: int, matrix: int, kind: int, expert: int) -> int:
    """Key of the byte stream for one (seed, layer, matrix, codes|scales, expert)."""
    k = fold(0, seed)
    k = fold(k, layer)
    k = fold(k, 2 * matrix + kind)
    return fold(k, expert)


def _words(key: int, n_words: int) -> np.ndarray:
    j = np.arange(1, n_words + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + j * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
        z = z ^ (z >> np.uint64(31))
    return z


def stream_bytes_numpy(key: int, n_bytes: int) -> np.ndarray:
    """Raw stream bytes computed with numpy (the definition, used to check hostgen.c)."""
    w = _words(key, (n_bytes + 7) // 8)
    return w.astype("<u8").view(np.uint8)[:n_bytes].copy()


_HERE = os.path.dirname(os.path.abspath(__file__))
_hostgen = None


def build_hostgen(force: bool = False) -> str:
    src = os.path.join(_HERE, "hostgen.c")
    so = os.path.join(_HERE, "libhostgen.so")
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        tmp = so + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src])
        os.replace(tmp, so)
    return so


def _hg():
    global _hostgen
    if _hostgen is None:
        _hostgen = ctypes.CDLL(build_hostgen())
        _hostgen.synth_host_stream.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int]
    return _hostgen


def stream_bytes(key: int, n_bytes: int, kind: int = CODES, lo: int = 0, hi: int = 0) -> np.ndarray:
    out = np.empty(n_bytes, np.uint8)
    _hg().synth_host_stream(out.ctypes.data, n_bytes, key, kind, lo, hi - lo + 1)
    return out


def code_bytes(seed, layer, matrix, expert, n_rows, k_cols) -> np.ndarray:
    """Packed E2M1 codes of one expert matrix, shape [n_rows][k_cols // 2]."""
    b = stream_bytes(stream_key(seed, layer, matrix, CODES, expert), n_rows * k_cols // 2)
    return b.reshape(n_rows, k_cols // 2)


def scale_bytes(seed, layer, matrix, expert, n_rows, k_cols, lo, hi) -> np.ndarray:
    """UE8M0 scale bytes of one expert matrix, shape [n_rows][k_cols // 32]."""
    b = stream_bytes(stream_key(seed, layer, matrix, SCALES, expert), n_rows * k_cols // 32,
                     SCALES, lo, hi)
    return b.reshape(n_rows, k_cols // 32)


def scale_bytes_numpy(seed, layer, matrix, expert, n_rows, k_cols, lo, hi) -> np.ndarray:
    b = stream_bytes_numpy(stream_key(seed, layer, matrix, SCALES, expert), n_rows * k_cols // 32)
    n = hi - lo + 1
    return (127 + lo + (b.astype(np.int32) % n)).astype(np.uint8).reshape(n_rows, k_cols // 32)


def host_expert(wl: "Workload", layer: int, expert: int) -> dict:
    """All six arrays of one expert (routed 0..E-1, shared E..E+n_shared-1)."""
    H, I, lo, hi, sd = wl.hidden, wl.inter, wl.scale_lo, wl.scale_hi, wl.seed
    return {
        "gate_codes": code_bytes(sd, layer, GATE, expert, I, H),
        "gate_scales": scale_bytes(sd, layer, GATE, expert, I, H, lo, hi),
        "up_codes": code_bytes(sd, layer, UP, expert, I, H),
        "up_scales": scale_bytes(sd, layer, UP, expert, I, H, lo, hi),
        "down_codes": code_bytes(sd, layer, DOWN, expert, H, I),
        "down_scales": scale_bytes(sd, layer, DOWN, expert, H, I, lo, hi),
    }


def host_experts(wl: "Workload", layer: int, ids) -> dict:
    """host_expert for several ids, generated on parallel host threads (the
    generator is C called through ctypes, which releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    ids = [int(e) for e in ids]
    if len(ids) <= 1:
        return {e: host_expert(wl, layer, e) for e in ids}
    with ThreadPoolExecutor(max_workers=min(len(ids), os.cpu_count() or 1)) as ex:
        return dict(zip(ids, ex.map(lambda e: host_expert(wl, layer, e), ids)))


# The shared-expert FP8 variant: E4M3 codes with one UE8M0 scale per 32 x 32
# block, drawn from streams of their own (matrix ids 4..6).  Scale exponents
# sit 6 below the MXFP4 range, since E4M3 reaches 448 where E2M1 reaches 6.
FP8_STREAM_OFFSET = 4


def fp8_code_bytes(seed, layer, matrix, expert, n_rows, k_cols) -> np.ndarray:
    """E4M3 codes of one FP8 matrix, [n_rows][k_cols]: uniform bytes with the two
    NaN codes (0x7F, 0xFF) moved to +-448 (0x7E, 0xFE)."""
    b = stream_bytes(stream_key(seed, layer, matrix + FP8_STREAM_OFFSET, CODES, expert), n_rows * k_cols)
    b = np.where((b & 0x7F) == 0x7F, b ^ 1, b).astype(np.uint8)
    return b.reshape(n_rows, k_cols)


def fp8_block_scale_bytes(seed, layer, matrix, expert, n_rows, k_cols, lo, hi) -> np.ndarray:
    """UE8M0 scale bytes of one FP8 matrix, one per 32 x 32 block: [n_rows/32][k_cols/32]."""
    n = (n_rows // 32) * (k_cols // 32)
    b = stream_bytes(stream_key(seed, layer, matrix + FP8_STREAM_OFFSET, SCALES, expert), n, SCALES, lo, hi)
    return b.reshape(n_rows // 32, k_cols // 32)


def host_expert_fp8(wl: "Workload", layer: int, expert: int) -> dict:
    """A shared expert in the FP8 (32 x 32 block) format; "fmt": 1 tells the oracle."""
    H, I, sd = wl.hidden, wl.inter, wl.seed
    lo, hi = wl.scale_lo - 6, wl.scale_hi - 6
    return {
        "fmt": 1,
        "gate_codes": fp8_code_bytes(sd, layer, GATE, expert, I, H),
        "gate_scales": fp8_block_scale_bytes(sd, layer, GATE, expert, I, H, lo, hi),
        "up_codes": fp8_code_bytes(sd, layer, UP, expert, I, H),
        "up_scales": fp8_block_scale_bytes(sd, layer, UP, expert, I, H, lo, hi),
        "down_codes": fp8_code_bytes(sd, layer, DOWN, expert, H, I),
        "down_scales": fp8_block_scale_bytes(sd, layer, DOWN, expert, H, I, lo, hi),
    }


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + r) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations(wl: "Workload", tokens: int | None = None, stream: int = 0) -> np.ndarray:
    """x ~ N(0, 1) rounded to bf16, as uint16 bit patterns [T][H]."""
    T = wl.tokens if tokens is None else tokens
    rng = np.random.default_rng([wl.seed, 1, stream])
    return f32_to_bf16_bits(rng.standard_normal((T, wl.hidden), dtype=np.float32))


def router_weights(wl: "Workload", layer: int = 0) -> np.ndarray:
    """W_r ~ N(0, 0.02), fp32 [E][H]."""
    rng = np.random.default_rng([wl.seed, 2, layer])
    w = rng.standard_normal((wl.n_experts, wl.hidden), dtype=np.float32)
    return (w * np.float32(0.02)).astype(np.float32)


def router_bias(wl: "Workload", layer: int = 0) -> np.ndarray | None:
    """Router bias giving Zipf(s) expert popularity, or None when unbiased.

    Logit noise W_r x has standard deviation sigma = 0.02 * sqrt(H) for unit
    activations; a Gumbel variable of the same variance has scale
    beta = sigma * sqrt(6) / pi, and top-1 selection under Gumbel noise picks
    expert e with probability proportional to exp(b_e / beta).  Choosing
    b_e = -s * beta * ln(rank(e) + 1) over a seeded permutation of ranks makes
    that proportional to (rank + 1) ** -s.
    """
    if wl.zipf is None:
        return None
    rng = np.random.default_rng([wl.seed, 3, layer])
    rank = rng.permutation(wl.n_experts)
    sigma = 0.02 * math.sqrt(wl.hidden)
    beta = sigma * math.sqrt(6.0) / math.pi
    return (-wl.zipf * beta * np.log(rank + 1.0)).astype(np.float32)
