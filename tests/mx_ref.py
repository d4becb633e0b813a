"""Independent helpers for pinning the oracle (tests only).

Nothing here is shared with the oracle or with the CUDA library: values come
from the golden E2M1 table (OCP MX specification), numpy's frexp/round and
torch's float8 casts, so a mistake in oracle.c does not cancel out.
"""
from __future__ import annotations

import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def e2m1_table() -> np.ndarray:
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                vals[int(c)] = float(v)
    return np.array([vals[c] for c in range(16)], dtype=np.float64)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[N][K] codes 0..15 -> [N][K/2] bytes, low nibble = even column."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def dequant_mx(code_bytes: np.ndarray, scale_bytes: np.ndarray) -> np.ndarray:
    """Dense fp64 matrix from packed E2M1 codes and UE8M0 scales (per 32 along K)."""
    tab = e2m1_table()
    cb = np.asarray(code_bytes, dtype=np.uint8)
    N = cb.shape[0]
    codes = np.empty((N, cb.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = cb & 15
    codes[:, 1::2] = cb >> 4
    scale = np.ldexp(1.0, np.asarray(scale_bytes, dtype=np.int64) - 127)
    return tab[codes] * np.repeat(scale, 32, axis=1)


def block_exponent_closed_form(amax: np.ndarray) -> np.ndarray:
    """Smallest e with amax <= 448 * 2**e: with amax = f * 2**E (f in [0.5, 1))
    and 448 = 0.875 * 2**9, e = E - 9 if f <= 0.875 else E - 8."""
    f, E = np.frexp(np.asarray(amax, dtype=np.float64))
    e = np.where(f <= 0.875, E - 9, E - 8)
    e = np.clip(e, -127, 127)
    return np.where(np.asarray(amax) == 0, 0, e).astype(np.int64)


def e4m3_round_closed_form(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value of fp64 inputs (ties to even), saturating at 448.

    Quantum of a value with binary exponent E is 2**(max(E, -6) - 3)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, E = np.frexp(a)           # a = f * 2**E, f in [0.5, 1) -> exponent E - 1
    Eb = np.maximum(E - 1, -6)
    q = np.ldexp(1.0, Eb - 3)
    r = np.round(a / q) * q      # numpy rounds half to even
    r = np.minimum(r, 448.0)
    return np.copysign(r, v)


def fp8_block_quant_torch(v: np.ndarray):
    """Per-32 dynamic FP8 quantisation of values exactly representable in fp32,
    encoding with torch's float8_e4m3fn cast.  Returns (codes, scale bytes)."""
    v = np.asarray(v, dtype=np.float64)
    blocks = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
    e = block_exponent_closed_form(np.abs(blocks).max(axis=-1))
    scaled = np.ldexp(blocks, -e[..., None])
    t = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn)
    codes = t.view(torch.uint8).numpy().reshape(v.shape)
    return codes, (e + 127).astype(np.uint8)


def fp8_block_dequant_torch(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    vals = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    vals = vals.to(torch.float64).numpy()
    return vals * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=-1)


def fp8_block_quant_f64(v: np.ndarray) -> np.ndarray:
    """Dequantised per-32 FP8 values of fp64 inputs (closed form, no fp32 step)."""
    v = np.asarray(v, dtype=np.float64)
    blocks = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
    e = block_exponent_closed_form(np.abs(blocks).max(axis=-1))
    r = e4m3_round_closed_form(np.ldexp(blocks, -e[..., None]))
    return np.ldexp(r, e[..., None]).reshape(v.shape)


def bf16_bits_torch(v: np.ndarray) -> np.ndarray:
    """fp32-representable values -> bf16 bit patterns with torch's RNE cast."""
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---- FP4-activation variant: closed forms for the E2M1 rounding and the
# block exponent (amax <= 6 * 2**e), independent of the oracle's search

def block_exponent4_closed_form(amax: np.ndarray) -> np.ndarray:
    """Smallest e with amax <= 6 * 2**e: with amax = f * 2**E (f in [0.5, 1))
    and 6 = 0.75 * 2**3, e = E - 3 if f <= 0.75 else E - 2."""
    f, E = np.frexp(np.asarray(amax, dtype=np.float64))
    e = np.where(f <= 0.75, E - 3, E - 2)
    e = np.clip(e, -127, 127)
    return np.where(np.asarray(amax) == 0, 0, e).astype(np.int64)


def e2m1_round_closed_form(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 value (grid 0, .5, 1, 1.5, 2, 3, 4, 6), ties to the even
    code, saturating at 6: spacing 0.5 below 2, 1 on [2, 4), 2 on [4, 6], and
    on each piece the code's parity is the parity of the grid index, so
    numpy's half-to-even rounding of a / spacing is the tie rule."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    r = np.where(a < 2, np.round(a * 2) / 2, np.where(a < 4, np.round(a), 2 * np.round(a / 2)))
    r = np.minimum(r, 6.0)
    return np.copysign(r, v)


def fp4_block_quant_f64(v: np.ndarray) -> np.ndarray:
    """Dequantised per-32 FP4 values of fp64 inputs (closed form)."""
    v = np.asarray(v, dtype=np.float64)
    blocks = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
    e = block_exponent4_closed_form(np.abs(blocks).max(axis=-1))
    r = e2m1_round_closed_form(np.ldexp(blocks, -e[..., None]))
    return np.ldexp(r, e[..., None]).reshape(v.shape)


def dequant_fp8_block32(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dense fp64 matrix from E4M3 codes [N][K] (torch's float8_e4m3fn decoding)
    and one UE8M0 scale per 32 x 32 block [N/32][K/32]."""
    vals = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    vals = vals.to(torch.float64).numpy()
    sc = np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    return vals * np.repeat(np.repeat(sc, 32, axis=0), 32, axis=1)
