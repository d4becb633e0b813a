"""Device-resident synthetic banks: the same bytes as synth.host_expert, filled
in place on the GPU by synth/fill.cu (counter-based, so a 7 GB layer fills in
milliseconds and any expert can be regenerated on the host for the oracle).
Holds no arithmetic of the MoE layer."""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


def _fill_lib():
    global _lib
    if _lib is None:
        path = os.path.join(_HERE, "libsynth_cuda.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} missing: run __graft_entry__.build()")
        _lib = C.CDLL(path)
        _lib.synth_fill.argtypes = [C.c_void_p, C.c_ulonglong, C.c_int, C.c_int, C.c_int, C.c_int,
                                    C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p]
        _lib.synth_fill.restype = C.c_int
    return _lib


def fill(t: torch.Tensor, n_experts: int, expert0: int, wl, layer: int, matrix: int, kind: int):
    per = t.numel() // n_experts
    rc = _fill_lib().synth_fill(t.data_ptr(), per, n_experts, expert0, wl.seed, layer, matrix, kind,
                                wl.scale_lo, wl.scale_hi, torch.cuda.current_stream().cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed with CUDA error {rc}")


def device_layer(wl, layer: int = 0, device: str = "cuda") -> dict:
    """All weights of one layer on the device, keyed like mxfp4_expert_ffn_gb300.Layer wants."""
    H, I, E, ns = wl.hidden, wl.inter, wl.n_experts, wl.n_shared
    shapes = {synth.GATE: (I, H), synth.UP: (I, H), synth.DOWN: (H, I)}
    names = {synth.GATE: "gate", synth.UP: "up", synth.DOWN: "down"}
    out = {}
    for m, (N, K) in shapes.items():
        for prefix, count, e0 in (("", E, 0), ("s_", ns, E)):
            if count == 0:
                continue
            c = torch.empty((count, N, K // 2), dtype=torch.uint8, device=device)
            s = torch.empty((count, N, K // 32), dtype=torch.uint8, device=device)
            fill(c, count, e0, wl, layer, m, synth.CODES)
            fill(s, count, e0, wl, layer, m, synth.SCALES)
            out[f"{prefix}{names[m]}_codes"] = c
            out[f"{prefix}{names[m]}_scales"] = s
    out["router_w"] = torch.from_numpy(synth.router_weights(wl, layer)).to(device)
    b = synth.router_bias(wl, layer)
    if b is not None:
        out["router_b"] = torch.from_numpy(b).to(device)
    return out


def host_experts(wl, layer: int, ids) -> dict:
    """Host copies (regenerated, not read back) of the given expert ids."""
    return synth.host_experts(wl, layer, ids)


def bf16_tensor(bits: np.ndarray, device: str = "cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(device)
