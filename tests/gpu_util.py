"""Shared helpers for the GPU parity tests: building a layer from the seeded
generators, running it through the C ABI, and the output tolerance of the
layer (max |dy| <= 2e-2 * max|y| and relative L2 <= 5e-3, bf16 output)."""
from __future__ import annotations

import numpy as np
import torch

import mxfp4_expert_ffn_gb300 as m
import oracle
import synth
from synth import gpu as sg

DEV = "cuda:0"
MAX_REL = 2e-2
REL_L2 = 5e-3


def make_layer(wl, layer: int = 0, max_tokens: int | None = None, weights=None):
    W = weights if weights is not None else sg.device_layer(wl, layer, DEV)
    L = m.Layer(wl.hidden, wl.inter, wl.n_experts, wl.top_k, wl.n_shared,
                max_tokens or max(wl.tokens, 1), W)
    return L, W


def fp8_shared_weights(wl, layer: int = 0, device: str = DEV) -> dict:
    """Device copies of the shared experts in the FP8 (32 x 32 block) format, keyed
    like the layer's weight dict (s_gate_codes, ...), stacked over the shared experts."""
    exs = [synth.host_expert_fp8(wl, layer, wl.n_experts + s) for s in range(wl.n_shared)]
    out = {}
    for mname in ("gate", "up", "down"):
        for kind in ("codes", "scales"):
            a = np.stack([e[f"{mname}_{kind}"] for e in exs])
            out[f"s_{mname}_{kind}"] = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return out


def make_layer_fp8_shared(wl, layer: int = 0, max_tokens: int | None = None):
    """A layer whose shared experts are FP8 with 32 x 32 block scales."""
    W = sg.device_layer(wl, layer, DEV)
    W.update(fp8_shared_weights(wl, layer))
    L, W = make_layer(wl, layer, max_tokens, weights=W)
    L.set_shared_format(m.MOE_SHARED_FP8_B32)
    return L, W


def bits_to_f64(bits) -> np.ndarray:
    if isinstance(bits, torch.Tensor):
        bits = bits.cpu().numpy()
    return synth.bf16_bits_to_f32(np.asarray(bits).view(np.uint16)).astype(np.float64)


def assert_y_close(got_bits, want_bits, what: str = "y"):
    g, w = bits_to_f64(got_bits), bits_to_f64(want_bits)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - w).max()
    scale = np.abs(w).max()
    l2 = np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30)
    assert err <= MAX_REL * scale, f"{what}: max|dy| {err:.4g} > {MAX_REL} * {scale:.4g}"
    assert l2 <= REL_L2, f"{what}: relative L2 {l2:.3g} > {REL_L2}"
    return err / max(scale, 1e-30), l2


def run_route(L, x_bits, T, E, k, logits_in=None):
    x = sg.bf16_tensor(x_bits, DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    lo = torch.empty((T, E), dtype=torch.float32, device=DEV)
    li = None if logits_in is None else torch.from_numpy(np.ascontiguousarray(logits_in)).to(DEV)
    L.route(x, T, idx, w, logits_in=li, logits_out=lo)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), lo.cpu().numpy()


def run_forward(L, x_bits, idx, w, residual_bits=None, H=None):
    T = x_bits.shape[0]
    x = sg.bf16_tensor(x_bits, DEV)
    y = torch.empty(x.shape, dtype=torch.int16, device=DEV)
    r = None if residual_bits is None else sg.bf16_tensor(residual_bits, DEV)
    L.forward(x, T, torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(DEV),
              torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).to(DEV), y, residual=r)
    st = L.sync()
    assert st == 0, m.status_string(st)
    return y.cpu().numpy().view(np.uint16)


def oracle_layer(wl, layer, x_bits, idx, w, residual=None, act4=False, shared_fp8=False):
    ids = np.unique(idx)
    ids = ids[(ids >= 0) & (ids < wl.n_experts)]
    experts = sg.host_experts(wl, layer, ids)
    gen = synth.host_expert_fp8 if shared_fp8 else synth.host_expert
    shared = [gen(wl, layer, wl.n_experts + s) for s in range(wl.n_shared)]
    y, _ = oracle.moe_layer(x_bits, idx, w, experts, shared, wl.n_experts, wl.inter,
                            residual=residual, act4=act4)
    return y
