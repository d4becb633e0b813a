"""Full-size DeepSeek-V4.1-shaped layers (hidden 5120, intermediate 2304, 384
routed experts top-6 + 1 shared) on the GPU, checked against the fp64 oracle:
routing bit-exact on every token given the oracle's logits, logits within
tolerance, outputs within the layer tolerance on every token (decode,
verification) or on sampled tokens (prefill, 8-layer stack; tokens are
independent, so a sample is exact).  The calls the benchmark times -- moe_step
per layer (the 8-layer stack with its input normalisation, as run), the
host-buffer entry points -- are checked the same way: their routing is the
oracle's top-k of the logits they report, and their outputs match the oracle's
layer on that routing."""
from __future__ import annotations

import gc

import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_gb300 as m
import oracle
import synth
from synth import gpu as sg
from synth.workloads import DECODE_T1, PREFILL_T4096, PREFILL_T64K, STACK8_T64, VERIFY_T5, VERIFY_T32
from tests import gpu_util as gu

DEV = gu.DEV

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _check_layer(wl, layer, L, x, sample):
    lg = oracle.router_logits(x, synth.router_weights(wl, layer), synth.router_bias(wl, layer))
    ridx, rw = oracle.topk(lg, wl.top_k)
    T = x.shape[0]
    # routing: bit-exact given the oracle's logits
    idx, w, _ = gu.run_route(L, x, T, wl.n_experts, wl.top_k, logits_in=lg)
    assert np.array_equal(idx, ridx)
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-7)
    # the GPU's own logits
    _, _, lo = gu.run_route(L, x, T, wl.n_experts, wl.top_k)
    assert (np.abs(lo - lg) <= 1e-5 * np.abs(lg).max(axis=1, keepdims=True)).all()
    # the layer on the oracle's routing, all T tokens in one launch
    y = gu.run_forward(L, x, idx, rw)
    ref = gu.oracle_layer(wl, layer, x[sample], ridx[sample], rw[sample])
    return gu.assert_y_close(y[sample], ref)


@pytest.mark.parametrize("path", [m.PATH_AUTO, m.PATH_SIMT, m.PATH_MMA])
@pytest.mark.parametrize("wl", [DECODE_T1, VERIFY_T5, VERIFY_T32], ids=lambda w: w.name)
def test_decode_and_verification_layers(wl, path):
    L, W = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, path)
    x = synth.activations(wl)
    sample = np.arange(wl.tokens) if wl.tokens <= 8 else np.random.default_rng(0).choice(
        wl.tokens, 8, replace=False)
    _check_layer(wl, 0, L, x, np.sort(sample))
    L.close()
    del W
    _free()


def test_prefill_4096_tokens():
    wl = PREFILL_T4096
    L, W = gu.make_layer(wl)
    x = synth.activations(wl)
    sample = np.sort(np.random.default_rng(1).choice(wl.tokens, 16, replace=False))
    _check_layer(wl, 0, L, x, sample)
    L.close()
    del W
    _free()


def test_prefill_65536_tokens():
    """The largest batch a layer takes: routing of every token bit-exact given
    the oracle's logits, the layer on sampled tokens."""
    wl = PREFILL_T64K
    L, W = gu.make_layer(wl)
    x = synth.activations(wl)
    sample = np.sort(np.random.default_rng(2).choice(wl.tokens, 8, replace=False))
    _check_layer(wl, 0, L, x, sample)
    L.close()
    del W
    _free()


def test_stack_of_8_layers_teacher_forced():
    """Layer l of the GPU stack gets the oracle's normalised input and
    residual for 8 sampled tokens (the other 56 rows are seeded activations;
    rows do not interact) and must match the oracle's next residual."""
    wl = STACK8_T64
    T = wl.tokens
    sample = np.sort(np.random.default_rng(2).choice(T, 8, replace=False))
    filler = synth.activations(wl, stream=9)
    xs = synth.activations(wl)[sample]                 # oracle residual stream, sampled rows
    for layer in range(wl.layers):
        L, W = gu.make_layer(wl, layer)
        xn = oracle.rmsnorm(xs, 1e-6)
        x_in = filler.copy()
        x_in[sample] = xn
        res = filler.copy()
        res[sample] = xs
        lg = oracle.router_logits(x_in, synth.router_weights(wl, layer), synth.router_bias(wl, layer))
        ridx, rw = oracle.topk(lg, wl.top_k)
        y = gu.run_forward(L, x_in, ridx, rw, residual_bits=res)
        xs = gu.oracle_layer(wl, layer, xn, ridx[sample], rw[sample], residual=xs)
        gu.assert_y_close(y[sample], xs, what=f"layer {layer}")
        L.close()
        del W
        _free()


def _step_checked(wl, layer, L, x_bits, sample, residual_bits=None):
    """Runs moe_step on T tokens and checks it against the oracle: top-k ids
    bit-exact and weights equal given the logits the step reports, those
    logits within 1e-5 of the oracle's fp64 router, y on the sampled tokens
    within the layer tolerance.  Returns y (bf16 bits)."""
    T, E, k = x_bits.shape[0], wl.n_experts, wl.top_k
    x = sg.bf16_tensor(x_bits, DEV)
    r = None if residual_bits is None else sg.bf16_tensor(residual_bits, DEV)
    y = torch.empty(x.shape, dtype=torch.int16, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    lo = torch.empty((T, E), dtype=torch.float32, device=DEV)
    L.step(x, T, y, residual=r, idx=idx, w=w, logits_out=lo)
    assert L.sync() == m.MOE_OK
    lg = lo.cpu().numpy()
    ridx, rw = oracle.topk(lg, k)
    ids = idx.cpu().numpy()
    assert np.array_equal(ids, ridx), f"layer {layer}: top-k differs from the oracle's on the step's logits"
    assert np.allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
    lref = oracle.router_logits(x_bits, synth.router_weights(wl, layer), synth.router_bias(wl, layer))
    assert (np.abs(lg - lref) <= 1e-5 * np.abs(lref).max(axis=1, keepdims=True)).all()
    yb = y.cpu().numpy().view(np.uint16)
    ref = gu.oracle_layer(wl, layer, x_bits[sample], ridx[sample], rw[sample],
                          residual=None if residual_bits is None else residual_bits[sample])
    gu.assert_y_close(yb[sample], ref, what=f"layer {layer} step")
    return yb


@pytest.mark.parametrize("wl", [DECODE_T1, VERIFY_T5, VERIFY_T32], ids=lambda w: w.name)
def test_step_full_size_matches_oracle(wl):
    """moe_step on the decode and verification workloads, as the benchmark
    times it (up to 64 tokens: one preparation launch, gate/up, down with the
    combine inside)."""
    L, W = gu.make_layer(wl)
    x = synth.activations(wl, stream=60)
    _step_checked(wl, 0, L, x, np.arange(wl.tokens))
    L.close()
    del W
    _free()


@pytest.mark.parametrize("wl", [DECODE_T1, VERIFY_T32], ids=lambda w: w.name)
def test_forward_host_full_size_matches_step_and_oracle(wl):
    """moe_forward_host (host buffers in and out, the end-to-end entry point):
    the same y bits as moe_step on the device, and the oracle's layer."""
    L, W = gu.make_layer(wl)
    x = synth.activations(wl, stream=61)
    y_dev = _step_checked(wl, 0, L, x, np.arange(wl.tokens))
    xh = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
    yh = torch.empty(xh.shape, dtype=torch.int16).pin_memory()
    for _ in range(2):  # a repeated call gives the same bits
        yh.fill_(0)
        L.forward_host(xh, wl.tokens, yh)
        assert np.array_equal(yh.numpy().view(np.uint16), y_dev)
    L.close()
    del W
    _free()


def test_stack_of_8_layers_as_benchmarked():
    """The 8-layer stack exactly as the benchmark runs it, on all 64 tokens:
    per layer moe_rmsnorm of the residual stream, then moe_step with the
    stream as residual.  Layer l is checked against the oracle given the GPU's
    own input of that layer (teacher forcing): the normalised input against
    oracle.rmsnorm, the routing against the oracle's top-k of the step's
    logits, y on 8 sampled tokens against the oracle's layer.  Then the
    host-buffer stack entry point (the end-to-end call) on the same input must
    give the same bits as the device loop."""
    wl = STACK8_T64
    T, H = wl.tokens, wl.hidden
    sample = np.sort(np.random.default_rng(3).choice(T, 8, replace=False))
    x0 = synth.activations(wl, stream=62)
    cur = x0
    layers = []
    for layer in range(wl.layers):
        L, W = gu.make_layer(wl, layer)
        layers.append((L, W))
        xn_t = torch.empty((T, H), dtype=torch.int16, device=DEV)
        m.moe_rmsnorm(sg.bf16_tensor(cur, DEV), T, H, 1e-6, xn_t)
        torch.cuda.synchronize()
        xn = xn_t.cpu().numpy().view(np.uint16)
        ref_n = gu.bits_to_f64(oracle.rmsnorm(cur, 1e-6))
        # fp32 on the GPU, fp64 in the oracle: within one bf16 step of each value
        assert np.all(np.abs(gu.bits_to_f64(xn) - ref_n) <= np.abs(ref_n) * 2.0 ** -7), f"layer {layer} rmsnorm"
        cur = _step_checked(wl, layer, L, xn, sample, residual_bits=cur)
    xh = torch.from_numpy(x0.view(np.int16).copy()).pin_memory()
    yh = torch.empty(xh.shape, dtype=torch.int16).pin_memory()
    m.moe_stack_forward_host([L for L, _ in layers], xh, T, 1e-6, yh)
    assert np.array_equal(yh.numpy().view(np.uint16), cur)
    for L, _ in layers:
        L.close()
    del layers
    _free()
