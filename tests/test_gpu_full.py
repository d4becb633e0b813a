"""Full-size DeepSeek-V4.1-shaped layers (hidden 5120, intermediate 2304, 384
routed experts top-6 + 1 shared) on the GPU, in the launch configuration the
benchmark times, checked against the fp64 oracle: routing bit-exact on every
token given the oracle's logits, logits within tolerance, outputs within the
layer tolerance on every token (decode, verification) or on sampled tokens
(prefill, 8-layer stack; tokens are independent, so a sample is exact)."""
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
