"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the golden
E2M1 table of the OCP MX specification, the byte counts printed on the pages,
torch's float8 casts, numpy/scipy routines, brute force, closed forms and
invariants.  No GPU needed.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
import synth
from synth.workloads import DECODE_T1, TINY
from tests import mx_ref

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ P1 codecs
def test_e2m1_all_16_codes_match_ocp_mx_table():
    tab = mx_ref.e2m1_table()
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert v == tab[c] and math.copysign(1, v) == math.copysign(1, tab[c]), c


def test_e2m1_structure():
    # 2 exponent bits (bias 1) + 1 mantissa bit: magnitudes strictly increase,
    # the normal values double every two codes, code 8 is negative zero.
    mags = [oracle.e2m1_value(c) for c in range(8)]
    assert all(a < b for a, b in zip(mags, mags[1:]))
    assert mags[1] == 0.5 and mags[7] == 6.0
    for c in range(2, 6):
        assert mags[c + 2] == 2 * mags[c]
    assert oracle.e2m1_value(8) == 0.0 and math.copysign(1, oracle.e2m1_value(8)) < 0
    # every E2M1 value is exactly an E4M3 value (so FP4 x FP8 products are exact)
    t = torch.tensor(mags, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float32)
    assert t.tolist() == mags


def test_ue8m0_all_256_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    for s in range(256):
        v = oracle.ue8m0_value(s)
        r = ref[s].item()
        assert (math.isnan(v) and math.isnan(r)) or v == r, s


def test_e4m3_all_256_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for c in range(256):
        v = oracle.e4m3_value(c)
        r = ref[c].item()
        assert (math.isnan(v) and math.isnan(r)) or (v == r and math.copysign(1, v) == math.copysign(1, r)), c
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(1) == 2.0 ** -9


def test_e4m3_encode_exhaustive_bf16_matches_torch():
    # every finite bf16 value with |v| <= 448, encoded by the oracle's nearest
    # search and by torch's round-to-nearest-even cast
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = mx_ref.bf16_to_f64(bits)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    vals = vals[keep]
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in vals], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(vals[i], got[i], ref[i]) for i in bad[:5]]


def test_e4m3_encode_saturates_and_keeps_sign():
    assert oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(464.0) == 0x7E      # above the last finite code: saturate
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-2.0 ** -11) == 0x80  # rounds to zero, sign kept
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00   # tie between 0 and 2^-9: even code
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 (x 2^-9): even


def test_e4m3_encode_random_doubles_match_closed_form():
    rng = np.random.default_rng(7)
    v = rng.standard_normal(4000) * np.ldexp(1.0, rng.integers(-12, 9, 4000))
    ref = mx_ref.e4m3_round_closed_form(v)
    got = np.array([oracle.e4m3_value(oracle.e4m3_encode(x)) for x in v])
    assert np.array_equal(got, ref)


def test_block_exponent_matches_closed_form():
    rng = np.random.default_rng(3)
    a = np.concatenate([
        np.abs(rng.standard_normal(2000)) * np.ldexp(1.0, rng.integers(-140, 140, 2000)),
        np.ldexp(448.0, np.arange(-130, 128)),                  # exactly on the boundary
        np.nextafter(np.ldexp(448.0, np.arange(-130, 127)), np.inf),
        [0.0, 2.0 ** -149, 3.3e38],
    ])
    ref = mx_ref.block_exponent_closed_form(a)
    got = np.array([oracle.block_exponent(x) for x in a])
    assert np.array_equal(got, ref)


def test_quantize_act_matches_torch_cast():
    rng = np.random.default_rng(11)
    x = synth.f32_to_bf16_bits(rng.standard_normal((5, 256)).astype(np.float32) *
                               np.ldexp(1.0, rng.integers(-20, 20, (5, 256))).astype(np.float32))
    x[0, :32] = 0            # all-zero block -> scale byte 127, codes 0
    x[1, 32:64] = 0x8000     # -0 block
    q, s = oracle.quantize_act(x)
    rq, rs = mx_ref.fp8_block_quant_torch(mx_ref.bf16_to_f64(x))
    assert np.array_equal(s, rs)
    assert np.array_equal(q, rq)
    assert s[0, 0] == 127 and not q[0, :32].any()
    assert (q[1, 32:64] == 0x80).all()


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(5)
    f = (rng.standard_normal(20000) * np.ldexp(1.0, rng.integers(-135, 128, 20000))).astype(np.float32)
    f = f[np.isfinite(f)]
    ref = mx_ref.bf16_bits_torch(f)
    got = np.array([oracle.bf16_round(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # exact ties go to even
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82


# ------------------------------------------------------------ P2 byte counts
def test_byte_accounting_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "byte_accounting.json")))
    H, I = g["hidden"], g["inter"]
    wl = DECODE_T1
    assert (wl.hidden, wl.inter, wl.n_experts, wl.top_k) == (H, I, g["n_routed"], g["top_k"])
    ex = synth.host_expert(wl, 0, 0)
    codes = sum(ex[f"{m}_codes"].nbytes for m in ("gate", "up", "down"))
    total = codes + sum(ex[f"{m}_scales"].nbytes for m in ("gate", "up", "down"))
    assert codes == 3 * H * I // 2 == 17_694_720
    assert round(codes / 2 ** 20, 2) == g["codes_mib_per_expert"]
    assert total == 18_800_640 == wl.expert_bytes
    assert round(total / 1e6, 2) == g["with_scales_mb_per_expert"]
    assert round(total / 2 ** 20, 2) == g["with_scales_mib_per_expert"]
    assert round(g["layers"] * g["n_routed"] * total / 2 ** 30) == g["routed_gib_total"]
    per_token = g["layers"] * g["top_k"] * total
    assert round(per_token / 1e9, 2) == g["routed_gb_per_token"]
    assert round(g["decode_bw_gbs"] * 1e9 / per_token) == g["decode_tok_s_estimate"]
    assert g["slots"] * codes / 2 ** 30 <= g["slot_cache_gib_approx"]


# -------------------------------------------------------------- P3/P4 top-k
def _brute_topk(row, k):
    key = [(-(-math.inf if math.isnan(v) else v), i) for i, v in enumerate(row)]
    return [i for _, i in sorted(key)[:k]]


@pytest.mark.parametrize("E,k", [(16, 2), (384, 6)])
def test_topk_matches_brute_force_sort(E, k):
    rng = np.random.default_rng(E + k)
    T = 64
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[1, :] = 0.5                                   # all tied
    lg[2, ::2] = 0.0
    lg[2, 1::2] = -0.0                               # +0 / -0 ties
    lg[3, : E // 2] = np.nan                         # NaN ranks last
    lg[4, :] = np.round(lg[4, :] * 2) / 2            # many ties
    lg[5, E - 1] = np.inf
    idx, _ = oracle.topk(lg, k)
    for t in range(T):
        assert idx[t].tolist() == _brute_topk(lg[t].tolist(), k), t


def test_combine_weights_renormalised_softmax():
    rng = np.random.default_rng(9)
    lg = (rng.standard_normal((50, 384)) * 1.4).astype(np.float32)
    idx, w = oracle.topk(lg, 6)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-15, rtol=0)
    assert (np.diff(w, axis=1) <= 0).all()
    full = softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, idx, axis=1)
    assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)


# ---- sigmoid scoring (selection on fp32 sigmoid(l) + bias, weights s / sum s * scale)

def test_sigmoid_f32_within_3_ulp_of_fp64_and_monotonic():
    l = np.linspace(-80, 80, 200001).astype(np.float32)
    s = oracle.sigmoid_f32(l).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert (np.abs(s - ref) / ulp).max() <= 3.0
    assert np.all(np.diff(s) >= 0)
    assert oracle.sigmoid_f32(np.float32([0.0]))[0] == 0.5
    assert oracle.sigmoid_f32(np.float32([30.0]))[0] == 1.0


def _brute_sigmoid(l, b, k, scale):
    s = oracle.sigmoid_f32(l)
    key = (s + b).astype(np.float32)
    order = sorted(range(len(l)), key=lambda e: (-(-math.inf if math.isnan(l[e]) or math.isnan(key[e])
                                                   else float(key[e])), e))
    sel = order[:k]
    sv = np.array([0.0 if math.isnan(l[e]) else float(s[e]) for e in sel])
    return sel, sv / sv.sum() * scale


@pytest.mark.parametrize("E,k", [(16, 2), (384, 6)])
def test_topk_sigmoid_matches_brute_force(E, k):
    rng = np.random.default_rng(100 + E)
    T = 32
    lg = (rng.standard_normal((T, E)) * 1.4).astype(np.float32)
    b = (rng.standard_normal(E) * 0.05).astype(np.float32)
    lg[1, :] = 0.25                                   # all tied before the bias
    lg[2, : E // 2] = np.nan                          # NaN logits rank last
    lg[3, :] = np.round(lg[3, :] * 2) / 2
    idx, w = oracle.topk_sigmoid(lg, b, k, 2.5)
    for t in range(T):
        sel, ww = _brute_sigmoid(lg[t], b, k, 2.5)
        assert idx[t].tolist() == sel, t
        assert np.allclose(w[t], ww, rtol=1e-12, atol=0), t
    assert np.allclose(w.sum(axis=1), 2.5, rtol=1e-12)


def test_topk_sigmoid_without_bias_selects_like_the_logits():
    # sigmoid is increasing: with no bias and no saturation ties the selection
    # is the logits' top-k (the softmax scoring's selection)
    rng = np.random.default_rng(7)
    lg = (rng.standard_normal((64, 384)) * 1.4).astype(np.float32)
    idx_s, _ = oracle.topk_sigmoid(lg, None, 6, 1.0)
    idx_l, _ = oracle.topk(lg, 6)
    s = oracle.sigmoid_f32(lg)
    for t in range(64):
        if len(np.unique(s[t])) == len(np.unique(lg[t])):
            assert idx_s[t].tolist() == idx_l[t].tolist(), t


def test_topk_sigmoid_bias_selects_but_does_not_weight():
    rng = np.random.default_rng(8)
    lg = (rng.standard_normal((4, 64)) * 1.4).astype(np.float32)
    b = np.zeros(64, np.float32)
    b[37] = 10.0                                      # forces expert 37 into first place
    idx, w = oracle.topk_sigmoid(lg, b, 4, 1.0)
    s = oracle.sigmoid_f32(lg).astype(np.float64)
    for t in range(4):
        assert idx[t, 0] == 37
        sel = s[t, idx[t]]
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-12)   # the bias is not in the weights


def test_router_logits_match_numpy_matmul():
    wl = TINY
    x = synth.activations(wl, tokens=16)
    W = synth.router_weights(wl)
    b = np.linspace(-1, 1, wl.n_experts).astype(np.float32)
    got = oracle.router_logits(x, W, b)
    ref = (mx_ref.bf16_to_f64(x) @ W.astype(np.float64).T + b.astype(np.float64)).astype(np.float32)
    ulps = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1


def test_segments_match_stable_argsort():
    rng = np.random.default_rng(4)
    E, T, k = 40, 100, 3
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    off, perm = oracle.segments(idx, E)
    flat = idx.ravel()
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))


# ------------------------------------------------------------ layer pins
def _tiny_bank(wl, seed_layer=0):
    experts = {e: synth.host_expert(wl, seed_layer, e) for e in range(wl.n_experts)}
    shared = [synth.host_expert(wl, seed_layer, wl.n_experts + s) for s in range(wl.n_shared)]
    return experts, shared


def _dense(ex):
    return {m: mx_ref.dequant_mx(ex[f"{m}_codes"], ex[f"{m}_scales"]) for m in ("gate", "up", "down")}


def _brute_dense_layer(x_bits, idx, w, experts, shared):
    """Independent evaluation: numpy matmuls over ALL experts, torch FP8 casts,
    non-selected experts masked with weight 0."""
    xf = mx_ref.bf16_to_f64(x_bits)
    xq, xs = mx_ref.fp8_block_quant_torch(xf)
    xh = mx_ref.fp8_block_dequant_torch(xq, xs)
    T = xf.shape[0]

    def ffn(d):
        g = xh @ d["gate"].T
        u = xh @ d["up"].T
        h = g / (1 + np.exp(-g)) * u
        return mx_ref.fp8_block_quant_f64(h) @ d["down"].T

    acc = sum(ffn(_dense(s)) for s in shared)
    for e, ex in experts.items():
        m = np.zeros(T)
        for j in range(idx.shape[1]):
            m += np.where(idx[:, j] == e, w[:, j], 0.0)
        acc = acc + m[:, None] * ffn(_dense(ex))
    return acc


def test_brute_force_dense_tiny_layer():
    wl = TINY
    experts, shared = _tiny_bank(wl)
    x = synth.activations(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl))
    idx, w = oracle.topk(lg, wl.top_k)
    y, y64 = oracle.moe_layer(x, idx, w, experts, shared, wl.n_experts, wl.inter)
    ref = _brute_dense_layer(x, idx, w, experts, shared)
    assert np.allclose(y64, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())
    # the bf16 output is the fp64 sum rounded once: within half a bf16 ulp
    assert np.all(np.abs(mx_ref.bf16_to_f64(y) - ref) <= np.abs(ref) * 2.0 ** -8)


def _identity_expert(H, I, a, b, c):
    """gate = 2^a P, up = 2^b P, down = 2^c P^T with P selecting coordinates 0..I-1."""
    one = 2  # E2M1 code of 1.0
    g = np.zeros((I, H), np.uint8)
    g[np.arange(I), np.arange(I)] = one
    d = np.zeros((H, I), np.uint8)
    d[np.arange(I), np.arange(I)] = one
    return {
        "gate_codes": mx_ref.pack_nibbles(g), "gate_scales": np.full((I, H // 32), 127 + a, np.uint8),
        "up_codes": mx_ref.pack_nibbles(g), "up_scales": np.full((I, H // 32), 127 + b, np.uint8),
        "down_codes": mx_ref.pack_nibbles(d), "down_scales": np.full((H, I // 32), 127 + c, np.uint8),
    }


def test_identity_like_expert_closed_form():
    H, I, E, k = 256, 128, 4, 2
    rng = np.random.default_rng(21)
    x = synth.f32_to_bf16_bits(rng.standard_normal((6, H)).astype(np.float32) * 3)
    experts = {e: _identity_expert(H, I, e - 1, 1 - e, e % 2) for e in range(E)}
    shared = [_identity_expert(H, I, 0, 0, -1)]
    idx = np.array([[0, 1], [2, 3], [1, 0], [3, 2], [0, 3], [2, 1]], np.int32)
    w = np.array([[0.75, 0.25]] * 6)
    y, y64 = oracle.moe_layer(x, idx, w, experts, shared, E, I)
    xq, xs = mx_ref.fp8_block_quant_torch(mx_ref.bf16_to_f64(x))
    xh = mx_ref.fp8_block_dequant_torch(xq, xs)[:, :I]

    def expert_out(a, b, c):
        h = (2.0 ** a * xh) / (1 + np.exp(-(2.0 ** a * xh))) * (2.0 ** b * xh)
        o = np.zeros((x.shape[0], H))
        o[:, :I] = 2.0 ** c * mx_ref.fp8_block_quant_f64(h)
        return o

    ref = expert_out(0, 0, -1)
    for j in range(k):
        for t in range(x.shape[0]):
            e = idx[t, j]
            ref[t] += w[t, j] * expert_out(e - 1, 1 - e, e % 2)[t]
    assert np.allclose(y64, ref, rtol=1e-12, atol=0)
    assert (y64[:, I:] == 0).all()


def test_all_experts_identical_routing_invariant():
    wl = TINY
    base = synth.host_expert(wl, 0, 3)
    experts = {e: base for e in range(wl.n_experts)}
    shared = [base]
    x = synth.activations(wl)
    w = np.array([[0.5, 0.5]] * wl.tokens)
    idx1 = np.array([[0, 1], [2, 3], [4, 5], [6, 7]], np.int32)
    idx2 = np.array([[15, 9], [1, 2], [11, 0], [3, 14]], np.int32)
    y1, a = oracle.moe_layer(x, idx1, w, experts, shared, wl.n_experts, wl.inter)
    y2, b = oracle.moe_layer(x, idx2, w, experts, shared, wl.n_experts, wl.inter)
    assert np.array_equal(y1, y2) and np.array_equal(a, b)
    # y = bf16(2 * f(x)): the shared expert plus weights summing to one
    y0, s = oracle.moe_layer(x, idx1, np.zeros_like(w), experts, shared, wl.n_experts, wl.inter)
    assert np.array_equal(a, 2 * s)


def test_zero_weights_zero_input_and_residual():
    wl = TINY
    experts, shared = _tiny_bank(wl)
    x = synth.activations(wl)
    idx = np.array([[0, 1], [2, 3], [4, 5], [6, 7]], np.int32)
    w0 = np.zeros((wl.tokens, 2))
    y_sh, y64 = oracle.moe_layer(x, idx, w0, experts, shared, wl.n_experts, wl.inter)
    y_only_shared, s64 = oracle.moe_layer(x, idx[:, :0], w0[:, :0], experts, shared, wl.n_experts, wl.inter)
    assert np.array_equal(y_sh, y_only_shared)
    z = np.zeros_like(x)
    yz, z64 = oracle.moe_layer(z, idx, np.full((wl.tokens, 2), 0.5), experts, shared, wl.n_experts, wl.inter)
    assert (z64 == 0).all() and (yz & 0x7FFF == 0).all()
    yr, _ = oracle.moe_layer(z, idx, np.full((wl.tokens, 2), 0.5), experts, shared, wl.n_experts,
                             wl.inter, residual=x)
    assert np.array_equal(yr, x)


def test_token_permutation_equivariance():
    wl = TINY.with_tokens(8)
    experts, shared = _tiny_bank(wl)
    x = synth.activations(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl))
    idx, w = oracle.topk(lg, wl.top_k)
    y, _ = oracle.moe_layer(x, idx, w, experts, shared, wl.n_experts, wl.inter)
    p = np.random.default_rng(1).permutation(wl.tokens)
    yp, _ = oracle.moe_layer(x[p], idx[p], w[p], experts, shared, wl.n_experts, wl.inter)
    assert np.array_equal(yp, y[p])


def test_residual_is_bf16_of_bf16_sum():
    wl = TINY
    experts, shared = _tiny_bank(wl)
    x = synth.activations(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl))
    idx, w = oracle.topk(lg, wl.top_k)
    y, _ = oracle.moe_layer(x, idx, w, experts, shared, wl.n_experts, wl.inter)
    r = synth.activations(wl, stream=5)
    yr, _ = oracle.moe_layer(x, idx, w, experts, shared, wl.n_experts, wl.inter, residual=r)
    ref = mx_ref.bf16_bits_torch((mx_ref.bf16_to_f64(y) + mx_ref.bf16_to_f64(r)).astype(np.float32))
    assert np.array_equal(yr, ref)


def test_expert_ffn_h_codes_match_closed_form():
    wl = TINY
    ex = synth.host_expert(wl, 0, 5)
    x = synth.activations(wl)
    q, s = oracle.quantize_act(x)
    r = oracle.expert_ffn(ex, q[0], s[0])
    d = _dense(ex)
    xh = mx_ref.fp8_block_dequant_torch(q[:1], s[:1])[0]
    g, u = d["gate"] @ xh, d["up"] @ xh
    h = g / (1 + np.exp(-g)) * u
    assert np.allclose(r["h"], h, rtol=1e-12, atol=1e-12 * np.abs(h).max())
    hh = mx_ref.fp8_block_dequant_torch(r["hq"][None], r["hs"][None])[0]
    assert np.array_equal(hh, mx_ref.fp8_block_quant_f64(h))
    assert np.allclose(r["o"], d["down"] @ hh, rtol=1e-12, atol=1e-12 * np.abs(r["o"]).max())


def test_rmsnorm_closed_form():
    rng = np.random.default_rng(2)
    x = synth.f32_to_bf16_bits((rng.standard_normal((4, 256)) * 300).astype(np.float32))
    out = oracle.rmsnorm(x, 1e-6)
    xf = mx_ref.bf16_to_f64(x)
    ref = xf / np.sqrt((xf ** 2).mean(axis=1, keepdims=True) + 1e-6)
    got = mx_ref.bf16_to_f64(out)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    assert np.allclose(np.sqrt((got ** 2).mean(axis=1)), 1.0, atol=5e-3)
    # scale invariance by a power of two is exact
    x2 = synth.f32_to_bf16_bits((mx_ref.bf16_to_f64(x) * 8).astype(np.float32))
    assert np.array_equal(oracle.rmsnorm(x2, 0.0), oracle.rmsnorm(x, 0.0))


# ---- FP4-activation variant (x and h as E2M1 per 32 with a UE8M0 scale)

def test_e2m1_encode_grid_midpoints_and_sign():
    tab = mx_ref.e2m1_table()
    for c in range(8):                       # every grid value encodes to itself
        assert oracle.e2m1_encode(tab[c]) == c
        assert oracle.e2m1_encode(-tab[c]) == c | 8
    # midpoints between neighbours go to the even code
    for lo, hi, want in [(0, 1, 0), (1, 2, 2), (2, 3, 2), (3, 4, 4), (4, 5, 4), (5, 6, 6), (6, 7, 6)]:
        assert oracle.e2m1_encode((tab[lo] + tab[hi]) / 2) == want, (lo, hi)
    assert oracle.e2m1_encode(7.0) == 7 and oracle.e2m1_encode(-100.0) == 15   # saturate
    assert oracle.e2m1_encode(-0.0) == 8 and oracle.e2m1_encode(-0.1) == 8      # sign kept at zero


def test_e2m1_encode_random_doubles_match_closed_form():
    rng = np.random.default_rng(17)
    v = rng.uniform(-7, 7, 20000)
    v[:64] = np.repeat(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]), 8) * np.tile([1, -1], 32)
    tab = mx_ref.e2m1_table()
    got = np.array([tab[oracle.e2m1_encode(x)] for x in v])
    assert np.array_equal(got, mx_ref.e2m1_round_closed_form(v))


def test_block_exponent4_matches_closed_form():
    rng = np.random.default_rng(19)
    a = np.concatenate([
        np.abs(rng.standard_normal(2000)) * np.ldexp(1.0, rng.integers(-140, 140, 2000)),
        6.0 * np.ldexp(1.0, np.arange(-127, 127)),            # exactly on the boundary
        np.nextafter(6.0 * np.ldexp(1.0, np.arange(-120, 120)), np.inf),
        [0.0, 1e-45, 3e38]])
    got = np.array([oracle.block_exponent4(x) for x in a])
    assert np.array_equal(got, mx_ref.block_exponent4_closed_form(a))


def test_quantize_act4_matches_closed_form_and_packs_low_nibble_first():
    wl = TINY
    x = synth.activations(wl, tokens=16)
    x[0, :32] = 0                          # an all-zero block: scale 2^0, codes 0
    q, s = oracle.quantize_act4(x)
    assert q.shape == (16, wl.hidden // 2) and s.shape == (16, wl.hidden // 32)
    assert s[0, 0] == 127 and (q[0, :16] == 0).all()
    tab = mx_ref.e2m1_table()
    codes = np.empty((16, wl.hidden), np.uint8)
    codes[:, 0::2], codes[:, 1::2] = q & 15, q >> 4
    deq = tab[codes] * np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)
    assert np.array_equal(deq, mx_ref.fp4_block_quant_f64(mx_ref.bf16_to_f64(x)))


def _brute_dense_layer4(x_bits, idx, w, experts, shared):
    """Independent evaluation of the FP4 variant: numpy matmuls over all
    experts with the closed-form FP4 activation rounding."""
    xh = mx_ref.fp4_block_quant_f64(mx_ref.bf16_to_f64(x_bits))
    T = xh.shape[0]

    def ffn(d):
        g = xh @ d["gate"].T
        u = xh @ d["up"].T
        h = g / (1 + np.exp(-g)) * u
        return mx_ref.fp4_block_quant_f64(h) @ d["down"].T

    acc = sum(ffn(_dense(s)) for s in shared)
    for e, ex in experts.items():
        m = np.zeros(T)
        for j in range(idx.shape[1]):
            m += np.where(idx[:, j] == e, w[:, j], 0.0)
        acc = acc + m[:, None] * ffn(_dense(ex))
    return acc


def test_brute_force_dense_tiny_layer_fp4_activations():
    wl = TINY
    experts, shared = _tiny_bank(wl)
    x = synth.activations(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl))
    idx, w = oracle.topk(lg, wl.top_k)
    y, y64 = oracle.moe_layer(x, idx, w, experts, shared, wl.n_experts, wl.inter, act4=True)
    ref = _brute_dense_layer4(x, idx, w, experts, shared)
    assert np.allclose(y64, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())
    # and it is a different layer from the FP8 one (the variant is not a no-op)
    _, y64_8 = oracle.moe_layer(x, idx, w, experts, shared, wl.n_experts, wl.inter)
    assert not np.allclose(y64, y64_8, rtol=1e-3, atol=0)


def test_identity_like_expert_closed_form_fp4_activations():
    H, I, E = 256, 128, 4
    rng = np.random.default_rng(23)
    x = synth.f32_to_bf16_bits(rng.standard_normal((6, H)).astype(np.float32) * 3)
    experts = {e: _identity_expert(H, I, e - 1, 1 - e, e % 2) for e in range(E)}
    shared = [_identity_expert(H, I, 0, 0, -1)]
    idx = np.array([[0, 1], [2, 3], [1, 0], [3, 2], [0, 3], [2, 1]], np.int32)
    w = np.array([[0.75, 0.25]] * 6)
    _, y64 = oracle.moe_layer(x, idx, w, experts, shared, E, I, act4=True)
    xh = mx_ref.fp4_block_quant_f64(mx_ref.bf16_to_f64(x))[:, :I]

    def expert_out(a, b, c):
        h = (2.0 ** a * xh) / (1 + np.exp(-(2.0 ** a * xh))) * (2.0 ** b * xh)
        o = np.zeros((x.shape[0], H))
        o[:, :I] = 2.0 ** c * mx_ref.fp4_block_quant_f64(h)
        return o

    ref = expert_out(0, 0, -1)
    for j in range(2):
        for t in range(x.shape[0]):
            e = idx[t, j]
            ref[t] += w[t, j] * expert_out(e - 1, 1 - e, e % 2)[t]
    assert np.allclose(y64, ref, rtol=1e-12, atol=0)
    assert (y64[:, I:] == 0).all()


# ---- FP8 shared expert (E4M3 weights, one UE8M0 scale per 32 x 32 block)

def _dense_any(ex):
    if ex.get("fmt", 0) == 1:
        return {m: mx_ref.dequant_fp8_block32(ex[f"{m}_codes"], ex[f"{m}_scales"]) for m in ("gate", "up", "down")}
    return _dense(ex)


def test_brute_force_dense_tiny_layer_fp8_shared_expert():
    wl = TINY
    experts, _ = _tiny_bank(wl)
    shared = [synth.host_expert_fp8(wl, 0, wl.n_experts)]
    x = synth.activations(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl))
    idx, w = oracle.topk(lg, wl.top_k)
    _, y64 = oracle.moe_layer(x, idx, w, experts, shared, wl.n_experts, wl.inter)
    xq, xs = mx_ref.fp8_block_quant_torch(mx_ref.bf16_to_f64(x))
    xh = mx_ref.fp8_block_dequant_torch(xq, xs)

    def ffn(d):
        g, u = xh @ d["gate"].T, xh @ d["up"].T
        return mx_ref.fp8_block_quant_f64(g / (1 + np.exp(-g)) * u) @ d["down"].T

    ref = ffn(_dense_any(shared[0]))
    for e, ex in experts.items():
        m = np.zeros(wl.tokens)
        for j in range(idx.shape[1]):
            m += np.where(idx[:, j] == e, w[:, j], 0.0)
        ref = ref + m[:, None] * ffn(_dense(ex))
    assert np.allclose(y64, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())


def test_fp8_shared_expert_identity_closed_form_and_block_scales():
    # gate = up = P (E4M3 code 0x38 = 1.0) with a different power of two in each
    # 32 x 32 block row, down = P^T: the closed form needs the block of each row
    H, I = 256, 128
    one = 0x38
    g = np.zeros((I, H), np.uint8)
    g[np.arange(I), np.arange(I)] = one
    d = np.zeros((H, I), np.uint8)
    d[np.arange(I), np.arange(I)] = one
    a = np.arange(I // 32) - 1                       # gate exponent per block row
    gs = np.repeat((127 + a)[:, None], H // 32, axis=1).astype(np.uint8)
    us = np.full((I // 32, H // 32), 127, np.uint8)
    ds = np.full((H // 32, I // 32), 126, np.uint8)   # down x 1/2
    shared = [{"fmt": 1, "gate_codes": g, "gate_scales": gs, "up_codes": g.copy(), "up_scales": us,
               "down_codes": d, "down_scales": ds}]
    rng = np.random.default_rng(29)
    x = synth.f32_to_bf16_bits(rng.standard_normal((5, H)).astype(np.float32) * 2)
    idx = np.zeros((5, 0), np.int32)
    w = np.zeros((5, 0))
    _, y64 = oracle.moe_layer(x, idx, w, {}, shared, 4, I)
    xq, xs = mx_ref.fp8_block_quant_torch(mx_ref.bf16_to_f64(x))
    xh = mx_ref.fp8_block_dequant_torch(xq, xs)[:, :I]
    ga = np.repeat(2.0 ** a, 32)[None, :] * xh
    h = ga / (1 + np.exp(-ga)) * xh
    ref = np.zeros((5, H))
    ref[:, :I] = 0.5 * mx_ref.fp8_block_quant_f64(h)
    assert np.allclose(y64, ref, rtol=1e-12, atol=0)
