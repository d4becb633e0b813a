"""GPU parity against the fp64 oracle through the C ABI, on small layers
that span several work units and ragged token chunks.  Routing, x codes and
segments are compared bit for bit; layer outputs within the layer tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_gb300 as m
import oracle
import synth
from synth import gpu as sg
from synth.workloads import TINY, Workload
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

SMALL = [
    TINY,
    Workload("ragged_h384_i256_e16_k2_t37", 384, 256, 16, 2, 1, 37, seed=11, scale_lo=-6, scale_hi=-2),
    Workload("h512_i384_e40_k6_s2_t13", 512, 384, 40, 6, 2, 13, seed=12, scale_lo=-7, scale_hi=-3),
    Workload("h256_i256_e8_k8_s0_t9", 256, 256, 8, 8, 0, 9, seed=13, scale_lo=-6, scale_hi=-2),
]


def _x(wl, T=None, stream=0):
    return synth.activations(wl, tokens=T, stream=stream)


# ------------------------------------------------------------- quantiser
def test_quantize_act_bit_exact_exhaustive_bf16():
    # every finite bf16 bit pattern, 32 per block, plus blocks with mixed
    # magnitudes so each value is quantised under many block scales
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = synth.bf16_bits_to_f32(bits)
    fin = bits[np.isfinite(vals)]
    rng = np.random.default_rng(0)
    a = fin[: fin.size // 256 * 256].reshape(-1, 256)
    b = rng.permutation(fin)[: fin.size // 256 * 256].reshape(-1, 256)
    x = np.concatenate([a, b, np.zeros((1, 256), np.uint16), np.full((1, 256), 0x8000, np.uint16)])
    wl = TINY
    L, _ = gu.make_layer(wl, max_tokens=x.shape[0])
    q = torch.empty(x.shape, dtype=torch.uint8, device=gu.DEV)
    s = torch.empty((x.shape[0], x.shape[1] // 32), dtype=torch.uint8, device=gu.DEV)
    L.quantize_act(sg.bf16_tensor(x), x.shape[0], q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_act(x)
    assert np.array_equal(s.cpu().numpy(), rs)
    qq = q.cpu().numpy()
    bad = np.argwhere(qq != rq)
    assert bad.size == 0, [(x[i, j], qq[i, j], rq[i, j]) for i, j in bad[:5]]
    L.close()


# ------------------------------------------------------------- routing
@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_route_bit_exact_given_oracle_logits(wl):
    L, W = gu.make_layer(wl)
    x = _x(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl), synth.router_bias(wl))
    ridx, rw = oracle.topk(lg, wl.top_k)
    idx, w, lo = gu.run_route(L, x, wl.tokens, wl.n_experts, wl.top_k, logits_in=lg)
    assert np.array_equal(idx, ridx)
    assert np.array_equal(lo, lg)
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-7)
    L.close()


def test_route_ties_nan_and_signed_zero():
    wl = Workload("ties_e384_k6", 256, 128, 384, 6, 1, 16, seed=14)
    L, _ = gu.make_layer(wl)
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((16, 384)).astype(np.float32)
    lg[1, :] = 0.25
    lg[2, ::2], lg[2, 1::2] = 0.0, -0.0
    lg[3, :200] = np.nan
    lg[4, :] = np.round(lg[4] * 2) / 2
    lg[5, 383] = np.inf
    lg[6, :] = -np.inf
    lg[6, 300] = 1.0
    ridx, _ = oracle.topk(lg, 6)
    idx, _, _ = gu.run_route(L, _x(wl), 16, 384, 6, logits_in=lg)
    assert np.array_equal(idx, ridx)
    L.close()


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_router_logits_and_selection(wl):
    L, _ = gu.make_layer(wl)
    x = _x(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl), synth.router_bias(wl))
    idx, w, lo = gu.run_route(L, x, wl.tokens, wl.n_experts, wl.top_k)
    tol = 1e-5 * np.abs(lg).max(axis=1, keepdims=True)
    assert (np.abs(lo - lg) <= tol).all()
    # selections agree wherever the oracle's k-th / (k+1)-th margin exceeds
    # twice the logit tolerance (the gate is a switch near ties)
    srt = -np.sort(-lg, axis=1)
    margin = srt[:, wl.top_k - 1] - (srt[:, wl.top_k] if wl.top_k < wl.n_experts else -np.inf)
    ridx, _ = oracle.topk(lg, wl.top_k)
    sure = margin > 2 * tol[:, 0]
    assert np.array_equal(np.sort(idx[sure], 1), np.sort(ridx[sure], 1))
    L.close()


# ------------------------------------------------------------- segments
@pytest.mark.parametrize("T,E,k", [(1, 384, 6), (37, 16, 2), (4096, 384, 6), (700, 512, 8)])
def test_segments_bit_exact(T, E, k):
    wl = Workload("seg", 128, 128, E, k, 1, T, seed=15)
    L, _ = gu.make_layer(wl)
    rng = np.random.default_rng(T + E)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[0] = np.arange(k)  # a few heavy experts
    off = torch.empty(E + 1, dtype=torch.int32, device=gu.DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=gu.DEV)
    L.segments(torch.from_numpy(idx).to(gu.DEV), T, off, perm)
    torch.cuda.synchronize()
    roff, rperm = oracle.segments(idx, E)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(perm.cpu().numpy(), rperm)
    L.close()


# ------------------------------------------------------------- layer
def _oracle_routing(wl, x, layer=0):
    lg = oracle.router_logits(x, synth.router_weights(wl, layer), synth.router_bias(wl, layer))
    return oracle.topk(lg, wl.top_k)


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("path", [m.PATH_AUTO, m.PATH_SIMT, m.PATH_MMA])
def test_layer_matches_oracle(wl, path):
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, path)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    y = gu.run_forward(L, x, idx, w)
    ref = gu.oracle_layer(wl, 0, x, idx, w)
    gu.assert_y_close(y, ref)
    L.close()


# Few work units with many K stages: the tensor-core GEMM cuts the units' K
# range across CTAs and the last CTA of each unit adds the partial tiles.
# gate/up split (K = 5120, 20 stages, ~10 pieces per unit); down split (K = 2304,
# 6 stages in 3-chunk steps, 2-3 pieces per unit); ragged token tiles.
SPLIT = [
    Workload("split_up_h5120_i256_e8_k2_t3", 5120, 256, 8, 2, 1, 3, seed=21, scale_lo=-8, scale_hi=-4),
    Workload("split_down_h1024_i2304_e8_k2_t3", 1024, 2304, 8, 2, 1, 3, seed=22, scale_lo=-8, scale_hi=-4),
    Workload("split_both_h5120_i2304_e6_k1_t2", 5120, 2304, 6, 1, 1, 2, seed=23, scale_lo=-8, scale_hi=-4),
    # 64-token tiles read by every token (40 tokens): pieces of units whose tile holds more than 32 slots
    Workload("split_dense_h5120_i256_e4_k2_t40", 5120, 256, 4, 2, 1, 40, seed=27, scale_lo=-8, scale_hi=-4),
]


@pytest.mark.parametrize("wl", SPLIT, ids=lambda w: w.name)
def test_split_partition_matches_oracle_and_is_deterministic(wl):
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, m.PATH_MMA)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    y = gu.run_forward(L, x, idx, w)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, w))
    for _ in range(3):  # partial tiles are added in piece order, whoever arrives last
        assert np.array_equal(gu.run_forward(L, x, idx, w), y)
    L.close()


def test_layer_with_residual_matches_oracle():
    wl = SMALL[1]
    L, _ = gu.make_layer(wl)
    x = _x(wl)
    r = _x(wl, stream=3)
    idx, w = _oracle_routing(wl, x)
    y = gu.run_forward(L, x, idx, w, residual_bits=r)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, w, residual=r))
    L.close()


@pytest.mark.parametrize("path", [m.PATH_SIMT, m.PATH_MMA])
def test_heavy_expert_duplicates_and_zero_weights(path):
    # every token on the same experts (long token chunks), a repeated id in a
    # row, and zero combine weights
    wl = SMALL[1]
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, path)
    x = _x(wl)
    T = wl.tokens
    idx = np.tile(np.array([[3, 3]], np.int32), (T, 1))
    idx[::5, 1] = 7
    w = np.tile(np.array([[0.6, 0.4]]), (T, 1))
    w[::3] = 0.0
    y = gu.run_forward(L, x, idx, w)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, w))
    L.close()


@pytest.mark.parametrize("path", [m.PATH_SIMT, m.PATH_MMA])
def test_deterministic_and_permutation_equivariant(path):
    wl = SMALL[2]
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, path)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    y1 = gu.run_forward(L, x, idx, w)
    y2 = gu.run_forward(L, x, idx, w)
    assert np.array_equal(y1, y2)
    p = np.random.default_rng(2).permutation(wl.tokens)
    yp = gu.run_forward(L, x[p], idx[p], w[p])
    assert np.array_equal(yp, y1[p])
    L.close()


def test_token_count_edges():
    wl = SMALL[1]
    L, _ = gu.make_layer(wl, max_tokens=wl.tokens)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    # T = 0 is a no-op, T = max_tokens works, T = max_tokens + 1 is rejected
    L.forward(sg.bf16_tensor(x), 0, torch.zeros(1, dtype=torch.int32, device=gu.DEV),
              torch.zeros(1, device=gu.DEV), torch.zeros(8, dtype=torch.int16, device=gu.DEV))
    with pytest.raises(m.MoeError) as e:
        L.forward(sg.bf16_tensor(x), wl.tokens + 1, torch.zeros(1, device=gu.DEV),
                  torch.zeros(1, device=gu.DEV), torch.zeros(8, device=gu.DEV))
    assert e.value.status == m.MOE_ERR_INVALID_ARG
    for T in (1, wl.tokens):
        y = gu.run_forward(L, x[:T], idx[:T], w[:T])
        gu.assert_y_close(y, gu.oracle_layer(wl, 0, x[:T], idx[:T], w[:T]))
    L.close()


@pytest.mark.parametrize("path", [m.PATH_SIMT, m.PATH_MMA])
def test_expert_id_out_of_range_is_reported_and_recovers(path):
    wl = SMALL[1]
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, path)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    bad = idx.copy()
    bad[1, 0] = wl.n_experts + 3
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    L.forward(xt, wl.tokens, torch.from_numpy(bad).to(gu.DEV),
              torch.from_numpy(w.astype(np.float32)).to(gu.DEV), y)
    assert L.sync() == m.MOE_ERR_INTERNAL
    assert L.sync() == m.MOE_OK  # the error word is cleared
    gu.assert_y_close(gu.run_forward(L, x, idx, w), gu.oracle_layer(wl, 0, x, idx, w))
    L.close()


@pytest.mark.parametrize("T", [37, 130])
def test_wait_that_gives_up_is_reported_and_recovers(T):
    """MOE_OPT_WAIT_LIMIT = 0: every pipeline wait of the tensor-core GEMMs gives
    up at once.  The call ends (each kernel lets its issued copies and MMAs
    finish, frees its tensor memory and returns), moe_sync reports
    MOE_ERR_TIMEOUT, and the next call with the default limit matches the
    oracle.  37 tokens: gathered 16-token tiles with the combine in the down
    GEMM; 130 tokens: 64-token tiles and the separate combine."""
    wl = SMALL[1].with_tokens(T)
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, m.PATH_MMA)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    xt = sg.bf16_tensor(x)
    it = torch.from_numpy(idx).to(gu.DEV)
    wt = torch.from_numpy(w.astype(np.float32)).to(gu.DEV)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    for call in ("forward", "step"):
        L.set_option(m.MOE_OPT_WAIT_LIMIT, 0)
        if call == "forward":
            L.forward(xt, T, it, wt, y)
        else:
            L.step(xt, T, y)
        assert L.sync() == m.MOE_ERR_TIMEOUT, call
        assert L.sync() == m.MOE_OK, call  # the error word is cleared
        L.set_option(m.MOE_OPT_WAIT_LIMIT, m.WAIT_LIMIT_DEFAULT)
        gu.assert_y_close(gu.run_forward(L, x, idx, w), gu.oracle_layer(wl, 0, x, idx, w), what=call)
    for bad in (-1, 1 << 31):
        with pytest.raises(m.MoeError) as e:
            L.set_option(m.MOE_OPT_WAIT_LIMIT, bad)
        assert e.value.status == m.MOE_ERR_INVALID_ARG
    L.close()


@pytest.mark.parametrize("norm_eps", [1e-6, -1.0])
def test_stack_forward_host_matches_device_loop_and_oracle(norm_eps):
    """moe_stack_forward_host over three layers (host x in, host y out) gives
    the same bits as the device loop of moe_rmsnorm + moe_step (or moe_step
    alone without normalisation), and each layer of that loop matches the
    oracle given its input (teacher forcing)."""
    base = SMALL[1]
    wls = [Workload(f"stack_l{i}", base.hidden, base.inter, base.n_experts, base.top_k, base.n_shared,
                    base.tokens, seed=30 + i, scale_lo=-6, scale_hi=-2) for i in range(3)]
    T, H = base.tokens, base.hidden
    Ls = [gu.make_layer(wl)[0] for wl in wls]
    x0 = _x(base, stream=7)
    cur = x0
    for wl, L in zip(wls, Ls):
        if norm_eps >= 0:
            xn_t = torch.empty((T, H), dtype=torch.int16, device=gu.DEV)
            m.moe_rmsnorm(sg.bf16_tensor(cur), T, H, norm_eps, xn_t)
            torch.cuda.synchronize()
            xin = xn_t.cpu().numpy().view(np.uint16)
        else:
            xin = cur
        y = torch.empty((T, H), dtype=torch.int16, device=gu.DEV)
        lo = torch.empty((T, wl.n_experts), dtype=torch.float32, device=gu.DEV)
        L.step(sg.bf16_tensor(xin), T, y, residual=sg.bf16_tensor(cur), logits_out=lo)
        assert L.sync() == m.MOE_OK
        ridx, rw = oracle.topk(lo.cpu().numpy(), wl.top_k)
        yb = y.cpu().numpy().view(np.uint16)
        gu.assert_y_close(yb, gu.oracle_layer(wl, 0, xin, ridx, rw, residual=cur), what=wl.name)
        cur = yb
    xh = torch.from_numpy(x0.view(np.int16).copy()).pin_memory()
    yh = torch.empty(xh.shape, dtype=torch.int16).pin_memory()
    for _ in range(2):
        yh.fill_(0)
        m.moe_stack_forward_host(Ls, xh, T, norm_eps, yh)
        assert np.array_equal(yh.numpy().view(np.uint16), cur)
    # a layer whose hidden size differs is refused before anything runs
    other, _ = gu.make_layer(TINY)
    with pytest.raises(m.MoeError) as e:
        m.moe_stack_forward_host([Ls[0], other], xh, T, norm_eps, yh)
    assert e.value.status == m.MOE_ERR_INVALID_ARG
    other.close()
    for L in Ls:
        L.close()


# ---- expert parallelism: rank layers over expert ranges, run one after the
# other on one GPU (their kernels never wait on each other), shares added by
# moe_combine_partials

EP_CASES = [
    (SMALL[1], 2),                                                             # 37 tokens, 16 experts
    (Workload("ep_h512_i256_e40_k6_s1_t130", 512, 256, 40, 6, 1, 130, seed=61,  # 64-token tiles
              scale_lo=-7, scale_hi=-3), 3),
    (Workload("ep_h256_i128_e16_k2_s1_t5", 256, 128, 16, 2, 1, 5, seed=62,      # decode-size tiles
              scale_lo=-6, scale_hi=-2), 4),
]


@pytest.mark.parametrize("wl,R", EP_CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_expert_parallel_shares_match_oracle_and_whole_layer(wl, R):
    from mxfp4_expert_ffn_gb300 import ep
    W = sg.device_layer(wl, 0, gu.DEV)
    T, H, E, k = wl.tokens, wl.hidden, wl.n_experts, wl.top_k
    x = _x(wl)
    xt = sg.bf16_tensor(x)
    ranges = ep.expert_ranges(E, R)
    layers = []
    for r, (lo, hi) in enumerate(ranges):
        Wr = {key: (v[lo:hi] if key.split("_")[0] in ("gate", "up", "down") else v)
              for key, v in W.items() if r == 0 or not key.startswith("s_")}
        layers.append(m.Layer(H, wl.inter, E, k, wl.n_shared if r == 0 else 0, T, Wr, expert_range=(lo, hi)))
    # every rank routes the batch the same way; the oracle's routing is used here
    idx, w = _oracle_routing(wl, x)
    it = torch.from_numpy(idx).to(gu.DEV)
    wt = torch.from_numpy(w.astype(np.float32)).to(gu.DEV)
    shares = torch.empty((R, T, H), dtype=torch.float32, device=gu.DEV)
    for r, L in enumerate(layers):
        L.forward_partial(xt, T, it, wt, shares[r])
        assert L.sync() == m.MOE_OK  # other ranks' experts are skipped without an error
    y = torch.empty((T, H), dtype=torch.int16, device=gu.DEV)
    res = sg.bf16_tensor(_x(wl, stream=5))
    m.moe_combine_partials(shares, R, T, H, res, y)
    torch.cuda.synchronize()
    yb = y.cpu().numpy().view(np.uint16)
    gu.assert_y_close(yb, gu.oracle_layer(wl, 0, x, idx, w, residual=_x(wl, stream=5)), what=f"EP x{R}")
    # the whole layer on one GPU: the same result up to the order of the fp32 sums
    full, _ = gu.make_layer(wl, weights=W)
    gu.assert_y_close(yb, gu.run_forward(full, x, idx, w, residual_bits=_x(wl, stream=5)), what="vs one layer")
    # a rank's share holds exactly its own experts: rank 1's share of a token
    # routed only to rank 0's experts is zero
    lo1, hi1 = ranges[1]
    only0 = [t for t in range(T) if not any(lo1 <= e < hi1 for e in idx[t])]
    if only0:
        assert np.all(shares[1, only0].cpu().numpy() == 0.0)
    full.close()
    for L in layers:
        L.close()


def test_fault_injection_launch_and_arg(monkeypatch):
    wl = TINY
    L, _ = gu.make_layer(wl)
    x = sg.bf16_tensor(_x(wl))
    z = torch.zeros((wl.tokens, wl.top_k), dtype=torch.int32, device=gu.DEV)
    zf = torch.zeros((wl.tokens, wl.top_k), device=gu.DEV)
    y = torch.empty_like(x)
    for mode, status in (("launch", m.MOE_ERR_CUDA), ("arg", m.MOE_ERR_INVALID_ARG)):
        monkeypatch.setenv("MOE_FAULT", mode)
        with pytest.raises(m.MoeError) as e:
            L.forward(x, wl.tokens, z, zf, y)
        assert e.value.status == status
    monkeypatch.delenv("MOE_FAULT")
    L.forward(x, wl.tokens, z, zf, y)
    assert L.sync() == m.MOE_OK
    L.close()


@pytest.mark.parametrize("wl", [SMALL[2], SMALL[1]], ids=lambda w: w.name)
def test_forward_host_matches_device_path(wl):
    # 13 tokens of 1 KB come back with the error word in one copy through the
    # pinned staging; 37 tokens of 768 B exceed the 16 KB staging and are
    # copied straight to the caller.  Repeated calls, a changed token count and
    # a changed option (the routing changes with it) must each match the
    # device path.
    L, _ = gu.make_layer(wl)
    T0 = wl.tokens
    calls = [T0, T0, T0, T0 - 4, T0 - 4, T0 - 4, T0, "sigmoid", T0, T0, T0]
    for i, T in enumerate(calls):
        if T == "sigmoid":
            L.set_scoring(m.MOE_SCORING_SIGMOID, 2.5)
            continue
        x = _x(wl, T=T, stream=i)
        xh = torch.from_numpy(x.view(np.int16)).pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        L.forward_host(xh, T, yh)
        idx, w, _ = gu.run_route(L, x, T, wl.n_experts, wl.top_k)
        yd = gu.run_forward(L, x, idx, w)
        assert np.array_equal(yh.numpy().view(np.uint16), yd), (i, T)
    L.close()


# at least 512 tokens: 112-token tiles (several per expert, ragged), both MMA issuers
# splitting the down tile's columns 64 + 48
PREFILL_SMALL = Workload("prefill_h512_i256_e16_k4_t600", 512, 256, 16, 4, 1, 600, seed=27,
                         scale_lo=-8, scale_hi=-4)


def test_prefill_tiles_match_oracle():
    wl = PREFILL_SMALL
    L, _ = gu.make_layer(wl)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    y = gu.run_forward(L, x, idx, w)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, w))
    assert np.array_equal(gu.run_forward(L, x, idx, w), y)
    L.close()


STEP = SMALL + [
    Workload("step_h1024_i256_e64_k6_t64", 1024, 256, 64, 6, 1, 64, seed=24, scale_lo=-8, scale_hi=-4),
    # up to 64 tokens with experts of more than 32 slots (one 64-token tile each) and two shared experts
    Workload("step_h512_i256_e8_k4_s2_t60", 512, 256, 8, 4, 2, 60, seed=28, scale_lo=-8, scale_hi=-4),
    Workload("step_h512_i256_e32_k4_t80", 512, 256, 32, 4, 1, 80, seed=25, scale_lo=-8, scale_hi=-4),
]


@pytest.mark.parametrize("wl", STEP, ids=lambda w: w.name)
@pytest.mark.parametrize("path", [m.PATH_AUTO, m.PATH_SIMT])
def test_step_equals_route_then_forward_and_matches_oracle(wl, path):
    """moe_step (one launch for router + top-k + x codes + segments at up to
    64 tokens) gives bit for bit what moe_route then moe_forward give; its
    routing is the oracle's given its own logits; y is within tolerance."""
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, path)
    x = _x(wl)
    T, E, k = wl.tokens, wl.n_experts, wl.top_k
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
    lo = torch.empty((T, E), dtype=torch.float32, device=gu.DEV)
    L.step(xt, T, y, idx=idx, w=w, logits_out=lo)
    assert L.sync() == m.MOE_OK
    y, idx, w, lo = (y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy(),
                     lo.cpu().numpy())
    idx2, w2, lo2 = gu.run_route(L, x, T, E, k)
    assert np.array_equal(lo, lo2) and np.array_equal(idx, idx2) and np.array_equal(w, w2)
    assert np.array_equal(gu.run_forward(L, x, idx2, w2), y)
    ridx, rw = oracle.topk(lo.astype(np.float32), k)
    assert np.array_equal(idx, ridx)
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-7)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, rw))
    # with a residual and without the optional outputs
    r = _x(wl, stream=5)
    y3 = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    L.step(xt, T, y3, residual=sg.bf16_tensor(r))
    assert L.sync() == m.MOE_OK
    assert np.array_equal(y3.cpu().numpy().view(np.uint16), gu.run_forward(L, x, idx2, w2, residual_bits=r))
    L.close()


# ---- 17 to 64 tokens with 64-token tiles and many down units: the kernel
# variant in which down starts per token tile (gate/up counts its finished
# units per tile) and takes whole units dynamically (units >= 4 per CTA:
# 40 row tiles of H = 5120 times ~60 active tiles)
EARLY = Workload("early_h5120_i256_e64_k6_t40", 5120, 256, 64, 6, 1, 40, seed=29, scale_lo=-8, scale_hi=-4)


def test_down_per_tile_matches_oracle_deterministic_and_equivariant():
    """The per-tile down start with dynamically taken units: y within the
    layer tolerance of the oracle, the same bits on every repeat (which CTA
    takes a unit changes nothing), moe_route + moe_forward bit for bit, and a
    permutation of the tokens permutes y bit for bit."""
    wl = EARLY
    L, _ = gu.make_layer(wl)
    x = _x(wl)
    T, E, k = wl.tokens, wl.n_experts, wl.top_k
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
    lo = torch.empty((T, E), dtype=torch.float32, device=gu.DEV)
    L.step(xt, T, y, idx=idx, w=w, logits_out=lo)
    assert L.sync() == m.MOE_OK
    y1 = y.cpu().numpy().view(np.uint16).copy()
    idx, w, lo = idx.cpu().numpy(), w.cpu().numpy(), lo.cpu().numpy()
    assert len(np.unique(idx)) * (wl.hidden // 128) >= 4 * torch.cuda.get_device_properties(0).multi_processor_count
    for _ in range(3):
        L.step(xt, T, y)
        assert L.sync() == m.MOE_OK
        assert np.array_equal(y.cpu().numpy().view(np.uint16), y1)
    idx2, w2, lo2 = gu.run_route(L, x, T, E, k)
    assert np.array_equal(lo, lo2) and np.array_equal(idx, idx2) and np.array_equal(w, w2)
    assert np.array_equal(gu.run_forward(L, x, idx2, w2), y1)
    ridx, rw = oracle.topk(lo.astype(np.float32), k)
    assert np.array_equal(idx, ridx)
    gu.assert_y_close(y1, gu.oracle_layer(wl, 0, x, idx, rw))
    p = np.random.default_rng(3).permutation(T)
    assert np.array_equal(gu.run_forward(L, x[p], idx[p], w[p]), y1[p])
    L.close()


# ---- sigmoid scoring with a selection-only bias and a routed scaling factor

SIG_ZIPF = Workload("sig_h512_i256_e64_k6_t20_zipf", 512, 256, 64, 6, 1, 20, seed=26, zipf=1.1,
                    scale_lo=-8, scale_hi=-4)

@pytest.mark.parametrize("wl", [SMALL[2], SIG_ZIPF, STEP[-1]], ids=lambda w: w.name)
def test_sigmoid_scoring_bit_exact_given_logits(wl):
    L, _ = gu.make_layer(wl)
    L.set_scoring(m.MOE_SCORING_SIGMOID, 2.5)
    x = _x(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl), None)   # unbiased logits
    lg[0, 3] = np.nan
    lg[1, :] = lg[1, 0]                                            # ties before the bias
    b = synth.router_bias(wl)
    b = np.zeros(wl.n_experts, np.float32) if b is None else b
    ridx, rw = oracle.topk_sigmoid(lg, b, wl.top_k, 2.5)
    idx, w, lo = gu.run_route(L, x, wl.tokens, wl.n_experts, wl.top_k, logits_in=lg)
    assert np.array_equal(idx, ridx)
    assert np.allclose(w, rw, rtol=1e-6, atol=0)
    L.close()


@pytest.mark.parametrize("wl", [SMALL[1], SIG_ZIPF, STEP[-1]], ids=lambda w: w.name)
@pytest.mark.parametrize("path", [m.PATH_AUTO, m.PATH_SIMT])
def test_sigmoid_scoring_layer_matches_oracle(wl, path):
    """The GPU's own (unbiased) logits, sigmoid selection reproduced by the oracle
    bit for bit, the layer within tolerance; moe_step equals route + forward."""
    L, _ = gu.make_layer(wl)
    L.set_option(m.MOE_OPT_PATH, path)
    L.set_scoring(m.MOE_SCORING_SIGMOID, 2.5)
    x = _x(wl)
    T, E, k = wl.tokens, wl.n_experts, wl.top_k
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
    lo = torch.empty((T, E), dtype=torch.float32, device=gu.DEV)
    L.step(xt, T, y, idx=idx, w=w, logits_out=lo)
    assert L.sync() == m.MOE_OK
    y, idx, w, lo = (y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy(), lo.cpu().numpy())
    ref_lo = oracle.router_logits(x, synth.router_weights(wl), None)
    assert (np.abs(lo - ref_lo) <= 1e-5 * (1 + np.abs(ref_lo))).all()
    b = synth.router_bias(wl)
    ridx, rw = oracle.topk_sigmoid(lo, b, k, 2.5)
    assert np.array_equal(idx, ridx)
    assert np.allclose(w, rw, rtol=1e-6, atol=0)
    idx2, w2, lo2 = gu.run_route(L, x, T, E, k)
    assert np.array_equal(lo2, lo) and np.array_equal(idx2, idx) and np.array_equal(w2, w)
    assert np.array_equal(gu.run_forward(L, x, idx2, w2), y)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, ridx, rw))
    L.close()


def test_scoring_options_are_validated():
    L, _ = gu.make_layer(TINY)
    for opt, val in ((m.MOE_OPT_SCORING, 2), (m.MOE_OPT_ROUTED_SCALE, 0x7FC00000),
                     (m.MOE_OPT_ROUTED_SCALE, 0xBF800000), (m.MOE_OPT_ROUTED_SCALE, 0)):
        with pytest.raises(m.MoeError) as e:
            L.set_option(opt, val)
        assert e.value.status == m.MOE_ERR_INVALID_ARG
    L.close()


def test_rmsnorm_matches_oracle():
    rng = np.random.default_rng(8)
    x = synth.f32_to_bf16_bits((rng.standard_normal((33, 5120)) * 200).astype(np.float32))
    out = torch.empty((33, 5120), dtype=torch.int16, device=gu.DEV)
    m.moe_rmsnorm(sg.bf16_tensor(x), 33, 5120, 1e-6, out)
    torch.cuda.synchronize()
    got = gu.bits_to_f64(out)
    ref = gu.bits_to_f64(oracle.rmsnorm(x, 1e-6))
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7)  # within one bf16 ulp
    assert (got != ref).mean() < 0.01


def test_gpu_bank_fill_equals_host_generator():
    wl = SMALL[2]
    W = sg.device_layer(wl, 1, gu.DEV)
    for e in (0, 17, wl.n_experts - 1):
        ex = synth.host_expert(wl, 1, e)
        for k in ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes", "down_scales"):
            assert np.array_equal(W[k][e].cpu().numpy(), ex[k]), (e, k)
    sh = synth.host_expert(wl, 1, wl.n_experts + 1)
    assert np.array_equal(W["s_down_codes"][1].cpu().numpy(), sh["down_codes"])


@pytest.mark.parametrize("wl", [
    Workload("router_t200_e40_h256", 256, 128, 40, 6, 1, 200, seed=31),
    Workload("router_t130_e384_h512", 512, 128, 384, 6, 1, 130, seed=32, zipf=1.1),
], ids=lambda w: w.name)
def test_router_many_tokens_tensor_core(wl):
    # more than 64 tokens: logits from the tensor-core router (three bf16 parts
    # of W_r, K split over CTAs), ragged expert and token tiles
    L, _ = gu.make_layer(wl)
    x = _x(wl)
    lg = oracle.router_logits(x, synth.router_weights(wl), synth.router_bias(wl))
    idx, w, lo = gu.run_route(L, x, wl.tokens, wl.n_experts, wl.top_k)
    tol = 1e-5 * np.abs(lg).max(axis=1, keepdims=True)
    assert (np.abs(lo - lg) <= tol).all(), np.abs(lo - lg).max()
    srt = -np.sort(-lg, axis=1)
    sure = srt[:, wl.top_k - 1] - srt[:, wl.top_k] > 2 * tol[:, 0]
    ridx, _ = oracle.topk(lg, wl.top_k)
    assert np.array_equal(np.sort(idx[sure], 1), np.sort(ridx[sure], 1))
    L.close()


# ---- small batches of at most 32 slots (the one-warp segments in the
# preparation launch), with repeated experts across tokens and no or two
# shared experts
TINY_SLOTS = [
    Workload("tiny_h256_i128_e16_k6_t1", 256, 128, 16, 6, 1, 1, seed=31, scale_lo=-6, scale_hi=-2),
    Workload("tiny_h256_i128_e8_k8_s0_t4", 256, 128, 8, 8, 0, 4, seed=32, scale_lo=-6, scale_hi=-2),
    Workload("tiny_h384_i256_e8_k6_s2_t5", 384, 256, 8, 6, 2, 5, seed=33, scale_lo=-6, scale_hi=-2),
]


@pytest.mark.parametrize("wl", TINY_SLOTS, ids=lambda w: w.name)
def test_tiny_batches_step_forward_and_oracle(wl):
    L, _ = gu.make_layer(wl)
    x = _x(wl)
    T, E, k = wl.tokens, wl.n_experts, wl.top_k
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
    lo = torch.empty((T, E), dtype=torch.float32, device=gu.DEV)
    L.step(xt, T, y, idx=idx, w=w, logits_out=lo)
    assert L.sync() == m.MOE_OK
    y, idx, w, lo = (y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy(),
                     lo.cpu().numpy())
    ridx, rw = oracle.topk(lo.astype(np.float32), k)
    assert np.array_equal(idx, ridx)
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-7)
    assert np.array_equal(gu.run_forward(L, x, idx, w), y)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, rw))
    # every token on the same few experts, in different slot orders
    dup = np.stack([np.roll(np.arange(k, dtype=np.int32), t) for t in range(T)])
    gu.assert_y_close(gu.run_forward(L, x, dup, rw), gu.oracle_layer(wl, 0, x, dup, rw))
    # an out-of-range id is reported, then the next call is clean
    bad = idx.copy()
    bad[T - 1, k - 1] = E + 1
    yb = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    L.forward(xt, T, torch.from_numpy(bad).to(gu.DEV), torch.from_numpy(rw.astype(np.float32)).to(gu.DEV), yb)
    assert L.sync() == m.MOE_ERR_INTERNAL
    assert np.array_equal(gu.run_forward(L, x, idx, w), y)
    L.close()


# ---- FP4-activation variant (MOE_OPT_ACT_FORMAT): x and h as E2M1 per 32,
# expert GEMMs on kind::mxf4

def test_quantize_act4_bit_exact_exhaustive_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = synth.bf16_bits_to_f32(bits)
    fin = bits[np.isfinite(vals)]
    rng = np.random.default_rng(4)
    a = fin[: fin.size // 256 * 256].reshape(-1, 256)
    b = rng.permutation(fin)[: fin.size // 256 * 256].reshape(-1, 256)
    x = np.concatenate([a, b, np.zeros((1, 256), np.uint16), np.full((1, 256), 0x8000, np.uint16)])
    wl = TINY  # hidden 256
    L, _ = gu.make_layer(wl, max_tokens=x.shape[0])
    q = torch.empty((x.shape[0], x.shape[1] // 2), dtype=torch.uint8, device=gu.DEV)
    s = torch.empty((x.shape[0], x.shape[1] // 32), dtype=torch.uint8, device=gu.DEV)
    L.quantize_act4(sg.bf16_tensor(x), x.shape[0], q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_act4(x)
    assert np.array_equal(s.cpu().numpy(), rs)
    qq = q.cpu().numpy()
    bad = np.argwhere(qq != rq)
    assert bad.size == 0, [(x[i, 2 * j:2 * j + 2], qq[i, j], rq[i, j]) for i, j in bad[:5]]
    L.close()


ACT4 = [
    Workload("a4_h512_i256_e16_k6_t3", 512, 256, 16, 6, 1, 3, seed=41, scale_lo=-6, scale_hi=-2),
    Workload("a4_h512_i256_e32_k4_s2_t80", 512, 256, 32, 4, 2, 80, seed=42, scale_lo=-6, scale_hi=-2),
    Workload("a4_h512_i256_e16_k4_t600", 512, 256, 16, 4, 1, 600, seed=43, scale_lo=-8, scale_hi=-4),
    Workload("a4_h512_i256_e8_k4_t48", 512, 256, 8, 4, 1, 48, seed=44, scale_lo=-6, scale_hi=-2),
    SPLIT[2],  # 5120 x 2304: the split partition on both GEMMs
]


@pytest.mark.parametrize("wl", ACT4, ids=lambda w: w.name)
def test_fp4_activation_layer_matches_oracle(wl):
    L, _ = gu.make_layer(wl)
    L.set_act_format(m.MOE_ACT_FP4)
    x = _x(wl)
    T, E, k = wl.tokens, wl.n_experts, wl.top_k
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
    L.step(xt, T, y, idx=idx, w=w)
    assert L.sync() == m.MOE_OK
    y, idx, w = y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy()
    # route then forward gives the same bits; the layer is the oracle's FP4 variant
    assert np.array_equal(gu.run_forward(L, x, idx, w), y)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, w, act4=True))
    # and not the FP8 layer
    y8 = gu.oracle_layer(wl, 0, x, idx, w)
    d4 = np.abs(synth.bf16_bits_to_f32(y) - synth.bf16_bits_to_f32(y8)).max()
    assert d4 > 0
    L.close()


def test_fp4_activation_option_rules():
    L, _ = gu.make_layer(TINY)  # inter 128: not a multiple of 256
    with pytest.raises(m.MoeError) as e:
        L.set_act_format(m.MOE_ACT_FP4)
    assert e.value.status == m.MOE_ERR_UNSUPPORTED
    L.close()
    L, _ = gu.make_layer(ACT4[0])
    L.set_act_format(m.MOE_ACT_FP4)
    with pytest.raises(m.MoeError) as e:
        L.set_option(m.MOE_OPT_PATH, m.PATH_SIMT)
    assert e.value.status == m.MOE_ERR_UNSUPPORTED
    with pytest.raises(m.MoeError):
        L.set_act_format(7)
    L.set_act_format(m.MOE_ACT_FP8)
    L.set_option(m.MOE_OPT_PATH, m.PATH_SIMT)  # allowed again with FP8 activations
    L.close()


# ---- FP8 shared expert (MOE_OPT_SHARED_FORMAT): E4M3 weights with one UE8M0
# scale per 32 x 32 block, routed experts MXFP4

FP8_SHARED = [
    Workload("s8_h512_i256_e16_k6_t3", 512, 256, 16, 6, 1, 3, seed=51, scale_lo=-6, scale_hi=-2),
    Workload("s8_h512_i256_e32_k4_s2_t80", 512, 256, 32, 4, 2, 80, seed=52, scale_lo=-6, scale_hi=-2),
    Workload("s8_h512_i256_e16_k4_t600", 512, 256, 16, 4, 1, 600, seed=53, scale_lo=-8, scale_hi=-4),
    Workload("s8_h512_i256_e8_k4_t48", 512, 256, 8, 4, 1, 48, seed=54, scale_lo=-6, scale_hi=-2),
    SPLIT[2],
]


@pytest.mark.parametrize("wl", FP8_SHARED, ids=lambda w: w.name)
def test_fp8_shared_expert_layer_matches_oracle(wl):
    L, _ = gu.make_layer_fp8_shared(wl)
    x = _x(wl)
    T, k = wl.tokens, wl.top_k
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
    L.step(xt, T, y, idx=idx, w=w)
    assert L.sync() == m.MOE_OK
    y, idx, w = y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy()
    assert np.array_equal(gu.run_forward(L, x, idx, w), y)
    gu.assert_y_close(y, gu.oracle_layer(wl, 0, x, idx, w, shared_fp8=True))
    # only the shared experts' contribution: zero routed weights
    w0 = np.zeros_like(w)
    gu.assert_y_close(gu.run_forward(L, x, idx, w0), gu.oracle_layer(wl, 0, x, idx, w0, shared_fp8=True))
    L.close()


def test_fp8_shared_expert_option_rules():
    wl = FP8_SHARED[0]
    L, _ = gu.make_layer_fp8_shared(wl)
    for bad in ((m.MOE_OPT_PATH, m.PATH_SIMT), (m.MOE_OPT_ACT_FORMAT, m.MOE_ACT_FP4)):
        with pytest.raises(m.MoeError) as e:
            L.set_option(*bad)
        assert e.value.status == m.MOE_ERR_UNSUPPORTED
    with pytest.raises(m.MoeError):
        L.set_shared_format(9)
    L.close()
    L, _ = gu.make_layer(SMALL[3])  # no shared expert
    with pytest.raises(m.MoeError) as e:
        L.set_shared_format(m.MOE_SHARED_FP8_B32)
    assert e.value.status == m.MOE_ERR_UNSUPPORTED
    L.close()


def test_expert_id_out_of_range_above_64_tokens():
    # the slot-ordered quantiser and the segments kernel (no preparation launch)
    wl = STEP[-1]  # 80 tokens
    L, _ = gu.make_layer(wl)
    x = _x(wl)
    idx, w = _oracle_routing(wl, x)
    bad = idx.copy()
    bad[3, 1] = -5
    bad[70, 0] = wl.n_experts
    xt = sg.bf16_tensor(x)
    y = torch.empty(xt.shape, dtype=torch.int16, device=gu.DEV)
    L.forward(xt, wl.tokens, torch.from_numpy(bad).to(gu.DEV),
              torch.from_numpy(w.astype(np.float32)).to(gu.DEV), y)
    assert L.sync() == m.MOE_ERR_INTERNAL
    # the invalid slots contribute nothing: the oracle with their weights zeroed
    w0 = w.copy()
    w0[3, 1] = 0.0
    w0[70, 0] = 0.0
    ok = bad.copy()
    ok[3, 1] = idx[3, 1]
    ok[70, 0] = idx[70, 0]
    gu.assert_y_close(y.cpu().numpy().view(np.uint16), gu.oracle_layer(wl, 0, x, ok, w0))
    gu.assert_y_close(gu.run_forward(L, x, idx, w), gu.oracle_layer(wl, 0, x, idx, w))
    L.close()
