"""moe_route_static: the router entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc (a runtime whose device
memory pool is owned by its own allocator, or a step that must not risk a
device-synchronising or failing allocation).  Its scratch is a fixed array
inside the library.  It must give the same routing as moe_route bit for bit
(the same split-K kernels), and that routing must be the oracle's top-k of
the logits moe_route reports.  This file is collected last so that a run
that stops at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_gb300 as m
import oracle
import synth
from synth import gpu as sg
from synth.workloads import VERIFY_T32, Workload
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = [
    VERIFY_T32.with_tokens(64),                                      # V4.1 router, 64 tokens, Zipf bias
    Workload("noalloc_h256_e16", 256, 128, 16, 2, 1, 7, seed=21),    # tiny, ragged token count
    # the largest request: T = MOE_ROUTE_STATIC_MAX_TOKENS tokens of E = 512 experts, k = 8
    Workload("noalloc_h1024_e512_t64", 1024, 128, 512, 8, 1, m.ROUTE_STATIC_MAX_TOKENS, seed=23),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_route_static_matches_route_and_oracle_on_two_calls(wl):
    W = {"router_w": torch.from_numpy(synth.router_weights(wl)).to(gu.DEV)}
    b = synth.router_bias(wl)
    if b is not None:
        W["router_b"] = torch.from_numpy(b).to(gu.DEV)
    # the existing entry point needs a layer; give it the real router and a
    # small dummy bank (the router does not read the experts)
    dummy = Workload("dummy", wl.hidden, 128, wl.n_experts, wl.top_k, 1, wl.tokens, seed=22)
    bank = sg.device_layer(dummy, 0, gu.DEV)
    bank.update(W)
    L = m.Layer(wl.hidden, 128, wl.n_experts, wl.top_k, 1, wl.tokens, bank)
    T, E, k = wl.tokens, wl.n_experts, wl.top_k
    for call in range(2):
        xb = synth.activations(wl, stream=40 + call)
        x = sg.bf16_tensor(xb, gu.DEV)
        idx_a = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
        w_a = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
        lo = torch.empty((T, E), dtype=torch.float32, device=gu.DEV)
        L.route(x, T, idx_a, w_a, logits_out=lo)
        # every row starts invalid, so an unwritten row (the last one included) fails
        idx_b = torch.full((T, k), -1, dtype=torch.int32, device=gu.DEV)
        w_b = torch.full((T, k), -1.0, dtype=torch.float32, device=gu.DEV)
        m.moe_route_static(x, T, wl.hidden, E, k, W["router_w"], W.get("router_b"), idx_b, w_b)
        torch.cuda.synchronize()
        ids, ws = idx_b.cpu().numpy(), w_b.cpu().numpy()
        # the same kernels as moe_route: identical bits
        assert np.array_equal(ids, idx_a.cpu().numpy()), call
        assert np.array_equal(ws.view(np.uint32), w_a.cpu().numpy().view(np.uint32)), call
        # the oracle's selection on those fp32 logits, and its weights
        lg = lo.cpu().numpy()
        ridx, rw = oracle.topk(lg, k)
        assert np.array_equal(ids, ridx), call
        assert np.allclose(ws, rw, rtol=2e-6, atol=1e-7), call
        # the logits themselves against the oracle's fp64 router
        lref = oracle.router_logits(xb, synth.router_weights(wl), b)
        assert (np.abs(lg - lref) <= 1e-5 * np.abs(lref).max(axis=1, keepdims=True)).all(), call
    L.close()


def test_route_static_rejects_oversize_and_bad_shapes():
    wl = VERIFY_T32
    T_max = m.ROUTE_STATIC_MAX_TOKENS
    x = torch.zeros((T_max + 1, wl.hidden), dtype=torch.int16, device=gu.DEV)
    Wr = torch.zeros((512 + 1, wl.hidden), device=gu.DEV)
    idx = torch.empty((T_max + 1, 8), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((T_max + 1, 8), device=gu.DEV)
    for args, want in [((x, T_max + 1, wl.hidden, wl.n_experts, 6), m.MOE_ERR_UNSUPPORTED),
                       ((x, 4, 200, wl.n_experts, 6), m.MOE_ERR_INVALID_ARG),    # H % 128
                       ((x, 4, wl.hidden, 513, 6), m.MOE_ERR_INVALID_ARG),       # E > 512
                       ((x, 4, wl.hidden, 4, 6), m.MOE_ERR_INVALID_ARG),         # k > E
                       ((x, 4, wl.hidden, wl.n_experts, 9), m.MOE_ERR_INVALID_ARG)]:  # k > 8
        with pytest.raises(m.MoeError) as e:
            m.moe_route_static(*args, Wr, None, idx, w)
        assert e.value.status == want, args[1:]
