"""moe_route_static: the router entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc (a runtime whose device
memory pool is owned by its own allocator, or a step that must not risk a
device-synchronising or failing allocation).  Its logits scratch is a fixed
array inside the library.  This file is collected last so that a run that
stops at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_gb300 as m
import synth
from synth import gpu as sg
from synth.workloads import VERIFY_T32, Workload
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [VERIFY_T32.with_tokens(64),
                                Workload("noalloc_h256_e16", 256, 128, 16, 2, 1, 7, seed=21)],
                         ids=lambda w: w.name)
def test_route_static_matches_route_on_two_calls(wl):
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
        x = sg.bf16_tensor(synth.activations(wl, stream=40 + call), gu.DEV)
        idx_a = torch.empty((T, k), dtype=torch.int32, device=gu.DEV)
        w_a = torch.empty((T, k), dtype=torch.float32, device=gu.DEV)
        L.route(x, T, idx_a, w_a)
        idx_b = torch.full((T, k), -1, dtype=torch.int32, device=gu.DEV)
        w_b = torch.full((T, k), -1.0, dtype=torch.float32, device=gu.DEV)
        m.moe_route_static(x, T, wl.hidden, E, k, W["router_w"], W.get("router_b"), idx_b, w_b)
        torch.cuda.synchronize()
        assert np.array_equal(idx_b.cpu().numpy(), idx_a.cpu().numpy()), call
        assert np.allclose(w_b.cpu().numpy(), w_a.cpu().numpy(), rtol=2e-6, atol=1e-7), call
    L.close()


def test_route_static_rejects_oversize_and_bad_shapes():
    wl = VERIFY_T32
    x = torch.zeros((129, wl.hidden), dtype=torch.int16, device=gu.DEV)
    Wr = torch.zeros((wl.n_experts, wl.hidden), device=gu.DEV)
    idx = torch.empty((129, 6), dtype=torch.int32, device=gu.DEV)
    w = torch.empty((129, 6), device=gu.DEV)
    T_over = m.ROUTE_STATIC_MAX_LOGITS // wl.n_experts + 1
    with pytest.raises(m.MoeError) as e:
        m.moe_route_static(x, T_over, wl.hidden, wl.n_experts, 6, Wr, None, idx, w)
    assert e.value.status == m.MOE_ERR_UNSUPPORTED
    with pytest.raises(m.MoeError) as e:
        m.moe_route_static(x, 4, 200, wl.n_experts, 6, Wr, None, idx, w)
    assert e.value.status == m.MOE_ERR_INVALID_ARG
