"""Expert parallelism over torch.distributed ranks: the partition of the routed
experts and the data plane of one layer step.

The routed experts are split in contiguous ranges over R ranks
(`expert_ranges`); one rank also holds the shared experts.  A layer step on
rank r, for its own batch of T tokens (every rank the same T):

  1. all-gather: the bf16 rows of every rank's batch (R*T tokens in all);
  2. route all R*T tokens (the router is replicated, so every rank gets the
     same routing: one fixed-order fp32 computation of the same inputs);
  3. the rank's share of y for all R*T tokens: its experts' weighted outputs
     (and the shared experts' on the rank that holds them), fp32;
  4. all-to-all: each token's R shares go to the token's rank;
  5. y of the rank's tokens = bf16(share_0 + share_1 + ... in rank order)
     (+ residual).

The exchange is x once (H * 2 bytes per token to every rank) and the fp32
shares (H * 4 bytes per token from every rank); each rank streams the weights
of its own experts only, so the decode cost per rank is its share of the
selected experts' bytes (FreeToken issue #444, janit's comment item 1: rate =
bandwidth / routed bytes).  Steps 2, 3 and 5 are the library's moe_route,
moe_forward_partial and moe_combine_partials (`library_step_fns`); this module
only moves the buffers.  The compute callables are injected, so the plan and
the exchange can be exercised on CPU ranks with any implementation of them.
"""
from __future__ import annotations

from typing import Callable

import torch


def expert_ranges(n_experts: int, n_ranks: int) -> list[tuple[int, int]]:
    """Contiguous ranges [lo, hi) of routed experts per rank, sizes differing by
    at most one (the lower ranks take the extra ones)."""
    if n_ranks < 1 or n_experts < n_ranks:
        raise ValueError("need 1 <= ranks <= experts")
    base, extra = divmod(n_experts, n_ranks)
    out, lo = [], 0
    for r in range(n_ranks):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def owner_of_expert(e: int, ranges: list[tuple[int, int]]) -> int:
    for r, (lo, hi) in enumerate(ranges):
        if lo <= e < hi:
            return r
    raise ValueError(f"expert {e} outside every range")


# route(x_all [N][H] int16) -> (idx [N][k] int32, w [N][k] fp32)
RouteFn = Callable[[torch.Tensor], tuple[torch.Tensor, torch.Tensor]]
# partial(x_all, idx, w) -> share [N][H] fp32
PartialFn = Callable[[torch.Tensor, torch.Tensor, torch.Tensor], torch.Tensor]
# combine(shares [R][T][H] fp32, residual [T][H] int16 or None) -> y [T][H] int16 (bf16 bits)
CombineFn = Callable[[torch.Tensor, torch.Tensor | None], torch.Tensor]


def ep_layer_step(pg, x_local: torch.Tensor, route: RouteFn, partial: PartialFn, combine: CombineFn,
                  residual_local: torch.Tensor | None = None) -> torch.Tensor:
    """One layer step of this rank's batch x_local [T][H] (bf16 bits in int16).
    pg: torch.distributed (initialised).  Returns y [T][H] (bf16 bits)."""
    R = pg.get_world_size()
    T, H = x_local.shape
    x_all = torch.empty((R * T, H), dtype=x_local.dtype, device=x_local.device)
    # as bytes: both backends (NCCL, gloo) move uint8, not every one 16-bit integers
    pg.all_gather_into_tensor(x_all.view(torch.uint8), x_local.contiguous().view(torch.uint8))
    idx, w = route(x_all)
    share = partial(x_all, idx, w)                    # [R*T][H], rows of rank q's tokens at q*T..
    shares = torch.empty_like(share)
    pg.all_to_all_single(shares, share.contiguous())  # now [R][T][H]: share of rank q for my tokens
    return combine(shares.view(R, T, H), residual_local)


def library_step_fns(layer, max_tokens_all: int, device) -> tuple[RouteFn, PartialFn, CombineFn]:
    """The three compute steps through the library, for a Layer created with
    its rank's expert range (Layer(..., expert_range=...)) on `device`, whose
    max_tokens is at least the step's tokens over all ranks (max_tokens_all)."""
    import mxfp4_expert_ffn_gb300 as m
    H, k = layer.cfg.hidden, layer.cfg.top_k
    idx = torch.empty((max_tokens_all, k), dtype=torch.int32, device=device)
    w = torch.empty((max_tokens_all, k), dtype=torch.float32, device=device)
    share = torch.empty((max_tokens_all, H), dtype=torch.float32, device=device)

    def route(x_all):
        N = x_all.shape[0]
        layer.route(x_all, N, idx[:N], w[:N])
        return idx[:N], w[:N]

    def partial(x_all, i, ww):
        N = x_all.shape[0]
        layer.forward_partial(x_all, N, i, ww, share[:N])
        return share[:N]

    def combine(shares, residual):
        R, T, _ = shares.shape
        y = torch.empty((T, H), dtype=torch.int16, device=device)
        m.moe_combine_partials(shares, R, T, H, residual, y)
        return y

    return route, partial, combine
