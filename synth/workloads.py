"""The synthetic workloads: one tiny layer, and DeepSeek-V4.1-Flash-shaped
MoE layers (hidden 5120, expert intermediate 2304, 384 routed experts top-6
plus one shared expert) at decode, verification-block, prefill and
8-layer-stack sizes.  Geometry from the FreeToken issue #444 ("Architecture
delta vs deepseek_v4": 384 routed + 1 shared, top-6, 3 x 5120 x 2304 FP4) and
the ai.rs article's table "What V4.1 Flash is, in bytes".
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    n_shared: int
    tokens: int
    seed: int
    layers: int = 1
    scale_lo: int = -8      # UE8M0 exponents uniform on [scale_lo, scale_hi]
    scale_hi: int = -4
    zipf: float | None = None   # router-bias Zipf exponent, None = unbiased
    rmsnorm: bool = False   # stack: normalise each layer's input

    def with_tokens(self, t: int) -> "Workload":
        return replace(self, tokens=t)

    @property
    def expert_bytes(self) -> int:
        """Bytes of one expert: codes (1/2 B) plus scales (1/32 B) per weight."""
        n = 3 * self.hidden * self.inter
        return n // 2 + n // 32


_V41 = dict(hidden=5120, inter=2304, n_experts=384, top_k=6, n_shared=1)

TINY = Workload("tiny_h256_e16_t4", 256, 128, 16, 2, 1, 4, seed=0, scale_lo=-6, scale_hi=-2)
DECODE_T1 = Workload("v41_layer_decode_t1", tokens=1, seed=1, **_V41)
VERIFY_T5 = Workload("v41_layer_verify_t5_zipf", tokens=5, seed=2, zipf=1.1, **_V41)
VERIFY_T32 = Workload("v41_layer_verify_t32_zipf", tokens=32, seed=3, zipf=1.1, **_V41)
PREFILL_T4096 = Workload("v41_layer_prefill_t4096", tokens=4096, seed=4, **_V41)
# a mid-size batch (64-token tiles, ~4 slots per expert): between decode and prefill
MID_T256 = Workload("v41_layer_t256", tokens=256, seed=11, **_V41)
# prefill sweep: tensor-pipe use as the tokens per expert grow (~64 at 4096)
PREFILL_T16K = Workload("v41_layer_prefill_t16384", tokens=16384, seed=8, **_V41)
PREFILL_T32K = Workload("v41_layer_prefill_t32768", tokens=32768, seed=9, **_V41)
PREFILL_T64K = Workload("v41_layer_prefill_t65536", tokens=65536, seed=10, **_V41)
STACK8_T64 = Workload("v41_stack8_decode_t64_zipf", tokens=64, seed=5, layers=8, zipf=1.1,
                      rmsnorm=True, **_V41)

# V4.1 expert shapes with a 24-expert bank (~450 MB, above the 126 MB L2): small
# enough for an ncu capture with memory save/restore; not a benchmark line.
NCU_DECODE_T1 = Workload("ncu_v41_e24_decode_t1", tokens=1, seed=6, **{**_V41, "n_experts": 24})
NCU_PREFILL = Workload("ncu_v41_e24_prefill_t512", tokens=512, seed=7, **{**_V41, "n_experts": 24})
# one layer of the decode stack's shape (64 tokens, Zipf(1.1) routing) with a 128-expert bank
# (~2.4 GB): small enough for a full ncu capture; not a benchmark line.
NCU_STACK_T64 = Workload("ncu_v41_e128_decode_t64_zipf", tokens=64, seed=12, zipf=1.1,
                         **{**_V41, "n_experts": 128})

WORKLOADS = {w.name: w for w in (TINY, DECODE_T1, VERIFY_T5, VERIFY_T32, MID_T256, PREFILL_T4096, PREFILL_T16K,
                                 PREFILL_T32K, PREFILL_T64K, STACK8_T64,
                                 NCU_DECODE_T1, NCU_PREFILL, NCU_STACK_T64)}
