"""The seeded generators: host C filler equals the numpy definition; the
workload shapes; Zipf bias sanity.  (The GPU filler is checked in
tests/test_gpu_parity.py.)"""
import numpy as np

import synth
from synth.workloads import DECODE_T1, STACK8_T64, TINY


def test_hostgen_matches_numpy_definition():
    for key in (synth.stream_key(0, 0, 0, 0, 0), synth.stream_key(5, 7, 2, 1, 384)):
        for n in (1, 7, 8, 1001, 4096):
            assert np.array_equal(synth.stream_bytes(key, n), synth.stream_bytes_numpy(key, n))
    assert np.array_equal(synth.scale_bytes(1, 0, 2, 5, 64, 2304, -8, -4),
                          synth.scale_bytes_numpy(1, 0, 2, 5, 64, 2304, -8, -4))


def test_codes_and_scales_distribution():
    ex = synth.host_expert(TINY, 0, 1)
    nib = np.concatenate([ex["gate_codes"].ravel() & 15, ex["gate_codes"].ravel() >> 4])
    assert set(np.unique(nib)) == set(range(16))
    s = ex["down_scales"].astype(int) - 127
    assert s.min() == TINY.scale_lo and s.max() == TINY.scale_hi


def test_experts_and_layers_differ():
    a = synth.host_expert(TINY, 0, 1)["gate_codes"]
    b = synth.host_expert(TINY, 0, 2)["gate_codes"]
    c = synth.host_expert(TINY, 1, 1)["gate_codes"]
    assert (a != b).mean() > 0.9 and (a != c).mean() > 0.9


def test_zipf_bias_is_monotone_in_rank():
    b = synth.router_bias(STACK8_T64, 0)
    assert b.shape == (384,) and b.max() == 0.0
    order = np.sort(b)[::-1]
    assert np.all(np.diff(order) < 0)
    assert synth.router_bias(DECODE_T1) is None
