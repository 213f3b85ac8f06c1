"""The seeded synthetic workloads have the structure of the regimes the pages
measure (CPU only).

"SM120 FP4 Kernel Research Campaign" studies the GLM-5 MoE at decode, where
each expert sees about 16-64 rows, a skewed expert popularity, and large
per-expert M; the workloads stand in for those regimes.  Routing the
host-drawn logits with the oracle router (weights are not drawn) checks
that each workload lands in its regime.
"""
import numpy as np
import pytest

from nvfp4_block_scaled_07_gb300 import workloads as W
from oracle import nvfp4_moe_oracle as O


def expert_rows(name, seed=0):
    w = W.WORKLOADS[name]
    inp = W.host_inputs(w, seed=seed, with_weights=False)
    bias = None if inp["bias"] is None else inp["bias"].numpy()
    idx, _ = O.route_topk(inp["logits"].numpy(), bias, w.k, w.score, w.renormalize)
    assert all(len(set(r)) == w.k for r in idx.tolist())
    c = np.bincount(idx.reshape(-1), minlength=w.E)
    assert c.sum() == w.T * w.k
    return c


def test_decode_t128_few_rows_per_expert():
    c = expert_rows("decode_t128")
    assert (c > 0).sum() >= 240                 # nearly every expert's weights stream
    assert 2 <= np.median(c) <= 8 and c.max() <= 16


def test_decode_t1024_in_the_16_to_64_row_regime():
    c = expert_rows("decode_t1024")
    assert c.min() >= 16 and c.max() <= 64


def test_skewed_t2048_has_hot_and_cold_experts():
    c = expert_rows("skewed_t2048")
    assert c.max() >= 1000                       # nearly every token routes to the hottest expert
    assert (c >= 100).sum() >= 20                # a group of compute-heavy experts ...
    assert (c <= 4).sum() >= 150                 # ... beside a long tail of cold ones


def test_prefill_t16384_large_per_expert_m():
    c = expert_rows("prefill_t16384")
    w = W.WORKLOADS["prefill_t16384"]
    mean = w.T * w.k / w.E
    assert np.all(np.abs(c - mean) <= 0.1 * mean)


@pytest.mark.parametrize("name", ["tiny", "ragged_small"])
def test_quantise_then_permute_equals_permute_then_quantise(name):
    """The quantiser works row by row once the per-tensor scale is fixed, so
    gathering quantised rows equals quantising gathered rows."""
    w = {**W.WORKLOADS, **W.TEST_WORKLOADS}[name]
    inp = W.host_inputs(w, seed=4, with_weights=False)
    x = inp["x"].float().numpy()
    idx, _ = O.route_topk(inp["logits"].numpy(), None, w.k, w.score, w.renormalize)
    _, _, p2f, _ = O.permute(idx, w.E)
    s = O.global_scale(x)
    xq, xs = O.quantize_nvfp4(x, s)
    gq, gs = O.quantize_nvfp4(x[p2f // w.k], s)
    assert np.array_equal(xq[p2f // w.k], gq) and np.array_equal(xs[p2f // w.k], gs)
