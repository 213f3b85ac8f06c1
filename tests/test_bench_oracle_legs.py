"""bench.py's CPU legs (cpu_baseline and the reference arm) time the oracle
layer itself, in the layer's format and routing (CPU only).

The timed sample runs the oracle's steps for a subset of experts (and, in
the reference arm, a slice of the intermediate dimension).  Over all
experts, and over all slices stitched together, it must give the oracle
layer's output; otherwise the CPU figures would time some other workload.
"""
import numpy as np
import pytest

import bench
from nvfp4_block_scaled_07_gb300 import workloads as W
from oracle import nvfp4_moe_oracle as O


def _case(name, fmt, k0):
    w = {**W.WORKLOADS, **W.TEST_WORKLOADS}[name]
    inp = W.host_inputs(w, seed=5)
    x32 = inp["x"].float().numpy()
    lg = inp["logits"].numpy()
    b = None if inp["bias"] is None else inp["bias"].numpy()
    q = bench.oracle_quantized_weights(inp["w_gu"], inp["w_d"], range(w.E), fmt)
    stack = lambda part, i: np.stack([q[(part, e)][i] for e in range(w.E)])
    if fmt == "mxfp4":
        ref, inter = O.moe_layer_mx(x32, lg, b, stack("gu", 0), stack("gu", 1), stack("d", 0), stack("d", 1), w.k,
                                    w.score, w.renormalize, k_primary=k0, return_intermediates=True)
    else:
        gg = np.array([q[("gu", e)][2] for e in range(w.E)], np.float32)
        dg = np.array([q[("d", e)][2] for e in range(w.E)], np.float32)
        ref, inter = O.moe_layer(x32, lg, b, stack("gu", 0), stack("gu", 1), gg, stack("d", 0), stack("d", 1), dg,
                                 w.k, w.score, np.float32(w.h_scale), w.renormalize, k_primary=k0,
                                 return_intermediates=True)
    full_sum = O.finalize(inter["y"], inter["flat_to_perm"], inter["w"], w.T, w.k)
    return w, x32, lg, b, q, ref, full_sum


@pytest.mark.parametrize("name,fmt,k0", [("ragged_small", "nvfp4", None), ("zipf_small", "nvfp4", 1),
                                         ("many_experts", "mxfp4", None), ("many_experts", "mxfp4", 2)])
def test_sample_over_all_experts_is_the_oracle_layer(name, fmt, k0):
    w, x32, lg, b, q, ref, full_sum = _case(name, fmt, k0)
    *_, rows, n_active, out = bench.oracle_sample(w, x32, lg, b, q, range(w.E), fmt=fmt, k_primary=k0,
                                                  return_out=True)
    assert rows == w.T * w.k
    # the same terms summed in expert order instead of slot order: equal up to
    # float64 reassociation (absolute, since some sums cancel to near zero)
    np.testing.assert_allclose(out, full_sum, rtol=1e-12, atol=1e-12 * np.abs(full_sum).max())
    # and after the bf16 rounding, the same output (reassociation can only move
    # a sum lying within a few float64 ulps of a bf16 midpoint)
    assert np.mean(O.round_to_bf16(out) != ref) < 1e-4


@pytest.mark.parametrize("name,fmt", [("ragged_small", "nvfp4"), ("many_experts", "mxfp4")])
def test_intermediate_slices_add_up_to_the_layer(name, fmt):
    """The reference arm's per-step sample: slices of the intermediate
    dimension whose partial down projections add up to the expert's output
    (each partial is rounded to bf16, so the sum matches to bf16 precision)."""
    w, x32, lg, b, q, ref, full_sum = _case(name, fmt, None)
    width = min(w.I, 256)
    total = np.zeros_like(full_sum)
    for a in range(0, w.I, width):
        *_, out = bench.oracle_sample(w, x32, lg, b, q, range(w.E), islice=(a, min(w.I, a + width)), fmt=fmt,
                                      return_out=True)
        total += out
    rel = np.linalg.norm(total - full_sum) / np.linalg.norm(full_sum)
    assert rel < 1e-2
