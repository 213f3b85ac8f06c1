"""The full-size parity tests compare sampled tokens with oracle values that
tests/oracle_samples.py assembles expert by expert (threads, row chunks).
Here, on CPU-sized layers, that assembly must reproduce the oracle's own
whole-layer functions (moe_layer, moe_layer_mx) on every sampled token: the
SwiGLU rows, their requantisation, the down-projection rows and the layer
output.  A dropped slot, a wrong expert, a transposed weight or a wrong
scale in the assembly fails here, on the CPU."""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_07_gb300 import workloads as W
from oracle import nvfp4_moe_oracle as O
from tests import nvfp4_testutil as U
from tests.oracle_samples import TokenSample


def _whole_layer(w, inp, fmt, k0):
    x32 = inp["x"].float().numpy()
    lg = inp["logits"].numpy()
    b = None if inp["bias"] is None else inp["bias"].numpy()
    if fmt == "mxfp4":
        gp, gs = U.oracle_quantize_experts_mx(inp["w_gu"])
        dp, ds = U.oracle_quantize_experts_mx(inp["w_d"])
        out, it = O.moe_layer_mx(x32, lg, b, gp, gs, dp, ds, w.k, w.score, w.renormalize, k_primary=k0,
                                 return_intermediates=True)
    else:
        gp, gs, gg = U.oracle_quantize_experts(inp["w_gu"])
        dp, ds, dg = U.oracle_quantize_experts(inp["w_d"])
        out, it = O.moe_layer(x32, lg, b, gp, gs, gg, dp, ds, dg, w.k, w.score, np.float32(w.h_scale),
                              w.renormalize, k_primary=k0, return_intermediates=True)
    return x32, out, it


@pytest.mark.parametrize("name,fmt,k0", [("ragged_small", "nvfp4", None), ("zipf_small", "nvfp4", None),
                                         ("many_experts", "mxfp4", None), ("many_experts", "nvfp4", 2)])
def test_token_sample_reproduces_the_oracle_layer(name, fmt, k0):
    w = W.TEST_WORKLOADS[name]
    inp = W.host_inputs(w, seed=11)
    x32, out, it = _whole_layer(w, inp, fmt, k0)
    tokens = np.arange(1, w.T, 7)
    s = TokenSample(tokens, x32, it["idx"], it["w"], inp["w_gu"], inp["w_d"], fmt=fmt,
                    s_x=None if fmt == "mxfp4" else it["s_x"], s_h=w.h_scale, threads=3)
    rows = it["flat_to_perm"][s.flat_ids(w.k)]          # the pairs' rows in the oracle's permuted order
    np.testing.assert_array_equal(s.experts, it["idx"].reshape(-1)[s.flat_ids(w.k)])
    np.testing.assert_array_equal(s.h, it["h"][rows])
    np.testing.assert_array_equal(s.h_codes, O.unpack_codes(it["hq"][rows]))
    np.testing.assert_array_equal(s.h_scales, it["hs"][rows])
    np.testing.assert_array_equal(s.y, it["y"][rows])
    np.testing.assert_array_equal(s.out, out[tokens])


def test_token_sample_accepts_device_style_weight_stacks():
    # the full-size tests hand torch tensors (on the GPU there); any [E, N, K] stack works
    w = W.TEST_WORKLOADS["ragged_small"]
    inp = W.host_inputs(w, seed=12)
    x32, out, it = _whole_layer(w, inp, "nvfp4", None)
    tokens = np.array([0, w.T - 1])
    a = TokenSample(tokens, x32, it["idx"], it["w"], inp["w_gu"], inp["w_d"], s_x=it["s_x"], s_h=w.h_scale,
                    threads=1)
    b = TokenSample(tokens, x32, it["idx"], it["w"], inp["w_gu"].float().numpy(), inp["w_d"].float().numpy(),
                    s_x=it["s_x"], s_h=w.h_scale, threads=2)
    np.testing.assert_array_equal(a.out, b.out)
    np.testing.assert_array_equal(a.out, out[tokens])
    assert isinstance(inp["w_gu"], torch.Tensor)
