"""Whole-layer parity (route -> quantise -> permute -> gate/up + SwiGLU +
requantise -> down -> finalize) of the CUDA library against the CPU oracle
on shapes the oracle runs in full: the tiny layer and medium layers with
ragged experts, several M tiles and partial K tiles."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


CASES = [W.WORKLOADS["tiny"]] + list(W.TEST_WORKLOADS.values())


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_layer_matches_oracle(B, w):
    inp = W.host_inputs(w, seed=0)
    cuda = torch.device("cuda")
    bias = inp["bias"]
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, w.renormalize, w.h_scale,
                       bias=None if bias is None else bias.to(cuda))
    out = layer(inp["x"].to(cuda), inp["logits"].to(cuda)).float().cpu().numpy()
    B.sync_status()

    gq = U.oracle_quantize_experts(inp["w_gu"])
    dq = U.oracle_quantize_experts(inp["w_d"])
    # the library's weight quantisation is bit-exact with the oracle's
    np.testing.assert_array_equal(U.packed_weights(layer.w_gu_packed), gq[0])
    np.testing.assert_array_equal(U.packed_weights(layer.w_d_packed), dq[0])
    np.testing.assert_array_equal(layer.w_gu_gscale.cpu().numpy(), gq[2])
    for e in range(w.E):
        np.testing.assert_array_equal(U.from_blocked(layer.w_d_scales[e].cpu().numpy(), w.H, w.I), dq[1][e])

    ref, it = O.moe_layer(inp["x"].float().numpy(), inp["logits"].numpy(),
                          None if bias is None else bias.numpy(), *gq, *dq, w.k, w.score,
                          np.float32(w.h_scale), renormalize=w.renormalize, return_intermediates=True)
    # bit-exact stages
    np.testing.assert_array_equal(layer.topk_idx.cpu().numpy(), it["idx"])
    assert layer.x_gscale.item() == it["s_x"]
    np.testing.assert_array_equal(layer.xq.cpu().numpy(), it["xq"])
    np.testing.assert_array_equal(layer.xs.cpu().numpy(), it["xs"])
    np.testing.assert_array_equal(layer.perm.counts.cpu().numpy(), it["counts"])
    # fused requantisation of the SwiGLU output
    roff = layer.perm.row_offsets.cpu().numpy()
    pos = np.concatenate([roff[e] + np.arange(it["counts"][e]) for e in range(w.E)])
    cap = layer.perm.rows_capacity
    U.check_requant(O.unpack_codes(layer.hq.cpu().numpy()[pos]),
                    U.from_blocked(layer.hs.cpu().numpy(), cap, w.I)[pos], O.unpack_codes(it["hq"]), it["hs"])
    # floating-point outputs
    U.check_close(layer.y.float().cpu().numpy()[pos], it["y"], what="down projection")
    U.check_close(out, ref, what="layer output")


def test_layer_is_deterministic(B):
    w = W.TEST_WORKLOADS["zipf_small"]
    inp = W.host_inputs(w, seed=5)
    cuda = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, w.renormalize, w.h_scale,
                       bias=inp["bias"].to(cuda))
    x, lg = inp["x"].to(cuda), inp["logits"].to(cuda)
    a = layer(x, lg).clone()
    b = layer(x, lg).clone()
    B.sync_status()
    assert torch.equal(a, b)


def test_layer_single_token(B):
    w = W.Workload("one_token", T=1, E=16, k=4, H=256, I=128, score="sigmoid")
    inp = W.host_inputs(w, seed=9)
    cuda = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, True, w.h_scale)
    out = layer(inp["x"].to(cuda), inp["logits"].to(cuda)).float().cpu().numpy()
    B.sync_status()
    ref = O.moe_layer(inp["x"].float().numpy(), inp["logits"].numpy(), None,
                      *U.oracle_quantize_experts(inp["w_gu"]), *U.oracle_quantize_experts(inp["w_d"]), w.k,
                      w.score, np.float32(w.h_scale))
    U.check_close(out, ref, what="single-token layer")


@pytest.mark.parametrize("tile_n", [(0, 0), (-1, -1), (-2, -2), (128, 128)],
                         ids=["autotuned", "token-major", "pairs", "weight-rows-as-M"])
def test_layer_all_tokens_on_two_experts(B, tile_n):
    """The most skewed routing: a bias of +8 on experts 3 and 11 of 16 sends
    every token to those two, so each holds all 600 tokens -- several token
    tiles and a ragged last one in every tile orientation (600 = 2 x 256 + 88
    = 4 x 128 + 88) -- and the other 14 experts are empty.  The down GEMM's K
    (I = 384) ends in a half stage."""
    w = W.Workload("two_hot", T=600, E=16, k=2, H=512, I=384, score="sigmoid")
    inp = W.host_inputs(w, seed=11)
    bias = np.zeros(w.E, np.float32)
    bias[[3, 11]] = 8.0
    cuda = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, True, w.h_scale,
                       bias=torch.from_numpy(bias).to(cuda), tile_n=tile_n)
    out = layer(inp["x"].to(cuda), inp["logits"].to(cuda)).float().cpu().numpy()
    B.sync_status()
    counts = layer.perm.counts.cpu().numpy()
    assert counts[3] == counts[11] == w.T and counts.sum() == w.T * w.k
    ref = O.moe_layer(inp["x"].float().numpy(), inp["logits"].numpy(), bias,
                      *U.oracle_quantize_experts(inp["w_gu"]), *U.oracle_quantize_experts(inp["w_d"]), w.k,
                      w.score, np.float32(w.h_scale))
    U.check_close(out, ref, what=f"layer output, tiles {tile_n}")


def test_layer_most_experts(B):
    """The largest expert count the library takes (E = 1024, k = 32): 64
    tokens over 1024 experts leave most of them empty or with a row or two,
    and the GEMMs' per-expert tile map fills 16 KB of their shared memory."""
    w = W.Workload("e1024", T=64, E=1024, k=32, H=256, I=128, score="softmax")
    inp = W.host_inputs(w, seed=13)
    cuda = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, True, w.h_scale)
    out = layer(inp["x"].to(cuda), inp["logits"].to(cuda)).float().cpu().numpy()
    B.sync_status()
    ref = O.moe_layer(inp["x"].float().numpy(), inp["logits"].numpy(), None,
                      *U.oracle_quantize_experts(inp["w_gu"]), *U.oracle_quantize_experts(inp["w_d"]), w.k,
                      w.score, np.float32(w.h_scale))
    U.check_close(out, ref, what="E = 1024 layer output")
