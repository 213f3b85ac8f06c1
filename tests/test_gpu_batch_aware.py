"""Batch-aware routing on the GPU (reading R8 of the oracle): the standalone
call and the fused prepare against the oracle's route_batch_aware (indices
bit-exact, weights within 1e-6), and the whole layer with batch-aware
routing against the oracle layer."""
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


def routing_inputs(T, E, bias, ties, seed):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        lg = (np.round(lg * 4) / 4).astype(np.float32)
    b = W.zipf_bias(E, 1.1) if bias else None
    return lg, b


def check_routing(idx, w, ridx, rw):
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    gw = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gw - rw) <= 1e-6 * np.abs(rw) + 1e-30)


ROUTE_CASES = [
    # T, E, k, k_primary, score, renorm, bias, ties
    (128, 256, 8, 4, "sigmoid", True, False, False),   # decode shape
    (128, 256, 8, 1, "sigmoid", True, False, False),
    (128, 256, 8, 8, "sigmoid", True, False, False),   # plain top-k
    (1, 64, 8, 2, "sigmoid", True, False, False),      # one token: falls back outside the set
    (40, 64, 8, 1, "sigmoid", True, True, True),       # skewed bias: fewer than k members, ties
    (33, 1024, 32, 3, "sigmoid", False, False, True),  # widest router
    (50, 64, 6, 2, "softmax", False, False, False),
    (16, 8, 2, 1, "softmax", True, False, False),
]


@pytest.mark.parametrize("T,E,k,k0,score,renorm,bias,ties", ROUTE_CASES)
def test_route_batch_aware(B, T, E, k, k0, score, renorm, bias, ties):
    lg, b = routing_inputs(T, E, bias, ties, seed=T + 7 * E + k0)
    cuda = torch.device("cuda")
    b_d = None if b is None else torch.from_numpy(b).to(cuda)
    idx, w = B.moe_route_batch_aware(torch.from_numpy(lg).to(cuda), k, k0, score, renorm, bias=b_d)
    B.sync_status()
    check_routing(idx, w, *O.route_batch_aware(lg, b, k, k0, score, renorm))
    if k0 == k:
        pidx, pw = B.moe_route_topk(torch.from_numpy(lg).to(cuda), k, score, renorm, bias=b_d)
        assert torch.equal(idx, pidx) and torch.equal(w, pw)


@pytest.mark.parametrize("T,E,k,k0,H", [(128, 256, 8, 4, 512), (300, 64, 8, 1, 256), (2100, 64, 8, 2, 128),
                                        (1, 32, 4, 1, 64)])
def test_prepare_batch_aware(B, T, E, k, k0, H):
    lg, b = routing_inputs(T, E, True, False, seed=T * 3 + k0)
    x = torch.from_numpy(np.random.default_rng(T).standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    cuda = torch.device("cuda")
    lg_d, b_d, x_d = torch.from_numpy(lg).to(cuda), torch.from_numpy(b).to(cuda), x.to(cuda)
    ws = B.alloc_prepare_workspace(T, E, k, cuda)
    for _ in range(2):   # the second call checks that the active set was cleared
        idx, w, gs, xq, xs, perm = B.moe_prepare(lg_d, x_d, k, "sigmoid", True, bias=b_d, workspace=ws,
                                                 k_primary=k0)
        B.sync_status()
        ridx, rw = O.route_batch_aware(lg, b, k, k0, "sigmoid")
        check_routing(idx, w, ridx, rw)
        x32 = x.float().numpy()
        s_x = O.global_scale(x32)
        rxq, rxs = O.quantize_nvfp4(x32, s_x)
        assert gs.item() == s_x
        U.check_permutation(perm, ridx, E, rxq, rxs)
        lg = lg[::-1].copy()          # a different batch on the same workspace
        lg_d = torch.from_numpy(lg).to(cuda)
    # the standalone calls give the same bits
    sidx, sw = B.moe_route_batch_aware(lg_d, k, k0, "sigmoid", True, bias=b_d)
    idx, w, *_ = B.moe_prepare(lg_d, x_d, k, "sigmoid", True, bias=b_d, workspace=ws, k_primary=k0)
    B.sync_status()
    assert torch.equal(idx, sidx) and torch.equal(w.view(torch.int32), sw.view(torch.int32))


@pytest.mark.parametrize("name,k0,fused", [("zipf_small", 1, True), ("many_experts", 2, True),
                                           ("many_experts", 2, False)])
def test_layer_batch_aware_matches_oracle(B, name, k0, fused):
    w = W.TEST_WORKLOADS[name]
    inp = W.host_inputs(w, seed=11)
    cuda = torch.device("cuda")
    bias = inp["bias"]
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, w.renormalize, w.h_scale,
                       bias=None if bias is None else bias.to(cuda), fused_prepare=fused, k_primary=k0)
    out = layer(inp["x"].to(cuda), inp["logits"].to(cuda)).float().cpu().numpy()
    B.sync_status()
    gq = U.oracle_quantize_experts(inp["w_gu"])
    dq = U.oracle_quantize_experts(inp["w_d"])
    ref, it = O.moe_layer(inp["x"].float().numpy(), inp["logits"].numpy(), None if bias is None else bias.numpy(),
                          *gq, *dq, w.k, w.score, np.float32(w.h_scale), renormalize=w.renormalize,
                          return_intermediates=True, k_primary=k0)
    np.testing.assert_array_equal(layer.topk_idx.cpu().numpy(), it["idx"])
    np.testing.assert_array_equal(layer.perm.counts.cpu().numpy(), it["counts"])
    U.check_close(out, ref, what="batch-aware layer output")
    # fewer active experts than plain top-k
    std, _ = O.route_topk(inp["logits"].numpy(), None if bias is None else bias.numpy(), w.k, w.score)
    assert len(np.unique(it["idx"])) <= len(np.unique(std))
