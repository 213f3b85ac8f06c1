"""Parity of moe_prepare -- route, quantise and permute in one cooperative
launch -- with the CPU oracle (router indices, global scale, quantised bytes,
permutation maps and gathered rows bit-exact; router weights within 1e-6)
and, bit for bit, with the three separate calls on the same inputs."""
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


def make_inputs(T, E, H, bias, ties, seed):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        lg = (np.round(lg * 4) / 4).astype(np.float32)   # many exactly equal logits
    b = W.zipf_bias(E, 1.1) if bias else None
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    return lg, b, x


CASES = [
    # T, E, k, H, score, renormalize, bias, ties
    (16, 8, 2, 256, "softmax", True, False, False),      # the tiny layer
    (128, 256, 8, 6144, "sigmoid", True, False, False),  # decode shape, one 256-id segment per 32 tokens
    (1, 16, 4, 256, "sigmoid", True, False, False),      # one token
    (33, 1, 1, 128, "softmax", True, False, False),      # one expert
    (40, 1024, 32, 64, "sigmoid", True, False, True),    # widest router (32 experts per lane), ties
    (700, 33, 5, 192, "sigmoid", False, True, True),     # ragged E, biased, unnormalised, ties
    (2100, 64, 8, 128, "sigmoid", True, True, False),    # T*k = 16800: 1024-id segments, scales by block
    (2100, 64, 8, 512, "sigmoid", True, False, False),   # the same with 16-byte scale gathers (8 words/row)
    (300, 4, 2, 1024, "softmax", True, False, False),    # few wide experts
]


@pytest.mark.parametrize("T,E,k,H,score,renorm,bias,ties", CASES)
def test_prepare_matches_oracle_and_separate_calls(B, T, E, k, H, score, renorm, bias, ties):
    lg, b, x = make_inputs(T, E, H, bias, ties, seed=T * 7 + E)
    cuda = torch.device("cuda")
    lg_d, x_d = torch.from_numpy(lg).to(cuda), x.to(cuda)
    b_d = None if b is None else torch.from_numpy(b).to(cuda)
    idx, w, gs, xq, xs, perm = B.moe_prepare(lg_d, x_d, k, score, renorm, bias=b_d)
    B.sync_status()

    # the oracle
    ridx, rw = O.route_topk(lg, b, k, score, renorm)
    x32 = x.float().numpy()
    s_x = O.global_scale(x32)
    rxq, rxs = O.quantize_nvfp4(x32, s_x)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    gw = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gw - rw) <= 1e-6 * np.abs(rw) + 1e-30)
    assert gs.item() == s_x
    np.testing.assert_array_equal(xq.cpu().numpy(), rxq)
    np.testing.assert_array_equal(xs.cpu().numpy(), rxs)
    U.check_permutation(perm, ridx, E, rxq, rxs)

    # the three separate calls, bit for bit
    sidx, sw = B.moe_route_topk(lg_d, k, score, renorm, bias=b_d)
    sxq, sxs, sgs = B.moe_quantize_nvfp4(x_d)
    sperm = B.moe_permute(sidx, E, sxq, sxs)
    B.sync_status()
    assert torch.equal(idx, sidx)
    assert torch.equal(w.view(torch.int32), sw.view(torch.int32))
    assert torch.equal(gs, sgs) and torch.equal(xq, sxq) and torch.equal(xs, sxs)
    for name in ("counts", "offsets", "row_offsets", "perm_to_flat", "flat_to_perm"):
        assert torch.equal(getattr(perm, name), getattr(sperm, name)), name
    rows = perm.flat_to_perm.long()
    assert torch.equal(perm.a_packed[rows], sperm.a_packed[rows])
    cap = perm.rows_capacity
    a = U.from_blocked(perm.a_scales.cpu().numpy(), cap, H)
    s = U.from_blocked(sperm.a_scales.cpu().numpy(), cap, H)
    np.testing.assert_array_equal(a[rows.cpu().numpy()], s[rows.cpu().numpy()])


def test_prepare_no_tokens(B):
    E, k, H = 12, 3, 128
    cuda = torch.device("cuda")
    idx, w, gs, xq, xs, perm = B.moe_prepare(torch.zeros((0, E), device=cuda),
                                             torch.zeros((0, H), dtype=torch.bfloat16, device=cuda), k)
    B.sync_status()
    assert gs.item() == 1.0
    U.check_permutation(perm, np.zeros((0, k), np.int32), E, np.zeros((0, H // 2), np.uint8),
                        np.zeros((0, H // 16), np.uint8))


def test_prepare_reuses_its_workspace(B):
    """Back-to-back calls on one workspace: the grid-barrier words are left
    at zero arrivals, and every call gives the same result as a fresh one."""
    T, E, k, H = 256, 64, 8, 512
    cuda = torch.device("cuda")
    ws = B.alloc_prepare_workspace(T, E, k, cuda)
    results = []
    for seed in (1, 2, 1):
        lg, b, x = make_inputs(T, E, H, True, False, seed=seed)
        lg_d, x_d, b_d = torch.from_numpy(lg).to(cuda), x.to(cuda), torch.from_numpy(b).to(cuda)
        r = B.moe_prepare(lg_d, x_d, k, "sigmoid", True, bias=b_d, workspace=ws)
        B.sync_status()
        assert ws[:4].view(torch.int32).item() == 0   # arrival counter back at zero
        results.append([t.clone() for t in r[:5]] + [r[5].perm_to_flat.clone(), r[5].flat_to_perm.clone()])
        fresh = B.moe_prepare(lg_d, x_d, k, "sigmoid", True, bias=b_d)
        B.sync_status()
        for got, ref in zip(results[-1], list(fresh[:5]) + [fresh[5].perm_to_flat, fresh[5].flat_to_perm]):
            assert torch.equal(got, ref)
    for a, c in zip(results[0], results[2]):
        assert torch.equal(a, c)


def test_prepare_rejects_small_or_misaligned_workspace(B):
    T, E, k, H = 8, 8, 2, 64
    cuda = torch.device("cuda")
    lg = torch.zeros((T, E), device=cuda)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device=cuda)
    need = B.moe_prepare_workspace_size(T, E, k)
    with pytest.raises(B.Nvfp4MoeError) as ei:
        B.moe_prepare(lg, x, k, workspace=torch.zeros((need - 256,), dtype=torch.uint8, device=cuda))
    assert ei.value.status == B.ERR_WORKSPACE
    big = torch.zeros((need + 512,), dtype=torch.uint8, device=cuda)
    with pytest.raises(B.Nvfp4MoeError) as ei:
        B.moe_prepare(lg, x, k, workspace=big[16:])
    assert ei.value.status == B.ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["zipf_small", "many_experts"])
def test_layer_fused_prepare_equals_separate_calls(B, name):
    w = W.TEST_WORKLOADS[name]
    inp = W.host_inputs(w, seed=4)
    cuda = torch.device("cuda")
    bias = None if inp["bias"] is None else inp["bias"].to(cuda)
    fused = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, w.renormalize, w.h_scale,
                       bias=bias, fused_prepare=True)
    sep = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, w.renormalize, w.h_scale,
                     bias=bias, fused_prepare=False)
    x, lg = inp["x"].to(cuda), inp["logits"].to(cuda)
    a = fused(x, lg).clone()
    c = sep(x, lg).clone()
    B.sync_status()
    assert torch.equal(a, c)
