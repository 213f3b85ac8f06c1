"""Full-size parity of the layer variants on the decode_t128 shape (T=128,
E=256, k=8, H=6144, I=2048), in the launch configuration bench.py times:
MXFP4 operands, and batch-aware routing (k_primary = 2).  Every token's
routing and the whole permutation are compared exactly; one token's layer
output is computed by the oracle, which quantises only that token's experts."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U

pytestmark = pytest.mark.gpu

TOKEN = 77


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


@pytest.fixture(scope="module", params=["mxfp4", "batch_aware_k2"])
def run(request, B):
    w = W.WORKLOADS["decode_t128"]
    inp = W.device_inputs(w, seed=0, device=torch.device("cuda"))
    mx = request.param == "mxfp4"
    k0 = None if mx else 2
    layer = B.MoELayer(inp["w_gu"], inp["w_d"], w.k, w.score, w.renormalize, w.h_scale, bias=inp["bias"], T=w.T,
                       fmt="mxfp4" if mx else "nvfp4", k_primary=k0)
    out = layer(inp["x"], inp["logits"]).float().cpu().numpy()
    B.sync_status()
    yield dict(w=w, inp=inp, layer=layer, out=out, mx=mx, k0=k0)
    del layer, inp
    torch.cuda.empty_cache()


def routing(r):
    w = r["w"]
    lg = r["inp"]["logits"].cpu().numpy()
    if r["k0"] is None:
        return O.route_topk(lg, None, w.k, w.score, w.renormalize)
    return O.route_batch_aware(lg, None, w.k, r["k0"], w.score, w.renormalize)


def test_routing_and_permutation(run):
    r = run
    w, L = r["w"], r["layer"]
    idx, wts = routing(r)
    np.testing.assert_array_equal(L.topk_idx.cpu().numpy(), idx)
    gw = L.topk_w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gw - wts) <= 1e-6 * np.abs(wts))
    counts, offsets, p2f, f2p = O.permute(idx, w.E)
    np.testing.assert_array_equal(L.perm.counts.cpu().numpy(), counts)
    np.testing.assert_array_equal(L.perm.offsets.cpu().numpy(), offsets)
    roff = L.perm.row_offsets.cpu().numpy()
    g_f2p = L.perm.flat_to_perm.cpu().numpy()
    e_of = idx.reshape(-1)
    np.testing.assert_array_equal(g_f2p - roff[e_of] + offsets[e_of], f2p)
    if r["k0"] is not None:
        std, _ = O.route_topk(r["inp"]["logits"].cpu().numpy(), None, w.k, w.score, w.renormalize)
        assert len(np.unique(idx)) < len(np.unique(std))   # fewer experts stream their weights


def test_one_token_output(run):
    r = run
    w = r["w"]
    idx, wts = routing(r)
    x32 = r["inp"]["x"].float().cpu().numpy()
    if r["mx"]:
        xq, xs = O.quantize_mxfp4(x32[TOKEN:TOKEN + 1])
        xd = O.dequantize_mxfp4(xq, xs)
    else:
        s_x = O.global_scale(x32)
        xq, xs = O.quantize_nvfp4(x32[TOKEN:TOKEN + 1], s_x)
        xd = O.dequantize_nvfp4(xq, xs, s_x)
    acc = np.zeros(w.H)
    for j in range(w.k):
        e = int(idx[TOKEN, j])
        a_gu = r["inp"]["w_gu"][e].float().cpu().numpy()
        a_d = r["inp"]["w_d"][e].float().cpu().numpy()
        if r["mx"]:
            gu = xd @ O.dequantize_mxfp4(*O.quantize_mxfp4(a_gu)).T
            h = O.swiglu(gu, w.I).astype(np.float32)
            hd = O.dequantize_mxfp4(*O.quantize_mxfp4(h))
            y = O.round_to_bf16(hd @ O.dequantize_mxfp4(*O.quantize_mxfp4(a_d)).T)
        else:
            g_gu, g_d = O.global_scale(a_gu), O.global_scale(a_d)
            gu = xd @ O.dequantize_nvfp4(*O.quantize_nvfp4(a_gu, g_gu), g_gu).T
            h = O.swiglu(gu, w.I).astype(np.float32)
            s_h = np.float32(w.h_scale)
            hd = O.dequantize_nvfp4(*O.quantize_nvfp4(h, s_h), s_h)
            y = O.round_to_bf16(hd @ O.dequantize_nvfp4(*O.quantize_nvfp4(a_d, g_d), g_d).T)
        acc += wts[TOKEN, j] * y[0]
    ref = O.round_to_bf16(acc)
    U.check_close(r["out"][TOKEN], ref, what=("MXFP4" if r["mx"] else "batch-aware") + " layer, one token")
