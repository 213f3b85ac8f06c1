"""Full-size parity of the layer variants on the decode_t128 shape (T=128,
E=256, k=8, H=6144, I=2048), in the launch configuration bench.py times:
MXFP4 operands, and batch-aware routing (k_primary = 2).  Every token's
routing and the whole permutation are compared exactly; for 16 spread tokens
the oracle (tests/oracle_samples.py) gives the SwiGLU requantisation of
their routed rows, their down-projection rows and their layer output,
quantising only the experts those tokens use."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U
from tests.oracle_samples import TokenSample

pytestmark = pytest.mark.gpu

TOKENS = np.arange(4, 128, 8)          # 16 spread tokens of the 128


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


@pytest.fixture(scope="module")
def sample(run):
    r = run
    w = r["w"]
    idx, wts = routing(r)
    x32 = r["inp"]["x"].float().cpu().numpy()
    return TokenSample(TOKENS, x32, idx, wts, r["inp"]["w_gu"], r["inp"]["w_d"],
                       fmt="mxfp4" if r["mx"] else "nvfp4", s_x=None if r["mx"] else O.global_scale(x32),
                       s_h=w.h_scale)


def _what(r):
    return "MXFP4" if r["mx"] else "batch-aware"


def test_sampled_rows_requant_and_down_projection(run, sample):
    r = run
    w, L = r["w"], r["layer"]
    rows = L.perm.flat_to_perm.cpu().numpy()[sample.flat_ids(w.k)]
    blk = 32 if r["mx"] else 16
    got_c = O.unpack_codes(L.hq[torch.from_numpy(rows).cuda()].cpu().numpy())
    got_s = U.from_blocked(L.hs.cpu().numpy(), L.perm.rows_capacity, w.I, blk)[rows]
    assert got_s.size >= 1000
    U.check_requant(got_c, got_s, sample.h_codes, sample.h_scales, block=blk)
    got_y = L.y[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    U.check_close(got_y, sample.y, what=_what(r) + " down rows")


def test_sampled_tokens_output(run, sample):
    U.check_close(run["out"][TOKENS], sample.out, what=_what(run) + f" layer, {len(TOKENS)} tokens")
