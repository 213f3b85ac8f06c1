"""Parity at the full workload sizes, in the launch configuration bench.py
times (MoELayer with the default tiles), on sampled outputs the oracle
computes (tests/oracle_samples.py, pinned against the oracle's whole-layer
functions on CPU).

Inputs come from the device generator (tens of GB of bf16 master weights);
the oracle quantises on the host only the expert matrices its samples need.
Checked per workload:
  * routing of every token (indices exact, weights to 1e-6 relative);
  * the activation's global scale (exact) and sampled quantised rows (exact);
  * the full permutation maps and counts (exact) and sampled gathered rows;
  * the sampled tokens' routed rows: every 16-feature block of the fused
    SwiGLU requantisation, and the whole down-projection row;
  * the layer output of the sampled tokens: 16 spread tokens of the decode
    and skewed batches, every 64th token of the prefill batch (256).
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U
from tests.oracle_samples import TokenSample

pytestmark = pytest.mark.gpu

FULL = ["decode_t128", "decode_t1024", "skewed_t2048", "prefill_t16384"]


def sampled_tokens(w):
    """Every 64th token of a batch of more than 1024 tokens, else 16 spread tokens."""
    step = 64 if w.T > 4096 else max(1, w.T // 16)
    return np.arange(step // 2, w.T, step)


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


class Case:
    def __init__(self, B, name):
        self.w = w = W.WORKLOADS[name]
        self.inp = W.device_inputs(w, seed=0, device=torch.device("cuda"))
        self.layer = B.MoELayer(self.inp["w_gu"], self.inp["w_d"], w.k, w.score, w.renormalize, w.h_scale,
                                bias=self.inp["bias"], T=w.T)
        self.out = self.layer(self.inp["x"], self.inp["logits"]).float().cpu().numpy()
        B.sync_status()
        self.x32 = self.inp["x"].float().cpu().numpy()
        self.s_x = O.global_scale(self.x32)
        self.bias = None if self.inp["bias"] is None else self.inp["bias"].cpu().numpy()
        self.idx, self.wts = O.route_topk(self.inp["logits"].cpu().numpy(), self.bias, w.k, w.score, w.renormalize)


@pytest.fixture(scope="module", params=FULL)
def case(request, B):
    c = Case(B, request.param)
    yield c
    del c
    torch.cuda.empty_cache()


def test_route_quantise_permute(case):
    w, L = case.w, case.layer
    np.testing.assert_array_equal(L.topk_idx.cpu().numpy(), case.idx)
    gw = L.topk_w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gw - case.wts) <= 1e-6 * case.wts)
    assert L.x_gscale.item() == case.s_x
    rows = np.linspace(0, w.T - 1, 8).astype(int)
    q, s = O.quantize_nvfp4(case.x32[rows], case.s_x)
    np.testing.assert_array_equal(L.xq.cpu().numpy()[rows], q)
    np.testing.assert_array_equal(L.xs.cpu().numpy()[rows], s)
    counts, offsets, p2f, f2p = O.permute(case.idx, w.E)
    np.testing.assert_array_equal(L.perm.counts.cpu().numpy(), counts)
    roff = L.perm.row_offsets.cpu().numpy()
    e_of = case.idx.reshape(-1)
    g_f2p = L.perm.flat_to_perm.cpu().numpy()
    np.testing.assert_array_equal(g_f2p - roff[e_of] + offsets[e_of], f2p)
    g_p2f = L.perm.perm_to_flat.cpu().numpy()
    for e in np.nonzero(counts)[0]:
        np.testing.assert_array_equal(g_p2f[roff[e]:roff[e] + counts[e]], p2f[offsets[e]:offsets[e + 1]])
    flats = np.linspace(0, w.R - 1, 16).astype(int)
    toks = flats // w.k
    qa, sa = O.quantize_nvfp4(case.x32[toks], case.s_x)
    np.testing.assert_array_equal(L.perm.a_packed[torch.from_numpy(g_f2p[flats]).cuda()].cpu().numpy(), qa)
    cap = L.perm.rows_capacity
    np.testing.assert_array_equal(U.from_blocked(L.perm.a_scales.cpu().numpy(), cap, w.H)[g_f2p[flats]], sa)


@pytest.fixture(scope="module")
def sample(case):
    w = case.w
    return TokenSample(sampled_tokens(w), case.x32, case.idx, case.wts, case.inp["w_gu"], case.inp["w_d"],
                       s_x=case.s_x, s_h=w.h_scale)


def test_gate_up_swiglu_requant_sampled_rows(case, sample):
    """Every 16-feature block of the fused SwiGLU requantisation of the
    sampled tokens' routed rows (2048 rows x 256 blocks at prefill)."""
    w, L = case.w, case.layer
    rows = L.perm.flat_to_perm.cpu().numpy()[sample.flat_ids(w.k)]
    cap = L.perm.rows_capacity
    got_c = O.unpack_codes(L.hq[torch.from_numpy(rows).cuda()].cpu().numpy())
    got_s = U.from_blocked(L.hs.cpu().numpy(), cap, w.I)[rows]
    assert got_s.size >= 1000
    eq, frac = U.check_requant(got_c, got_s, sample.h_codes, sample.h_scales)
    print(f"{w.name}: {got_s.size} blocks, scales equal {eq:.6f}, codes one step apart {frac:.2e}")


def test_down_projection_sampled_rows(case, sample):
    """The whole bf16 down-projection row of every sampled routed row."""
    w, L = case.w, case.layer
    rows = L.perm.flat_to_perm.cpu().numpy()[sample.flat_ids(w.k)]
    got = L.y[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    U.check_close(got, sample.y, what=f"{w.name} down rows")


def test_layer_output_sampled_tokens(case, sample):
    U.check_close(case.out[sample.tokens], sample.out, what=f"{case.w.name} layer, {len(sample.tokens)} tokens")
