"""Parity at the full workload sizes, in the launch configuration bench.py
times (MoELayer with the default tiles), on sampled outputs the oracle
computes one by one.

Inputs come from the device generator (tens of GB of bf16 master weights);
the oracle quantises on the host only the expert matrices its samples need.
Checked per workload:
  * routing of every token (indices exact, weights to 1e-6 relative);
  * the activation's global scale (exact) and sampled quantised rows (exact);
  * the full permutation maps and counts (exact) and sampled gathered rows;
  * sampled 16-feature blocks of the fused SwiGLU requantisation;
  * sampled down-projection outputs of two routed rows;
  * the layer output of one token (decode and skewed workloads).
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U

pytestmark = pytest.mark.gpu

FULL = ["decode_t128", "decode_t1024", "skewed_t2048", "prefill_t16384"]
TOKEN_CHECK = {"decode_t128", "skewed_t2048"}


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
        self._q = {}

    def expert(self, which, e):
        """Oracle NVFP4 of one expert matrix ('gu' or 'd'), cached."""
        key = (which, e)
        if key not in self._q:
            a = self.inp["w_gu" if which == "gu" else "w_d"][e].float().cpu().numpy()
            g = O.global_scale(a)
            p, s = O.quantize_nvfp4(a, g)
            self._q[key] = (p, s, g)
        return self._q[key]

    def expert_rows(self, which, e, rows):
        """Oracle NVFP4 of selected rows of one expert matrix (scale from the whole matrix)."""
        a = self.inp["w_gu" if which == "gu" else "w_d"][e].float().cpu().numpy()
        g = O.global_scale(a)
        p, s = O.quantize_nvfp4(a[rows], g)
        return p, s, g

    def x_deq(self, t):
        q, s = O.quantize_nvfp4(self.x32[t:t + 1], self.s_x)
        return O.dequantize_nvfp4(q, s, self.s_x)

    def h_row(self, t, e):
        """float32 SwiGLU output of token t through expert e (oracle)."""
        gp, gs, gg = self.expert("gu", e)
        gu = self.x_deq(t) @ O.dequantize_nvfp4(gp, gs, gg).T
        return O.swiglu(gu, self.w.I).astype(np.float32)


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


def test_gate_up_swiglu_requant_samples(case):
    """Sampled (routed row, 16-feature block) pairs of the fused epilogue."""
    w, L = case.w, case.layer
    rng = np.random.default_rng(1)
    g_f2p = L.perm.flat_to_perm.cpu().numpy()
    cap = L.perm.rows_capacity
    hq = L.hq.cpu().numpy()
    hs = U.from_blocked(L.hs.cpu().numpy(), cap, w.I)
    experts = rng.choice(np.unique(case.idx), size=min(4, len(np.unique(case.idx))), replace=False)
    got_c, ref_c, got_s, ref_s = [], [], [], []
    for e in experts:
        flats = np.nonzero(case.idx.reshape(-1) == e)[0][:3]
        blocks = rng.choice(w.I // 16, size=4, replace=False)
        feats = (blocks[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)
        gp, gs, gg = case.expert_rows("gu", e, np.concatenate([feats, w.I + feats]))
        wdq = O.dequantize_nvfp4(gp, gs, gg)
        for f in flats:
            gu = case.x_deq(f // w.k) @ wdq.T
            h = O.swiglu(gu, feats.size).astype(np.float32)          # [1, 64]: 4 blocks of 16
            rq, rs = O.quantize_nvfp4(h, np.float32(w.h_scale))
            row = g_f2p[f]
            codes = O.unpack_codes(hq[row:row + 1])[0]
            got_c.append(codes[feats]), ref_c.append(O.unpack_codes(rq)[0])
            got_s.append(hs[row, blocks]), ref_s.append(rs[0])
    U.check_requant(np.concatenate(got_c)[None], np.concatenate(got_s)[None], np.concatenate(ref_c)[None],
                    np.concatenate(ref_s)[None], max_flip_frac=0.02, min_scale_eq=0.95)


def test_down_projection_samples(case):
    """Sampled outputs of the down projection for two routed rows."""
    w, L = case.w, case.layer
    g_f2p = L.perm.flat_to_perm.cpu().numpy()
    y = L.y
    cols = np.linspace(0, w.H - 1, 96).astype(int)
    for f in [0, w.R // 2 + 1]:
        t, e = f // w.k, int(case.idx.reshape(-1)[f])
        h = case.h_row(t, e)
        hq, hsc = O.quantize_nvfp4(h, np.float32(w.h_scale))
        dp, ds, dg = case.expert_rows("d", e, cols)
        ref = O.round_to_bf16(O.dequantize_nvfp4(hq, hsc, np.float32(w.h_scale)) @ O.dequantize_nvfp4(dp, ds, dg).T)
        got = y[int(g_f2p[f])].float().cpu().numpy()[cols]
        U.check_close(got[None], ref, what=f"{w.name} down row {f}")


def test_layer_output_one_token(case):
    if case.w.name not in TOKEN_CHECK:
        pytest.skip("token-level check runs on the decode and skewed workloads")
    w = case.w
    t = w.T // 3
    acc = np.zeros(w.H)
    for j in range(w.k):
        e = int(case.idx[t, j])
        h = case.h_row(t, e)
        hq, hsc = O.quantize_nvfp4(h, np.float32(w.h_scale))
        dp, ds, dg = case.expert("d", e)
        y = O.round_to_bf16(O.dequantize_nvfp4(hq, hsc, np.float32(w.h_scale)) @ O.dequantize_nvfp4(dp, ds, dg).T)
        acc += case.wts[t, j] * y[0]
    ref = O.round_to_bf16(acc)[None]
    U.check_close(case.out[t:t + 1], ref, what=f"{w.name} token {t}")
