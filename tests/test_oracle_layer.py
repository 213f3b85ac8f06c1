"""Pins of the oracle's routing, permutation, grouped GEMM and whole layer
(CPU only).

Routing follows "SM120 FP4 Kernel Research Campaign" (key finding 8: sigmoid
expert scoring); the expert-first permutation and the weighted reduce follow
its section 6 (expert-first layout, token reordering with fused reduction);
the grouped GEMM is the array block-scaled GEMM of "Uncovering SM120 CUTLASS
Collective Implementations" (Context).  Every check below compares against an
independent computation: torch.topk / torch.softmax, pure-Python loops, or
a dense float64 FFN built with library matmuls.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W


def test_route_matches_torch_topk_and_softmax():
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    idx, w = O.route_topk(logits, None, 16, "softmax", renormalize=True)
    ref = torch.softmax(torch.from_numpy(logits).double(), dim=1)
    assert np.allclose(np.take_along_axis(ref.numpy(), idx, 1), w, rtol=1e-13, atol=0)
    idx4, _ = O.route_topk(logits, None, 4, "sigmoid")
    tv, _ = torch.topk(torch.from_numpy(logits), 4, dim=1, sorted=True)
    assert np.array_equal(np.take_along_axis(logits, idx4, 1), tv.numpy())
    # not renormalised softmax over all experts
    _, w_nr = O.route_topk(logits, None, 4, "softmax", renormalize=False)
    assert np.allclose(w_nr, np.take_along_axis(ref.numpy(), idx4, 1), rtol=1e-13)


def test_route_ties_go_to_lower_index():
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.5]], np.float32)
    idx, _ = O.route_topk(logits, None, 4, "sigmoid")
    assert idx.tolist() == [[1, 2, 4, 3]]
    # a bias can create a tie in logit + bias
    idx, _ = O.route_topk(np.array([[1.0, 0.5]], np.float32), np.array([0.0, 0.5], np.float32), 1, "sigmoid")
    assert idx.tolist() == [[0]]


def test_route_sigmoid_weights_and_invariants():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((200, 64)).astype(np.float32)
    bias = W.zipf_bias(64, 1.1)
    idx, w = O.route_topk(logits, bias, 8, "sigmoid")
    assert np.allclose(w.sum(1), 1.0, atol=1e-12, rtol=0)
    assert all(len(set(r)) == 8 for r in idx.tolist())
    v = (logits + bias).astype(np.float64)
    sig = 1 / (1 + np.exp(-np.take_along_axis(v, idx, 1)))
    assert np.allclose(w, sig / sig.sum(1, keepdims=True), rtol=1e-14)
    # slots in descending order of logit + bias
    sel = np.take_along_axis((logits + bias).astype(np.float32), idx, 1)
    assert np.all(np.diff(sel, axis=1) <= 0)
    _, w_raw = O.route_topk(logits, bias, 8, "sigmoid", renormalize=False)
    assert np.allclose(w_raw, sig, rtol=1e-14)


def test_permute_brute_force():
    rng = np.random.default_rng(12)
    for T, E, k in [(1, 4, 1), (37, 8, 3), (128, 64, 8)]:
        idx = W.random_routing(T, E, k, seed=int(rng.integers(1 << 30)))
        counts, offsets, p2f, f2p = O.permute(idx, E)
        flat = idx.reshape(-1).tolist()
        order = [f for e in range(E) for f in range(len(flat)) if flat[f] == e]
        assert p2f.tolist() == order
        assert counts.tolist() == [flat.count(e) for e in range(E)]
        assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) == counts)
        assert np.array_equal(p2f[f2p], np.arange(T * k))
        # every token appears exactly k times
        assert np.all(np.bincount(p2f // k, minlength=T) == k)


def _brute_gemm_row(a_codes, a_sc, s_a, w_codes, w_sc, s_w):
    # independent decode: literal E2M1 table and torch's e4m3 for the scales
    tab = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    f8 = torch.arange(128, dtype=torch.uint8).view(torch.float8_e4m3fn).double().tolist()
    acc = 0.0
    for kk in range(len(a_codes)):
        av = tab[a_codes[kk]] * f8[a_sc[kk // 16]] * float(s_a)
        wv = tab[w_codes[kk]] * f8[w_sc[kk // 16]] * float(s_w)
        acc += av * wv
    return acc


def test_grouped_gemm_brute_force():
    rng = np.random.default_rng(13)
    E, K, N = 3, 64, 5
    counts = [2, 0, 3]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    R = offsets[-1]
    ap, asc, s_a = W.random_nvfp4_operand(R, K, seed=1)
    wp = np.stack([W.random_nvfp4_operand(N, K, seed=10 + e)[0] for e in range(E)])
    wsc = np.stack([W.random_nvfp4_operand(N, K, seed=20 + e)[1] for e in range(E)])
    s_w = np.float32(rng.uniform(0.01, 0.1, size=E))
    out = O.grouped_gemm(ap, asc, s_a, offsets, wp, wsc, s_w)
    ac = O.unpack_codes(ap)
    for e in range(E):
        wc = O.unpack_codes(wp[e])
        for r in range(offsets[e], offsets[e + 1]):
            for n in range(N):
                ref = _brute_gemm_row(ac[r].tolist(), asc[r].tolist(), s_a, wc[n].tolist(), wsc[e][n].tolist(), s_w[e])
                assert abs(out[r, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def _quantize_weights(w_bf16):
    E = w_bf16.shape[0]
    ps, ss, gs = [], [], []
    for e in range(E):
        we = w_bf16[e].float().numpy()
        g = O.global_scale(we)
        p, s = O.quantize_nvfp4(we, g)
        ps.append(p), ss.append(s), gs.append(g)
    return np.stack(ps), np.stack(ss), np.array(gs, np.float32)


def test_single_expert_layer_is_dense_swiglu_ffn():
    """E = 1, k = 1: the layer is one dense SwiGLU FFN on the quantised
    operands, computed here with torch float64 matmuls."""
    w = W.Workload("dense", T=24, E=1, k=1, H=128, I=64, score="softmax")
    inp = W.host_inputs(w, seed=3)
    x = inp["x"].float().numpy()
    gp, gs, gg = _quantize_weights(inp["w_gu"])
    dp, ds, dg = _quantize_weights(inp["w_d"])
    out = O.moe_layer(x, inp["logits"].numpy(), None, gp, gs, gg, dp, ds, dg, 1, "softmax", np.float32(w.h_scale))
    s_x = O.global_scale(x)
    xd = torch.from_numpy(O.dequantize_nvfp4(*O.quantize_nvfp4(x, s_x), s_x))
    Wg = torch.from_numpy(O.dequantize_nvfp4(gp[0], gs[0], gg[0]))
    Wd = torch.from_numpy(O.dequantize_nvfp4(dp[0], ds[0], dg[0]))
    gu = xd @ Wg.T
    h = (torch.nn.functional.silu(gu[:, :64]) * gu[:, 64:]).float().numpy()
    hq, hs = O.quantize_nvfp4(h, np.float32(w.h_scale))
    y = torch.from_numpy(O.dequantize_nvfp4(hq, hs, np.float32(w.h_scale))) @ Wd.T
    ref = y.to(torch.bfloat16).double().numpy()        # softmax over one expert: weight 1
    assert np.array_equal(out, ref)


def test_layer_token_subset_matches_full_layer():
    w = W.TEST_WORKLOADS["zipf_small"]
    inp = W.host_inputs(w, seed=7)
    x = inp["x"].float().numpy()
    gp, gs, gg = _quantize_weights(inp["w_gu"])
    dp, ds, dg = _quantize_weights(inp["w_d"])
    s_h = np.float32(w.h_scale)
    bias = inp["bias"].numpy()
    out, inter = O.moe_layer(x, inp["logits"].numpy(), bias, gp, gs, gg, dp, ds, dg, w.k, w.score, s_h,
                             return_intermediates=True)
    toks = [0, 5, 77, 255]
    sub = O.moe_layer_tokens(toks, x, inp["logits"].numpy(), bias,
                             lambda e: (gp[e], gs[e], gg[e]), lambda e: (dp[e], ds[e], dg[e]),
                             w.k, w.score, s_h, inter["s_x"])
    assert np.array_equal(sub, out[toks])
    # the skewed bias gives a few hot experts and many cold ones
    c = inter["counts"]
    assert c.max() >= 4 * np.median(c)
    # the static SwiGLU scale keeps every block scale below saturation
    assert inter["hs"].max() < 0x7E


def test_finalize_hand_worked():
    """The router-weighted sum back to token order ("SM120 FP4 Kernel Research
    Campaign", Sections 5-6: token reordering with a fused reduction) on a
    case worked by hand: dyadic values, so every product and sum is exact.

    Y rows (expert order): r0 = (1, 2, 3), r1 = (0.5, -1, 4), r2 = (8, 0, -2),
    r3 = (0.25, 0.25, 0.25).  Token 0 sends slot 0 to row 2 and slot 1 to row
    0, weights 0.75 and 0.25; token 1 sends slot 0 to row 3 and slot 1 to
    row 1, weights 0.5 and 0.5.
      out[0] = 0.75 r2 + 0.25 r0 = (6.25, 0.5, -0.75)
      out[1] = 0.5 r3 + 0.5 r1   = (0.375, -0.375, 2.125)"""
    y = np.array([[1, 2, 3], [0.5, -1, 4], [8, 0, -2], [0.25, 0.25, 0.25]])
    flat_to_perm = np.array([2, 0, 3, 1])
    w = np.array([[0.75, 0.25], [0.5, 0.5]])
    out = O.finalize(y, flat_to_perm, w, 2, 2)
    assert np.array_equal(out, [[6.25, 0.5, -0.75], [0.375, -0.375, 2.125]])
    # a one-hot weight picks out exactly the row its slot points at
    for t in range(2):
        for j in range(2):
            oh = np.zeros((2, 2))
            oh[t, j] = 1.0
            got = O.finalize(y, flat_to_perm, oh, 2, 2)
            assert np.array_equal(got[t], y[flat_to_perm[2 * t + j]])
            assert not got[1 - t].any()


def test_layer_invariant_to_token_order_within_expert():
    """Permuting tokens permutes the output rows (the layer is row-wise)."""
    w = W.TEST_WORKLOADS["many_experts"]
    inp = W.host_inputs(w, seed=8)
    x = inp["x"].float().numpy()
    lg = inp["logits"].numpy()
    gp, gs, gg = _quantize_weights(inp["w_gu"])
    dp, ds, dg = _quantize_weights(inp["w_d"])
    s_h = np.float32(w.h_scale)
    out = O.moe_layer(x, lg, None, gp, gs, gg, dp, ds, dg, w.k, w.score, s_h)
    perm = np.random.default_rng(0).permutation(w.T)
    out2 = O.moe_layer(x[perm], lg[perm], None, gp, gs, gg, dp, ds, dg, w.k, w.score, s_h)
    assert np.array_equal(out2, out[perm])


@pytest.mark.parametrize("name", ["tiny"])
def test_tiny_workload_statistics(name):
    w = W.WORKLOADS[name]
    inp = W.host_inputs(w, seed=0)
    x = inp["x"].float().numpy()
    gp, gs, gg = _quantize_weights(inp["w_gu"])
    dp, ds, dg = _quantize_weights(inp["w_d"])
    out, inter = O.moe_layer(x, inp["logits"].numpy(), None, gp, gs, gg, dp, ds, dg, w.k, w.score,
                             np.float32(w.h_scale), return_intermediates=True)
    assert out.shape == (16, 256) and np.all(np.isfinite(out))
    assert inter["counts"].sum() == 32
    assert 0 < inter["hs"].max() < 0x7E
