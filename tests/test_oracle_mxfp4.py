"""Pins of the oracle's MXFP4 codec, GEMM and layer (reading R9; the MXFP4
grouped GEMM named in "SM120 FP4 Kernel Research Campaign", sections 2-4).
Checked against torch's independent float8_e8m0fnu decode, the defining
inequality of the shared exponent, brute-force nearest-code search,
hand-worked blocks, idempotence, a pure-Python GEMM and the dense-FFN case."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e8m0_decode_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = O.e8m0_decode(np.arange(256))
    assert np.array_equal(got[:255], ref[:255]) and np.isnan(got[255]) and np.isnan(ref[255])


def test_scale_exponent_defining_inequality():
    rng = np.random.default_rng(0)
    a = np.concatenate([np.abs(rng.standard_normal(2000)) * 10.0 ** rng.integers(-40, 38, 2000),
                        [2.0 ** -149, 2.0 ** -130, 2.0 ** -126, 4.0, 7.999, 8.0, 6.0, 3.4e38]]).astype(np.float32)
    X = O.mx_scale_exponent(a)
    for ai, xi in zip(a.astype(np.float64), X):
        # unclamped: 2**(X+2) <= amax < 2**(X+3); clamped at -127 below that
        if xi > -127:
            assert 2.0 ** (xi + 2) <= ai < 2.0 ** (xi + 3), (ai, xi)
        else:
            assert ai < 2.0 ** -124
    assert O.mx_scale_exponent(np.float32(0.0)) == -127


def test_hand_worked_blocks():
    # amax 6 -> X = 0 (byte 127): 0.3 -> 0.5, -1.7 -> -1.5, 6 -> 6
    p, s = O.quantize_mxfp4(np.array([[0.3, -1.7, 6.0] + [0.0] * 29], np.float32))
    assert s.tolist() == [[127]] and p[0, :2].tolist() == [0x1 | 0xB << 4, 0x7]
    # amax 7 -> X = 0 as well: 7 saturates to 6 (code 7); 5 is a tie between 4 and 6 -> even code 6 (value 4)
    p, s = O.quantize_mxfp4(np.array([[7.0, 5.0] + [0.0] * 30], np.float32))
    assert s.tolist() == [[127]] and p[0, 0] == 0x7 | 0x6 << 4
    # amax 0.75 -> floor(log2) = -1 -> X = -3 (byte 124), q = 8x: 0.75 -> 6, 0.1 -> 0.8 -> 1, -0.2 -> -1.6 -> -1.5
    p, s = O.quantize_mxfp4(np.array([[0.75, 0.1, -0.2, 0.0] + [0.0] * 28], np.float32))
    assert s.tolist() == [[124]] and p[0, :2].tolist() == [0x7 | 0x2 << 4, 0xB | 0x0 << 4]
    # an all-zero block: byte 0 (2**-127), codes 0
    p, s = O.quantize_mxfp4(np.zeros((1, 32), np.float32))
    assert s.tolist() == [[0]] and not p.any()


def _nearest_code(q):
    """Brute force: scan the 8 magnitudes; ties to the even code; saturate at 6."""
    m = min(abs(q), 6.0)
    best = None
    for c, v in enumerate(E2M1):
        d = abs(m - v)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1] | (8 if np.signbit(q) else 0)


def test_brute_force_codes():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((40, 64)) * 10.0 ** rng.integers(-3, 4, (40, 1))).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()       # bf16 values, as the layer sees them
    x[3, :32] = np.round(x[3, :32] * 4) / 4                            # many exact ties
    p, s = O.quantize_mxfp4(x)
    codes = O.unpack_codes(p)
    for r in range(x.shape[0]):
        for b in range(2):
            blk = x[r, 32 * b:32 * b + 32].astype(np.float64)
            X = int(s[r, b]) - 127
            for i in range(32):
                assert codes[r, 32 * b + i] == _nearest_code(blk[i] / 2.0 ** X), (r, b, i)


def test_idempotent():
    x = np.random.default_rng(2).standard_normal((16, 128)).astype(np.float32)
    p, s = O.quantize_mxfp4(x)
    p2, s2 = O.quantize_mxfp4(O.dequantize_mxfp4(p, s).astype(np.float32))
    assert np.array_equal(p, p2) and np.array_equal(s, s2)


def test_gemm_brute_force():
    rng = np.random.default_rng(3)
    E, K, N = 2, 64, 3
    counts = [2, 1]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    a = rng.integers(0, 256, (3, K // 2), dtype=np.uint8)
    asc = rng.integers(120, 135, (3, K // 32), dtype=np.uint8)
    w = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    wsc = rng.integers(118, 131, (E, N, K // 32), dtype=np.uint8)
    out = O.grouped_gemm_mx(a, asc, offsets, w, wsc)
    tab = E2M1 + [-v for v in E2M1]
    for e in range(E):
        for r in range(offsets[e], offsets[e + 1]):
            for n in range(N):
                acc = 0.0
                for kk in range(K):
                    ca = (int(a[r, kk // 2]) >> (4 * (kk % 2))) & 15
                    cw = (int(w[e, n, kk // 2]) >> (4 * (kk % 2))) & 15
                    acc += tab[ca] * 2.0 ** (int(asc[r, kk // 32]) - 127) * tab[cw] * 2.0 ** (int(wsc[e, n, kk // 32]) - 127)
                assert out[r, n] == acc


def test_single_expert_mx_layer_is_dense_swiglu_ffn():
    w = W.Workload("dense", T=20, E=1, k=1, H=128, I=64, score="softmax")
    inp = W.host_inputs(w, seed=4)
    x = inp["x"].float().numpy()
    gp, gs = O.quantize_mxfp4(inp["w_gu"][0].float().numpy())
    dp, ds = O.quantize_mxfp4(inp["w_d"][0].float().numpy())
    out = O.moe_layer_mx(x, inp["logits"].numpy(), None, gp[None], gs[None], dp[None], ds[None], 1, "softmax")
    xd = torch.from_numpy(O.dequantize_mxfp4(*O.quantize_mxfp4(x)))
    gu = xd @ torch.from_numpy(O.dequantize_mxfp4(gp, gs)).T
    h = (torch.nn.functional.silu(gu[:, :64]) * gu[:, 64:]).float().numpy()
    y = torch.from_numpy(O.dequantize_mxfp4(*O.quantize_mxfp4(h))) @ torch.from_numpy(O.dequantize_mxfp4(dp, ds)).T
    assert np.array_equal(out, y.to(torch.bfloat16).double().numpy())
