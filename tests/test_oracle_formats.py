"""Pins of the oracle's number formats and quantiser (CPU only).

Each test checks the oracle against something other than itself: the format
definitions written out as literal tables, torch's own float8_e4m3fn cast,
hand-worked blocks (tests/golden/nvfp4_blocks.txt) and brute-force nearest
searches.  The format is the one the block-scaled MMA of "SM120 FP4 Kernel
Research Campaign", section 1, takes: e2m1 data, ue4m3 scales, 16-element
blocks.
"""
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")


def load_golden():
    blocks, cur = [], {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line.startswith("#"):
                continue
            if not line:
                if cur:
                    blocks.append(cur)
                cur = {}
                continue
            key, _, val = line.partition(":")
            if key == "why":
                continue
            cur[key.strip()] = val.strip()
    if cur:
        blocks.append(cur)
    return blocks


def test_e2m1_table_exhaustive():
    # The 16 E2M1 values, written out from the format (sign, 2-bit exponent,
    # 1-bit mantissa, bias 1): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
             -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    got = O.e2m1_decode(np.arange(16))
    assert np.array_equal(got, np.array(table))
    assert np.array_equal(np.signbit(got), np.signbit(np.array(table)))


def test_ue4m3_table_against_torch_float8():
    # torch's float8_e4m3fn decoder is an independent implementation; the
    # unsigned scale format is its non-negative half.
    ref = torch.arange(128, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = O.ue4m3_decode(np.arange(128))
    assert np.isnan(got[0x7F]) and np.isnan(ref[0x7F])
    assert np.array_equal(got[:0x7F], ref[:0x7F])
    assert got[0x7E] == 448.0 and got[0x38] == 1.0 and got[0x01] == 2.0 ** -9
    assert np.all(np.isnan(O.ue4m3_decode(np.arange(128, 256))))


def test_ue4m3_rounding_matches_torch_cast():
    rng = np.random.default_rng(1)
    # log-uniform over the whole ue4m3 range plus exact midpoints (ties)
    t = np.exp2(rng.uniform(-14, np.log2(463.9), size=200000)).astype(np.float32)
    vals = O.ue4m3_decode(np.arange(0x7F))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    t = np.concatenate([t, mids, vals.astype(np.float32), np.float32([0.0, 2.0 ** -10, 460.0])])
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.round_to_ue4m3(t)
    assert np.array_equal(got, ref)


def test_ue4m3_saturation():
    # torch maps values past the last midpoint (464) to NaN; the scale
    # rounding saturates at 448 instead (reading R2).
    t = np.float32([448.0, 464.0, 465.0, 1e6, np.inf])
    assert np.all(O.round_to_ue4m3(t) == 0x7E)


def test_e2m1_rounding_brute_force():
    rng = np.random.default_rng(2)
    q = np.concatenate([rng.uniform(-7, 7, 100000),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 6.5, 100.0])]).astype(np.float32)
    q = np.concatenate([q, -q])
    got = O.round_to_e2m1(q, np.signbit(q))
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for qi, gi in zip(q[::37].tolist() + q[-20:].tolist(), np.concatenate([got[::37], got[-20:]]).tolist()):
        a = min(abs(qi), 6.0)
        dist = [abs(a - m) for m in mags]
        best = min(dist)
        cands = [c for c in range(8) if dist[c] == best]
        code = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        code |= 8 if np.signbit(np.float32(qi)) else 0
        assert gi == code, (qi, gi, code)


@pytest.mark.parametrize("blk", load_golden(), ids=lambda b: b["x"][:24])
def test_golden_blocks(blk):
    s = np.float32(float(blk["s"]))
    x = np.array([float(v) for v in blk["x"].split()], dtype=np.float32)
    # inputs are bf16 values
    assert np.array_equal(torch.from_numpy(x).to(torch.bfloat16).float().numpy(), x)
    packed, scales = O.quantize_nvfp4(x[None, :], s)
    assert scales[0, 0] == int(blk["scale"], 16)
    codes = O.unpack_codes(packed)[0]
    assert [int(c) for c in codes] == [int(c, 16) for c in blk["codes"].split()]
    assert [int(b) for b in packed[0]] == [int(b, 16) for b in blk["packed"].split()]


def test_global_scale_definition():
    x = np.zeros((2, 32), np.float32)
    x[1, 3] = -1344.0
    assert O.global_scale(x) == np.float32(0.5)
    assert O.global_scale(np.zeros((1, 16), np.float32)) == np.float32(1.0)
    # the largest block scale any tensor gets is 448
    rng = np.random.default_rng(3)
    y = (rng.standard_normal((64, 256)) * 3).astype(np.float32)
    y = torch.from_numpy(y).to(torch.bfloat16).float().numpy()
    _, sc = O.quantize_nvfp4(y, O.global_scale(y))
    assert sc.max() <= 0x7E and O.ue4m3_decode(sc.max()) <= 448.0


def test_quantize_nearest_property():
    """Every code is the nearest representable value to x/d (brute force)."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((40, 64)) * np.exp2(rng.integers(-8, 8, size=(40, 1)))).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    s = O.global_scale(x)
    packed, scales = O.quantize_nvfp4(x, s)
    codes = O.unpack_codes(packed).reshape(40, 4, 16)
    d = (O.ue4m3_decode(scales).astype(np.float32) * s).astype(np.float32)
    q = (x.reshape(40, 4, 16) / d[..., None]).astype(np.float64)
    allv = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])[codes & 7]
    err = np.abs(np.minimum(np.abs(q), 6.0) - mag)
    best = np.min(np.abs(np.minimum(np.abs(q), 6.0)[..., None] - allv), axis=-1)
    assert np.all(err == best)
    assert np.all(((codes >> 3) & 1) == np.signbit(x.reshape(40, 4, 16)))
    # the block scale is the nearest ue4m3 to (amax/6)/s (brute force over all 127 values)
    t = ((np.abs(x.reshape(40, 4, 16)).max(-1) / np.float32(6)) / s).astype(np.float64)
    vals = O.ue4m3_decode(np.arange(0x7F))
    dist = np.abs(t[..., None] - vals)
    assert np.all(dist[np.arange(40)[:, None], np.arange(4)[None, :], scales] == dist.min(-1))


def test_requantise_is_idempotent():
    """Quantising dequantised data reproduces the codes (power-of-two s keeps
    every intermediate exact)."""
    rng = np.random.default_rng(5)
    for s in (np.float32(1.0), np.float32(2.0 ** -4), np.float32(8.0)):
        packed = rng.integers(0, 256, size=(32, 64), dtype=np.uint8)
        codes = O.unpack_codes(packed)
        codes[:, ::16] = 0x7                       # each block has a +6, so amax = 6 * scale
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        scales = rng.integers(0x10, 0x60, size=(32, 8), dtype=np.uint8)
        x = O.dequantize_nvfp4(packed, scales, s).astype(np.float32)
        p2, s2 = O.quantize_nvfp4(x, s)
        assert np.array_equal(s2, scales)
        c1, c2 = O.unpack_codes(packed), O.unpack_codes(p2)
        # -0 and +0 decode alike; the requantised sign follows the value
        same = (c1 == c2) | (((c1 & 7) == 0) & ((c2 & 7) == 0))
        assert same.all()


def test_bf16_rounding_matches_torch_for_float32_inputs():
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(100000) * np.exp2(rng.integers(-30, 30, 100000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.round_to_bf16(v.astype(np.float64)), ref)
    # a float64 value just above a bf16 midpoint rounds up although its
    # float32 rounding would land exactly on the midpoint
    mid = 1.0 + 2.0 ** -8
    assert O.round_to_bf16(np.float64(mid + 2.0 ** -40)) == 1.0 + 2.0 ** -7
    assert O.round_to_bf16(np.float64(mid)) == 1.0


def _bf16_value(bits):
    """Exact value of a bf16 bit pattern (the top half of a float32)."""
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


def _nearest_bf16_brute(v):
    """Nearest bfloat16 to the float64 v by exact rational comparison of the
    bf16 patterns around it; ties to the even pattern; beyond the largest
    finite bf16 by half a step or more, infinity."""
    from fractions import Fraction
    if v == 0:
        return v
    a = abs(v)
    top = 0x7F7F                                     # largest finite bf16
    if Fraction(a) >= Fraction(_bf16_value(top)) + Fraction(2) ** (127 - 8):
        return float(np.copysign(np.inf, v))
    f32 = np.float32(min(a, float(np.finfo(np.float32).max)))
    b = int(np.array([f32], np.float32).view(np.uint32)[0]) >> 16
    best = None
    for c in range(max(0, b - 2), min(top, b + 2) + 1):
        d = abs(Fraction(_bf16_value(c)) - Fraction(a))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return float(np.copysign(_bf16_value(best[1]), v))


def test_bf16_rounding_of_float64_brute_force():
    """round_to_bf16 against the exact nearest bf16: normal values, the bf16
    subnormal range, exact midpoints, points just off them, and the overflow
    boundary.  Reading R7 rounds the down projection's float64 sum and the
    finalize sum straight to bfloat16 (round to nearest, ties to even), so
    the inputs here are float64, not float32."""
    rng = np.random.default_rng(16)
    vals = list(rng.standard_normal(1500) * np.exp2(rng.integers(-140, 128, 1500)))
    for b in rng.integers(1, 0x7F7F, 300):
        lo, hi = _bf16_value(int(b)), _bf16_value(int(b) + 1)
        mid = (lo + hi) / 2                            # exact in float64
        vals += [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), -mid]
    top = _bf16_value(0x7F7F)
    vals += [top, top + 2.0 ** (127 - 8), np.nextafter(top + 2.0 ** (127 - 8), 0), 2.0 ** -133, 2.0 ** -134,
             3 * 2.0 ** -135, 2.0 ** -200, -2.0 ** -126]
    vals = np.array(vals, np.float64)
    got = O.round_to_bf16(vals)
    ref = np.array([_nearest_bf16_brute(float(v)) for v in vals])
    assert np.array_equal(got, ref, equal_nan=False), vals[got != ref][:5]
