"""The oracle's pins catch plausible mistakes (CPU only).

Each case below plants one mistake in the oracle -- a swapped table entry, a
wrong tie rule, a dropped sign, a transposed nibble order, a wrong scale
divisor, a bias left out, a reversed order, a swapped gate and up, a double
rounding -- by replacing one function of the oracle module for the duration
of the case, and runs the pins that cover that function.  At least one of
them must fail; otherwise that part of the oracle would be unpinned.  The
mistakes are planted in the oracle only, never in the library.  Each one
breaks a reading the oracle follows: the E2M1 and ue4m3 formats ("SM120 FP4
Kernel Research Campaign", section 1), the block scale and element code
rules (R2, R3), the nibble order (R4), the per-tensor scale (R1), routing
(R5), the permutation order (R6), the layer's SwiGLU, bf16 rounding and
slot-order finalize (R7), batch-aware routing (R8) and the MX exponent (R9).
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from tests import test_oracle_batch_aware as PB
from tests import test_oracle_formats as PF
from tests import test_oracle_layer as PL
from tests import test_oracle_mxfp4 as PM

ORIG = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}


def golden_blocks():
    for blk in PF.load_golden():
        PF.test_golden_blocks(blk)


# ---- planted mistakes: each keeps the signature of the function it replaces ----
def e2m1_decode_swapped(codes):
    v = ORIG["e2m1_decode"](codes)
    return np.where(np.abs(v) == 3.0, np.sign(v) * 4.0, np.where(np.abs(v) == 4.0, np.sign(v) * 3.0, v))


def ue4m3_decode_bias8(b):
    return ORIG["ue4m3_decode"](b) / 2.0


def round_to_ue4m3_ties_up(t):
    t32 = np.asarray(t, dtype=np.float32)
    vals = O.ue4m3_decode(np.arange(0x7F))
    x = np.minimum(t32.astype(np.float64), 448.0)
    hi = np.clip(np.searchsorted(vals, x, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    pick_hi = np.abs(vals[hi] - x) <= np.abs(x - vals[lo])
    return np.where(t32 >= 448.0, 0x7E, np.where(pick_hi, hi, lo)).astype(np.uint8)


def round_to_e2m1_ties_down(q, negative):
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    a = np.minimum(np.abs(np.asarray(q, dtype=np.float32).astype(np.float64)), 6.0)
    code = np.argmin(np.abs(a[..., None] - mags), axis=-1)      # first (lower) code on ties
    return (code | (np.asarray(negative, dtype=np.int64) << 3)).astype(np.uint8)


def round_to_e2m1_unsigned(q, negative):
    return ORIG["round_to_e2m1"](q, np.zeros_like(np.asarray(negative)))


def quantize_nvfp4_high_nibble_first(x, s):
    packed, scales = ORIG["quantize_nvfp4"](x, s)
    return ((packed >> 4) | (packed << 4)).astype(np.uint8), scales


def quantize_nvfp4_divisor4(x, s):
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    blk = x.reshape(rows, cols // 16, 16)
    b = O.round_to_ue4m3((np.max(np.abs(blk), axis=-1) / np.float32(4.0)) / np.float32(s))
    d = O.ue4m3_decode(b).astype(np.float32) * np.float32(s)
    q = blk / np.where(d == 0, np.float32(1.0), d)[..., None]
    codes = np.where((d == 0)[..., None], np.uint8(0), O.round_to_e2m1(q, np.signbit(blk))).reshape(rows, cols)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), b.reshape(rows, cols // 16)


def global_scale_448(x):
    return np.float32(ORIG["global_scale"](x) * np.float32(6.0))


def route_topk_ties_high(logits, bias, k, score_fn, renormalize=True):
    v = O._router_values(logits, bias)
    E = v.shape[1]
    order = (E - 1 - np.argsort(-v[:, ::-1], axis=1, kind="stable"))   # equal values: higher index first
    idx = order[:, :k].astype(np.int32)
    return idx, O._route_weights(v, idx, score_fn, renormalize)


def route_topk_unbiased_weights(logits, bias, k, score_fn, renormalize=True):
    idx, _ = ORIG["route_topk"](logits, bias, k, score_fn, renormalize)
    return idx, O._route_weights(O._router_values(logits, None), idx, score_fn, renormalize)


def route_weights_always_renormalised(v, idx, score_fn, renormalize):
    return ORIG["_route_weights"](v, idx, score_fn, True)


def permute_descending(topk_idx, E):
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    p2f = np.concatenate([np.nonzero(flat == e)[0][::-1] for e in range(E)]).astype(np.int64)
    f2p = np.empty_like(p2f)
    f2p[p2f] = np.arange(flat.size)
    return counts, offsets, p2f, f2p


def grouped_gemm_first_expert_scale(a_packed, a_scales, s_a, offsets, w_packed, w_scales, s_w):
    s = np.asarray(s_w, np.float32)
    return ORIG["grouped_gemm"](a_packed, a_scales, s_a, offsets, w_packed, w_scales, np.full_like(s, s[0]))


def swiglu_swapped(gu, I):
    return O.silu(gu[:, I:2 * I]) * gu[:, :I]


def silu_without_z(z):
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def finalize_reversed_weights(y, flat_to_perm, w, T, k):
    return ORIG["finalize"](y, flat_to_perm, np.asarray(w, np.float64).reshape(T, k)[:, ::-1], T, k)


def finalize_slot_major(y, flat_to_perm, w, T, k):
    # the flat ids read as slot-major (j * T + t) instead of token-major (t * k + j)
    f2p = np.asarray(flat_to_perm).reshape(k, T).T.reshape(-1)
    return ORIG["finalize"](y, f2p, w, T, k)


def round_to_bf16_via_float32(v):
    return torch.from_numpy(np.asarray(v, np.float64).astype(np.float32)).to(torch.bfloat16).double().numpy()


def mx_scale_exponent_minus1(amax):
    return np.clip(ORIG["mx_scale_exponent"](amax) + 1, -127, 127)


def route_batch_aware_plain(logits, bias, k, k_primary, score_fn, renormalize=True):
    return ORIG["route_topk"](logits, bias, k, score_fn, renormalize)


MUTATIONS = {
    "e2m1 table with 3 and 4 swapped": (
        "e2m1_decode", e2m1_decode_swapped, [PF.test_e2m1_table_exhaustive]),
    "ue4m3 exponent bias 8": (
        "ue4m3_decode", ue4m3_decode_bias8, [PF.test_ue4m3_table_against_torch_float8]),
    "ue4m3 rounding ties upward": (
        "round_to_ue4m3", round_to_ue4m3_ties_up, [PF.test_ue4m3_rounding_matches_torch_cast]),
    "e2m1 rounding ties to the lower code": (
        "round_to_e2m1", round_to_e2m1_ties_down, [PF.test_e2m1_rounding_brute_force, golden_blocks]),
    "e2m1 sign bit dropped": (
        "round_to_e2m1", round_to_e2m1_unsigned, [PF.test_e2m1_rounding_brute_force, golden_blocks]),
    "packing high nibble first": (
        "quantize_nvfp4", quantize_nvfp4_high_nibble_first, [golden_blocks]),
    "block scale amax/4 instead of amax/6": (
        "quantize_nvfp4", quantize_nvfp4_divisor4, [golden_blocks, PF.test_quantize_nearest_property]),
    "per-tensor scale amax/448": (
        "global_scale", global_scale_448, [PF.test_global_scale_definition]),
    "router ties to the higher index": (
        "route_topk", route_topk_ties_high, [PL.test_route_ties_go_to_lower_index]),
    "router weights from the unbiased logit": (
        "route_topk", route_topk_unbiased_weights, [PL.test_route_sigmoid_weights_and_invariants]),
    "softmax always renormalised over the top k": (
        "_route_weights", route_weights_always_renormalised, [PL.test_route_matches_torch_topk_and_softmax]),
    "permutation in descending flat id": (
        "permute", permute_descending, [PL.test_permute_brute_force]),
    "every expert takes expert 0's weight scale": (
        "grouped_gemm", grouped_gemm_first_expert_scale, [PL.test_grouped_gemm_brute_force]),
    "gate and up swapped": (
        "swiglu", swiglu_swapped, [PL.test_single_expert_layer_is_dense_swiglu_ffn]),
    "silu without the z factor": (
        "silu", silu_without_z, [PL.test_single_expert_layer_is_dense_swiglu_ffn]),
    "finalize weights in reversed slot order": (
        "finalize", finalize_reversed_weights,
        [PL.test_layer_token_subset_matches_full_layer, PL.test_finalize_hand_worked]),
    "finalize reads flat ids slot-major": (
        "finalize", finalize_slot_major, [PL.test_finalize_hand_worked]),
    "bf16 rounding through float32": (
        "round_to_bf16", round_to_bf16_via_float32, [PF.test_bf16_rounding_of_float64_brute_force]),
    "MX shared exponent floor(log2 amax) - 1": (
        "mx_scale_exponent", mx_scale_exponent_minus1,
        [PM.test_scale_exponent_defining_inequality, PM.test_hand_worked_blocks]),
    "batch-aware routing ignores the active set": (
        "route_batch_aware", route_batch_aware_plain, [PB.test_hand_worked_batch]),
}


def _fails(pin):
    try:
        pin()
    except Exception:                      # an assertion, or the mistake breaking the pin outright
        return True
    return False


@pytest.mark.parametrize("case", sorted(MUTATIONS))
def test_planted_mistake_is_caught(case, monkeypatch):
    name, mutated, pins = MUTATIONS[case]
    # the pins pass on the oracle as it stands ...
    assert not any(_fails(p) for p in pins), f"a pin for {name} fails without a planted mistake"
    # ... and at least one fails with the mistake planted
    monkeypatch.setattr(O, name, mutated)
    assert any(_fails(p) for p in pins), f"planted mistake not caught: {case}"
