"""Plain CPU oracle for the NVFP4 block-scaled Mixture-of-Experts expert layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code, table or helper
with the CUDA library; both sides only share the seeded input generators.

What it computes (source pages, cited by title and section):

* "SM120 FP4 Kernel Research Campaign", section 1 (CUTLASS kernels): the
  block-scaled MMA operand types -- E2M1 data, unsigned E4M3 (ue4m3) scales,
  four scales per 64-element K step, so one scale per 16 consecutive K
  elements, FP32 accumulation.
* same page, section 6 (actionable techniques): expert-first layout and token
  reordering with a fused (router-weighted) reduction.
* same page, key finding 8 and the closing paragraph: sigmoid expert scoring.
* "Uncovering SM120 CUTLASS Collective Implementations", Context section:
  the grouped ("array") block-scaled GEMM over experts and the finalize
  (weighted reduce) epilogue.

Everything the pages leave open is fixed by one stated reading; each function
below names the readings it uses:

  R1  per-tensor scale s = amax(|x|) / 2688 (2688 = 6 * 448), s = 1 when the
      tensor is all zero; one s per expert weight matrix; the activation's s
      is computed from the whole [T, H] input; the SwiGLU output uses a static
      caller-supplied s (the fused epilogue cannot know its amax in advance).
  R2  block scale: t = (amax_block / 6) / s in float32, rounded to the nearest
      ue4m3 value, ties to the even code, saturating at 448.
  R3  element code: q = x / (ue4m3(b) * s) in float32, rounded to the nearest
      E2M1 magnitude, ties to the even code, saturating at 6; the sign bit is
      the sign of x; a zero block scale gives code 0 for the whole block.
  R4  packing: element 2i in the low nibble of byte i.
  R5  routing: select on float32 (logit + bias), descending, lower index on
      ties; weights in float64 after selection; sigmoid is applied to the
      biased logit.
  R6  permutation: an expert's rows are its flat ids t*k+j in ascending order.
  R7  gate/up weight rows [0, I) are the gate, [I, 2I) the up projection;
      h = silu(gate) * up with no clamp; h is rounded to float32 before
      requantisation; the down projection output and the layer output are
      rounded to bfloat16; the finalize sum runs in slot order.
  R8  batch-aware routing (the pages name the technique -- at decode, a token
      trades its least-weighted experts for experts the batch already uses --
      but give no algorithm): every token keeps its top
      k_primary experts; the union of those over the batch is the active
      set S; each token's k experts are its best within S (then, only if S
      has fewer than k experts, its best outside S); see route_batch_aware.
  R9  MXFP4 (the pages name an MXFP4 grouped GEMM and nothing more; the
      format is the OCP microscaling one): E2M1 values, one E8M0 scale
      2**X per 32 elements along K, X = floor(log2(block amax)) - 2 clamped
      to [-127, 127] (-127 for an all-zero block), codes by reading R3 on
      x / 2**X, no per-tensor scale; the layer's SwiGLU output is
      requantised the same way.

Precision: values are decoded exactly to float64, GEMMs accumulate in float64
(numpy matmul on exactly dequantised operands), the few steps that must
mirror a float32 decision (scale and code rounding) are done in float32
round-to-nearest exactly as the reading defines them.

Pinned by tests/test_oracle_*.py against: hand-worked blocks
(tests/golden/nvfp4_blocks.txt), the exhaustive E2M1 and E4M3 tables,
torch's independent float8_e4m3fn cast, brute-force nearest-value search,
a pure-Python triple-loop GEMM on tiny shapes, the dense-FFN special case
(E=1, k=1), torch.softmax / torch.topk, and routing invariants.
Parity unpinned: the absolute end-to-end values at full size (the pages print
no worked example of a layer output).
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# Formats ("SM120 FP4 Kernel Research Campaign", section 1: operand types
# e2m1 and ue4m3 of the block-scaled MMA).
# ----------------------------------------------------------------------------


def e2m1_decode(codes):
    """Decode 4-bit E2M1 codes (1 sign, 2 exponent, 1 mantissa bit, bias 1).

    exponent 0 is subnormal: value = mantissa * 0.5; otherwise
    (1 + mantissa/2) * 2**(exponent - 1).  Returns float64.
    """
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0))
    return sign * mag


def ue4m3_decode(b):
    """Decode unsigned E4M3 scale bytes (4 exponent bits, bias 7, 3 mantissa).

    exponent 0 is subnormal: m/8 * 2**-6.  0x7F is NaN.  Bytes with the top
    bit set are not valid unsigned scales and decode to NaN.  float64.
    """
    b = np.asarray(b).astype(np.int64)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    bad = (b == 0x7F) | (b >= 0x80)
    return np.where(bad, np.nan, val)


_UE4M3_VALUES = ue4m3_decode(np.arange(0x7F))          # codes 0..0x7E, ascending
_E2M1_MAGS = e2m1_decode(np.arange(8))                  # 0, .5, 1, 1.5, 2, 3, 4, 6

UE4M3_MAX = 448.0
E2M1_MAX = 6.0
GLOBAL_SCALE_DIVISOR = np.float32(E2M1_MAX * UE4M3_MAX)  # 2688


def _nearest_even(values_sorted, x):
    """Index of the nearest entry of an ascending value table; ties -> even index.

    Adjacent codes of both formats differ by one in their integer encoding, so
    "even index" is "even code" (the round-to-nearest-even rule).  x >= 0.
    Distances are taken in float64, where they are exact for these tables.
    """
    x = np.asarray(x, dtype=np.float64)
    hi = np.searchsorted(values_sorted, x, side="left")
    hi = np.clip(hi, 0, len(values_sorted) - 1)
    lo = np.clip(hi - 1, 0, len(values_sorted) - 1)
    d_lo = np.abs(x - values_sorted[lo])
    d_hi = np.abs(values_sorted[hi] - x)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo)


def round_to_ue4m3(t):
    """Round non-negative float32 values to ue4m3 bytes (reading R2).

    Round to nearest, ties to even code; values at or above 448 saturate to
    0x7E (448); tiny values round to 0 (2**-10, half the smallest subnormal,
    is a tie and goes to the even code 0).
    """
    t = np.asarray(t, dtype=np.float32).astype(np.float64)
    if np.any(t < 0) or np.any(np.isnan(t)):
        raise ValueError("ue4m3 rounding takes non-negative finite values")
    idx = _nearest_even(_UE4M3_VALUES, np.minimum(t, UE4M3_MAX))
    return np.where(t >= UE4M3_MAX, 0x7E, idx).astype(np.uint8)


def round_to_e2m1(q, negative):
    """E2M1 code of float32 quotients q (reading R3).

    Magnitude: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code,
    saturating at 6.  The sign bit is ``negative`` (the sign of the original
    element, so a small negative element gives code 0x8, "-0").
    """
    mag = np.abs(np.asarray(q, dtype=np.float32).astype(np.float64))
    code = _nearest_even(_E2M1_MAGS, np.minimum(mag, E2M1_MAX))
    return (code | (np.asarray(negative, dtype=np.int64) << 3)).astype(np.uint8)


# ----------------------------------------------------------------------------
# Quantisation: FP4 E2M1 values, one unsigned E4M3 scale per 16-element block
# along K and a per-tensor FP32 scale ("SM120 FP4 Kernel Research Campaign",
# section 1, operand types of the block-scaled MMA).
# ----------------------------------------------------------------------------


def global_scale(x):
    """Per-tensor FP32 scale s = amax(|x|) / 2688 (reading R1); 1 if amax is 0.

    2688 = 6 * 448, so the largest block scale a tensor needs is at most 448.
    """
    a = np.float32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) if np.size(x) else np.float32(0)
    if a == 0:
        return np.float32(1.0)
    return np.float32(a / GLOBAL_SCALE_DIVISOR)


def quantize_nvfp4(x, s):
    """Quantise rows of x (float32 values, [rows, cols], cols % 16 == 0).

    Per 16-element block along the row (readings R2, R3):
      a = max |x| over the block (exact), t = (a / 6) / s in float32,
      b = round_to_ue4m3(t), d = value(b) * s in float32,
      code = round_to_e2m1(x / d) with the sign of x; d == 0 gives code 0.
    Packing (reading R4): element 2i in the low nibble of byte i.
    Returns (packed uint8 [rows, cols/2], scales uint8 [rows, cols/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    if cols % 16:
        raise ValueError("cols must be a multiple of 16")
    s = np.float32(s)
    blk = x.reshape(rows, cols // 16, 16)
    a = np.max(np.abs(blk), axis=-1)
    t = (a / np.float32(6.0)) / s
    b = round_to_ue4m3(t)
    d = ue4m3_decode(b).astype(np.float32) * s
    safe_d = np.where(d == 0, np.float32(1.0), d).astype(np.float32)
    q = blk / safe_d[..., None]
    codes = round_to_e2m1(q, np.signbit(blk))
    codes = np.where((d == 0)[..., None], np.uint8(0), codes).reshape(rows, cols)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, b.reshape(rows, cols // 16)


def unpack_codes(packed):
    """Split packed bytes into codes: low nibble first (reading R4)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequantize_nvfp4(packed, scales, s):
    """Exact float64 value of NVFP4 data: e2m1(code) * ue4m3(scale) * s."""
    codes = unpack_codes(packed)
    rows, cols = codes.shape
    v = e2m1_decode(codes).reshape(rows, cols // 16, 16)
    v = v * ue4m3_decode(scales)[..., None] * np.float64(np.float32(s))
    return v.reshape(rows, cols)


# ----------------------------------------------------------------------------
# MXFP4: E2M1 values with one power-of-two (E8M0) scale per 32-element block
# along K and no per-tensor scale -- the second block-scaled FP4 format for
# grouped GEMMs the pages name ("SM120 FP4 Kernel Research Campaign",
# section 2-4: FlashInfer's MXFP4 grouped GEMM).  Reading R9.
# ----------------------------------------------------------------------------
MX_BLOCK = 32
E2M1_EMAX = 2          # 6 = 1.5 * 2**2: exponent of E2M1's largest normal


def e8m0_decode(b):
    """Value of E8M0 scale bytes: 2**(b - 127); 0xFF is NaN."""
    b = np.asarray(b, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def mx_scale_exponent(amax):
    """Shared exponent of an MX block from its float32 amax (reading R9):
    X = floor(log2(amax)) - 2, clamped to the E8M0 range [-127, 127];
    an all-zero block takes X = -127."""
    a = np.asarray(amax, dtype=np.float32).astype(np.float64)
    _, e = np.frexp(np.where(a > 0, a, 1.0))        # a = m * 2**e, m in [0.5, 1): floor(log2 a) = e - 1
    x = np.where(a > 0, e - 1 - E2M1_EMAX, -127)
    return np.clip(x, -127, 127).astype(np.int64)


def quantize_mxfp4(x):
    """Quantise rows of x (float32 values, [rows, cols], cols % 32 == 0) to MXFP4.

    Per 32-element block along the row (reading R9): X = mx_scale_exponent(
    max |x|), scale byte X + 127, q = x / 2**X (exact in float32), code =
    round_to_e2m1(q) with the sign of x (reading R3: nearest, ties to the
    even code, saturating at 6).  Packing as reading R4.
    Returns (packed uint8 [rows, cols/2], scales uint8 [rows, cols/32]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    if cols % MX_BLOCK:
        raise ValueError("cols must be a multiple of 32")
    blk = x.reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    X = mx_scale_exponent(np.max(np.abs(blk), axis=-1))
    q = (blk.astype(np.float64) * np.ldexp(1.0, -X)[..., None]).astype(np.float32)   # exact power-of-two scaling
    codes = round_to_e2m1(q, np.signbit(blk)).reshape(rows, cols)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, (X + 127).astype(np.uint8).reshape(rows, cols // MX_BLOCK)


def dequantize_mxfp4(packed, scales):
    """float64 values of MXFP4 data: e2m1(code) * 2**(scale - 127)."""
    codes = unpack_codes(packed)
    vals = e2m1_decode(codes)
    sc = np.repeat(e8m0_decode(scales), MX_BLOCK, axis=-1)
    return vals * sc


# ----------------------------------------------------------------------------
# Routing (key finding 8 / conclusion of the research page: sigmoid scoring;
# softmax for the tiny configuration).  Reading R5.
# ----------------------------------------------------------------------------


def route_topk(logits, bias, k, score_fn, renormalize=True):
    """Top-k expert selection and routing weights.

    Selection compares v = logits + bias in float32, descending, lower expert
    index first on ties; slots are in that order.  Weights in float64:
      softmax: exp(v_j - max v) / sum(...) over the selected k (renormalised)
               or over all E (not renormalised);
      sigmoid: sigma(v_j), divided by the sum over the selected k when
               renormalised.
    Returns (idx int32 [T,k], w float64 [T,k]).
    """
    v = _router_values(logits, bias)
    T, E = v.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    order = np.argsort(-v, axis=1, kind="stable")   # stable: equal values keep ascending index
    idx = order[:, :k].astype(np.int32)
    return idx, _route_weights(v, idx, score_fn, renormalize)


def _router_values(logits, bias):
    """v = logits + bias in float32 (reading R5)."""
    v = np.asarray(logits, dtype=np.float32)
    if bias is not None:
        v = (v + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    return v


def _route_weights(v, idx, score_fn, renormalize):
    """Routing weights of the selected experts idx [T, k] (see route_topk)."""
    vs = np.take_along_axis(v, idx.astype(np.int64), axis=1).astype(np.float64)
    if score_fn == "softmax":
        vmax = v.max(axis=1, keepdims=True).astype(np.float64)
        num = np.exp(vs - vmax)
        den = num.sum(axis=1, keepdims=True) if renormalize else \
            np.exp(v.astype(np.float64) - vmax).sum(axis=1, keepdims=True)
        w = num / den
    elif score_fn == "sigmoid":
        sig = 1.0 / (1.0 + np.exp(-vs))
        w = sig / sig.sum(axis=1, keepdims=True) if renormalize else sig
    else:
        raise ValueError(score_fn)
    return w


def route_batch_aware(logits, bias, k, k_primary, score_fn, renormalize=True):
    """Batch-aware ("opportunistic") expert routing, reading R8.

    "SM120 FP4 Kernel Research Campaign" (Introduction; key finding 6; section
    6, batch-aware routing) names the technique -- during decode a token
    trades the experts it weights least for experts other tokens of the
    batch use already, so fewer experts' weights are streamed -- but gives
    no algorithm.  Reading R8, step by step:
      1. each token's primary experts are its top-k_primary by
         v = logit + bias (order and ties as in route_topk);
      2. the batch's active set S is the union of every token's primary
         experts;
      3. each token takes k experts ranked by (member of S first, then v
         descending, then lower index): its top-k within S, followed -- only
         when S holds fewer than k experts -- by its best experts outside S;
         slots keep that rank order;
      4. weights as route_topk over the chosen experts.
    k_primary == k gives route_topk.  Returns (idx int32 [T,k], w float64 [T,k]).
    """
    v = _router_values(logits, bias)
    T, E = v.shape
    if not 1 <= k_primary <= k <= E:
        raise ValueError("need 1 <= k_primary <= k <= E")
    order = np.argsort(-v, axis=1, kind="stable")          # per token: v descending, lower index first
    in_s = np.zeros(E, dtype=bool)
    in_s[order[:, :k_primary].reshape(-1)] = True           # steps 1-2
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):                                       # step 3
        members = [int(e) for e in order[t] if in_s[e]]
        others = [int(e) for e in order[t] if not in_s[e]]
        idx[t] = (members + others)[:k]
    return idx, _route_weights(v, idx, score_fn, renormalize)   # step 4


# ----------------------------------------------------------------------------
# Permutation (section 6: expert-first layout, token reordering).  Reading R6.
# ----------------------------------------------------------------------------


def permute(topk_idx, E):
    """Expert-first order of the routed rows.

    Flat id f = t*k + j.  Rows of expert e are the flat ids routed to e in
    ascending f; offsets is the exclusive scan of the per-expert counts.
    Returns counts [E], offsets [E+1], perm_to_flat [R], flat_to_perm [R].
    """
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    perm_to_flat = np.argsort(flat, kind="stable").astype(np.int64)
    flat_to_perm = np.empty_like(perm_to_flat)
    flat_to_perm[perm_to_flat] = np.arange(flat.size)
    return counts, offsets, perm_to_flat, flat_to_perm


# ----------------------------------------------------------------------------
# Grouped GEMM, SwiGLU, finalize ("Uncovering SM120 CUTLASS Collective
# Implementations", Context: grouped block-scaled GEMM and finalize epilogue).
# ----------------------------------------------------------------------------


def grouped_gemm(a_packed, a_scales, s_a, offsets, w_packed, w_scales, s_w):
    """out[r] = A_r . W[e]^T for r in expert e's row range, float64.

    A [R, K/2] packed with scales [R, K/16] and per-tensor scale s_a;
    W [E, N, K/2] with scales [E, N, K/16] and per-expert scales s_w [E].
    Both operands are dequantised exactly; the product is a float64 matmul.
    """
    E, N = w_packed.shape[0], w_packed.shape[1]
    R = a_packed.shape[0]
    out = np.zeros((R, N), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        A = dequantize_nvfp4(a_packed[r0:r1], a_scales[r0:r1], s_a)
        W = dequantize_nvfp4(w_packed[e], w_scales[e], s_w[e])
        out[r0:r1] = A @ W.T
    return out


def grouped_gemm_mx(a_packed, a_scales, offsets, w_packed, w_scales):
    """grouped_gemm for MXFP4 operands (no per-tensor scales):
    C[r, n] = sum_K A[r, :] * W[e, n, :] for rows r of expert e, float64."""
    offsets = np.asarray(offsets, dtype=np.int64)
    E = w_packed.shape[0]
    out = np.zeros((a_packed.shape[0], w_packed.shape[1]), dtype=np.float64)
    a = dequantize_mxfp4(a_packed, a_scales)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            out[r0:r1] = a[r0:r1] @ dequantize_mxfp4(w_packed[e], w_scales[e]).T
    return out


def silu(z):
    """z / (1 + exp(-z)), float64 (reading R7: SwiGLU, no clamp, no alpha)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(gu, I):
    """h = silu(gate) * up with gate = columns [0, I), up = columns [I, 2I)."""
    return silu(gu[:, :I]) * gu[:, I:2 * I]


def round_to_bf16(v):
    """Round float64 values to the nearest bfloat16 (ties to even), as float64.

    One rounding straight from float64 (8 significant bits; overflow to inf;
    below 2**-126 the spacing stays 2**-133, the bf16 subnormal step).
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                       # v = m * 2**e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # subnormal region keeps a fixed step
    r = np.rint(np.ldexp(v, 8 - e))          # rint: round half to even
    out = np.ldexp(r, e - 8)
    out = np.where(np.abs(out) > 3.3895313892515355e38, np.copysign(np.inf, v), out)
    return np.where(v == 0, v, out)


def finalize(y, flat_to_perm, w, T, k):
    """out[t] = sum_j w[t,j] * y[flat_to_perm[t*k+j]] in slot order, float64."""
    y = np.asarray(y, dtype=np.float64)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    w = np.asarray(w, dtype=np.float64).reshape(T, k)
    for j in range(k):
        out += w[:, j:j + 1] * y[np.asarray(flat_to_perm).reshape(T, k)[:, j]]
    return out


def moe_layer(x, logits, bias, w_gu_packed, w_gu_scales, s_gu, w_d_packed, w_d_scales, s_d,
              k, score_fn, s_h, renormalize=True, s_x=None, return_intermediates=False, k_primary=None):
    """The whole expert layer, steps in the pages' order (route, quantise,
    permute, gate/up GEMM + SwiGLU + requantise, down GEMM, finalize).

    x: float32 [T, H] (bf16 values); weights already NVFP4 with per-expert
    scales.  s_h is the static per-tensor scale of the SwiGLU output
    (reading R1); s_x defaults to the dynamic amax/2688 of x.  k_primary
    (None = k) selects batch-aware routing (route_batch_aware).
    Returns bf16-rounded float64 out [T, H] (and intermediates on request).
    """
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    E = w_gu_packed.shape[0]
    I = w_gu_packed.shape[1] // 2
    if k_primary is None or k_primary == k:
        idx, w = route_topk(logits, bias, k, score_fn, renormalize)
    else:
        idx, w = route_batch_aware(logits, bias, k, k_primary, score_fn, renormalize)
    if s_x is None:
        s_x = global_scale(x)
    xq, xs = quantize_nvfp4(x, s_x)
    counts, offsets, p2f, f2p = permute(idx, E)
    tok = p2f // k
    a_packed, a_scales = xq[tok], xs[tok]
    gu = grouped_gemm(a_packed, a_scales, s_x, offsets, w_gu_packed, w_gu_scales, s_gu)
    h = swiglu(gu, I).astype(np.float32)           # the GEMM result is a float32 accumulator
    hq, hs = quantize_nvfp4(h, s_h)
    y = round_to_bf16(grouped_gemm(hq, hs, s_h, offsets, w_d_packed, w_d_scales, s_d))
    out = round_to_bf16(finalize(y, f2p, w, T, k))
    if not return_intermediates:
        return out
    return out, dict(idx=idx, w=w, s_x=np.float32(s_x), xq=xq, xs=xs, counts=counts, offsets=offsets,
                     perm_to_flat=p2f, flat_to_perm=f2p, gu=gu, h=h, hq=hq, hs=hs, y=y)


def moe_layer_mx(x, logits, bias, w_gu_packed, w_gu_scales, w_d_packed, w_d_scales, k, score_fn,
                 renormalize=True, k_primary=None, return_intermediates=False):
    """moe_layer with MXFP4 operands (reading R9): x and the SwiGLU output
    quantised by quantize_mxfp4 (no per-tensor scales), weights MXFP4."""
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    E = w_gu_packed.shape[0]
    I = w_gu_packed.shape[1] // 2
    if k_primary is None or k_primary == k:
        idx, w = route_topk(logits, bias, k, score_fn, renormalize)
    else:
        idx, w = route_batch_aware(logits, bias, k, k_primary, score_fn, renormalize)
    xq, xs = quantize_mxfp4(x)
    counts, offsets, p2f, f2p = permute(idx, E)
    tok = p2f // k
    gu = grouped_gemm_mx(xq[tok], xs[tok], offsets, w_gu_packed, w_gu_scales)
    h = swiglu(gu, I).astype(np.float32)
    hq, hs = quantize_mxfp4(h)
    y = round_to_bf16(grouped_gemm_mx(hq, hs, offsets, w_d_packed, w_d_scales))
    out = round_to_bf16(finalize(y, f2p, w, T, k))
    if not return_intermediates:
        return out
    return out, dict(idx=idx, w=w, xq=xq, xs=xs, counts=counts, offsets=offsets, perm_to_flat=p2f,
                     flat_to_perm=f2p, gu=gu, h=h, hq=hq, hs=hs, y=y)


def moe_layer_tokens(token_ids, x, logits, bias, w_gu, w_d, k, score_fn, s_h, s_x, renormalize=True,
                     routing=None):
    """Layer output for a subset of tokens, computed one token at a time.

    Each output row depends only on its own token once s_x and the routing
    are fixed, so this equals the matching rows of moe_layer().  w_gu / w_d
    are callables e -> (packed, scales, s) so that only the experts those
    tokens use are ever quantised.  routing = (idx, w) of the whole batch
    (needed for batch-aware routing); None routes each token by route_topk.
    Returns bf16-rounded float64 [len(token_ids), H].
    """
    x = np.asarray(x, dtype=np.float32)
    I = None
    outs = []
    for t in token_ids:
        if routing is None:
            idx, w = route_topk(logits[t:t + 1], bias, k, score_fn, renormalize)
        else:
            idx, w = routing[0][t:t + 1], routing[1][t:t + 1]
        xq, xs = quantize_nvfp4(x[t:t + 1], s_x)
        xd = dequantize_nvfp4(xq, xs, s_x)
        acc = np.zeros(x.shape[1], dtype=np.float64)
        for j in range(k):
            e = int(idx[0, j])
            gp, gsc, gs = w_gu(e)
            I = gp.shape[0] // 2
            gu = xd @ dequantize_nvfp4(gp, gsc, gs).T
            h = swiglu(gu, I).astype(np.float32)
            hq, hs = quantize_nvfp4(h, s_h)
            dp, dsc, ds = w_d(e)
            y = round_to_bf16(dequantize_nvfp4(hq, hs, s_h) @ dequantize_nvfp4(dp, dsc, ds).T)
            acc += w[0, j] * y[0]
        outs.append(round_to_bf16(acc))
    return np.stack(outs)
