"""Test-side helpers: the blocked scale layout as a pure index map, NVFP4 code
comparisons and the floating-point tolerances.

The blocked layout (declared in include/nvfp4moe.h): rows in blocks of 128,
K in blocks of 64 elements; block (rb, kb) is 512 bytes at
(rb * cols/64 + kb) * 512; row r of a block keeps its 4 scales at
(r % 32) * 16 + (r / 32) * 4.
"""
import numpy as np

from oracle import nvfp4_moe_oracle as O

# Floating-point parity bar for GEMM and layer outputs (bf16): relative
# Frobenius error and per-element error relative to max(|ref|, rms(ref)).
FROB_TOL = 5e-3
ELEM_TOL = 2e-2


def ceil_to(a, b):
    return -(-a // b) * b


def blocked_index(rows_pad, cols, block=16):
    """Byte offset of scale (row, c) in the blocked layout; block = elements
    per scale (16 for NVFP4, 32 for MXFP4), four scales per 512-byte group row."""
    r = np.arange(rows_pad, dtype=np.int64)[:, None]
    c = np.arange(cols // block, dtype=np.int64)[None, :]
    return ((r // 128) * (cols // (4 * block)) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)


def to_blocked(scales, cols, block=16):
    rows = scales.shape[0]
    rp = max(ceil_to(rows, 128), 128)
    out = np.zeros(rp * (cols // block), dtype=np.uint8)
    out[blocked_index(rp, cols, block)[:rows].ravel()] = np.asarray(scales, dtype=np.uint8).ravel()
    return out


def from_blocked(buf, rows, cols, block=16):
    rp = max(ceil_to(rows, 128), 128)
    return np.asarray(buf)[blocked_index(rp, cols, block)[:rows]]


def untile_weights(tiled, E, N, K):
    """Row-major [E, N, K/2] packed weights from the tiled layout (as the
    library header defines it): box (rb, kc) of 128 rows x 128 bytes at byte
    (rb * KC + kc) * 16384, KC = ceil(K / 256), bytes past K/2 zero."""
    KC = (K + 255) // 256
    t = np.asarray(tiled, dtype=np.uint8).reshape(E * N // 128, KC, 128, 128)
    rows = t.transpose(0, 2, 1, 3).reshape(E * N, KC * 128)
    assert not rows[:, K // 2:].any(), "bytes past K/2 must be zero"
    return rows[:, :K // 2].reshape(E, N, K // 2)


def packed_weights(w):
    """Row-major [E, N, K/2] codes of a layer's packed weights (tiled or not)."""
    if hasattr(w, "data") and hasattr(w, "K"):
        return untile_weights(w.data.cpu().numpy(), w.E, w.N, w.K)
    return w.cpu().numpy()


def signed_rank(codes):
    """Position of each E2M1 code on the ordered value line (-7..7; +-0 -> 0)."""
    c = np.asarray(codes).astype(np.int64)
    mag = c & 7
    return np.where((c >> 3) & 1, -mag, mag)


def check_close(got, ref, frob_tol=FROB_TOL, elem_tol=ELEM_TOL, what="output"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    frob = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    worst = np.max(np.abs(got - ref) / np.maximum(np.abs(ref), rms)) if ref.size else 0.0
    assert frob <= frob_tol, f"{what}: relative Frobenius error {frob:.3e} > {frob_tol}"
    assert worst <= elem_tol, f"{what}: worst element error {worst:.3e} > {elem_tol} (x max(|ref|, rms))"
    return frob, worst


def check_requant(got_codes, got_scales, ref_codes, ref_scales, max_flip_frac=0.01, min_scale_eq=0.99, block=16):
    """Fused SwiGLU requantisation vs the oracle's: float32 accumulation order
    may move a value across an E2M1 or ue4m3 midpoint, so codes may differ by
    one step on a small fraction of elements and scales may differ in a
    small fraction of blocks."""
    eq = np.mean(np.asarray(got_scales) == np.asarray(ref_scales)) if np.size(ref_scales) else 1.0
    assert eq >= min_scale_eq, f"only {eq:.4f} of block scales equal"
    same_scale = np.repeat(np.asarray(got_scales) == np.asarray(ref_scales), block, axis=-1)
    d = np.abs(signed_rank(got_codes) - signed_rank(ref_codes))
    d = d[same_scale]
    assert d.size == 0 or d.max() <= 1, f"a code differs by {d.max()} steps"
    frac = np.mean(d != 0) if d.size else 0.0
    assert frac <= max_flip_frac, f"{frac:.4f} of codes differ by one step"
    return eq, frac


def oracle_quantize_experts_mx(w_bf16):
    """Oracle MXFP4 quantisation of bf16 expert weights [E, N, K] (CPU tensor)."""
    ps, ss = [], []
    for e in range(w_bf16.shape[0]):
        p, s = O.quantize_mxfp4(w_bf16[e].float().numpy())
        ps.append(p), ss.append(s)
    return np.stack(ps), np.stack(ss)


def oracle_quantize_experts(w_bf16):
    """Oracle NVFP4 quantisation of bf16 expert weights [E, N, K] (CPU tensor)."""
    ps, ss, gs = [], [], []
    for e in range(w_bf16.shape[0]):
        a = w_bf16[e].float().numpy()
        g = O.global_scale(a)
        p, s = O.quantize_nvfp4(a, g)
        ps.append(p), ss.append(s), gs.append(g)
    return np.stack(ps), np.stack(ss), np.array(gs, np.float32)


def check_permutation(out, idx, E, xq, xs, block=16):
    """A Permutation (CUDA) against the oracle's stable expert-first order
    of `idx` [T, k], with the gathered packed rows `xq` and row-major scales
    `xs` of the tokens: counts, offsets, 128-aligned row offsets, both maps,
    -1 on every padding row, and the gathered rows and blocked scales."""
    T, k = idx.shape
    H = xq.shape[1] * 2
    counts, offsets, p2f, f2p = O.permute(idx, E)
    np.testing.assert_array_equal(out.counts.cpu().numpy(), counts)
    np.testing.assert_array_equal(out.offsets.cpu().numpy(), offsets)
    roff = out.row_offsets.cpu().numpy()
    np.testing.assert_array_equal(roff, np.concatenate([[0], np.cumsum(ceil_to(counts, 128))]))
    g_p2f = out.perm_to_flat.cpu().numpy()
    g_f2p = out.flat_to_perm.cpu().numpy()
    cap = out.rows_capacity
    assert g_p2f.shape == (cap,)
    valid = np.zeros(cap, bool)
    for e in range(E):
        rows = roff[e] + np.arange(counts[e])
        valid[rows] = True
        np.testing.assert_array_equal(g_p2f[rows], p2f[offsets[e]:offsets[e + 1]])
    assert np.all(g_p2f[~valid] == -1)
    if T * k == 0:
        return
    e_of = idx.reshape(-1)
    np.testing.assert_array_equal(g_f2p - roff[e_of] + offsets[e_of], f2p)
    a = out.a_packed.cpu().numpy()
    np.testing.assert_array_equal(a[g_f2p], xq[np.arange(T * k) // k])
    sc = from_blocked(out.a_scales.cpu().numpy(), cap, H, block)
    np.testing.assert_array_equal(sc[g_f2p], xs[np.arange(T * k) // k])
