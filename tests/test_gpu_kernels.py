"""Per-kernel parity of the CUDA library against the CPU oracle (GB300).

Integer and byte outputs (router indices, permutation maps, offsets,
gathered rows, quantiser bytes, scale bytes, global scales) must be
bit-exact; floating-point outputs use the bar in nvfp4_testutil.  Every
input comes from the seeded generators; no expected value comes from the
CUDA path.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


def dev(a, dtype=None):
    t = torch.as_tensor(a) if not isinstance(a, torch.Tensor) else a
    t = t.to("cuda")
    return t if dtype is None else t.to(dtype)


def bf16_from_bits(bits16):
    return torch.from_numpy(np.ascontiguousarray(bits16.astype(np.uint16)).view(np.int16)).view(torch.bfloat16)


# ---------------------------------------------------------------------------
# quantiser
# ---------------------------------------------------------------------------
ALL_FINITE_BF16 = np.array([b for b in range(65536) if ((b >> 7) & 0xFF) != 0xFF], dtype=np.uint32)


@pytest.mark.parametrize("s", [1.0, 2.0 ** -30, 2.0 ** 30, 0.0123, 2.0 ** -120, 3.0e12, 2.0 ** -4])
@pytest.mark.parametrize("order", ["sorted", "shuffled"])
def test_quantize_every_bf16_value(B, s, order):
    bits = ALL_FINITE_BF16.copy()
    if order == "shuffled":
        np.random.default_rng(1).shuffle(bits)
    bits = np.concatenate([bits, np.zeros((-len(bits)) % 1024, np.uint32)])
    xb = bf16_from_bits(bits).reshape(-1, 1024)
    x32 = xb.float().numpy()
    gs = torch.tensor([s], dtype=torch.float32)
    packed, scales, _ = B.moe_quantize_nvfp4(dev(xb), global_scale=dev(gs), compute_global=False)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        rp, rs = O.quantize_nvfp4(x32, np.float32(s))
    np.testing.assert_array_equal(scales.cpu().numpy(), rs)
    np.testing.assert_array_equal(packed.cpu().numpy(), rp)


@pytest.mark.parametrize("rows,cols", [(1, 64), (16, 256), (129, 6144), (300, 1024)])
def test_quantize_global_scale_and_blocked_layout(B, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = torch.from_numpy((rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-6, 6, (rows, 1))))
                         .astype(np.float32)).to(torch.bfloat16)
    x32 = x.float().numpy()
    p1, s1, g1 = B.moe_quantize_nvfp4(dev(x))
    p2, s2, g2 = B.moe_quantize_nvfp4(dev(x), blocked=True)
    rg = O.global_scale(x32)
    rp, rs = O.quantize_nvfp4(x32, rg)
    assert g1.item() == rg and g2.item() == rg
    np.testing.assert_array_equal(p1.cpu().numpy(), rp)
    np.testing.assert_array_equal(p2.cpu().numpy(), rp)
    np.testing.assert_array_equal(s1.cpu().numpy(), rs)
    blk = s2.cpu().numpy()
    np.testing.assert_array_equal(U.from_blocked(blk, rows, cols), rs)
    # padding rows of the last 128-row block are zero
    rp_rows = U.ceil_to(rows, 128)
    full = blk[U.blocked_index(rp_rows, cols)]
    assert np.all(full[rows:] == 0)


def test_quantize_all_zero_tensor(B):
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    p, s, g = B.moe_quantize_nvfp4(dev(x))
    assert g.item() == 1.0 and not p.any().item() and not s.any().item()


def test_scales_to_blocked(B):
    rng = np.random.default_rng(3)
    for rows, cols in [(1, 64), (130, 384), (256, 6144)]:
        sc = rng.integers(0, 127, size=(rows, cols // 16), dtype=np.uint8)
        got = B.moe_scales_to_blocked(dev(torch.from_numpy(sc)), cols).cpu().numpy()
        np.testing.assert_array_equal(got, U.to_blocked(sc, cols))


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,score,renorm,bias,ties", [
    (16, 8, 2, "softmax", True, False, False),
    (64, 8, 8, "softmax", True, False, True),
    (37, 256, 8, "sigmoid", True, True, False),
    (128, 256, 8, "sigmoid", True, False, True),
    (50, 64, 6, "softmax", False, False, False),
    (40, 33, 5, "sigmoid", False, True, True),
    (9, 1024, 32, "sigmoid", True, False, True),
    (5, 1, 1, "softmax", True, False, False),
])
def test_route_topk(B, T, E, k, score, renorm, bias, ties):
    rng = np.random.default_rng(T * 131 + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        lg = (np.round(lg * 4) / 4).astype(np.float32)   # many exactly equal logits
    b = W.zipf_bias(E, 1.1) if bias else None
    idx, w = B.moe_route_topk(dev(torch.from_numpy(lg)), k, score, renorm,
                              bias=dev(torch.from_numpy(b)) if bias else None)
    ridx, rw = O.route_topk(lg, b, k, score, renorm)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    gw = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gw - rw) <= 1e-6 * np.abs(rw) + 1e-30), np.max(np.abs(gw - rw) / rw)


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,H,skew", [
    (16, 8, 2, 256, False),
    (700, 16, 4, 128, True),     # several 1024-id segments, skewed counts
    (128, 256, 8, 6144, False),
    (33, 1, 1, 64, False),       # one expert
    (40, 1024, 3, 64, False),    # many empty experts
    (2048, 64, 8, 512, True),
])
def test_permute(B, T, E, k, H, skew):
    rng = np.random.default_rng(T + E)
    hint = 1.0 / np.arange(1, E + 1) ** 1.1 if skew else None
    idx = W.random_routing(T, E, k, seed=T * E, counts_hint=hint)
    xq = rng.integers(0, 256, size=(T, H // 2), dtype=np.uint8)
    xs = rng.integers(0, 127, size=(T, H // 16), dtype=np.uint8)
    out = B.moe_permute(dev(torch.from_numpy(idx)), E, dev(torch.from_numpy(xq)), dev(torch.from_numpy(xs)))
    B.sync_status()
    counts, offsets, p2f, f2p = O.permute(idx, E)
    np.testing.assert_array_equal(out.counts.cpu().numpy(), counts)
    np.testing.assert_array_equal(out.offsets.cpu().numpy(), offsets)
    roff = out.row_offsets.cpu().numpy()
    np.testing.assert_array_equal(roff, np.concatenate([[0], np.cumsum(U.ceil_to(counts, 128))]))
    g_p2f = out.perm_to_flat.cpu().numpy()
    g_f2p = out.flat_to_perm.cpu().numpy()
    cap = out.rows_capacity
    valid = np.zeros(cap, bool)
    for e in range(E):
        rows = roff[e] + np.arange(counts[e])
        valid[rows] = True
        np.testing.assert_array_equal(g_p2f[rows], p2f[offsets[e]:offsets[e + 1]])
    assert np.all(g_p2f[~valid] == -1)
    e_of = idx.reshape(-1)
    np.testing.assert_array_equal(g_f2p - roff[e_of] + offsets[e_of], f2p)
    a = out.a_packed.cpu().numpy()
    np.testing.assert_array_equal(a[g_f2p], xq[np.arange(T * k) // k])
    sc = U.from_blocked(out.a_scales.cpu().numpy(), cap, H)
    np.testing.assert_array_equal(sc[g_f2p], xs[np.arange(T * k) // k])


def test_permute_rejects_bad_expert_ids(B):
    idx = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32)
    xq = torch.zeros((2, 32), dtype=torch.uint8)
    xs = torch.zeros((2, 4), dtype=torch.uint8)
    B.moe_permute(dev(idx), 4, dev(xq), dev(xs))
    with pytest.raises(B.Nvfp4MoeError) as ei:
        B.sync_status()
    assert ei.value.status == B.ERR_DEVICE_DATA
    B.sync_status()   # the flag is cleared once read


# ---------------------------------------------------------------------------
# finalize
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,k,H", [(16, 2, 256), (129, 8, 6144), (1, 1, 8)])
def test_finalize(B, T, k, H):
    rng = np.random.default_rng(T * k)
    cap = U.ceil_to(T * k + 50, 128)
    y = torch.from_numpy(rng.standard_normal((cap, H)).astype(np.float32)).to(torch.bfloat16)
    f2p = rng.permutation(cap)[:T * k].astype(np.int32)
    w = rng.uniform(0, 1, size=(T, k)).astype(np.float32)
    got = B.moe_finalize(dev(y), dev(torch.from_numpy(f2p)), dev(torch.from_numpy(w))).float().cpu().numpy()
    ref = O.round_to_bf16(O.finalize(y.float().numpy(), f2p, w, T, k))
    U.check_close(got, ref, frob_tol=1e-3, elem_tol=2 ** -7, what="finalize")


# ---------------------------------------------------------------------------
# grouped GEMM (operands: random NVFP4 bytes from the generator)
# ---------------------------------------------------------------------------
def gemm_case(E, N, K, counts, seed):
    counts = np.asarray(counts, dtype=np.int64)
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)])
    roff = np.concatenate([[0], np.cumsum(U.ceil_to(counts, 128))])
    cap = max(int(roff[-1]), 128)
    ap, asc, s_a = W.random_nvfp4_operand(R, K, seed)
    wp = np.empty((E, N, K // 2), np.uint8)
    wsc = np.empty((E, N, K // 16), np.uint8)
    for e in range(E):
        wp[e], wsc[e], _ = W.random_nvfp4_operand(N, K, seed + 1 + e)
    s_w = np.float32(np.random.default_rng(seed).uniform(0.01, 0.1, size=E))
    # expert-padded device layout
    a_pad = np.zeros((cap, K // 2), np.uint8)
    s_pad = np.zeros((cap, K // 16), np.uint8)
    pos = np.concatenate([roff[e] + np.arange(counts[e]) for e in range(E)]).astype(np.int64)
    a_pad[pos] = ap
    s_pad[pos] = asc
    g = dict(
        a_packed=dev(torch.from_numpy(a_pad)), a_scales=dev(torch.from_numpy(U.to_blocked(s_pad, K))),
        a_gscale=dev(torch.tensor([s_a])), counts=dev(torch.from_numpy(counts.astype(np.int32))),
        row_offsets=dev(torch.from_numpy(roff.astype(np.int32))), w_packed=dev(torch.from_numpy(wp)),
        w_scales=dev(torch.from_numpy(np.stack([U.to_blocked(wsc[e], K) for e in range(E)]))),
        w_gscale=dev(torch.from_numpy(s_w)))
    ref = O.grouped_gemm(ap, asc, s_a, offsets, wp, wsc, s_w)
    return g, ref, pos, R


GEMM_SHAPES = [
    # E, N, K, counts, tile_n (widest token tile); tile widths follow the counts
    (3, 256, 256, [5, 0, 40], 0),                 # widths 32 and 64
    (4, 384, 448, [1, 33, 64, 129], 0),           # partial last K tile, 3 M tiles, 128 + 32
    (2, 128, 128, [7, 200], 128),                 # K below one stage
    (2, 256, 1024, [300, 17], 256),               # a 256-wide tile, a one-block tail
    (5, 128, 64, [3, 3, 3, 3, 3], 0),
    (2, 512, 2048, [64, 64], 0),
    (8, 256, 768, [0, 1, 2, 3, 130, 0, 31, 257], 0),
    (3, 128, 512, [256, 129, 96], 256),           # 256, 128 + 32 ... under the 256 cap
    (6, 256, 512, [200, 1, 2, 3, 4, 5], 0),       # tile order: one multi-tile expert among single-tile ones
]


@pytest.mark.parametrize("E,N,K,counts,tile_n", GEMM_SHAPES)
def test_grouped_gemm_bf16(B, E, N, K, counts, tile_n):
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=E * 1000 + K)
    out = B.moe_grouped_gemm_nvfp4(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"],
                                   g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=R,
                                   tile_n=tile_n)
    B.sync_status()
    got = out.float().cpu().numpy()[pos]
    U.check_close(got, O.round_to_bf16(ref), what="bf16 GEMM")


SWIGLU_SHAPES = [
    # E, I, K, counts, tile_n
    (3, 128, 512, [9, 70, 0], 0),                 # one single-slot and one double-slot tile
    (2, 256, 320, [130, 1], 0),
    (4, 128, 1024, [128, 5, 64, 200], 128),       # slot sequence mixes 32/64/128-wide tiles
    (2, 384, 256, [40, 41], 0),
]


@pytest.mark.parametrize("E,I,K,counts,tile_n", SWIGLU_SHAPES)
def test_grouped_gemm_swiglu(B, E, I, K, counts, tile_n):
    g, ref, pos, R = gemm_case(E, 2 * I, K, counts, seed=E * 777 + K)
    h_ref = O.swiglu(ref, I)
    args = (g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"], g["w_packed"],
            g["w_scales"], g["w_gscale"])
    hf = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_F32, m_total=R, tile_n=tile_n)
    s_h = np.float32(2.0 ** -4)
    hq, hs = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_NVFP4, c_gscale=dev(torch.tensor([s_h])), m_total=R,
                                      tile_n=tile_n)
    B.sync_status()
    U.check_close(hf.cpu().numpy()[pos], h_ref, frob_tol=1e-5, elem_tol=1e-4, what="SwiGLU float32")
    rq, rs = O.quantize_nvfp4(h_ref.astype(np.float32), s_h)
    cap = hq.shape[0]
    codes = O.unpack_codes(hq.cpu().numpy()[pos])
    scales = U.from_blocked(hs.cpu().numpy(), cap, I)[pos]
    U.check_requant(codes, scales, O.unpack_codes(rq), rs)


TM = -1  # binding.TILE_TOKEN_MAJOR: 128 tokens as M, two 128-row weight tiles as one N = 256 operand
TM_GEMM_SHAPES = [
    # E, N, K, counts: partial token tiles, empty experts, several M tiles, a partial last K stage
    (3, 256, 256, [5, 0, 40]),
    (2, 512, 1024, [300, 17]),
    (8, 256, 768, [0, 1, 2, 3, 130, 0, 31, 257]),
    (2, 768, 320, [128, 129]),
    (6, 256, 512, [200, 1, 2, 3, 4, 5]),          # more single-tile than multi-tile work
]


@pytest.mark.parametrize("E,N,K,counts", TM_GEMM_SHAPES)
def test_grouped_gemm_bf16_token_major(B, E, N, K, counts):
    """Token-major tiles (tokens as M, N = 256 weight rows per MMA) against
    the oracle: a partial token tile still computes 128 rows and stores only
    the expert's."""
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=E * 1300 + K)
    out = B.moe_grouped_gemm_nvfp4(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"],
                                   g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=R,
                                   tile_n=B.TILE_TOKEN_MAJOR)
    B.sync_status()
    U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="bf16 GEMM, token-major")


@pytest.mark.parametrize("E,I,K,counts", [(3, 128, 512, [9, 70, 0]), (2, 256, 320, [130, 1]),
                                          (4, 128, 1024, [128, 5, 64, 200]), (2, 384, 256, [40, 41])])
def test_grouped_gemm_swiglu_token_major(B, E, I, K, counts):
    g, ref, pos, R = gemm_case(E, 2 * I, K, counts, seed=E * 701 + K)
    h_ref = O.swiglu(ref, I)
    args = (g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"], g["w_packed"],
            g["w_scales"], g["w_gscale"])
    hf = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_F32, m_total=R, tile_n=B.TILE_TOKEN_MAJOR)
    s_h = np.float32(2.0 ** -4)
    hq, hs = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_NVFP4, c_gscale=dev(torch.tensor([s_h])), m_total=R,
                                      tile_n=B.TILE_TOKEN_MAJOR)
    B.sync_status()
    U.check_close(hf.cpu().numpy()[pos], h_ref, frob_tol=1e-5, elem_tol=1e-4, what="SwiGLU float32, token-major")
    rq, rs = O.quantize_nvfp4(h_ref.astype(np.float32), s_h)
    cap = hq.shape[0]
    U.check_requant(O.unpack_codes(hq.cpu().numpy()[pos]), U.from_blocked(hs.cpu().numpy(), cap, I)[pos],
                    O.unpack_codes(rq), rs)


def test_grouped_gemm_token_major_chosen_automatically(B):
    """tile_n = 0 picks token-major tiles once experts average 64 rows
    (m_total >= 64 E); the result is the explicit token-major call's, bit for
    bit, with the dynamic schedule as with static stripes."""
    E, N, K, counts = 3, 512, 512, [150, 5, 60]
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=91)
    assert R >= 64 * E
    args = (g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"], g["w_packed"],
            g["w_scales"], g["w_gscale"])
    ws = B.alloc_gemm_workspace(torch.device("cuda"))
    auto = B.moe_grouped_gemm_nvfp4(*args, B.EPI_BF16, m_total=R, tile_n=0, workspace=ws)
    tm = B.moe_grouped_gemm_nvfp4(*args, B.EPI_BF16, m_total=R, tile_n=B.TILE_TOKEN_MAJOR)
    B.sync_status()
    assert not ws.any().item()
    rows = torch.from_numpy(pos).cuda()
    assert torch.equal(auto[rows], tm[rows])
    U.check_close(auto.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="bf16 GEMM, automatic tiles")


@pytest.mark.parametrize("E,N,K,counts,tile_n", [(3, 256, 320, [5, 0, 140], 0), (2, 512, 1024, [300, 17], TM),
                                                  (4, 384, 448, [1, 33, 64, 129], 0), (2, 256, 256, [7, 200], 256)])
def test_grouped_gemm_tiled_weights(B, E, N, K, counts, tile_n):
    """nvfp4moe_tile_weights writes the layout the header defines (checked by
    undoing it), and the GEMMs read tiled weights to the same bits as
    row-major ones: same operands, same arithmetic."""
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=E * 3 + K)
    tiled = B.tile_expert_weights(g["w_packed"])
    B.sync_status()
    np.testing.assert_array_equal(U.untile_weights(tiled.data.cpu().numpy(), E, N, K), g["w_packed"].cpu().numpy())
    args = (g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"])
    rows = torch.from_numpy(pos).cuda()
    y0 = B.moe_grouped_gemm_nvfp4(*args, g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=R,
                                  tile_n=tile_n)
    y1 = B.moe_grouped_gemm_nvfp4(*args, tiled, g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=R, tile_n=tile_n)
    B.sync_status()
    assert torch.equal(y0[rows], y1[rows])
    U.check_close(y1.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="bf16 GEMM, tiled weights")
    if N % 256 == 0 and tile_n != 256:
        s_h = dev(torch.tensor([2.0 ** -4]))
        h0, hs0 = B.moe_grouped_gemm_nvfp4(*args, g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_SWIGLU_NVFP4,
                                           c_gscale=s_h, m_total=R, tile_n=tile_n)
        h1, hs1 = B.moe_grouped_gemm_nvfp4(*args, tiled, g["w_scales"], g["w_gscale"], B.EPI_SWIGLU_NVFP4,
                                           c_gscale=s_h, m_total=R, tile_n=tile_n)
        B.sync_status()
        assert torch.equal(h0[rows], h1[rows])
        cap = h0.shape[0]
        np.testing.assert_array_equal(U.from_blocked(hs0.cpu().numpy(), cap, N // 2)[pos],
                                      U.from_blocked(hs1.cpu().numpy(), cap, N // 2)[pos])


@pytest.mark.parametrize("E,N,K,counts,tile_n", GEMM_SHAPES[:4])
def test_grouped_gemm_dynamic_schedule_matches_static(B, E, N, K, counts, tile_n):
    """Tiles claimed from the launch-wide counter give the same bits as the
    static stripes (each tile's arithmetic does not depend on its CTA), and
    the workspace is left zeroed for the next call."""
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=E * 55 + K)
    args = (g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"], g["w_packed"],
            g["w_scales"], g["w_gscale"])
    ws = B.alloc_gemm_workspace(torch.device("cuda"))
    static = B.moe_grouped_gemm_nvfp4(*args, B.EPI_BF16, m_total=R, tile_n=tile_n)
    for _ in range(3):
        dyn = B.moe_grouped_gemm_nvfp4(*args, B.EPI_BF16, m_total=R, tile_n=tile_n, workspace=ws)
        B.sync_status()
        assert not ws.any().item()
        assert torch.equal(dyn[torch.from_numpy(pos).cuda()], static[torch.from_numpy(pos).cuda()])
    I = N // 2
    if N % 256 == 0:
        hq0, hs0 = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_NVFP4, c_gscale=dev(torch.tensor([2.0 ** -4])),
                                            m_total=R)
        hq1, hs1 = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_NVFP4, c_gscale=dev(torch.tensor([2.0 ** -4])),
                                            m_total=R, workspace=ws)
        B.sync_status()
        rows = torch.from_numpy(pos).cuda()
        assert torch.equal(hq0[rows], hq1[rows])
        cap = hq0.shape[0]
        np.testing.assert_array_equal(U.from_blocked(hs0.cpu().numpy(), cap, I)[pos],
                                      U.from_blocked(hs1.cpu().numpy(), cap, I)[pos])
        assert not ws.any().item()
