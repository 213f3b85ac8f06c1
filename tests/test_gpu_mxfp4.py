"""MXFP4 variant (reading R9 of the oracle): quantiser, permutation, grouped
GEMM (both epilogues) and the whole layer against the CPU oracle.  Quantiser
bytes, scales and permutation maps bit-exact; floating-point outputs with the
bar in nvfp4_testutil."""
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


def dev(a):
    return (torch.as_tensor(a) if not isinstance(a, torch.Tensor) else a).to("cuda")


ALL_FINITE_BF16 = np.array([b for b in range(65536) if ((b >> 7) & 0xFF) != 0xFF], dtype=np.uint32)


def bf16_from_bits(bits16):
    return torch.from_numpy(np.ascontiguousarray(bits16.astype(np.uint16)).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("order", ["sorted", "shuffled"])
def test_quantize_mx_every_bf16_value(B, order):
    bits = ALL_FINITE_BF16.copy()
    if order == "shuffled":
        np.random.default_rng(2).shuffle(bits)
    bits = np.concatenate([bits, np.zeros((-len(bits)) % 1024, np.uint32)])
    xb = bf16_from_bits(bits).reshape(-1, 1024)
    packed, scales = B.moe_quantize_mxfp4(dev(xb))
    rp, rs = O.quantize_mxfp4(xb.float().numpy())
    np.testing.assert_array_equal(scales.cpu().numpy(), rs)
    np.testing.assert_array_equal(packed.cpu().numpy(), rp)


@pytest.mark.parametrize("rows,cols", [(1, 128), (16, 256), (129, 6144), (300, 1024)])
def test_quantize_mx_blocked_layout(B, rows, cols):
    rng = np.random.default_rng(rows + cols)
    x = torch.from_numpy((rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-20, 20, (rows, 1))))
                         .astype(np.float32)).to(torch.bfloat16)
    rp, rs = O.quantize_mxfp4(x.float().numpy())
    p1, s1 = B.moe_quantize_mxfp4(dev(x))
    p2, s2 = B.moe_quantize_mxfp4(dev(x), blocked=True)
    np.testing.assert_array_equal(p1.cpu().numpy(), rp)
    np.testing.assert_array_equal(p2.cpu().numpy(), rp)
    np.testing.assert_array_equal(s1.cpu().numpy(), rs)
    blk = s2.cpu().numpy()
    np.testing.assert_array_equal(U.from_blocked(blk, rows, cols, 32), rs)
    full = blk[U.blocked_index(U.ceil_to(rows, 128), cols, 32)]
    assert np.all(full[rows:] == 0)


@pytest.mark.parametrize("T,E,k,H", [(16, 8, 2, 256), (700, 16, 4, 128), (128, 256, 8, 6144)])
def test_permute_mx(B, T, E, k, H):
    rng = np.random.default_rng(T + E)
    idx = W.random_routing(T, E, k, seed=T * E)
    xq = rng.integers(0, 256, size=(T, H // 2), dtype=np.uint8)
    xs = rng.integers(100, 150, size=(T, H // 32), dtype=np.uint8)
    out = B.moe_permute_mxfp4(dev(torch.from_numpy(idx)), E, dev(torch.from_numpy(xq)), dev(torch.from_numpy(xs)))
    B.sync_status()
    U.check_permutation(out, idx, E, xq, xs, block=32)


def mx_operand(rows, K, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8),
            rng.integers(118, 133, size=(rows, K // 32), dtype=np.uint8))


def gemm_case_mx(E, N, K, counts, seed):
    counts = np.asarray(counts, dtype=np.int64)
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)])
    roff = np.concatenate([[0], np.cumsum(U.ceil_to(counts, 128))])
    cap = max(int(roff[-1]), 128)
    ap, asc = mx_operand(R, K, seed)
    wp = np.empty((E, N, K // 2), np.uint8)
    wsc = np.empty((E, N, K // 32), np.uint8)
    for e in range(E):
        wp[e], wsc[e] = mx_operand(N, K, seed + 1 + e)
    a_pad = np.zeros((cap, K // 2), np.uint8)
    s_pad = np.zeros((cap, K // 32), np.uint8)
    pos = np.concatenate([roff[e] + np.arange(counts[e]) for e in range(E)]).astype(np.int64)
    a_pad[pos] = ap
    s_pad[pos] = asc
    g = dict(a_packed=dev(torch.from_numpy(a_pad)), a_scales=dev(torch.from_numpy(U.to_blocked(s_pad, K, 32))),
             counts=dev(torch.from_numpy(counts.astype(np.int32))),
             row_offsets=dev(torch.from_numpy(roff.astype(np.int32))), w_packed=dev(torch.from_numpy(wp)),
             w_scales=dev(torch.from_numpy(np.stack([U.to_blocked(wsc[e], K, 32) for e in range(E)]))))
    return g, O.grouped_gemm_mx(ap, asc, offsets, wp, wsc), pos, R


MX_GEMM_SHAPES = [
    # E, N, K, counts, tile_n
    (3, 256, 256, [5, 0, 40], 0),
    (4, 384, 384, [1, 33, 64, 129], 0),           # partial last K stage (one k128 scale block)
    (2, 128, 128, [7, 200], 128),                 # K below one stage
    (2, 256, 1024, [300, 17], 256),               # a 256-wide tile
    (8, 256, 768, [0, 1, 2, 3, 130, 0, 31, 257], 0),
]


@pytest.mark.parametrize("E,N,K,counts,tile_n", MX_GEMM_SHAPES)
def test_grouped_gemm_mx_bf16(B, E, N, K, counts, tile_n):
    g, ref, pos, R = gemm_case_mx(E, N, K, counts, seed=E * 100 + K)
    out = B.moe_grouped_gemm_mxfp4(g["a_packed"], g["a_scales"], g["counts"], g["row_offsets"], g["w_packed"],
                                   g["w_scales"], B.EPI_BF16, m_total=R, tile_n=tile_n)
    B.sync_status()
    U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="MXFP4 bf16 GEMM")


@pytest.mark.parametrize("E,N,K,counts", [(3, 256, 256, [5, 0, 40]), (2, 256, 1024, [300, 17]),
                                          (4, 512, 384, [1, 33, 64, 129])])
def test_grouped_gemm_mx_bf16_token_major(B, E, N, K, counts):
    g, ref, pos, R = gemm_case_mx(E, N, K, counts, seed=E * 170 + K)
    out = B.moe_grouped_gemm_mxfp4(g["a_packed"], g["a_scales"], g["counts"], g["row_offsets"], g["w_packed"],
                                   g["w_scales"], B.EPI_BF16, m_total=R, tile_n=B.TILE_TOKEN_MAJOR)
    B.sync_status()
    U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="MXFP4 bf16 GEMM, token-major")


@pytest.mark.parametrize("tile_n", [0, -1])  # -1: binding.TILE_TOKEN_MAJOR
def test_grouped_gemm_mx_tiled_weights(B, tile_n):
    """MXFP4 codes in the tiled layout: the same bits as row-major weights."""
    E, N, K, counts = 3, 512, 640, [9, 140, 1]
    g, ref, pos, R = gemm_case_mx(E, N, K, counts, seed=77)
    tiled = B.tile_expert_weights(g["w_packed"])
    args = (g["a_packed"], g["a_scales"], g["counts"], g["row_offsets"])
    y0 = B.moe_grouped_gemm_mxfp4(*args, g["w_packed"], g["w_scales"], B.EPI_BF16, m_total=R, tile_n=tile_n)
    y1 = B.moe_grouped_gemm_mxfp4(*args, tiled, g["w_scales"], B.EPI_BF16, m_total=R, tile_n=tile_n)
    B.sync_status()
    rows = torch.from_numpy(pos).cuda()
    assert torch.equal(y0[rows], y1[rows])
    U.check_close(y1.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="MXFP4 bf16 GEMM, tiled weights")


@pytest.mark.parametrize("tile_n", [0, -1])  # -1: binding.TILE_TOKEN_MAJOR
@pytest.mark.parametrize("E,I,K,counts", [(3, 128, 512, [9, 70, 0]), (2, 256, 384, [130, 1]),
                                          (4, 128, 1024, [128, 5, 64, 200])])
def test_grouped_gemm_mx_swiglu(B, E, I, K, counts, tile_n):
    g, ref, pos, R = gemm_case_mx(E, 2 * I, K, counts, seed=E * 31 + K)
    h_ref = O.swiglu(ref, I)
    args = (g["a_packed"], g["a_scales"], g["counts"], g["row_offsets"], g["w_packed"], g["w_scales"])
    hf = B.moe_grouped_gemm_mxfp4(*args, B.EPI_SWIGLU_F32, m_total=R, tile_n=tile_n)
    hq, hs = B.moe_grouped_gemm_mxfp4(*args, B.EPI_SWIGLU_MXFP4, m_total=R, tile_n=tile_n)
    B.sync_status()
    U.check_close(hf.cpu().numpy()[pos], h_ref, frob_tol=1e-5, elem_tol=1e-4, what="MXFP4 SwiGLU float32")
    rq, rs = O.quantize_mxfp4(h_ref.astype(np.float32))
    cap = hq.shape[0]
    U.check_requant(O.unpack_codes(hq.cpu().numpy()[pos]), U.from_blocked(hs.cpu().numpy(), cap, I, 32)[pos],
                    O.unpack_codes(rq), rs, block=32)


@pytest.mark.parametrize("T,E,k,H,k0", [(16, 8, 2, 256, None), (128, 256, 8, 6144, None), (2100, 64, 8, 128, None),
                                        (2100, 64, 8, 512, None), (300, 16, 4, 512, 1), (1, 4, 2, 128, None)])
def test_prepare_mx_matches_separate_calls_and_oracle(B, T, E, k, H, k0):
    rng = np.random.default_rng(T + H)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    cuda = torch.device("cuda")
    lg_d, x_d = torch.from_numpy(lg).to(cuda), x.to(cuda)
    idx, w, xq, xs, perm = B.moe_prepare_mxfp4(lg_d, x_d, k, "sigmoid", True, k_primary=k0)
    B.sync_status()
    ridx, _ = (O.route_topk(lg, None, k, "sigmoid") if k0 is None else
               O.route_batch_aware(lg, None, k, k0, "sigmoid"))
    rxq, rxs = O.quantize_mxfp4(x.float().numpy())
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(xq.cpu().numpy(), rxq)
    np.testing.assert_array_equal(xs.cpu().numpy(), rxs)
    U.check_permutation(perm, ridx, E, rxq, rxs, block=32)
    sidx, sw = (B.moe_route_topk(lg_d, k, "sigmoid", True) if k0 is None else
                B.moe_route_batch_aware(lg_d, k, k0, "sigmoid", True))
    sxq, sxs = B.moe_quantize_mxfp4(x_d)
    sperm = B.moe_permute_mxfp4(sidx, E, sxq, sxs)
    B.sync_status()
    assert torch.equal(idx, sidx) and torch.equal(w.view(torch.int32), sw.view(torch.int32))
    assert torch.equal(xq, sxq) and torch.equal(xs, sxs)
    for name in ("counts", "offsets", "row_offsets", "perm_to_flat", "flat_to_perm"):
        assert torch.equal(getattr(perm, name), getattr(sperm, name)), name


@pytest.mark.parametrize("fused", [True, False], ids=["fused_prepare", "separate_calls"])
@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"]] + list(W.TEST_WORKLOADS.values()), ids=lambda w: w.name)
def test_layer_mx_matches_oracle(B, w, fused):
    inp = W.host_inputs(w, seed=2)
    cuda = torch.device("cuda")
    bias = inp["bias"]
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, w.renormalize, w.h_scale,
                       bias=None if bias is None else bias.to(cuda), fmt="mxfp4", fused_prepare=fused)
    out = layer(inp["x"].to(cuda), inp["logits"].to(cuda)).float().cpu().numpy()
    B.sync_status()
    gq = U.oracle_quantize_experts_mx(inp["w_gu"])
    dq = U.oracle_quantize_experts_mx(inp["w_d"])
    np.testing.assert_array_equal(U.packed_weights(layer.w_gu_packed), gq[0])
    np.testing.assert_array_equal(U.packed_weights(layer.w_d_packed), dq[0])
    for e in range(w.E):
        np.testing.assert_array_equal(U.from_blocked(layer.w_d_scales[e].cpu().numpy(), w.H, w.I, 32), dq[1][e])
    ref, it = O.moe_layer_mx(inp["x"].float().numpy(), inp["logits"].numpy(),
                             None if bias is None else bias.numpy(), gq[0], gq[1], dq[0], dq[1], w.k, w.score,
                             renormalize=w.renormalize, return_intermediates=True)
    np.testing.assert_array_equal(layer.xq.cpu().numpy(), it["xq"])
    np.testing.assert_array_equal(layer.xs.cpu().numpy(), it["xs"])
    np.testing.assert_array_equal(layer.perm.counts.cpu().numpy(), it["counts"])
    roff = layer.perm.row_offsets.cpu().numpy()
    pos = np.concatenate([roff[e] + np.arange(it["counts"][e]) for e in range(w.E)])
    cap = layer.perm.rows_capacity
    U.check_requant(O.unpack_codes(layer.hq.cpu().numpy()[pos]),
                    U.from_blocked(layer.hs.cpu().numpy(), cap, w.I, 32)[pos], O.unpack_codes(it["hq"]), it["hs"],
                    block=32)
    U.check_close(layer.y.float().cpu().numpy()[pos], it["y"], what="MXFP4 down projection")
    U.check_close(out, ref, what="MXFP4 layer output")


def test_grouped_gemm_mx_dynamic_schedule(B):
    g, ref, pos, R = gemm_case_mx(4, 256, 512, [3, 300, 0, 77], seed=9)
    args = (g["a_packed"], g["a_scales"], g["counts"], g["row_offsets"], g["w_packed"], g["w_scales"])
    ws = B.alloc_gemm_workspace(torch.device("cuda"))
    a = B.moe_grouped_gemm_mxfp4(*args, B.EPI_BF16, m_total=R)
    b = B.moe_grouped_gemm_mxfp4(*args, B.EPI_BF16, m_total=R, workspace=ws)
    B.sync_status()
    rows = torch.from_numpy(pos).cuda()
    assert torch.equal(a[rows], b[rows]) and not ws.any().item()
    U.check_close(b.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="MXFP4 GEMM, dynamic schedule")


@pytest.mark.parametrize("tile_n", [(0, 0), (-1, -1), (-2, -2), (128, 128)],
                         ids=["autotuned", "token-major", "pairs", "weight-rows-as-M"])
def test_layer_mx_all_tokens_on_two_experts(B, tile_n):
    """MXFP4 counterpart of the most skewed routing case: every one of 600
    tokens on experts 3 and 11 of 16 (a +8 bias), ragged last tiles in each
    orientation, 14 empty experts, a half K stage in the down GEMM."""
    w = W.Workload("two_hot", T=600, E=16, k=2, H=512, I=384, score="sigmoid")
    inp = W.host_inputs(w, seed=12)
    bias = np.zeros(w.E, np.float32)
    bias[[3, 11]] = 8.0
    cuda = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(cuda), inp["w_d"].to(cuda), w.k, w.score, True, w.h_scale,
                       bias=torch.from_numpy(bias).to(cuda), fmt="mxfp4", tile_n=tile_n)
    out = layer(inp["x"].to(cuda), inp["logits"].to(cuda)).float().cpu().numpy()
    B.sync_status()
    counts = layer.perm.counts.cpu().numpy()
    assert counts[3] == counts[11] == w.T and counts.sum() == w.T * w.k
    gq = U.oracle_quantize_experts_mx(inp["w_gu"])
    dq = U.oracle_quantize_experts_mx(inp["w_d"])
    ref = O.moe_layer_mx(inp["x"].float().numpy(), inp["logits"].numpy(), bias, gq[0], gq[1], dq[0], dq[1], w.k,
                         w.score)
    U.check_close(out, ref, what=f"MXFP4 layer output, tiles {tile_n}")
