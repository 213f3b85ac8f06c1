"""Token-major tiles on a CTA pair (tile_n = TILE_TOKEN_MAJOR_PAIR): two
CTAs on neighbouring SMs run one 256-token x 256-weight-row tile with
cta_group::2 MMAs, each SM staging 128 tokens and one of the two weight
tiles.  Checked against the oracle like the single-SM orientations, on
shapes that leave the second CTA's token half partial or empty, put several
pair tiles on one expert, leave experts empty and end K in a partial stage,
with row-major and tiled weights, NVFP4 and MXFP4, every epilogue."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U
from tests.test_gpu_kernels import gemm_case, dev
from tests.test_gpu_mxfp4 import gemm_case_mx

pytestmark = pytest.mark.gpu

PAIR = -2   # binding.TILE_TOKEN_MAJOR_PAIR

PAIR_SHAPES = [
    # E, N, K, counts
    (3, 256, 256, [5, 0, 40]),                    # second CTA's half empty in every tile
    (2, 512, 1024, [300, 17]),                    # 256 + a 44-row pair tile; a 17-row one
    (8, 256, 768, [0, 1, 2, 3, 130, 0, 31, 257]),  # 130: the second half holds 2 rows; 257: one row past a tile
    (2, 768, 320, [128, 129]),                    # partial last K stage; exactly one half; one row into the second
    (3, 512, 512, [256, 512, 600]),               # whole pair tiles
]


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    assert binding.TILE_TOKEN_MAJOR_PAIR == PAIR
    return binding


@pytest.mark.parametrize("tiled", [False, True])
@pytest.mark.parametrize("E,N,K,counts", PAIR_SHAPES)
def test_pair_bf16(B, E, N, K, counts, tiled):
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=E * 1900 + K)
    w = B.tile_expert_weights(g["w_packed"]) if tiled else g["w_packed"]
    out = B.moe_grouped_gemm_nvfp4(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"], w,
                                   g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=R, tile_n=PAIR)
    B.sync_status()
    U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="bf16 GEMM, CTA pair")


@pytest.mark.parametrize("tiled", [False, True])
@pytest.mark.parametrize("E,I,K,counts", [(3, 128, 512, [9, 70, 0]), (2, 256, 320, [130, 1]),
                                          (4, 128, 1024, [128, 5, 300, 200]), (2, 384, 256, [256, 41])])
def test_pair_swiglu(B, E, I, K, counts, tiled):
    g, ref, pos, R = gemm_case(E, 2 * I, K, counts, seed=E * 907 + K)
    h_ref = O.swiglu(ref, I)
    w = B.tile_expert_weights(g["w_packed"]) if tiled else g["w_packed"]
    args = (g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"], w, g["w_scales"],
            g["w_gscale"])
    hf = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_F32, m_total=R, tile_n=PAIR)
    s_h = np.float32(2.0 ** -4)
    hq, hs = B.moe_grouped_gemm_nvfp4(*args, B.EPI_SWIGLU_NVFP4, c_gscale=dev(torch.tensor([s_h])), m_total=R,
                                      tile_n=PAIR)
    B.sync_status()
    U.check_close(hf.cpu().numpy()[pos], h_ref, frob_tol=1e-5, elem_tol=1e-4, what="SwiGLU float32, CTA pair")
    rq, rs = O.quantize_nvfp4(h_ref.astype(np.float32), s_h)
    cap = hq.shape[0]
    U.check_requant(O.unpack_codes(hq.cpu().numpy()[pos]), U.from_blocked(hs.cpu().numpy(), cap, I)[pos],
                    O.unpack_codes(rq), rs)


@pytest.mark.parametrize("E,N,K,counts", [(3, 256, 256, [5, 0, 40]), (2, 256, 1024, [300, 17]),
                                          (4, 512, 384, [1, 33, 264, 129])])
def test_pair_mx_bf16(B, E, N, K, counts):
    g, ref, pos, R = gemm_case_mx(E, N, K, counts, seed=E * 190 + K)
    out = B.moe_grouped_gemm_mxfp4(g["a_packed"], g["a_scales"], g["counts"], g["row_offsets"], g["w_packed"],
                                   g["w_scales"], B.EPI_BF16, m_total=R, tile_n=PAIR)
    B.sync_status()
    U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="MXFP4 bf16 GEMM, CTA pair")


@pytest.mark.parametrize("E,I,K,counts", [(3, 128, 512, [9, 70, 0]), (2, 256, 384, [130, 300])])
def test_pair_mx_swiglu(B, E, I, K, counts):
    g, ref, pos, R = gemm_case_mx(E, 2 * I, K, counts, seed=E * 37 + K)
    h_ref = O.swiglu(ref, I)
    args = (g["a_packed"], g["a_scales"], g["counts"], g["row_offsets"], g["w_packed"], g["w_scales"])
    hf = B.moe_grouped_gemm_mxfp4(*args, B.EPI_SWIGLU_F32, m_total=R, tile_n=PAIR)
    hq, hs = B.moe_grouped_gemm_mxfp4(*args, B.EPI_SWIGLU_MXFP4, m_total=R, tile_n=PAIR)
    B.sync_status()
    U.check_close(hf.cpu().numpy()[pos], h_ref, frob_tol=1e-5, elem_tol=1e-4, what="MXFP4 SwiGLU float32, CTA pair")
    rq, rs = O.quantize_mxfp4(h_ref.astype(np.float32))
    cap = hq.shape[0]
    U.check_requant(O.unpack_codes(hq.cpu().numpy()[pos]), U.from_blocked(hs.cpu().numpy(), cap, I, 32)[pos],
                    O.unpack_codes(rq), rs, block=32)


def test_pair_all_experts_empty(B):
    """No tiles at all: every pair finds the end marker at once and exits."""
    E, N, K = 4, 512, 256
    g, ref, pos, R = gemm_case(E, N, K, [0, 0, 0, 0], seed=5)
    out = B.moe_grouped_gemm_nvfp4(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"],
                                   g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=0, tile_n=PAIR)
    B.sync_status()
    assert out.shape[1] == N


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_pair_layer_matches_oracle(B, fmt):
    """The whole layer with both GEMMs on CTA pairs against the oracle layer."""
    w = W.TEST_WORKLOADS["wide_experts"]          # 300 tokens, 4 experts, k = 2: ~150 rows per expert
    inp = W.host_inputs(w, seed=3)
    d = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(d), inp["w_d"].to(d), w.k, w.score, w.renormalize, w.h_scale,
                       tile_n=(PAIR, PAIR), fmt=fmt)
    out = layer(inp["x"].to(d), inp["logits"].to(d)).float().cpu().numpy()
    B.sync_status()
    x32, lg = inp["x"].float().numpy(), inp["logits"].numpy()
    if fmt == "mxfp4":
        gp, gs = U.oracle_quantize_experts_mx(inp["w_gu"])
        dp, ds = U.oracle_quantize_experts_mx(inp["w_d"])
        ref = O.moe_layer_mx(x32, lg, None, gp, gs, dp, ds, w.k, w.score, w.renormalize)
    else:
        ref = O.moe_layer(x32, lg, None, *U.oracle_quantize_experts(inp["w_gu"]),
                          *U.oracle_quantize_experts(inp["w_d"]), w.k, w.score, np.float32(w.h_scale), w.renormalize)
    U.check_close(out, ref, what=f"{fmt} layer, CTA pairs")
