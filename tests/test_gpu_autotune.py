"""Grouped GEMM launches restricted to an expert row range, and the layer's
tile autotuner, which chooses among launch plans built from them.

A plan is a list of (tile_n, (min_rows, max_rows)) launches covering every
expert.  Every plan the autotuner may choose must compute the oracle's
layer (up to float32 summation order), and a launch must leave the rows of
experts outside its range untouched."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U
from tests.test_gpu_kernels import gemm_case, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


@pytest.mark.parametrize("hot_tile", [-1, -2])
def test_complementary_row_ranges_cover_every_expert(B, hot_tile):
    E, N, K, counts = 6, 512, 512, [300, 0, 3, 129, 128, 40]
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=808)
    args = (g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"], g["w_packed"],
            g["w_scales"], g["w_gscale"], B.EPI_BF16)
    out = torch.full((g["a_packed"].shape[0], N), 7.0, dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm_nvfp4(*args, m_total=R, tile_n=hot_tile, out=out, rows=(128, 2 ** 31 - 1))
    B.sync_status()
    # experts with fewer than 128 rows are untouched by the first launch
    roff = np.concatenate([[0], np.cumsum(U.ceil_to(np.array(counts), 128))])
    cold = np.concatenate([roff[e] + np.arange(c) for e, c in enumerate(counts) if c < 128]).astype(np.int64)
    assert torch.all(out[torch.from_numpy(cold).cuda()] == 7.0)
    B.moe_grouped_gemm_nvfp4(*args, m_total=R, tile_n=128, out=out, rows=(1, 128))
    B.sync_status()
    U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="bf16 GEMM over two row ranges")


def test_row_range_is_validated(B):
    E, N, K, counts = 2, 256, 256, [5, 40]
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=809)
    for rows in ((0, 10), (10, 5)):
        with pytest.raises(B.Nvfp4MoeError) as ei:
            B.moe_grouped_gemm_nvfp4(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"],
                                     g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=R, rows=rows)
        assert ei.value.status == B.ERR_INVALID_ARG


def _oracle_layer(w, inp, fmt):
    x32, lg = inp["x"].float().numpy(), inp["logits"].numpy()
    b = None if inp["bias"] is None else inp["bias"].numpy()
    if fmt == "mxfp4":
        gp, gs = U.oracle_quantize_experts_mx(inp["w_gu"])
        dp, ds = U.oracle_quantize_experts_mx(inp["w_d"])
        return O.moe_layer_mx(x32, lg, b, gp, gs, dp, ds, w.k, w.score, w.renormalize)
    return O.moe_layer(x32, lg, b, *U.oracle_quantize_experts(inp["w_gu"]), *U.oracle_quantize_experts(inp["w_d"]),
                       w.k, w.score, np.float32(w.h_scale), w.renormalize)


@pytest.mark.parametrize("name,fmt", [("zipf_small", "nvfp4"), ("wide_experts", "nvfp4"), ("zipf_small", "mxfp4")])
def test_every_candidate_plan_computes_the_oracle_layer(B, name, fmt):
    w = W.TEST_WORKLOADS[name]
    inp = W.host_inputs(w, seed=21)
    d = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(d), inp["w_d"].to(d), w.k, w.score, w.renormalize, w.h_scale,
                       bias=None if inp["bias"] is None else inp["bias"].to(d), T=w.T, fmt=fmt, autotune=False)
    ref = _oracle_layer(w, inp, fmt)
    x, lg = inp["x"].to(d), inp["logits"].to(d)
    gu_plans, down_plans = layer.candidate_plans("gate_up"), layer.candidate_plans("down")
    assert len(gu_plans) >= 4 and any(len(p) == 2 for p in gu_plans)
    for i in range(max(len(gu_plans), len(down_plans))):
        gu, dn = gu_plans[i % len(gu_plans)], down_plans[i % len(down_plans)]
        layer.prepare(x, lg)
        layer.gemm_gate_up(gu)
        layer.gemm_down(dn)
        out = layer.finalize().float().cpu().numpy()
        B.sync_status()
        U.check_close(out, ref, what=f"{name} {fmt} layer, plans {gu} / {dn}")


def test_autotuner_chooses_once_per_batch_size(B):
    w = W.TEST_WORKLOADS["zipf_small"]
    inp = W.host_inputs(w, seed=22)
    d = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(d), inp["w_d"].to(d), w.k, w.score, w.renormalize, w.h_scale,
                       bias=inp["bias"].to(d))
    assert layer.autotune_enabled and not layer.plans
    out = layer(inp["x"].to(d), inp["logits"].to(d)).float().cpu().numpy()
    B.sync_status()
    assert w.T in layer.plans
    gu, dn = layer.plans[w.T]
    assert gu in layer.candidate_plans("gate_up") and dn in layer.candidate_plans("down")
    U.check_close(out, _oracle_layer(w, inp, "nvfp4"), what="autotuned layer")
    chosen = layer.plans[w.T]
    layer(inp["x"].to(d), inp["logits"].to(d))
    assert layer.plans[w.T] is chosen                   # cached: no second tuning
    assert layer.launches_per_forward == 1 + len(gu) + len(dn) + 1
    # explicit tiles switch the tuner off
    fixed = B.MoELayer(inp["w_gu"].to(d), inp["w_d"].to(d), w.k, w.score, w.renormalize, w.h_scale,
                       bias=inp["bias"].to(d), tile_n=(128, 128))
    assert not fixed.autotune_enabled
