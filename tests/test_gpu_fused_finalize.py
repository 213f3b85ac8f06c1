"""The finalize fused into the down GEMM's epilogue (NVFP4MOE_EPI_FINALIZE_F32):
each routed row's bf16 down projection, times its routing weight, is added
by float32 atomics into its token's row, and moe_finalize_f32 converts the
accumulator to bf16 and zeroes it.  Checked against the oracle at the GEMM
and layer level, in every tile orientation; the sum order of a token's k
rows is not fixed, so results are compared within the usual bar."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U
from tests.test_gpu_kernels import gemm_case, dev
from tests.test_gpu_autotune import _oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


@pytest.mark.parametrize("tile_n", [128, -1, -2])
@pytest.mark.parametrize("E,N,K,counts,k", [(4, 512, 512, [40, 0, 300, 60], 4), (3, 768, 256, [129, 128, 7], 2)])
def test_fused_finalize_gemm(B, tile_n, E, N, K, counts, k):
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=E * 31 + N + k)
    T = R // k
    assert T * k == R
    rng = np.random.default_rng(7)
    flat_of_row = rng.permutation(R).astype(np.int32)          # routed row -> flat id t * k + j
    cap = g["a_packed"].shape[0]
    p2f = np.full(cap, -1, np.int32)
    p2f[pos] = flat_of_row
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    acc = torch.zeros((T, N), dtype=torch.float32, device="cuda")
    B.moe_grouped_gemm_nvfp4_finalize(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"],
                                      g["w_packed"], g["w_scales"], g["w_gscale"], dev(torch.from_numpy(p2f)),
                                      dev(torch.from_numpy(w)), acc, m_total=R, tile_n=tile_n)
    out = B.moe_finalize_f32(acc)
    B.sync_status()
    assert not acc.any().item()                                 # zeroed for the next call
    y = O.round_to_bf16(ref)                                    # [R, N] in expert row order
    expect = np.zeros((T, N))
    np.add.at(expect, flat_of_row // k, w.reshape(-1)[flat_of_row][:, None] * y)
    U.check_close(out.float().cpu().numpy(), O.round_to_bf16(expect), what=f"fused finalize, tile_n {tile_n}")


@pytest.mark.parametrize("name,tile_n", [("zipf_small", (0, 0)), ("wide_experts", (-2, -2)), ("wide_experts", (0, 128))])
def test_fused_finalize_layer(B, name, tile_n):
    w = W.TEST_WORKLOADS[name]
    inp = W.host_inputs(w, seed=33)
    d = torch.device("cuda")
    layer = B.MoELayer(inp["w_gu"].to(d), inp["w_d"].to(d), w.k, w.score, w.renormalize, w.h_scale,
                       bias=None if inp["bias"] is None else inp["bias"].to(d), tile_n=tile_n, fused_finalize=True)
    ref = _oracle_layer(w, inp, "nvfp4")
    for _ in range(2):                                          # the accumulator is reused
        out = layer(inp["x"].to(d), inp["logits"].to(d)).float().cpu().numpy()
        B.sync_status()
        U.check_close(out, ref, what=f"{name} layer with the fused finalize")
    assert layer.y is None and not layer.acc.any().item()
