"""Every launch plan of the grouped GEMMs computes the same numbers bit for bit.

The three tile orientations (weight rows as M with token tiles up to 128,
token-major 128 x 256 tiles on one SM, token-major 256 x 256 tiles on a CTA
pair) and the hot/cold splits of an expert row range over two launches all
form each output element as the same fp32 sum over the same K steps, so the
SwiGLU requantisation (codes and block scales), the bf16 down rows and the
layer output must agree exactly with the reference plan (weight rows as M).
This checks the tilings' pipelines (stage rings, scale slots, tile maps)
against one another at sizes where the oracle would be slow: a scale block
read from the wrong stage or a slot overwritten before it was read changes
whole token tiles while every plan still looks plausible on its own.  The
oracle pins the reference plan elsewhere (test_gpu_kernels, test_gpu_pair,
test_gpu_fullsize)."""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_07_gb300 import workloads as W
from tests import nvfp4_testutil as U

pytestmark = pytest.mark.gpu

ALL = (1, 2 ** 31 - 1)
# plans as (gate/up plan, down plan), each a list of (tile_n, (min_rows, max_rows))
PLANS = {
    "token-major": ([(-1, ALL)], [(-1, ALL)]),
    "pairs": ([(-2, ALL)], [(-2, ALL)]),
    "pairs gate/up, token-major down": ([(-2, ALL)], [(-1, ALL)]),
    "hot pairs, cold weight rows as M": ([(-2, (512, ALL[1])), (128, (1, 512))],
                                         [(-2, (512, ALL[1])), (128, (1, 512))]),
    "hot token-major, cold weight rows as M": ([(-1, (96, ALL[1])), (128, (1, 96))],
                                               [(-1, (96, ALL[1])), (128, (1, 96))]),
}

CASES = {
    # 2048 rows per expert: several pair tiles per expert, 28 / 16 K stages per tile
    "prefill_e8": W.PROFILE_WORKLOADS["profile_prefill_e8"],
    # Zipf-skewed routing: hot experts with many token tiles next to cold ones with a few rows
    "skewed_e32": W.Workload("skewed_e32", T=1024, E=32, k=8, H=2048, I=1536, score="sigmoid", zipf_s=1.1),
}


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


def snapshot(L, w):
    """Valid rows of h (codes, block scales) and y, and the layer output."""
    counts = L.perm.counts.cpu().numpy()
    offs = L.perm.row_offsets.cpu().numpy()
    rows = np.concatenate([np.arange(o, o + c) for o, c in zip(offs, counts)])
    hq = L.hq.cpu().numpy()[rows]
    hs = U.from_blocked(L.hs.cpu().numpy(), L.perm.rows_capacity, w.I)[rows]
    y = L.y.cpu().view(torch.int16).numpy()[rows]
    return rows, hq, hs, y, L.out.cpu().view(torch.int16).numpy().copy()


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request, B):
    w = CASES[request.param]
    inp = W.device_inputs(w, seed=3, device=torch.device("cuda"))
    L = B.MoELayer(inp["w_gu"], inp["w_d"], w.k, w.score, w.renormalize, w.h_scale, bias=inp["bias"], T=w.T,
                   tile_n=(128, 128), autotune=False)
    L(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    B.sync_status()
    ref = snapshot(L, w)
    yield w, L, ref
    del L, inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("plan", sorted(PLANS))
def test_plan_matches_reference_bit_for_bit(B, case, plan):
    w, L, ref = case
    gu, dn = PLANS[plan]
    for buf in (L.hq, L.hs, L.y):
        buf.fill_(0x55 if buf.dtype == torch.uint8 else 7)   # stale values must not pass
    L.gemm_gate_up(gu)
    L.gemm_down(dn)
    L.finalize()
    torch.cuda.synchronize()
    B.sync_status()
    rows, hq, hs, y, out = snapshot(L, w)
    assert np.array_equal(rows, ref[0])
    for what, got, want in (("h codes", hq, ref[1]), ("h scales", hs, ref[2]), ("down rows", y, ref[3]),
                            ("layer output", out, ref[4])):
        bad = np.nonzero(np.any(got.reshape(len(got), -1) != want.reshape(len(want), -1), axis=1))[0]
        assert bad.size == 0, f"{plan}: {what} differ in {bad.size} of {len(got)} rows, first {bad[:8]}"
