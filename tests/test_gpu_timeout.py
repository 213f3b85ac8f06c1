"""Bounded device waits end in a status, not a hang or a fault.

The library's wait limit is set from the host (nvfp4moe_set_wait_limit_us).
The self-test kernel waits, through the grouped GEMM's own bounded mbarrier
wait, for a phase that host inputs make impossible (an mbarrier expecting
two arrivals that receives one): the wait must give up after the limit,
the kernel must return without trapping, sync_status must report
ERR_TIMEOUT once, and the context must stay usable -- the next self-test
with a reachable phase and a full grouped GEMM and layer must then pass.
Nothing here can hang the GPU: the only wait that cannot complete is
bounded by a 1 ms limit (the default limit, 2 s, applies to everything
else)."""
import time

import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from tests import nvfp4_testutil as U
from tests.test_gpu_kernels import gemm_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    yield binding
    binding.set_wait_limit_us(0)


def test_wait_that_cannot_complete_times_out_and_the_context_survives(B):
    B.sync_status()                                   # nothing pending
    B.set_wait_limit_us(1000)
    try:
        assert B.wait_limit_us() == 1000
        t0 = time.perf_counter()
        B.wait_selftest(expected_arrivals=2, arrivals=1)
        with pytest.raises(B.Nvfp4MoeError) as ei:
            B.sync_status()
        elapsed = time.perf_counter() - t0
        assert ei.value.status == B.ERR_TIMEOUT
        assert elapsed < 1.0, f"the 1 ms wait took {elapsed:.3f} s"
        B.sync_status()                               # the flag was read and cleared
        B.wait_selftest(expected_arrivals=1, arrivals=1)
        B.sync_status()
    finally:
        B.set_wait_limit_us(0)
    assert B.wait_limit_us() == 2000000
    # the context is intact: a grouped GEMM still matches the oracle
    E, N, K, counts = 3, 256, 512, [5, 0, 140]
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=404)
    out = B.moe_grouped_gemm_nvfp4(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"], g["row_offsets"],
                                   g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_BF16, m_total=R)
    B.sync_status()
    U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what="GEMM after a timeout")


def test_short_limit_leaves_healthy_calls_alone(B):
    """A 100 ms limit is far above every wait a healthy call makes."""
    E, N, K, counts = 2, 512, 1024, [300, 17]
    g, ref, pos, R = gemm_case(E, N, K, counts, seed=405)
    B.set_wait_limit_us(100000)
    try:
        for tile in (0, B.TILE_TOKEN_MAJOR, B.TILE_TOKEN_MAJOR_PAIR):
            out = B.moe_grouped_gemm_nvfp4(g["a_packed"], g["a_scales"], g["a_gscale"], g["counts"],
                                           g["row_offsets"], g["w_packed"], g["w_scales"], g["w_gscale"], B.EPI_BF16,
                                           m_total=R, tile_n=tile)
            B.sync_status()
            U.check_close(out.float().cpu().numpy()[pos], O.round_to_bf16(ref), what=f"GEMM tile_n {tile}")
    finally:
        B.set_wait_limit_us(0)


def test_wait_limit_is_validated(B):
    with pytest.raises(B.Nvfp4MoeError) as ei:
        B.set_wait_limit_us(60000001)
    assert ei.value.status == B.ERR_INVALID_ARG
    with pytest.raises(B.Nvfp4MoeError):
        B.wait_selftest(expected_arrivals=0, arrivals=0)
    assert B.wait_limit_us() == 2000000
