"""moe_permute_no_alloc: the permutation on the library's own scratch, for
callers that cannot allocate device memory when they call (a fixed memory
arena, a plugin handed tensors but no allocator, a loop where cudaMalloc is
not acceptable).  Its outputs must equal those of moe_permute, which runs on
a caller-provided workspace, on two calls in a row (the second runs on
scratch left over from the first).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_07_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_block_scaled_07_gb300 import build
    build.build()
    from nvfp4_block_scaled_07_gb300 import binding
    binding.device_check()
    return binding


def _zeroed(B, T, E, k, H):
    p = B.alloc_permutation(T, E, k, H, torch.device("cuda"))
    for name in ("counts", "offsets", "row_offsets", "perm_to_flat", "flat_to_perm", "a_packed", "a_scales"):
        getattr(p, name).zero_()
    return p


def test_no_alloc_permute_matches_workspace_permute(B):
    # two calls in a row with different shapes; the second reuses the scratch of the first
    for T, E, k, H, seed in [(700, 16, 4, 128, 1), (128, 256, 8, 6144, 2), (16384, 64, 8, 256, 3)]:
        rng = np.random.default_rng(seed)
        idx = torch.from_numpy(W.random_routing(T, E, k, seed=seed)).cuda()
        xq = torch.from_numpy(rng.integers(0, 256, size=(T, H // 2), dtype=np.uint8)).cuda()
        xs = torch.from_numpy(rng.integers(0, 127, size=(T, H // 16), dtype=np.uint8)).cuda()
        ref = B.moe_permute(idx, E, xq, xs, out=_zeroed(B, T, E, k, H))
        got = B.moe_permute_no_alloc(idx, E, xq, xs, out=_zeroed(B, T, E, k, H))
        B.sync_status()
        for name in ("counts", "offsets", "row_offsets", "perm_to_flat", "flat_to_perm", "a_packed", "a_scales"):
            assert torch.equal(getattr(got, name), getattr(ref, name)), (T, E, name)


def test_no_alloc_permute_at_the_segment_counter_limit(B):
    # E = 1024, k = 8, T = 8192: 64 segments of 1024 routed rows x 1024
    # experts = 65536 per-segment counters, exactly the scratch's limit
    T, E, k, H = 8192, 1024, 8, 64
    rng = np.random.default_rng(4)
    idx = torch.from_numpy(W.random_routing(T, E, k, seed=4)).cuda()
    xq = torch.from_numpy(rng.integers(0, 256, size=(T, H // 2), dtype=np.uint8)).cuda()
    xs = torch.from_numpy(rng.integers(0, 127, size=(T, H // 16), dtype=np.uint8)).cuda()
    for _ in range(2):
        ref = B.moe_permute(idx, E, xq, xs, out=_zeroed(B, T, E, k, H))
        got = B.moe_permute_no_alloc(idx, E, xq, xs, out=_zeroed(B, T, E, k, H))
        B.sync_status()
        for name in ("counts", "offsets", "row_offsets", "perm_to_flat", "flat_to_perm", "a_packed", "a_scales"):
            assert torch.equal(getattr(got, name), getattr(ref, name)), name


def test_no_alloc_permute_rejects_one_segment_past_the_counter_limit(B):
    T, E, k, H = 8193, 1024, 8, 64         # 65 segments x 1024 experts = 66560 counters > 65536
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    xq = torch.zeros((T, H // 2), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((T, H // 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(B.Nvfp4MoeError) as ei:
        B.moe_permute_no_alloc(idx, E, xq, xs)
    assert ei.value.status == B.ERR_UNSUPPORTED
    assert "static scratch" in str(ei.value)


def test_no_alloc_permute_rejects_sizes_beyond_its_scratch(B):
    T, E, k, H = 16385, 64, 8, 64          # 131080 routed rows > 131072
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    xq = torch.zeros((T, H // 2), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((T, H // 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(B.Nvfp4MoeError) as ei:
        B.moe_permute_no_alloc(idx, E, xq, xs)
    assert ei.value.status == B.ERR_UNSUPPORTED
    assert "static scratch" in str(ei.value)
