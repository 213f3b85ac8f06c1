"""The whole layer captured into one CUDA graph (MoELayer.capture) replays
exactly the eager forward: the same outputs bit for bit, on the captured
inputs and on new inputs copied into the same tensors.  This checks that no
step of the path synchronises the host, allocates, or bakes per-call host
state (tensor maps, launch plans, tile-scheduler counters, the prepare
kernel's barrier words) into a launch in a way that goes stale on replay.
The eager forward itself is pinned to the oracle in test_gpu_layer."""
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


CASES = [("ragged_small", "nvfp4", None), ("many_experts", "nvfp4", None), ("zipf_small", "nvfp4", None),
         ("ragged_small", "mxfp4", None), ("many_experts", "nvfp4", 2)]


@pytest.mark.parametrize("name,fmt,k_primary", CASES, ids=lambda v: str(v))
def test_graph_replay_matches_eager(B, name, fmt, k_primary):
    w = W.TEST_WORKLOADS[name]
    cuda = torch.device("cuda")
    a = W.device_inputs(w, seed=5, device=cuda)
    b = W.device_inputs(w, seed=6, device=cuda, with_weights=False)
    layer = B.MoELayer(a["w_gu"], a["w_d"], w.k, w.score, w.renormalize, w.h_scale, bias=a["bias"], T=w.T,
                       fmt=fmt, k_primary=k_primary)
    x, lg = a["x"].clone(), a["logits"].clone()
    graph = layer.capture(x, lg)
    for inp in (a, b):
        want = layer(inp["x"], inp["logits"]).clone()   # eager, on the inputs' own tensors
        layer.out.fill_(7)
        x.copy_(inp["x"])
        lg.copy_(inp["logits"])
        graph.replay()
        torch.cuda.synchronize()
        B.sync_status()
        assert torch.equal(layer.out.view(torch.int16), want.view(torch.int16)), f"{name} {fmt}: replay differs"
