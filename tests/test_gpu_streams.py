"""Two layers on two CUDA streams at once give the same outputs, bit for
bit, as the same calls one after the other: every piece of per-call device
state (the prepare workspace and its barrier words, the GEMMs' tile-scheduler
counters, the permutation, the intermediate buffers) belongs to the layer
that owns it, so calls on different streams may overlap on the GPU.  (The
no-allocation permute's library-owned scratch is the one exception and is
documented as such; the layer does not use it.)"""
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


@pytest.mark.parametrize("names", [("zipf_small", "many_experts"), ("ragged_small", "ragged_small")],
                         ids=lambda v: "+".join(v))
def test_two_streams_match_sequential(B, names):
    cuda = torch.device("cuda")
    layers, inputs = [], []
    for i, name in enumerate(names):
        w = W.TEST_WORKLOADS[name]
        inp = W.device_inputs(w, seed=20 + i, device=cuda)
        layer = B.MoELayer(inp["w_gu"], inp["w_d"], w.k, w.score, w.renormalize, w.h_scale, bias=inp["bias"],
                           T=w.T)
        layer(inp["x"], inp["logits"])     # launch plans chosen (autotune synchronises) before the overlap
        layers.append(layer)
        inputs.append(inp)
    torch.cuda.synchronize()
    want = [L(inp["x"], inp["logits"]).clone() for L, inp in zip(layers, inputs)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in layers]
    outs = [[] for _ in layers]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for step in range(4):
        for L, inp, s, o in zip(layers, inputs, streams, outs):
            with torch.cuda.stream(s):
                o.append(L(inp["x"], inp["logits"]).clone())
    torch.cuda.synchronize()
    B.sync_status()
    for i, o in enumerate(outs):
        for step, got in enumerate(o):
            assert torch.equal(got.view(torch.int16), want[i].view(torch.int16)), f"layer {i}, step {step}"
