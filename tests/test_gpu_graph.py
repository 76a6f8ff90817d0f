"""The fused forward captured in a CUDA graph and replayed (GB300).

moe_layer_forward forks the shared expert onto a second stream with events and joins
it before the combine, allocates nothing and never synchronises with the host, so a
stream capture of the caller's stream takes in both streams' launches.  A replay with
new x in the captured input buffer must give the same y, bit for bit, as an eager
call on that x, and a second replay the same again.
"""
import pytest
import torch

import routing_shared_expert_gb300 as moe
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

SHAPES = {
    # bf16: tensor-core router, CTA-pair (olmo_g) and one-SM (dsv3_g) expert tiles, a
    # learned shared gate (qwen2_g); fp32: the CUDA-core path
    "olmo_g": CONFIGS["olmo"].replace(T=1100, d_model=448, N=4, K=2, alpha=2.0, d_expert=320,
                                      d_shared=192),
    "dsv3_g": CONFIGS["dsv3"].replace(T=600, d_model=448, d_expert=128, d_shared=128),
    "qwen2_g": CONFIGS["qwen2"].replace(T=777, d_model=256, d_expert=200, d_shared=320),
    "tiny": CONFIGS["tiny"],
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_forward_graph_replay(name):
    spec = SHAPES[name]
    inp = make_inputs(spec, "cuda")
    x2 = make_inputs(spec.replace(N=1, d_expert=64, d_shared=0), "cuda", seed=7)["x"]
    layer = moe.MoELayer(moe.config_from_spec(spec), inp, "cuda")
    x_static = inp["x"].clone()

    # eager references for both inputs
    y1 = layer.forward(inp["x"]).clone()
    y2 = layer.forward(x2).clone()
    torch.cuda.synchronize()
    assert layer.status() == 0

    # warm-up on a side stream, then capture one forward of the static input buffer
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(x_static)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        y_graph = layer.forward(x_static)

    x_static.copy_(x2)
    graph.replay()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y_graph, y2), f"{name}: graph replay on x2 differs from the eager call"

    x_static.copy_(inp["x"])
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y1), f"{name}: second replay differs from the eager call"
