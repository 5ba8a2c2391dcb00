"""The layer inside a CUDA graph: every call of the C ABI only enqueues work
on the caller's stream (kernel launches, memsets; tensor maps are encoded on
the host into the kernel parameters), so a whole forward + backward step can
be captured once and replayed.  A replay with new input values copied into the
captured buffers must give, bit for bit, what the eager calls give."""

import pytest
import torch

import synth_inputs as si

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_graph_replay_equals_eager(precision):
    from mixture_experts_layer_17_gb300 import MoeLayer
    sh = si.custom_shape(517, 512, 384, 16, 4, seed=71, precision=precision)
    inp = si.make_inputs(sh, "cuda")
    other = si.make_inputs(si.custom_shape(517, 512, 384, 16, 4, seed=72, precision=precision),
                           "cuda")
    W = (inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"])
    layer = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, precision)
    x = inp["x"].clone()
    dY = inp["dY"].clone()
    y = torch.empty_like(x)
    grads = {"dx": torch.empty_like(x), "dW_r": torch.empty_like(W[0]),
             "dW_gate": torch.empty_like(W[1]), "dW_up": torch.empty_like(W[2]),
             "dW_down": torch.empty_like(W[3])}

    def step():
        layer.forward(x, *W, y=y)
        layer.backward(x, *W, dY, grads=grads)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                       # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    # replay on other inputs, compare with eager calls on the same inputs
    x.copy_(other["x"])
    dY.copy_(other["dY"])
    graph.replay()
    torch.cuda.synchronize()
    got = {"y": y.clone(), **{k: v.clone() for k, v in grads.items()}}
    step()
    torch.cuda.synchronize()
    assert layer.device_status("fwd") == 0 and layer.device_status("bwd") == 0
    assert torch.equal(got["y"], y)
    for k, v in grads.items():
        assert torch.equal(got[k], v), k
