"""The forward and backward are stream-ordered and capturable: captured into a
CUDA graph on a side stream and replayed, they give bitwise the same results as
eager calls."""
import pytest
import torch

import jsd_inputs

pytestmark = pytest.mark.gpu


def test_forward_backward_in_a_cuda_graph():
    from lm_head_jsd_gb300 import FusedLinearJSD

    w = jsd_inputs.custom("graph", 71, 300, 128, 5000, "bf16", ignore_frac=0.1)
    x_s, w_s, x_t, w_t, labels = (t.cuda() for t in jsd_inputs.make_inputs(w, "cpu"))
    run = FusedLinearJSD(300, 128, 128, 5000, torch.bfloat16, beta=0.3, temperature=1.5)
    g_out = torch.full((1,), 0.5, device="cuda")
    eager = run.alloc_outputs()
    run.forward(x_s, w_s, x_t, w_t, labels, out=eager)
    run.backward(g_out, eager[1], eager[2])
    torch.cuda.synchronize()

    out = run.alloc_outputs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        run.forward(x_s, w_s, x_t, w_t, labels, out=out, stream=side)  # warm-up on the stream
        run.backward(g_out, out[1], out[2], stream=side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            run.forward(x_s, w_s, x_t, w_t, labels, out=out, stream=side)
            run.backward(g_out, out[1], out[2], stream=side)
    for _ in range(3):
        for t in out:
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for e, o in zip(eager, out):
            assert torch.equal(e, o)
