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


def test_two_problems_on_two_streams_at_once():
    """Two independent problems (different shapes, chunking and the CTA-pair
    and one-CTA schedules among their GEMMs), each with its own workspace,
    launched on two streams so that their kernels overlap, give bitwise the
    results of running them one after the other: the library keeps no state
    between calls that concurrent calls could share."""
    from lm_head_jsd_gb300 import FusedLinearJSD

    specs = [("conc_a", 81, 1024, 256, 20000, 0.5, 1.0, 0),
             ("conc_b", 82, 640, 128, 33001, 0.0, 2.0, 256)]
    runs, inputs, seq = [], [], []
    for name, seed, bt, h, v, beta, t, chunk in specs:
        w = jsd_inputs.custom(name, seed, bt, h, v, "bf16", ignore_frac=0.1)
        inp = tuple(x.cuda() for x in jsd_inputs.make_inputs(w, "cpu"))
        run = FusedLinearJSD(bt, h, h, v, torch.bfloat16, beta=beta, temperature=t,
                             chunk_rows=chunk)
        out = run.forward(*inp)
        torch.cuda.synchronize()
        runs.append(run)
        inputs.append(inp)
        seq.append([o.clone() for o in out])
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [r.alloc_outputs() for r in runs]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(3):
        for o in outs:
            for x in o:
                x.fill_(float("nan"))
        for run, inp, o, s in zip(runs, inputs, outs, streams):
            with torch.cuda.stream(s):
                run.forward(*inp, out=o, stream=s)
        torch.cuda.synchronize()
        for ref, o in zip(seq, outs):
            for a, b in zip(ref, o):
                assert torch.equal(a, b), f"repeat {rep}"
