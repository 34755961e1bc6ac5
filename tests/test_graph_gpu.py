"""The Ulysses step captured in a CUDA graph and replayed: the library's calls only
enqueue work on the current stream (no allocation, no host synchronisation), so a whole
forward + backward can be captured once and replayed.  Replay runs the same kernels on
the same inputs: o, dk, dv equal the eager step's bit for bit, dq (fp32 additions in
any order) within the gradient bar."""
import pytest
import torch

from gpu_util import check_grad, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import UlyssesAttention, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_equals_eager(fused):
    need_gpu()
    w = workloads.Workload("graph", 97, b=1, h=8, d=128, s=2048, N=4, causal=True, scale=1.0)
    ins = workloads.make_inputs(w, device="cuda")
    step = UlyssesAttention(w.N, w.b, w.s, w.h, w.d, w.causal, fused=fused)

    def one_step():
        step.forward(ins["q"], ins["k"], ins["v"])
        step.backward(ins["dout"])

    one_step()
    torch.cuda.synchronize()
    check_status()
    eager = [t.clone() for t in (step.o, step.dq, step.dk, step.dv)]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            one_step()
    torch.cuda.current_stream().wait_stream(side)
    for t in (step.o, step.dq, step.dk, step.dv):
        t.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    check_status()
    for name, a, b in zip(("o", "dk", "dv"), (eager[0], eager[2], eager[3]),
                          (step.o, step.dk, step.dv)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
    check_grad(f64(step.dq), f64(eager[1]), "dq")
