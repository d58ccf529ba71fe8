"""The library's calls are capture-safe: no allocation, no synchronisation and no host copies on
the stream, so the fused allreduce-mean (both quantise kernels) and the segmented form can be
recorded into a CUDA graph and replayed, with results bit-identical to the eager calls (a
launch-bound small problem is where replaying a graph pays)."""
import pytest

from gpu_common import EXP, INF, LINEAR, gq_module
from allreduce_compatible_gradient_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    return gq_module()


@pytest.mark.parametrize("n,d", [(4, 65_536), (8, 1_200_000)])  # direct-load and bulk-copy paths
@pytest.mark.parametrize("scheme,s,q", [(LINEAR, 15, 2), (EXP, 8, INF)])
def test_fused_call_in_a_graph(gq, n, d, scheme, s, q):
    import torch
    x = workloads.device_inputs("normal", n, d, seed=n)
    ws = gq.gq_workspace()
    out = torch.empty(d, device="cuda")
    norm = torch.empty(1, device="cuda")
    eager = gq.gq_allreduce_mean(x, q, q, scheme, s, 1, 9, ws=ws).clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        gq.gq_allreduce_mean(x, q, q, scheme, s, 1, 9, out=out, norm=norm, ws=ws, stream=stream)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gq.gq_allreduce_mean(x, q, q, scheme, s, 1, 9, out=out, norm=norm, ws=ws,
                             stream=torch.cuda.current_stream())
    for _ in range(3):
        out.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert gq.gq_get_status(ws) == 0


def test_segments_in_a_graph(gq):
    import torch
    sizes = workloads.resnet50_layer_sizes()[:40]
    segs = workloads.segment_tensors(8, sizes, seed=5)
    outs = [torch.empty(sz, device="cuda") for sz in sizes]
    ws = gq.gq_workspace()
    eager = [o.clone() for o in gq.gq_allreduce_mean_segments(segs, INF, INF, LINEAR, 127, 1, 2,
                                                               ws=ws)]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gq.gq_allreduce_mean_segments(segs, INF, INF, LINEAR, 127, 1, 2, outs=outs, ws=ws,
                                      stream=torch.cuda.current_stream())
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)
