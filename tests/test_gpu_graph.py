"""A forward+backward captured into a CUDA graph and replayed gives bitwise the results of the same
calls made directly: the launches take everything they need from their arguments (tensor maps
encoded on the host, tile-scheduler counters that every launch resets, the workspace header
cleared by a memset node), so a training step can replay the whole strip loop without host work."""

import pytest
import torch

from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,mode", [("n4096-d2048-v151936", "exact"),
                                       ("n32768-d6144-v151552-outliers", "exact"),
                                       ("tiny-fp32", "tf32x3")],
                         ids=["bf16-overlapped", "bf16", "tf32x3"])
def test_forward_backward_replay_in_cuda_graph(cuda_lib, name, mode):
    base = WORKLOADS[name]
    w = base.with_sizes(N=700, d=192, V=3000, strip_V=1024)
    if name.startswith("n32768"):
        w = base.with_sizes(N=4352, d=8192, V=1500, strip_V=512)  # 17 x 32 dH tiles: large steps
    H, W, y = make_inputs(w, "cuda")
    N, d, V = w.N, w.d, w.V
    dt = "tf32x3" if mode == "tf32x3" else w.dtype
    ws = torch.empty(api.lce_workspace_size(N, d, V, w.strip_V, dt), dtype=torch.uint8,
                     device="cuda")
    loss = torch.empty((), device="cuda")
    lse = torch.empty(N, device="cuda")
    nv = torch.empty((), dtype=torch.int64, device="cuda")
    dH = torch.empty(N, d, device="cuda")
    dW = torch.empty(V, d, device="cuda")
    one = torch.ones((), device="cuda")

    def step():
        api.lce_forward(H, W, y, strip_V=w.strip_V, reduction=w.reduction, workspace=ws,
                        out=(loss, lse, nv), f32_mode=mode)
        api.lce_backward(H, W, y, lse, nv, one, strip_V=w.strip_V, reduction=w.reduction,
                         workspace=ws, dH=dH, dW=dW, f32_mode=mode)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # direct calls (also the first launch of every kernel, before any capture)
    torch.cuda.current_stream().wait_stream(side)
    api.lce_check_error(ws)
    ref = [t.clone() for t in (loss, lse, nv, dH, dW)]

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in (loss, lse, dH, dW):
        t.fill_(float("nan"))
    nv.fill_(-1)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        api.lce_check_error(ws)
        for a, b in zip((loss, lse, nv, dH, dW), ref):
            assert torch.equal(a, b)
