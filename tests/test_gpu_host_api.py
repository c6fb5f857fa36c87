"""The host-buffer entry point (lce_forward_backward_host): inputs and results in host memory, one
caller-owned device buffer.  Through the C ABI, its results must be bitwise those of
lce_forward + lce_backward on device copies of the same inputs (the same kernels run on the same
values), for every input format and both backward schedules, and match the float64 oracle;
device-side errors come back through the flags output; results not asked for are not copied;
two calls in flight on two streams with two buffers do not disturb each other."""

import numpy as np
import pytest
import torch

from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

from ._parity import assert_parity, run_oracle

pytestmark = pytest.mark.gpu

W2 = WORKLOADS["n4096-d2048-v151936"]
W3 = WORKLOADS["n16384-d4096-v131072-ignore10"]
WT = WORKLOADS["tiny-fp32"]

CASES = [
    (W3.with_sizes(N=517, d=256, V=2048, strip_V=512), "exact"),     # bf16, overlapped backward
    (W2.with_sizes(N=4352, d=8192, V=700, strip_V=512), "exact"),    # bf16, separate launches
    (WT.with_sizes(N=300, d=136, V=1000, strip_V=384), "exact"),     # fp32 on the CUDA cores
    (WT.with_sizes(N=300, d=136, V=1000, strip_V=384, reduction="sum"), "tf32x3"),
]
IDS = ["bf16-overlap", "bf16-large-step", "f32", "tf32x3-sum"]


def _host_outputs(N, d, V):
    return {"loss": torch.full((), float("nan")).pin_memory(),
            "lse": torch.full((N,), float("nan")).pin_memory(),
            "n_valid": torch.full((), -1, dtype=torch.int64).pin_memory(),
            "dH": torch.full((N, d), float("nan")).pin_memory(),
            "dW": torch.full((V, d), float("nan")).pin_memory(),
            "flags": torch.full((1,), 0x7F7F7F7F, dtype=torch.int32).pin_memory()}


def _host_run(H, W, y, w, mode, skip=(), stream=None, buffer=None, outs=None, after=None,
              done=None):
    dt = "tf32x3" if (w.dtype == "f32" and mode == "tf32x3") else w.dtype
    N, d, V = w.N, w.d, w.V
    if buffer is None:
        buffer = torch.empty(api.lce_host_buffer_size(N, d, V, w.strip_V, dt), dtype=torch.uint8,
                             device="cuda")
    outs = outs or _host_outputs(N, d, V)
    kw = {k: (None if k in skip else v) for k, v in outs.items()}
    # the pinned inputs and the device buffer must outlive the copies the call enqueued: they are
    # returned with the outputs and kept until the caller has synchronised
    pinned = (H.pin_memory(), W.pin_memory(), y.pin_memory(),
              torch.ones((), dtype=torch.float32).pin_memory())
    api.lce_forward_backward_host(*pinned, device_buffer=buffer, strip_V=w.strip_V,
                                  reduction=w.reduction, f32_mode=mode, stream=stream,
                                  compute_after=after, compute_done=done, **kw)
    outs["_keep"] = (pinned, buffer)
    return outs


def _device_run(H, W, y, w, mode):
    Hd, Wd, yd = H.cuda(), W.cuda(), y.cuda()
    loss, lse, nv, ws = api.lce_forward(Hd, Wd, yd, strip_V=w.strip_V, reduction=w.reduction,
                                        f32_mode=mode)
    dH, dW, _ = api.lce_backward(Hd, Wd, yd, lse, nv, torch.ones((), device="cuda"),
                                 strip_V=w.strip_V, reduction=w.reduction, workspace=ws,
                                 f32_mode=mode)
    torch.cuda.synchronize()
    return {"loss": loss.cpu(), "lse": lse.cpu(), "n_valid": nv.cpu(), "dH": dH.cpu(),
            "dW": dW.cpu()}


@pytest.mark.parametrize("w,mode", CASES, ids=IDS)
def test_host_entry_point_matches_device_entry_points_bitwise(cuda_lib, w, mode):
    H, W, y = make_inputs(w, "cpu", seed=11)
    out = _host_run(H, W, y, w, mode)
    torch.cuda.synchronize()
    ref = _device_run(H, W, y, w, mode)
    assert int(out["flags"].item()) == 0
    for k in ("loss", "lse", "n_valid", "dH", "dW"):
        assert torch.equal(out[k], ref[k]), k
    g = {"loss": out["loss"].item(), "lse": out["lse"].double().numpy(),
         "n_valid": int(out["n_valid"].item()), "dH": out["dH"].double().numpy(),
         "dW": out["dW"].double().numpy()}
    r = run_oracle(H, W, y, w.reduction)
    assert_parity(g, r, "tf32x3" if mode == "tf32x3" else w.dtype)


@pytest.mark.parametrize("w,mode", [CASES[0], CASES[3]], ids=["bf16", "tf32x3"])
def test_host_entry_point_reports_bad_label(cuda_lib, w, mode):
    H, W, y = make_inputs(w, "cpu", seed=12)
    y[3] = w.V
    y[w.N - 1] = -5
    out = _host_run(H, W, y, w, mode)
    torch.cuda.synchronize()
    assert int(out["flags"].item()) == 1
    r = run_oracle(H, W, y, w.reduction)
    assert int(out["n_valid"].item()) == r["n_valid"]
    assert torch.count_nonzero(out["dH"][[3, w.N - 1]]).item() == 0


def test_host_entry_point_skips_results_not_asked_for(cuda_lib):
    w, mode = CASES[0]
    H, W, y = make_inputs(w, "cpu", seed=13)
    out = _host_run(H, W, y, w, mode, skip=("lse", "dW", "flags"))
    torch.cuda.synchronize()
    ref = _device_run(H, W, y, w, mode)
    assert torch.isnan(out["lse"]).all() and torch.isnan(out["dW"]).all()
    assert int(out["flags"].item()) == 0x7F7F7F7F
    assert torch.equal(out["loss"], ref["loss"]) and torch.equal(out["dH"], ref["dH"])


def test_two_host_calls_in_flight_on_two_streams(cuda_lib):
    """Two calls, each with its own device buffer, enqueued on two streams back to back: each
    returns its own inputs' results."""
    w, mode = CASES[1]
    inputs = [make_inputs(w, "cpu", seed=s) for s in (21, 22)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for (H, W, y), st in zip(inputs, streams):
        outs.append(_host_run(H, W, y, w, mode, stream=st))
    torch.cuda.synchronize()
    for (H, W, y), out in zip(inputs, outs):
        ref = _device_run(H, W, y, w, mode)
        assert int(out["flags"].item()) == 0
        for k in ("loss", "lse", "dH", "dW"):
            assert torch.equal(out[k], ref[k]), k
    assert not np.array_equal(outs[0]["dW"].numpy(), outs[1]["dW"].numpy())


def test_host_calls_chained_by_compute_events(cuda_lib):
    """Four calls alternating between two streams and two buffers, each call's kernels waiting
    for the previous call's (compute_after / compute_done), as a pipelined caller runs them: every
    call returns its own inputs' results, and the kernels of consecutive calls do not overlap in
    time."""
    w, mode = CASES[0]
    inputs = [make_inputs(w, "cpu", seed=s) for s in (31, 32, 33, 34)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    done = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    dt = "bf16"
    buffers = [torch.empty(api.lce_host_buffer_size(w.N, w.d, w.V, w.strip_V, dt),
                           dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = []
    for i, (H, W, y) in enumerate(inputs):
        outs.append(_host_run(H, W, y, w, mode, stream=streams[i % 2], buffer=buffers[i % 2],
                              after=done[i - 1] if i else None, done=done[i]))
    torch.cuda.synchronize()
    for (H, W, y), out in zip(inputs, outs):
        ref = _device_run(H, W, y, w, mode)
        assert int(out["flags"].item()) == 0
        for k in ("loss", "lse", "dH", "dW"):
            assert torch.equal(out[k], ref[k]), k
    # each compute_done comes after the previous one
    for i in range(1, 4):
        assert done[i - 1].elapsed_time(done[i]) > 0.0


def _same(a, b):
    """Bitwise equality that treats NaN as equal to NaN (the mean loss of an empty batch)."""
    if a.shape != b.shape or not torch.equal(torch.isnan(a), torch.isnan(b)):
        return False
    return torch.equal(torch.nan_to_num(a, nan=0.0), torch.nan_to_num(b, nan=0.0))


@pytest.mark.parametrize("fmt,mode", [("bf16", "exact"), ("f32", "exact"), ("f32", "tf32x3")],
                         ids=["bf16", "f32", "tf32x3"])
def test_host_entry_point_degenerate_shapes(cuda_lib, fmt, mode):
    """An empty batch, one token, and a one-word vocabulary through the host entry point: every
    result bitwise that of the device entry points on the same inputs, no error flag, and the
    closed forms of those cases (no valid row: n_valid 0 and dW 0; V = 1: loss and gradients
    0 within rounding)."""
    base = W2 if fmt == "bf16" else WT
    for N, d, V in [(0, 64, 300), (1, 16, 2), (130, 24, 1)]:
        w = base.with_sizes(N=N, d=d, V=V, strip_V=128)
        H, W, y = make_inputs(w, "cpu", seed=3)
        out = _host_run(H, W, y, w, mode)
        torch.cuda.synchronize()
        ref = _device_run(H, W, y, w, mode)
        assert int(out["flags"].item()) == 0, (N, d, V)
        for k in ("loss", "lse", "n_valid", "dH", "dW"):
            assert _same(out[k], ref[k]), (N, d, V, k)
        if N == 0:
            assert int(out["n_valid"].item()) == 0 and torch.count_nonzero(out["dW"]).item() == 0
        if V == 1:  # zero up to the rounding of the base-2 log-sum-exp
            assert abs(out["loss"].item()) < 1e-6
            assert out["dH"].abs().max().item() < 1e-6 and out["dW"].abs().max().item() < 1e-6
