"""The forward entry point that allocates nothing (lce_forward_static_scratch).

It exists for callers that may not call cudaMalloc themselves -- an engine plugin that only gets
the buffers its host planned, a service whose device memory budget is fixed at start-up,
latency-critical code that cannot take an allocation's cost or a free's device-wide
synchronisation.  These tests call it through the C ABI, twice in a row on the same device (the
library's scratch array keeps the first call's contents when the second call starts), and check
each call's outputs against the workspace-taking lce_forward within the tolerances of the other
parity tests, for each input format; a planted bad label must come back in the device error
flags; the device's free memory must not change across a call.  This file is collected last so
that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from memory_bounded_linear_gb300 import _lib, api
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

from ._parity import TOL, max_rel, run_oracle

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # LCE_STATIC_SCRATCH_BYTES in include/lce.h

# (input format of H and W, arithmetic): bf16 tensor cores, fp32 exact on the CUDA cores, fp32 as
# three tf32 products on the tensor cores
FORMATS = [("bf16", "bf16"), ("f32", "f32"), ("f32", "tf32x3")]


def _static_forward(lib, H, W, y, strip_V, reduction, dt):
    N, d = H.shape
    V = W.shape[0]
    loss = torch.full((), float("nan"), device="cuda")
    lse = torch.full((N,), float("nan"), device="cuda")
    nv = torch.full((), -1, dtype=torch.int64, device="cuda")
    flags = torch.full((1,), 0x7F7F7F7F, dtype=torch.int32, device="cuda")
    st = lib.lce_forward_static_scratch(
        H.data_ptr(), W.data_ptr(), y.data_ptr(), N, d, V, -100, strip_V,
        _lib.REDUCTIONS[reduction], _lib.DTYPES[dt], loss.data_ptr(), lse.data_ptr(),
        nv.data_ptr(), flags.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, loss.item(), lse.cpu().double().numpy(), int(nv.item()), int(flags.item())


def _workload(fmt):
    # six strips with a ragged tail; the tf32x3 workspace (13.9 MiB) also fits the array
    w = WORKLOADS["n16384-d4096-v131072-ignore10"].with_sizes(N=1000, d=256, V=3001,
                                                               strip_V=512)
    return w if fmt == "bf16" else w.with_sizes(dtype="f32")


@pytest.mark.parametrize("fmt,dt", FORMATS, ids=["bf16", "f32", "tf32x3"])
def test_static_scratch_forward_matches_workspace_forward(cuda_lib, fmt, dt):
    lib = _lib.load()
    w = _workload(fmt)
    tl = TOL[dt][0]
    assert api.lce_workspace_size(w.N, w.d, w.V, w.strip_V, dt) <= SCRATCH_BYTES
    H, W, y = make_inputs(w, "cuda", seed=3)

    mode = "tf32x3" if dt == "tf32x3" else "exact"
    ref_loss, ref_lse, ref_nv, ws = api.lce_forward(H, W, y, strip_V=w.strip_V,
                                                    reduction=w.reduction, f32_mode=mode)
    api.lce_check_error(ws)
    ref_loss = ref_loss.item()
    ref_lse = ref_lse.cpu().double().numpy()
    ref_nv = int(ref_nv.item())
    orc = run_oracle(H.cpu(), W.cpu(), y.cpu(), w.reduction)

    for call in range(2):
        st, loss, lse, nv, flags = _static_forward(lib, H, W, y, w.strip_V, w.reduction, dt)
        assert st == 0, (call, _lib.STATUS_NAMES.get(st))
        assert flags == 0
        assert nv == ref_nv == orc["n_valid"]
        assert abs(loss - ref_loss) <= tl * abs(ref_loss)
        assert max_rel(lse, ref_lse) <= tl
        assert abs(loss - orc["loss"]) <= tl * abs(orc["loss"])
        assert max_rel(lse, orc["lse"]) <= tl

    # a shape whose workspace does not fit the array is refused before anything is enqueued
    big_N = SCRATCH_BYTES // (2 * 1024) + 1
    st = lib.lce_forward_static_scratch(H.data_ptr(), W.data_ptr(), y.data_ptr(), big_N, w.d,
                                        w.V, -100, 1024, 0, _lib.DTYPES[dt], None, None, None,
                                        None, None)
    assert _lib.STATUS_NAMES[st] == "LCE_ERR_WORKSPACE_TOO_SMALL"


@pytest.mark.parametrize("fmt,dt", FORMATS, ids=["bf16", "f32", "tf32x3"])
def test_static_scratch_reports_bad_label(cuda_lib, fmt, dt):
    """A label outside [0, V) sets bit 0 of the returned device flags; that row is left out of the
    loss and n_valid, as in lce_forward; the next clean call reports 0 again."""
    lib = _lib.load()
    w = _workload(fmt)
    H, W, y = make_inputs(w, "cuda", seed=5)
    y_bad = y.clone()
    y_bad[7] = w.V
    y_bad[900] = -3
    st, loss, lse, nv, flags = _static_forward(lib, H, W, y_bad, w.strip_V, w.reduction, dt)
    assert st == 0
    assert flags == 1
    orc = run_oracle(H.cpu(), W.cpu(), y_bad.cpu(), w.reduction)
    assert nv == orc["n_valid"]
    tl = TOL[dt][0]
    assert abs(loss - orc["loss"]) <= tl * abs(orc["loss"])
    assert max_rel(lse, orc["lse"]) <= tl
    st, _, _, _, flags = _static_forward(lib, H, W, y, w.strip_V, w.reduction, dt)
    assert st == 0 and flags == 0


def test_static_scratch_call_allocates_nothing(cuda_lib):
    """After a first call on the device (its set-up), a call leaves the device's free memory
    unchanged: no allocation, no release."""
    lib = _lib.load()
    w = _workload("bf16")
    H, W, y = make_inputs(w, "cuda", seed=3)
    _static_forward(lib, H, W, y, w.strip_V, w.reduction, "bf16")
    N, d, V = w.N, w.d, w.V
    loss = torch.empty((), device="cuda")
    lse = torch.empty((N,), device="cuda")
    nv = torch.empty((), dtype=torch.int64, device="cuda")
    flags = torch.empty((1,), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        st = lib.lce_forward_static_scratch(
            H.data_ptr(), W.data_ptr(), y.data_ptr(), N, d, V, -100, w.strip_V,
            _lib.REDUCTIONS[w.reduction], _lib.DTYPES["bf16"], loss.data_ptr(), lse.data_ptr(),
            nv.data_ptr(), flags.data_ptr(),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(flags.item()) == 0 and np.isfinite(loss.item())
