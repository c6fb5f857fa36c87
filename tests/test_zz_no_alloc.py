"""The forward entry point that allocates nothing (lce_forward_static_scratch).

It exists for callers that may not call cudaMalloc themselves -- an engine plugin that only gets
the buffers its host planned, code enqueuing work during CUDA-graph capture, latency-critical code
that cannot take an allocation's device synchronisation.  This test calls it through the C ABI,
twice in a row on the same device (the library's scratch array keeps the first call's contents
when the second call starts), and checks each call's outputs against the workspace-taking
lce_forward within the bf16 tolerances used by the other parity tests.  This file is collected
last so that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from memory_bounded_linear_gb300 import _lib, api
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # LCE_STATIC_SCRATCH_BYTES in include/lce.h


def _static_forward(lib, H, W, y, strip_V, reduction):
    N, d = H.shape
    V = W.shape[0]
    loss = torch.full((), float("nan"), device="cuda")
    lse = torch.full((N,), float("nan"), device="cuda")
    nv = torch.full((), -1, dtype=torch.int64, device="cuda")
    flags = torch.full((1,), 0x7F7F7F7F, dtype=torch.int32, device="cuda")
    st = lib.lce_forward_static_scratch(
        H.data_ptr(), W.data_ptr(), y.data_ptr(), N, d, V, -100, strip_V,
        _lib.REDUCTIONS[reduction], _lib.DTYPES["bf16"], loss.data_ptr(), lse.data_ptr(),
        nv.data_ptr(), flags.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, loss.item(), lse.cpu().double().numpy(), int(nv.item()), int(flags.item())


def test_static_scratch_forward_matches_workspace_forward(cuda_lib):
    lib = _lib.load()
    w = WORKLOADS["n16384-d4096-v131072-ignore10"].with_sizes(N=1000, d=256, V=3001,
                                                               strip_V=1024)
    assert api.lce_workspace_size(w.N, w.d, w.V, w.strip_V) <= SCRATCH_BYTES
    H, W, y = make_inputs(w, "cuda", seed=3)

    ref_loss, ref_lse, ref_nv, ws = api.lce_forward(H, W, y, strip_V=w.strip_V,
                                                    reduction=w.reduction)
    api.lce_check_error(ws)
    ref_loss = ref_loss.item()
    ref_lse = ref_lse.cpu().double().numpy()
    ref_nv = int(ref_nv.item())

    for call in range(2):
        st, loss, lse, nv, flags = _static_forward(lib, H, W, y, w.strip_V, w.reduction)
        assert st == 0, (call, _lib.STATUS_NAMES.get(st))
        assert flags == 0
        assert nv == ref_nv
        assert abs(loss - ref_loss) <= 1e-3 * abs(ref_loss)
        assert np.max(np.abs(lse - ref_lse) / np.abs(ref_lse)) <= 1e-3

    # a shape whose workspace does not fit the array is refused before anything is enqueued
    big_N = SCRATCH_BYTES // (2 * 1024) + 1
    st = lib.lce_forward_static_scratch(H.data_ptr(), W.data_ptr(), y.data_ptr(), big_N, w.d,
                                        w.V, -100, 1024, 0, 0, None, None, None, None, None)
    assert _lib.STATUS_NAMES[st] == "LCE_ERR_WORKSPACE_TOO_SMALL"
