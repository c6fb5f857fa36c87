"""The kernels' timeout path, exercised without faulting or hanging the GPU: a launch whose first
operand load is withheld (a barrier nothing will complete) must give up after its 2 s wait limit,
report LCE_ERR_TIMEOUT through the workspace, and leave the context fully usable."""

import time

import pytest
import torch

from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300._lib import LceError
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

from ._parity import parity_case

pytestmark = pytest.mark.gpu

W2 = WORKLOADS["n4096-d2048-v151936"]
WT = WORKLOADS["tiny-fp32"]
# (workload sizes, f32_mode): bf16 operands, and fp32 operands as tf32 parts on the tensor cores
FORMATS = [(W2.with_sizes(N=600, d=128, V=1100, strip_V=512), "exact"),
           (WT.with_sizes(N=600, d=128, V=1100, strip_V=512), "tf32x3")]


@pytest.mark.parametrize("fmt", [0, 1], ids=["bf16", "tf32x3"])
@pytest.mark.parametrize("cfg", [1, 2], ids=["single-cta", "cta-pair"])
def test_withheld_load_times_out_and_context_stays_usable(cuda_lib, cfg, fmt):
    w, mode = FORMATS[fmt]
    H, W, y = make_inputs(w, "cuda")
    assert cuda_lib.lce_set_tile_config(cfg) == 0
    try:
        assert cuda_lib.lce_test_inject_stall(1) == 0
        t0 = time.monotonic()
        loss, lse, nv, ws = api.lce_forward(H, W, y, strip_V=w.strip_V, f32_mode=mode)
        with pytest.raises(LceError) as e:
            api.lce_check_error(ws)
        elapsed = time.monotonic() - t0
        assert e.value.name == "LCE_ERR_TIMEOUT"
        assert 1.5 < elapsed < 60.0
        # the hook cleared itself; the same workspace and the context work normally again
        loss, lse, nv, ws = api.lce_forward(H, W, y, strip_V=w.strip_V, workspace=ws,
                                            f32_mode=mode)
        api.lce_check_error(ws)
        parity_case(w, seed=1, f32_mode=mode)
    finally:
        cuda_lib.lce_test_inject_stall(0)
        cuda_lib.lce_set_tile_config(0)


@pytest.mark.parametrize("fmt", [0, 1], ids=["bf16", "tf32x3"])
def test_withheld_load_in_backward_times_out(cuda_lib, fmt):
    """The same in the backward kernels: the gradient launch (the first tensor-core launch of the
    backward) withholds its first k-block; the backward reports LCE_ERR_TIMEOUT and the next one
    matches the oracle."""
    w, mode = FORMATS[fmt]
    H, W, y = make_inputs(w, "cuda")
    loss, lse, nv, ws = api.lce_forward(H, W, y, strip_V=w.strip_V, f32_mode=mode)
    api.lce_check_error(ws)
    one = torch.ones((), device="cuda")
    try:
        assert cuda_lib.lce_test_inject_stall(1) == 0
        t0 = time.monotonic()
        api.lce_backward(H, W, y, lse, nv, one, strip_V=w.strip_V, workspace=ws, f32_mode=mode)
        with pytest.raises(LceError) as e:
            api.lce_check_error(ws)
        assert e.value.name == "LCE_ERR_TIMEOUT"
        assert 1.5 < time.monotonic() - t0 < 60.0
    finally:
        cuda_lib.lce_test_inject_stall(0)
    api.lce_backward(H, W, y, lse, nv, one, strip_V=w.strip_V, workspace=ws, f32_mode=mode)
    api.lce_check_error(ws)
    parity_case(w, seed=2, f32_mode=mode)


def test_hook_rejects_other_values(cuda_lib):
    assert cuda_lib.lce_test_inject_stall(2) == 1
    assert cuda_lib.lce_test_inject_stall(-1) == 1
    assert cuda_lib.lce_test_inject_stall(0) == 0
