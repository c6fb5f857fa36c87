"""GPU parity where the logits are large: valid rows with logits up to a few hundred, and ignored
and bad-label rows whose logits reach several hundred.

exp(Z) overflows fp32 once Z is above about 88.7.  A valid row never evaluates it unshifted (the
forward folds exp(Z - running max), the backward exp(Z - lse) with lse >= every logit of the
row), but a row that is ignored or carries a bad label has no lse to shift by and must come out
as exact zeros in G, dH and dW's sums, not as 0 * inf.  The cross-entropy definition the oracle
writes out ("Flattening Every Memory Peak in Long-Context Mixture-of-Experts Training", section
2: the replaced implementation's values and gradients) gives G = 0 on those rows at any logit
size.

Inputs: the seeded workload draws, then each token row of H multiplied by a power of two (exact
in bf16 and fp32): valid rows by 1, 4, 16 or 64 (logits with standard deviation up to 64, maxima
in the hundreds), ignored and bad-label rows by 128 (maxima of several hundred).  A few valid
rows get labels outside [0, V) (the bad-label rows).
"""

import numpy as np
import pytest
import torch

from memory_bounded_linear_gb300 import _lib
from memory_bounded_linear_gb300._lib import LceError
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

from ._parity import assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

W2 = WORKLOADS["n4096-d2048-v151936"]
WT = WORKLOADS["tiny-fp32"]


def large_logit_inputs(w, seed=0):
    """H, W, labels of workload ``w`` (10% ignored rows) with rows of H scaled as described in
    the module docstring, plus the indices of the ignored and of the bad-label rows."""
    w = w.with_sizes(ignore_frac=0.1)
    H, W, y = make_inputs(w, "cpu", seed=seed)
    rng = np.random.default_rng(seed + 1000)
    yn = y.numpy()
    ignored = np.nonzero(yn == -100)[0]
    live = np.nonzero(yn != -100)[0]
    bad = rng.choice(live, 3, replace=False)
    y[torch.from_numpy(bad)] = torch.tensor([w.V, -7, 10**9])
    scale = np.ones(w.N)
    scale[live] = 2.0 ** (2 * rng.integers(0, 4, live.size))   # 1, 4, 16, 64
    scale[ignored] = 128.0
    scale[bad] = 128.0
    dt = H.dtype
    H = (H.double() * torch.from_numpy(scale)[:, None]).to(dt)  # powers of two: exact
    return H, W, y, ignored, bad


def _case(w, fmt, mode, reduction):
    H, W, y, ignored, bad = large_logit_inputs(w)
    with pytest.raises(LceError) as e:
        run_gpu(H, W, y, w.strip_V, reduction, f32_mode=mode)
    assert e.value.name == "LCE_ERR_LABEL_OUT_OF_RANGE"
    g = run_gpu(H, W, y, w.strip_V, reduction, check=False, f32_mode=mode)
    r = run_oracle(H, W, y, reduction)
    # the inputs really are in the overflow regime of an unshifted exp
    assert r["lse"][ignored].max() > 150.0 and r["lse"][bad].max() > 150.0
    assert r["lse"][np.setdiff1d(np.arange(w.N), np.concatenate([ignored, bad]))].max() > 100.0
    assert np.isfinite(g["dH"]).all() and np.isfinite(g["dW"]).all()
    assert np.isfinite(g["lse"]).all() and np.isfinite(g["loss"])
    assert np.all(g["dH"][ignored] == 0.0) and np.all(g["dH"][bad] == 0.0)
    assert_parity(g, r, "tf32x3" if mode == "tf32x3" else fmt)


@pytest.fixture
def tile_config(cuda_lib):
    def set_(cfg):
        assert cuda_lib.lce_set_tile_config(cfg) == 0
    yield set_
    cuda_lib.lce_set_tile_config(0)


@pytest.mark.parametrize("cfg", [1, 2], ids=["single-cta", "cta-pair"])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_bf16_overlapped_backward(cuda_lib, tile_config, cfg, reduction):
    """bf16, a backward small enough that each launch overlaps dH and dW of one strip with the
    next strip's gradient."""
    tile_config(cfg)
    _case(W2.with_sizes(N=517, d=256, V=2048, strip_V=512), "bf16", "exact", reduction)


@pytest.mark.parametrize("cfg", [1, 2], ids=["single-cta", "cta-pair"])
def test_bf16_large_backward_step(cuda_lib, tile_config, cfg):
    """bf16, 17 x 32 dH tiles per strip: the gradient launch, then dW and dH in a second launch."""
    tile_config(cfg)
    w = W2.with_sizes(N=4352, d=8192, V=700, strip_V=512)
    assert _lib.load().lce_workspace_size(w.N, w.d, w.V, w.strip_V, 0) == \
        256 + ((w.N * 512 * 2 + 255) // 256) * 256  # one gradient strip: not overlapped
    _case(w, "bf16", "exact", "mean")


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_fp32_exact(cuda_lib, reduction):
    """fp32 inputs on the CUDA cores, fp32 tolerances."""
    _case(WT.with_sizes(N=300, d=136, V=1000, strip_V=384), "f32", "exact", reduction)


@pytest.mark.parametrize("cfg", [1, 2], ids=["single-cta", "cta-pair"])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_fp32_tf32x3(cuda_lib, tile_config, cfg, reduction):
    """fp32 inputs as three tf32 products on the tensor cores, fp32 tolerances."""
    tile_config(cfg)
    _case(WT.with_sizes(N=300, d=136, V=1000, strip_V=384), "f32", "tf32x3", reduction)
