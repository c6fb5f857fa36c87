"""Full-size parity at the benchmark's launch configuration (same workloads, strip widths and
C-ABI calls as bench.py), against the float64 oracle on every configuration:

* lse of EVERY token against the oracle's lse (formed a block of tokens at a time; the oracle
  result is computed once per workload and shared by the strip widths and arithmetics that run
  it);
* n_valid exactly, and the loss against the oracle's loss (its lse and target logits);
* dH on seeded samples of token rows (each row needs only its own logits);
* dW on samples of vocabulary rows: the most frequent labels, outlier rows of W (rows whose norm
  stands out), the rows on both sides of every strip boundary (lce_strip_columns), the last row, and seeded random
  rows -- a dW tile written to the wrong place, or a wrong long reduction over the tokens, shows
  there;
* and, on the full gradients, properties that hold at any size: sum_v dW_v = 0 and
  <dW, W> = <dH, H>.
"""

import time

import numpy as np
import pytest
import torch

import oracle
from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

from ._parity import TOL, max_rel, rel_fro

pytestmark = pytest.mark.gpu

# oracle lse of every token, per (workload, input dtype): shared by the tests of one workload
_ORACLE_LSE = {}


def _oracle_lse(key, Hn, Wn, block=1024):
    if key not in _ORACLE_LSE:
        t0 = time.perf_counter()
        _ORACLE_LSE[key] = np.concatenate([oracle.lse_rows(Hn[i:i + block], Wn)[0]
                                           for i in range(0, Hn.shape[0], block)])
        print(f"oracle lse of {Hn.shape[0]} tokens x {Wn.shape[0]} x {Wn.shape[1]}: "
              f"{time.perf_counter() - t0:.1f} s")
    return _ORACLE_LSE[key]


def _run(w, strip_V, f32_mode="exact"):
    H, W, y = make_inputs(w, "cuda", seed=0)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    loss, lse, nv, ws = api.lce_forward(H, W, y, strip_V=strip_V, reduction=w.reduction,
                                        f32_mode=f32_mode)
    dH, dW, _ = api.lce_backward(H, W, y, lse, nv, torch.ones((), device="cuda"),
                                 strip_V=strip_V, reduction=w.reduction, workspace=ws,
                                 f32_mode=f32_mode)
    api.lce_check_error(ws)
    torch.cuda.synchronize()
    _run.extra_peak = torch.cuda.max_memory_allocated() - base
    return H, W, y, loss.item(), lse, int(nv.item()), dH, dW


def _check(w, strip_V, n_rows=48, n_vocab=24, f32_mode="exact"):
    tl, tg = TOL["tf32x3" if f32_mode == "tf32x3" else w.dtype]
    H, W, y, loss, lse, nv, dH, dW = _run(w, strip_V, f32_mode)
    peak_after_run = _run.extra_peak  # device memory the forward+backward added
    Hn = H.cpu().double().numpy()
    Wn = W.cpu().double().numpy()
    yn = y.cpu().numpy()
    valid, bad = oracle.row_masks(yn, w.V, -100)
    assert not bad.any()
    assert nv == int(valid.sum())
    scale = 1.0 / nv if w.reduction == "mean" else 1.0
    rng = np.random.default_rng(1234)
    rows = np.unique(np.concatenate([[0, w.N - 1, (w.N // 128) * 128 - 1],
                                     rng.choice(w.N, n_rows, replace=False)]))
    rows = rows[(rows >= 0) & (rows < w.N)]
    dH_ref, lse_ref = oracle.dH_rows(Hn[rows], Wn, yn[rows], scale)
    lse_gpu = lse.cpu().double().numpy()
    assert max_rel(lse_gpu[rows], lse_ref) <= tl
    assert rel_fro(dH.cpu().double().numpy()[rows], dH_ref) <= tg

    # every token's lse and the loss against the oracle
    lse_all = _oracle_lse((w.name, w.dtype), Hn, Wn)
    assert max_rel(lse_gpu, lse_all) <= tl
    t = np.einsum("ij,ij->i", Hn[valid], Wn[yn[valid]])
    total = float((lse_all[valid] - t).sum())
    ref_loss = total / nv if w.reduction == "mean" else total
    assert abs(loss - ref_loss) <= tl * abs(ref_loss), (loss, ref_loss)

    # dW on sampled vocabulary rows
    counts = np.bincount(yn[valid], minlength=w.V)
    norms = np.linalg.norm(Wn, axis=1)
    outliers = np.nonzero(norms > 4.0 * np.median(norms))[0]
    assert (outliers.size > 0) == (w.outlier_frac > 0)
    width = api.lce_strip_columns(w.V, strip_V, "tf32x3" if f32_mode == "tf32x3" else w.dtype)
    bounds = np.arange(width, w.V, width)
    vs = np.concatenate([np.argsort(-counts)[:8], outliers[:8], bounds - 1, bounds, [w.V - 1],
                         rng.choice(w.V, n_vocab, replace=False)])
    vs = np.unique(vs[(vs >= 0) & (vs < w.V)])
    dW_ref = oracle.dW_rows(Hn, Wn, yn, lse_all, vs, scale)
    assert rel_fro(dW.cpu().double().numpy()[vs], dW_ref) <= tg
    if outliers.size:
        ov = outliers[:8]
        assert rel_fro(dW.cpu().double().numpy()[ov], dW_ref[np.searchsorted(vs, ov)]) <= tg

    # invariants on the full gradients (computed on the device, fp64)
    dWd, dHd = dW.double(), dH.double()
    colsum = dWd.sum(dim=0).abs().max().item()
    assert colsum <= tg * dWd.abs().sum(dim=0).max().item()
    a = (dWd * W.double()).sum().item()
    b = (dHd * H.double()).sum().item()
    assert abs(a - b) <= tg * max(abs(a), abs(b))
    assert torch.isfinite(dWd).all() and torch.isfinite(dHd).all()
    return peak_after_run


def test_n4096_d2048_v151936_strip8192(cuda_lib):
    _check(WORKLOADS["n4096-d2048-v151936"], 8192)


def test_n16384_d4096_v131072_ignore10_strip16384(cuda_lib):
    _check(WORKLOADS["n16384-d4096-v131072-ignore10"], 16384)


@pytest.mark.parametrize("strip", [4096, 8192, 16384, 32768])
def test_n65536_d2048_v151936_strip_sweep(cuda_lib, strip):
    """The longest batch, at every strip width of the sweep; peak device memory grows with the
    strip width and stays far below the N x V fp32 logits."""
    w = WORKLOADS["n65536-d2048-v151936"]
    torch.cuda.empty_cache()
    extra = _check(w, strip, n_rows=32, n_vocab=16)
    outputs = w.N * 4 + w.N * w.d * 4 + w.V * w.d * 4       # lse, dH, dW
    ws = api.lce_workspace_size(w.N, w.d, w.V, strip)
    width = api.lce_strip_columns(w.V, strip)
    assert width <= strip and -(-w.V // width) == -(-w.V // strip)  # as many strips, none wider
    assert ws >= w.N * width * 2                            # one bf16 gradient strip
    assert extra <= outputs + ws + 4 * 1024 * 1024
    assert extra - outputs < w.N * w.V * 4 / 4              # far below the N x V fp32 logits


def test_n32768_d6144_v151552_outliers_sum_strip16384(cuda_lib):
    _check(WORKLOADS["n32768-d6144-v151552-outliers"], 16384)


def test_n16384_d7168_v200000_fp32_strip16384(cuda_lib):
    """The pages' FP32 benchmark shape (Ring-DTP, appendix C), exact fp32 path, fp32 tolerances."""
    _check(WORKLOADS["n16384-d7168-v200000-fp32"], 16384, n_rows=24, n_vocab=16)


def test_n16384_d7168_v200000_fp32_tf32x3_strip16384(cuda_lib):
    """The same shape on the tensor cores (three tf32 products per fp32 product), fp32
    tolerances."""
    _check(WORKLOADS["n16384-d7168-v200000-fp32"], 16384, n_rows=24, n_vocab=16,
           f32_mode="tf32x3")


def test_n4096_d2048_v151936_single_cta_tiles(cuda_lib):
    """The single-CTA 128x256 tile variant at a full benchmark shape (the default picks CTA
    pairs here): the same sampled checks."""
    assert cuda_lib.lce_set_tile_config(1) == 0
    try:
        _check(WORKLOADS["n4096-d2048-v151936"], 8192)
    finally:
        cuda_lib.lce_set_tile_config(0)


def test_n4096_d2048_v151936_fp32_tf32x3_strip8192(cuda_lib):
    """fp32 inputs at the N=4096 shape on the tensor cores: 19 strips of the split-and-launch
    loop, exact loss and sampled dW rows against the oracle's full lse, fp32 tolerances."""
    w = WORKLOADS["n4096-d2048-v151936"].with_sizes(dtype="f32")
    _check(w, 8192, f32_mode="tf32x3")
