"""Full-size parity at the benchmark's launch configuration (same workloads, strip widths and
C-ABI calls as bench.py), on outputs the float64 oracle can compute one by one:

* lse and dH on seeded samples of token rows (each row needs only its own logits);
* n_valid exactly, and the loss: exactly against the oracle where its full lse is affordable
  (N=4096 and N=16384), else through the identity loss = reduce(lse_i - t_i) with the target
  logits t_i = h_i . w_{y_i} computed by the oracle;
* dW on seeded samples of vocabulary rows (including the most frequent labels) where the
  oracle's full lse is affordable; elsewhere through properties that hold at any size:
  sum_v dW_v = 0 and <dW, W> = <dH, H>.
"""

import numpy as np
import pytest
import torch

import oracle
from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

from ._parity import TOL, max_rel, rel_fro

pytestmark = pytest.mark.gpu


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


def _check(w, strip_V, full_lse: bool, n_rows=48, n_vocab=24, f32_mode="exact"):
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

    t = np.einsum("ij,ij->i", Hn[valid], Wn[yn[valid]])
    if full_lse:
        lse_all = np.concatenate([oracle.lse_rows(Hn[i:i + 1024], Wn)[0]
                                  for i in range(0, w.N, 1024)])
        total = float((lse_all[valid] - t).sum())
        ref_loss = total / nv if w.reduction == "mean" else total
        assert abs(loss - ref_loss) <= tl * abs(ref_loss)
        counts = np.bincount(yn[valid], minlength=w.V)
        vs = np.unique(np.concatenate([np.argsort(-counts)[:8],
                                       rng.choice(w.V, n_vocab, replace=False), [w.V - 1]]))
        dW_ref = oracle.dW_rows(Hn, Wn, yn, lse_all, vs, scale)
        assert rel_fro(dW.cpu().double().numpy()[vs], dW_ref) <= tg
        assert max_rel(lse_gpu, lse_all) <= tl
    else:
        total = float((lse_gpu[valid] - t).sum())
        ident = total / nv if w.reduction == "mean" else total
        assert abs(loss - ident) <= tl * abs(ident)
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
    _check(WORKLOADS["n4096-d2048-v151936"], 8192, full_lse=True)


def test_n16384_d4096_v131072_ignore10_strip16384(cuda_lib):
    _check(WORKLOADS["n16384-d4096-v131072-ignore10"], 16384, full_lse=True)


@pytest.mark.parametrize("strip", [4096, 8192, 16384, 32768])
def test_n65536_d2048_v151936_strip_sweep(cuda_lib, strip):
    """The longest batch, at every strip width of the sweep; peak device memory grows with the
    strip width and stays far below the N x V fp32 logits."""
    w = WORKLOADS["n65536-d2048-v151936"]
    torch.cuda.empty_cache()
    extra = _check(w, strip, full_lse=False, n_rows=32, n_vocab=0)
    outputs = w.N * 4 + w.N * w.d * 4 + w.V * w.d * 4       # lse, dH, dW
    ws = api.lce_workspace_size(w.N, w.d, w.V, strip)
    assert ws >= w.N * strip * 2                            # one bf16 gradient strip
    assert extra <= outputs + ws + 4 * 1024 * 1024
    assert extra - outputs < w.N * w.V * 4 / 4              # far below the N x V fp32 logits


def test_n32768_d6144_v151552_outliers_sum_strip16384(cuda_lib):
    _check(WORKLOADS["n32768-d6144-v151552-outliers"], 16384, full_lse=False)


def test_n16384_d7168_v200000_fp32_strip16384(cuda_lib):
    """The pages' FP32 benchmark shape (Ring-DTP, appendix C), exact fp32 path, fp32 tolerances."""
    _check(WORKLOADS["n16384-d7168-v200000-fp32"], 16384, full_lse=False, n_rows=24, n_vocab=0)


def test_n16384_d7168_v200000_fp32_tf32x3_strip16384(cuda_lib):
    """The same shape on the tensor cores (three tf32 products per fp32 product), fp32
    tolerances."""
    _check(WORKLOADS["n16384-d7168-v200000-fp32"], 16384, full_lse=False, n_rows=24, n_vocab=0,
           f32_mode="tf32x3")


def test_n4096_d2048_v151936_single_cta_tiles(cuda_lib):
    """The single-CTA 128x256 tile variant at a full benchmark shape (the default picks CTA
    pairs here): the same sampled checks."""
    assert cuda_lib.lce_set_tile_config(1) == 0
    try:
        _check(WORKLOADS["n4096-d2048-v151936"], 8192, full_lse=True)
    finally:
        cuda_lib.lce_set_tile_config(0)


def test_n4096_d2048_v151936_fp32_tf32x3_strip8192(cuda_lib):
    """fp32 inputs at the N=4096 shape on the tensor cores: 19 strips of the split-and-launch
    loop, exact loss and sampled dW rows against the oracle's full lse, fp32 tolerances."""
    w = WORKLOADS["n4096-d2048-v151936"].with_sizes(dtype="f32")
    _check(w, 8192, full_lse=True, f32_mode="tf32x3")
