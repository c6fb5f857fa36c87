"""Bit-exact checks of the three-product tf32 path's operand copies, read back from the workspace
after a call (its layout is the one include/lce.h describes for LCE_F32_TF32X3).

The split is a rounding decision, so it is checked exactly: hi must be x rounded to the nearest
value with 10 explicit mantissa bits, ties away from zero (the low 13 bits of the fp32 pattern
cleared after adding half of their range to the magnitude), and lo the same rounding of x - hi
(exact in fp32).  The transposed copies must be the transposes, bit for bit, and the gradient
strip's transposed hi / lo parts the transposes of its hi / lo parts."""

import numpy as np
import pytest
import torch

from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def rna_tf32(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest value with 10 explicit mantissa bits, ties away from zero."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    sign = u & np.uint32(0x80000000)
    mag = u & np.uint32(0x7FFFFFFF)
    mag = (mag + np.uint32(0x1000)) & np.uint32(0xFFFFE000)
    return (sign | mag).view(np.float32)


def r256(x: int) -> int:
    return (x + 255) // 256 * 256


def _f32(ws: np.ndarray, off: int, rows: int, cols: int, ld: int) -> np.ndarray:
    a = ws[off:off + rows * ld * 4].view(np.float32).reshape(rows, ld)
    return a[:, :cols]


@pytest.mark.parametrize("N,d,V", [(130, 72, 300), (517, 256, 1000), (64, 8, 129), (50, 12, 200)])
def test_split_parts_and_transposes_are_exact(cuda_lib, N, d, V):
    w = WORKLOADS["tiny-fp32"].with_sizes(N=N, d=d, V=V, strip_V=1024)  # one strip: V <= 1024
    H, W, y = make_inputs(w, "cuda")
    loss, lse, nv, ws = api.lce_forward(H, W, y, strip_V=1024, f32_mode="tf32x3")
    api.lce_backward(H, W, y, lse, nv, torch.ones((), device="cuda"), strip_V=1024,
                     workspace=ws, f32_mode="tf32x3")
    api.lce_check_error(ws)
    torch.cuda.synchronize()
    wsn = ws.cpu().numpy()
    Hn, Wn = H.cpu().numpy(), W.cpu().numpy()

    # layout of LCE_F32_TF32X3 (include/lce.h): header | H hi, lo | W strip hi, lo | backward:
    # H^T hi, lo | W strip^T hi, lo | G hi, lo | G^T hi, lo
    wcols = min(1024, V)
    ldg = (wcols + 255) // 256 * 256
    ldt = (N + 31) // 32 * 32
    h_part, w_part = r256(N * d * 4), r256(wcols * d * 4)
    ht_part, wt_part = r256(d * ldt * 4), r256(d * ldg * 4)
    g_part, gt_part = r256(N * ldg * 4), r256(ldg * ldt * 4)
    off_h = 256
    off_w = off_h + 2 * h_part
    base = off_w + 2 * w_part
    off_ht = base
    off_wt = off_ht + 2 * ht_part
    off_g = off_wt + 2 * wt_part
    off_gt = off_g + 2 * g_part
    assert off_gt + 2 * gt_part <= wsn.size

    for x, off, part, rows, cols, ld in [(Hn, off_h, h_part, N, d, d), (Wn, off_w, w_part, V, d, d)]:
        hi = _f32(wsn, off, rows, cols, ld)
        lo = _f32(wsn, off + part, rows, cols, ld)
        want_hi = rna_tf32(x)
        want_lo = rna_tf32(x - want_hi)
        assert np.array_equal(hi.view(np.uint32), want_hi.view(np.uint32))
        assert np.array_equal(lo.view(np.uint32), want_lo.view(np.uint32))
        # x = hi + lo + r with |r| <= about 2^-22 |x|
        assert np.all(np.abs(x.astype(np.float64) - hi - lo) <= 2.0**-21 * np.abs(x) + 1e-38)

    for x, off, part, rows, cols, ld in [(Hn, off_ht, ht_part, d, N, ldt),
                                         (Wn, off_wt, wt_part, d, V, ldg)]:
        hi_t = _f32(wsn, off, rows, cols, ld)
        lo_t = _f32(wsn, off + part, rows, cols, ld)
        want_hi = rna_tf32(x)
        want_lo = rna_tf32(x - want_hi)
        assert np.array_equal(hi_t.view(np.uint32), want_hi.T.view(np.uint32))
        assert np.array_equal(lo_t.view(np.uint32), want_lo.T.view(np.uint32))

    g_hi = _f32(wsn, off_g, N, V, ldg)
    g_lo = _f32(wsn, off_g + g_part, N, V, ldg)
    gt_hi = _f32(wsn, off_gt, V, N, ldt)
    gt_lo = _f32(wsn, off_gt + gt_part, V, N, ldt)
    assert np.array_equal(gt_hi.view(np.uint32), g_hi.T.view(np.uint32))
    assert np.array_equal(gt_lo.view(np.uint32), g_lo.T.view(np.uint32))
    # the parts themselves are a tf32 split: hi has no bit below the 10 kept ones, and so does lo
    assert np.all((g_hi.view(np.uint32) & np.uint32(0x1FFF)) == 0)
    assert np.all((g_lo.view(np.uint32) & np.uint32(0x1FFF)) == 0)
    assert np.array_equal(rna_tf32(g_hi).view(np.uint32), g_hi.view(np.uint32))
