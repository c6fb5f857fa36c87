"""Pins for the float64 oracle: checks against facts that do not come from the oracle itself.

Each pin is a plain function so that ``test_planted_mistakes_are_caught`` can re-run the whole
set against deliberately broken copies of the oracle (mistakes planted in the oracle, on the CPU)
and show that every one of them is caught.
"""

import math
import os

import numpy as np
import pytest

from oracle import lce_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(N, d, V, seed, h=1.0, w=None):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, d)) * h
    W = rng.standard_normal((V, d)) * (1.0 / math.sqrt(d) if w is None else w)
    y = rng.integers(0, V, size=N)
    return H, W, y


# ----------------------------------------------------------------------------------- pins

def pin_zero_weights_closed_form():
    """W = 0: every logit is 0, so lse = ln V, loss = ln V (mean), P = 1/V, dH = 0 and
    dW_v = scale * (sum_i h_i / V - sum_{i: y_i = v} h_i)."""
    N, d, V = 7, 5, 11
    H, _, y = _rand(N, d, V, 1)
    W = np.zeros((V, d))
    f = R.forward_backward(H, W, y, reduction="mean")
    assert np.allclose(f["lse"], math.log(V), rtol=0, atol=1e-14)
    assert abs(f["loss"] - math.log(V)) < 1e-14
    assert np.abs(f["dH"]).max() == 0.0
    scale = 1.0 / N
    expect = np.zeros((V, d))
    hsum = H.sum(axis=0)
    for v in range(V):
        expect[v] = scale * hsum / V
        for i in range(N):
            if y[i] == v:
                expect[v] -= scale * H[i]
    assert np.allclose(f["dW"], expect, rtol=0, atol=1e-14)


def pin_two_classes_is_logistic_loss():
    """V = 2: l_i = softplus(z_other - z_target) (the logistic loss)."""
    N, d, V = 9, 4, 2
    H, W, y = _rand(N, d, V, 2, w=1.0)
    f = R.forward(H, W, y, reduction="sum")
    Z = H @ W.T
    other = 1 - y
    margin = Z[np.arange(N), other] - Z[np.arange(N), y]
    expect = np.logaddexp(0.0, margin)
    assert np.allclose(f["per_token"], expect, rtol=1e-13, atol=1e-13)
    assert abs(f["loss"] - expect.sum()) < 1e-12


def pin_single_class_is_zero():
    """V = 1: softmax is 1 on the only class, so the loss and both gradients are 0."""
    H, W, y = _rand(5, 3, 1, 3)
    f = R.forward_backward(H, W, y)
    assert abs(f["loss"]) < 1e-15
    assert np.abs(f["dH"]).max() < 1e-15 and np.abs(f["dW"]).max() < 1e-15
    Z = H @ W.T
    assert np.allclose(f["lse"], Z[:, 0], rtol=0, atol=1e-15)


def pin_gradient_rows_sum_to_zero():
    """Each row of softmax - onehot sums to 0, hence sum_v dW_v = 0 (a vector of zeros)."""
    H, W, y = _rand(13, 6, 17, 4)
    f = R.forward_backward(H, W, y)
    assert np.abs(f["dW"].sum(axis=0)).max() < 1e-14 * max(1.0, np.abs(f["dW"]).max() * 17)


def pin_ignored_rows_contribute_nothing():
    """Rows with ignore_index: zero loss and exactly zero dH; changing their hidden state leaves
    the loss and dW unchanged; mean divides by the number of valid rows."""
    H, W, y = _rand(10, 5, 9, 5)
    y = y.copy()
    y[[1, 4, 7]] = -100
    f = R.forward_backward(H, W, y)
    assert f["n_valid"] == 7
    assert np.all(f["per_token"][[1, 4, 7]] == 0.0)
    assert np.all(f["dH"][[1, 4, 7]] == 0.0)
    H2 = H.copy()
    H2[[1, 4, 7]] += 3.0
    f2 = R.forward_backward(H2, W, y)
    assert abs(f2["loss"] - f["loss"]) < 1e-14
    assert np.allclose(f2["dW"], f["dW"], rtol=0, atol=1e-14)
    assert abs(f["loss"] - f["per_token"].sum() / 7) < 1e-14


def pin_brute_force_python_loops():
    """Pure-Python loops with math.exp/math.log on a tiny case: loss, lse, dH, dW."""
    N, d, V = 4, 3, 5
    H, W, y = _rand(N, d, V, 6)
    y = y.copy()
    y[2] = -100
    for reduction in ("mean", "sum"):
        Z = [[sum(H[i][k] * W[v][k] for k in range(d)) for v in range(V)] for i in range(N)]
        lse = [math.log(sum(math.exp(z) for z in Z[i])) for i in range(N)]
        valid = [y[i] != -100 for i in range(N)]
        nv = sum(valid)
        tot = sum(lse[i] - Z[i][y[i]] for i in range(N) if valid[i])
        loss = tot / nv if reduction == "mean" else tot
        sc = 1.0 / nv if reduction == "mean" else 1.0
        G = [[(sc * (math.exp(Z[i][v] - lse[i]) - (1.0 if v == y[i] else 0.0))) if valid[i] else 0.0
              for v in range(V)] for i in range(N)]
        dH = [[sum(G[i][v] * W[v][k] for v in range(V)) for k in range(d)] for i in range(N)]
        dW = [[sum(G[i][v] * H[i][k] for i in range(N)) for k in range(d)] for v in range(V)]
        f = R.forward_backward(H, W, y, reduction=reduction)
        assert abs(f["loss"] - loss) < 1e-12
        assert np.allclose(f["lse"], lse, rtol=0, atol=1e-12)
        assert np.allclose(f["dH"], dH, rtol=0, atol=1e-12)
        assert np.allclose(f["dW"], dW, rtol=0, atol=1e-12)


def pin_central_finite_differences():
    """Central differences (step 1e-6, float64) of the loss against dH and dW, N=6, d=8, V=16,
    one ignored row, both reductions: relative error <= 1e-6."""
    N, d, V = 6, 8, 16
    H, W, y = _rand(N, d, V, 7, w=0.5)
    y = y.copy()
    y[3] = -100
    eps = 1e-6
    for reduction in ("mean", "sum"):
        f = R.forward_backward(H, W, y, reduction=reduction)

        def L(Hx, Wx):
            return R.forward(Hx, Wx, y, reduction=reduction)["loss"]

        num_dH = np.zeros_like(H)
        for i in range(N):
            for k in range(d):
                Hp = H.copy(); Hp[i, k] += eps
                Hm = H.copy(); Hm[i, k] -= eps
                num_dH[i, k] = (L(Hp, W) - L(Hm, W)) / (2 * eps)
        num_dW = np.zeros_like(W)
        for v in range(V):
            for k in range(d):
                Wp = W.copy(); Wp[v, k] += eps
                Wm = W.copy(); Wm[v, k] -= eps
                num_dW[v, k] = (L(H, Wp) - L(H, Wm)) / (2 * eps)
        assert np.linalg.norm(num_dH - f["dH"]) <= 1e-6 * np.linalg.norm(f["dH"])
        assert np.linalg.norm(num_dW - f["dW"]) <= 1e-6 * np.linalg.norm(f["dW"])


def pin_library_cross_entropy():
    """torch.nn.functional.cross_entropy in float64 on the CPU, with autograd gradients, on the
    same inputs: the textbook routine this operator replaces."""
    torch = pytest.importorskip("torch")
    N, d, V = 12, 6, 10
    H, W, y = _rand(N, d, V, 8)
    y = y.copy()
    y[[0, 5]] = -100
    for reduction in ("mean", "sum"):
        Ht = torch.tensor(H, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        loss = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=-100,
                                                 reduction=reduction)
        loss.backward()
        f = R.forward_backward(H, W, y, reduction=reduction)
        assert abs(f["loss"] - loss.item()) < 1e-12
        assert np.allclose(f["dH"], Ht.grad.numpy(), rtol=0, atol=1e-13)
        assert np.allclose(f["dW"], Wt.grad.numpy(), rtol=0, atol=1e-13)
        lse_t = torch.logsumexp(Ht.detach() @ Wt.detach().T, dim=1).numpy()
        assert np.allclose(f["lse"], lse_t, rtol=0, atol=1e-12)


def pin_scipy_logsumexp_large_logits():
    """lse against scipy.special.logsumexp with logits far beyond exp's range (overflow safe)."""
    special = pytest.importorskip("scipy.special")
    H, W, y = _rand(8, 4, 30, 9, h=40.0, w=10.0)
    f = R.forward(H, W, y)
    Z = H @ W.T
    assert np.isfinite(f["lse"]).all()
    assert np.allclose(f["lse"], special.logsumexp(Z, axis=1), rtol=1e-14, atol=1e-10)


def pin_strip_order_matches_dense():
    """The strip fold gives the dense result for every strip width (only the order changes)."""
    H, W, y = _rand(9, 5, 37, 10, w=2.0)
    y = y.copy()
    y[4] = -100
    for reduction in ("mean", "sum"):
        dense = R.forward(H, W, y, reduction=reduction)
        for strip in (1, 3, 8, 36, 37, 64):
            s = R.strip_forward(H, W, y, strip, reduction=reduction)
            assert np.allclose(s["lse"], dense["lse"], rtol=1e-14, atol=1e-13)
            assert abs(s["loss"] - dense["loss"]) < 1e-12
            assert s["n_valid"] == dense["n_valid"]


def pin_sampled_forms_match_dense():
    """Row/column-sampled forms (used at full sizes) agree with the dense definition."""
    H, W, y = _rand(11, 6, 50, 11)
    y = y.copy()
    y[3] = -100
    f = R.forward_backward(H, W, y, reduction="mean")
    scale = 1.0 / f["n_valid"]
    rows = np.array([0, 3, 7, 10])
    dHr, lser = R.dH_rows(H[rows], W, y[rows], scale)
    assert np.allclose(lser, f["lse"][rows], rtol=0, atol=1e-13)
    assert np.allclose(dHr, f["dH"][rows], rtol=0, atol=1e-14)
    lse_only, _ = R.lse_rows(H[rows], W, vocab_chunk=7)
    assert np.allclose(lse_only, f["lse"][rows], rtol=0, atol=1e-13)
    vs = np.array([0, 1, 17, 49, int(y[0])])
    dWr = R.dW_rows(H, W, y, f["lse"], vs, scale)
    assert np.allclose(dWr, f["dW"][vs], rtol=0, atol=1e-14)
    # token blocks are independent: their dH rows and dW contributions add up to the dense result
    dW_acc = np.zeros_like(W)
    for b0 in range(0, 11, 4):
        pt, lse_b, dH_b, dW_b = R.token_block_fwd_bwd(H[b0:b0 + 4], W, y[b0:b0 + 4], scale)
        assert np.allclose(dH_b, f["dH"][b0:b0 + 4], rtol=0, atol=1e-14)
        assert np.allclose(pt, f["per_token"][b0:b0 + 4], rtol=0, atol=1e-13)
        dW_acc += dW_b
    assert np.allclose(dW_acc, f["dW"], rtol=0, atol=1e-14)


def pin_mean_with_no_valid_row():
    """Mean over zero valid rows: loss NaN (0/0); G has no valid row, so dH = dW = 0."""
    H, W, y = _rand(4, 3, 6, 12)
    y = np.full(4, -100)
    f = R.forward_backward(H, W, y, reduction="mean")
    assert math.isnan(f["loss"]) and f["n_valid"] == 0
    assert np.all(f["dH"] == 0) and np.all(f["dW"] == 0)
    assert np.isfinite(f["lse"]).all()


def pin_bad_labels_are_reported_and_excluded():
    """Labels outside [0, V) that are not ignore_index are reported and left out."""
    H, W, y = _rand(6, 3, 8, 13)
    y = y.copy()
    y[1] = 8
    y[2] = -5
    f = R.forward_backward(H, W, y)
    assert list(np.nonzero(f["bad"])[0]) == [1, 2]
    assert f["n_valid"] == 4
    assert np.all(f["dH"][[1, 2]] == 0)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_golden_full_logits_bytes():
    """The blog's worked example: 65,536 x 124,160 x 4 B and 32,768 x 248,320 x 4 B, both
    printed as approximately 32.55 GB."""
    from memory_bounded_linear_gb300 import full_logits_bytes as pkg_bytes
    rows = [l.split() for l in open(os.path.join(GOLDEN, "full_logits_bytes.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for tok, voc, gb in rows:
        b = R.full_logits_bytes(int(tok), int(voc))
        assert b == 32_547_799_040
        assert round(b / 1e9, 2) == float(gb)
        assert pkg_bytes(int(tok), int(voc)) == b


# ----------------------------------------------------------------------- planted mistakes

def _mut_lse_drops_max(Z):
    M = Z.max(axis=1)
    return np.log(np.exp(Z - M[:, None]).sum(axis=1))


def _mut_onehot_sign(Z, lse, labels, valid, scale):
    P = np.exp(Z - lse[:, None])
    rows = np.nonzero(valid)[0]
    y = np.asarray(labels, dtype=np.int64)
    P[rows, y[rows]] += 1.0
    G = np.zeros_like(P)
    G[rows] = scale * P[rows]
    return G


def _mut_ignored_rows_kept(Z, lse, labels, valid, scale):
    P = np.exp(Z - lse[:, None])
    y = np.asarray(labels, dtype=np.int64)
    rows = np.nonzero(valid)[0]
    P[rows, y[rows]] -= 1.0
    return scale * P


def _mut_mean_over_all_rows(reduction, dloss, n_valid):
    return dloss / (n_valid + 1) if reduction == "mean" else dloss


def _mut_backward_transposed(H, W, labels, lse, n_valid, dloss=1.0, ignore_index=-100,
                             reduction="mean"):
    Z = R.logits(H, W)
    valid, _ = R.row_masks(labels, W.shape[0], ignore_index)
    G = R.grad_logits(Z, np.asarray(lse, float), labels, valid, R._scale(reduction, dloss, n_valid))
    return G @ W, (H.T @ G).T[:, ::-1].copy()   # dW columns reversed: a transposed/flipped operand


def _mut_masks_swap(labels, V, ignore_index):
    y = np.asarray(labels, dtype=np.int64)
    in_range = (y >= 0) & (y <= V)        # off-by-one in the range check
    not_ignored = y != ignore_index
    return in_range & not_ignored, (~in_range) & not_ignored


MUTANTS = {
    "lse drops the max term": ("row_logsumexp", _mut_lse_drops_max),
    "onehot subtracted with the wrong sign": ("grad_logits", _mut_onehot_sign),
    "ignored rows keep a gradient": ("grad_logits", _mut_ignored_rows_kept),
    "mean divides by the wrong count": ("_scale", _mut_mean_over_all_rows),
    "dW built from a flipped operand": ("backward", _mut_backward_transposed),
    "label range check off by one": ("row_masks", _mut_masks_swap),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(R, attr, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake: {name}"
