"""Float64 CPU oracle for linear cross-entropy (vocabulary projection + cross-entropy).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
shares no code with the CUDA library (no kernels, headers, helpers or tables).

What it computes, and where the definition comes from
-----------------------------------------------------
"Running 128K-Sequence MoE RL on 32 H100s" (blog), section "Linear CE: Avoiding
Materialization of Full Logits": the logits are the linear layer's output laid out along the
vocabulary, followed by cross-entropy; Linear CE only avoids *holding* the N x V logits.
"Flattening Every Memory Peak in Long-Context Mixture-of-Experts Training",
section 2: an
operator of this kind must return the replaced (dense) implementation's forward values and
gradients and change only the order of computation.  So the oracle is the plain dense
definition, written out in float64:

    Z      = H W^T                                  (N x V logits, materialised)
    lse_i  = M_i + log sum_v exp(Z_iv - M_i),  M_i = max_v Z_iv
    l_i    = lse_i - Z_{i, y_i}     for valid rows, 0 for rows with y_i == ignore_index
    loss   = sum_i l_i / n_valid   (mean)   or   sum_i l_i   (sum)
    G      = scale * (softmax(Z) - onehot(y))  on valid rows, 0 on the others,
             scale = dloss / n_valid (mean) or dloss (sum)
    dH     = G W,   dW = G^T H

Readings where the pages are silent (each is also listed in the design notes):
  * reduction semantics follow the usual cross-entropy convention: mean over non-ignored rows;
  * a label outside [0, V) that is not ignore_index is an error; that row is left out of the
    loss, of n_valid and of the gradients (``bad`` reports those rows);
  * with mean reduction and no valid row, loss = 0/0 = NaN and dH = dW = 0 (G has no valid row);
  * lse is reported for every row, ignored or not (it does not depend on the label).

``strip_forward`` follows the method's own order instead ("Flattening Every Memory Peak in Long-Context Mixture-of-Experts Training",
section 3.2 and appendix C, Ring-DTP): the vocabulary is cut into strips, each strip of
logits is folded into a running per-token state and released.  The state is read as
(running max m, running sum of exp(z - m), target logit t), an online log-sum-exp.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "logits", "row_logsumexp", "row_masks", "forward", "grad_logits", "backward",
    "forward_backward", "strip_forward", "lse_rows", "dH_rows", "dW_rows",
    "token_block_fwd_bwd", "full_logits_bytes",
]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def logits(H, W):
    """Z = H W^T: the linear output along the vocabulary (blog, "Linear CE" section)."""
    return _f64(H) @ _f64(W).T


def row_logsumexp(Z):
    """lse_i = M_i + log sum_v exp(Z_iv - M_i) with M_i the row maximum (log-softmax normaliser)."""
    M = Z.max(axis=1)
    return M + np.log(np.exp(Z - M[:, None]).sum(axis=1))


def row_masks(labels, V, ignore_index):
    """(valid, bad): valid rows carry a label in [0, V); bad rows carry neither such a label
    nor ignore_index."""
    y = np.asarray(labels, dtype=np.int64)
    in_range = (y >= 0) & (y < V)
    not_ignored = y != ignore_index
    return in_range & not_ignored, (~in_range) & not_ignored


def _scale(reduction, dloss, n_valid):
    if reduction == "mean":
        return dloss / n_valid if n_valid > 0 else np.inf  # only multiplies valid rows
    if reduction == "sum":
        return dloss
    raise ValueError(f"unknown reduction {reduction!r}")


def forward(H, W, labels, ignore_index=-100, reduction="mean"):
    """Dense forward: loss, per-token lse and loss, n_valid, bad-label mask."""
    Z = logits(H, W)
    N, V = Z.shape
    lse = row_logsumexp(Z)
    valid, bad = row_masks(labels, V, ignore_index)
    y = np.asarray(labels, dtype=np.int64)
    per_token = np.zeros(N)
    rows = np.nonzero(valid)[0]
    per_token[rows] = lse[rows] - Z[rows, y[rows]]
    n_valid = int(valid.sum())
    total = per_token.sum()
    if reduction == "mean":
        loss = total / n_valid if n_valid > 0 else float("nan")
    elif reduction == "sum":
        loss = total
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    return {"loss": float(loss), "lse": lse, "per_token": per_token,
            "n_valid": n_valid, "bad": bad}


def grad_logits(Z, lse, labels, valid, scale):
    """dloss/dZ = scale * (softmax(Z) - onehot(y)) on valid rows, 0 on every other row."""
    P = np.exp(Z - lse[:, None])
    rows = np.nonzero(valid)[0]
    y = np.asarray(labels, dtype=np.int64)
    P[rows, y[rows]] -= 1.0
    G = np.zeros_like(P)
    G[rows] = scale * P[rows]
    return G


def backward(H, W, labels, lse, n_valid, dloss=1.0, ignore_index=-100, reduction="mean"):
    """Dense backward from the saved lse: dH = G W, dW = G^T H."""
    H = _f64(H)
    W = _f64(W)
    Z = logits(H, W)
    valid, _ = row_masks(labels, W.shape[0], ignore_index)
    G = grad_logits(Z, _f64(lse), labels, valid, _scale(reduction, dloss, n_valid))
    return G @ W, G.T @ H


def forward_backward(H, W, labels, ignore_index=-100, reduction="mean", dloss=1.0):
    f = forward(H, W, labels, ignore_index, reduction)
    dH, dW = backward(H, W, labels, f["lse"], f["n_valid"], dloss, ignore_index, reduction)
    f["dH"] = dH
    f["dW"] = dW
    return f


def strip_forward(H, W, labels, strip_V, ignore_index=-100, reduction="mean"):
    """Forward in the method's order: one vocabulary strip at a time, each strip's logits
    folded into a running per-token (m, s, t) state and then dropped ("Flattening Every
    Memory Peak", section 3.2; appendix C).

    For strip [c0, c1): Z_s = H W[c0:c1]^T; m' = max(m, max_v Z_s);
    s' = s exp(m - m') + sum_v exp(Z_s - m'); t picks Z_{i,y_i} when y_i falls in the strip.
    At the end lse = m + log s.
    """
    H = _f64(H)
    W = _f64(W)
    N, V = H.shape[0], W.shape[0]
    y = np.asarray(labels, dtype=np.int64)
    m = np.full(N, -np.inf)
    s = np.zeros(N)
    t = np.zeros(N)
    for c0 in range(0, V, strip_V):
        c1 = min(c0 + strip_V, V)
        Zs = H @ W[c0:c1].T
        m_new = np.maximum(m, Zs.max(axis=1))
        s = s * np.exp(m - m_new) + np.exp(Zs - m_new[:, None]).sum(axis=1)
        m = m_new
        hit = (y >= c0) & (y < c1)
        t[hit] = Zs[np.nonzero(hit)[0], y[hit] - c0]
        del Zs  # the strip is released before the next one is formed
    lse = m + np.log(s)
    valid, bad = row_masks(y, V, ignore_index)
    per_token = np.where(valid, lse - t, 0.0)
    n_valid = int(valid.sum())
    total = per_token.sum()
    if reduction == "mean":
        loss = total / n_valid if n_valid > 0 else float("nan")
    else:
        loss = total
    return {"loss": float(loss), "lse": lse, "per_token": per_token,
            "n_valid": n_valid, "bad": bad}


# ---------------------------------------------------------------------------------------------
# Row- and column-sampled forms of the same definition, for sizes where the N x V logits do not
# fit in host memory.  Each token row is computed exactly as in ``forward``/``backward``; only the
# set of rows (or vocabulary entries) evaluated is restricted.
# ---------------------------------------------------------------------------------------------

def lse_rows(H_rows, W, vocab_chunk=32768):
    """lse for the given token rows (the row's logits are formed a vocabulary chunk at a time
    only to bound host memory; the maximum and the sum are taken over the whole row)."""
    H_rows = _f64(H_rows)
    W = _f64(W)
    V = W.shape[0]
    Zrow = np.empty((H_rows.shape[0], V))
    for c0 in range(0, V, vocab_chunk):
        Zrow[:, c0:c0 + vocab_chunk] = H_rows @ W[c0:c0 + vocab_chunk].T
    return row_logsumexp(Zrow), Zrow


def dH_rows(H_rows, W, labels_rows, scale, ignore_index=-100):
    """dH for the given token rows: G_rows W with G_rows = scale (softmax - onehot)."""
    W = _f64(W)
    lse, Zrow = lse_rows(H_rows, W)
    valid, _ = row_masks(labels_rows, W.shape[0], ignore_index)
    G = grad_logits(Zrow, lse, labels_rows, valid, scale)
    return G @ W, lse


def dW_rows(H, W, labels, lse, v_idx, scale, ignore_index=-100):
    """dW for the given vocabulary rows v: dW_v = sum_i G_iv h_i, using lse for every token."""
    H = _f64(H)
    W = _f64(W)
    y = np.asarray(labels, dtype=np.int64)
    valid, _ = row_masks(y, W.shape[0], ignore_index)
    v_idx = np.asarray(v_idx, dtype=np.int64)
    Zc = H @ W[v_idx].T                          # N x |v_idx| logit columns
    G = np.exp(Zc - _f64(lse)[:, None])
    G -= (y[:, None] == v_idx[None, :]).astype(np.float64)
    G *= np.where(valid, scale, 0.0)[:, None]
    return G.T @ H


def token_block_fwd_bwd(H_blk, W, labels_blk, scale, ignore_index=-100):
    """One block of tokens through the dense definition: its logits, lse, per-token loss, its
    dH rows and its contribution G^T H_blk to dW.  Used to time the oracle on a bounded sample."""
    H_blk = _f64(H_blk)
    W = _f64(W)
    Z = H_blk @ W.T
    lse = row_logsumexp(Z)
    valid, _ = row_masks(labels_blk, W.shape[0], ignore_index)
    y = np.asarray(labels_blk, dtype=np.int64)
    rows = np.nonzero(valid)[0]
    per_token = np.zeros(Z.shape[0])
    per_token[rows] = lse[rows] - Z[rows, y[rows]]
    G = grad_logits(Z, lse, y, valid, scale)
    return per_token, lse, G @ W, G.T @ H_blk


def full_logits_bytes(tokens, vocab, bytes_per_element=4):
    """Size of a materialised fp32 logits tensor: local_tokens x vocab_partition x 4 bytes
    (blog, "Linear CE" section, the full-logits estimate)."""
    return int(tokens) * int(vocab) * int(bytes_per_element)
