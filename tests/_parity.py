"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and the oracle on
the same seeded inputs, and compare with the stated tolerances."""

import numpy as np
import torch

import oracle
from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300.workloads import make_inputs, to_float64_numpy

# Tolerances: bf16 inputs -> loss and lse relative error <= 1e-3, dH and dW relative Frobenius
# error <= 1e-2; fp32 inputs -> 1e-5 and 1e-4, for the exact fp32 path and for the three-product
# tf32 path alike (its products carry about 2^-21 relative error, below the fp32 summation
# error at these depths).
TOL = {"bf16": (1e-3, 1e-2), "f32": (1e-5, 1e-4), "tf32x3": (1e-5, 1e-4)}


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def max_rel(a, b):
    return float(np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-30)))


def run_gpu(H, W, y, strip_V, reduction, ignore_index=-100, check=True, dev="cuda",
            f32_mode="exact"):
    Hd, Wd, yd = H.to(dev), W.to(dev), y.to(dev)
    loss, lse, nv, ws = api.lce_forward(Hd, Wd, yd, ignore_index=ignore_index, strip_V=strip_V,
                                        reduction=reduction, f32_mode=f32_mode)
    dH, dW, _ = api.lce_backward(Hd, Wd, yd, lse, nv, torch.ones((), device=dev),
                                 ignore_index=ignore_index, strip_V=strip_V,
                                 reduction=reduction, workspace=ws, f32_mode=f32_mode)
    if check:
        api.lce_check_error(ws)
    torch.cuda.synchronize()
    return {"loss": loss.item(), "lse": lse.cpu().double().numpy(), "n_valid": int(nv.item()),
            "dH": dH.cpu().double().numpy(), "dW": dW.cpu().double().numpy(), "ws": ws}


def run_oracle(H, W, y, reduction, ignore_index=-100):
    return oracle.forward_backward(to_float64_numpy(H), to_float64_numpy(W), y.numpy(),
                                   ignore_index=ignore_index, reduction=reduction)


def assert_parity(g, r, dtype):
    tl, tg = TOL[dtype]
    assert g["n_valid"] == r["n_valid"]
    if np.isnan(r["loss"]):
        assert np.isnan(g["loss"])
    else:
        assert abs(g["loss"] - r["loss"]) <= tl * max(abs(r["loss"]), 1e-30), (g["loss"], r["loss"])
    assert max_rel(g["lse"], r["lse"]) <= tl
    assert rel_fro(g["dH"], r["dH"]) <= tg, rel_fro(g["dH"], r["dH"])
    assert rel_fro(g["dW"], r["dW"]) <= tg, rel_fro(g["dW"], r["dW"])


def parity_case(w, seed=0, ignore_index=-100, f32_mode="exact"):
    H, W, y = make_inputs(w, "cpu", seed=seed)
    g = run_gpu(H, W, y, w.strip_V, w.reduction, ignore_index, f32_mode=f32_mode)
    r = run_oracle(H, W, y, w.reduction, ignore_index)
    assert_parity(g, r, "tf32x3" if (w.dtype == "f32" and f32_mode == "tf32x3") else w.dtype)
    return g, r
