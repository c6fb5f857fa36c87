"""Input recipe checks (host only): determinism, shapes, and the stated distributions."""

import math

import pytest
import torch

from memory_bounded_linear_gb300.workloads import (IGNORE_INDEX, WORKLOADS, make_inputs,
                                                   zipf_ranks)


def test_workloads_with_stated_sizes():
    sizes = {(w.N, w.d, w.V, w.strip_V, w.dtype, w.reduction) for w in WORKLOADS.values()}
    assert sizes == {
        (256, 256, 4096, 512, "f32", "mean"),
        (4096, 2048, 151936, 8192, "bf16", "mean"),
        (16384, 4096, 131072, 16384, "bf16", "mean"),
        (65536, 2048, 151936, 8192, "bf16", "mean"),
        (32768, 6144, 151552, 16384, "bf16", "sum"),
        # the pages' FP32 benchmark shape (Ring-DTP, appendix C)
        (16384, 7168, 200000, 16384, "f32", "mean"),
    }
    assert WORKLOADS["n65536-d2048-v151936"].strip_sweep == (4096, 8192, 16384, 32768)


def test_seeded_draws_repeat():
    w = WORKLOADS["tiny-fp32"]
    a = make_inputs(w, "cpu", seed=0)
    b = make_inputs(w, "cpu", seed=0)
    c = make_inputs(w, "cpu", seed=1)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])


def test_tiny_distributions():
    H, W, y = make_inputs(WORKLOADS["tiny-fp32"], "cpu")
    assert H.dtype == torch.float32 and W.dtype == torch.float32 and y.dtype == torch.int64
    assert abs(H.std().item() - 1.0) < 0.02
    assert abs(W.std().item() - 1.0 / math.sqrt(256)) < 0.002
    assert int(y.min()) >= 0 and int(y.max()) < 4096


def test_ignore_fraction_and_outliers_reduced_size():
    w = WORKLOADS["n16384-d4096-v131072-ignore10"].with_sizes(N=1000, d=64, V=3000)
    H, W, y = make_inputs(w, "cpu")
    assert H.dtype == torch.bfloat16
    assert int((y == IGNORE_INDEX).sum()) == 100
    assert abs(W.float().std().item() - 0.02) < 0.002
    w5 = WORKLOADS["n32768-d6144-v151552-outliers"].with_sizes(N=64, d=64, V=5000)
    H5, W5, _ = make_inputs(w5, "cpu")
    norms = W5.float().norm(dim=1)
    big = norms > 4.0 * norms.median()
    assert int(big.sum()) == 50           # floor(1% of 5000) rows scaled x8
    assert abs(H5.float().std().item() - 0.5) < 0.05


def test_zipf_head_frequencies():
    g = torch.Generator().manual_seed(0)
    r = zipf_ranks(200000, 1000, 1.1, g, "cpu")
    k = torch.arange(1, 1001, dtype=torch.float64)
    p = k.pow(-1.1) / k.pow(-1.1).sum()
    counts = torch.bincount(r, minlength=1000).double() / 200000
    assert torch.allclose(counts[:5], p[:5], rtol=0.03)
    assert int(r.min()) >= 0 and int(r.max()) < 1000


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_flops_count(name):
    w = WORKLOADS[name]
    assert w.flops == 8 * w.N * w.d * w.V
