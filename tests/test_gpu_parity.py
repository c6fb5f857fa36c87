"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle, element by element,
on seeded inputs small enough for the oracle, spanning several tiles with ragged tails."""

import numpy as np
import pytest
import torch

from memory_bounded_linear_gb300 import api
from memory_bounded_linear_gb300._lib import LceError
from memory_bounded_linear_gb300.workloads import WORKLOADS, make_inputs

from ._parity import assert_parity, parity_case, rel_fro, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

W2 = WORKLOADS["n4096-d2048-v151936"]
W3 = WORKLOADS["n16384-d4096-v131072-ignore10"]
W4 = WORKLOADS["n65536-d2048-v151936"]
W5 = WORKLOADS["n32768-d6144-v151552-outliers"]
WT = WORKLOADS["tiny-fp32"]


def test_tiny_fp32_workload_full(cuda_lib):
    parity_case(WT)


@pytest.mark.parametrize("w", [
    W2.with_sizes(N=300, d=136, V=1000, strip_V=384),      # ragged N, d (K tail), V, strips
    W3.with_sizes(N=517, d=256, V=2048, strip_V=512),      # 10% ignored rows
    W5.with_sizes(N=400, d=320, V=2500, strip_V=1024),     # outlier W rows, sum reduction
    W2.with_sizes(N=256, d=1024, V=512, strip_V=256),      # long K loop, exact tiles
    W2.with_sizes(N=129, d=64, V=257, strip_V=128),        # one past a tile in every direction
    W4.with_sizes(N=1000, d=192, V=3001, strip_V=4096),    # one strip wider than V
], ids=["ragged", "ignore10", "outliers-sum", "longK", "tile+1", "strip>V"])
def test_bf16_reduced_workloads(cuda_lib, w):
    parity_case(w)


@pytest.fixture
def tile_config(cuda_lib):
    """Force one tile variant of the tensor-core kernels for a test, then restore automatic."""
    def set_(cfg):
        assert cuda_lib.lce_set_tile_config(cfg) == 0
    yield set_
    cuda_lib.lce_set_tile_config(0)


@pytest.mark.parametrize("cfg", [1, 2], ids=["single-cta", "cta-pair"])
@pytest.mark.parametrize("w", [
    W2.with_sizes(N=300, d=136, V=1000, strip_V=384),
    W3.with_sizes(N=517, d=256, V=2048, strip_V=512),
    W5.with_sizes(N=640, d=320, V=2500, strip_V=1024),
    W2.with_sizes(N=129, d=64, V=257, strip_V=128),
    W2.with_sizes(N=40, d=64, V=700, strip_V=384),
], ids=["ragged", "ignore10", "outliers-sum", "tile+1", "N<128"])
def test_bf16_each_tile_variant(cuda_lib, tile_config, cfg, w):
    """Both tile variants (single-CTA 128x256 and CTA-pair 256x256) match the oracle on ragged
    shapes, including GEMMs with fewer rows than one tile of the variant."""
    tile_config(cfg)
    parity_case(w)


def test_tile_variants_agree(cuda_lib, tile_config):
    w = W4.with_sizes(N=700, d=192, V=3000, strip_V=1024)
    H, W, y = make_inputs(w, "cpu")
    out = {}
    for cfg in (1, 2):
        tile_config(cfg)
        out[cfg] = run_gpu(H, W, y, 1024, "mean")
    assert abs(out[1]["loss"] - out[2]["loss"]) <= 1e-5 * abs(out[1]["loss"])
    assert np.max(np.abs(out[1]["lse"] - out[2]["lse"])) <= 1e-4
    assert rel_fro(out[2]["dH"], out[1]["dH"]) <= 1e-3
    assert rel_fro(out[2]["dW"], out[1]["dW"]) <= 1e-3


@pytest.mark.parametrize("w", [
    WT.with_sizes(N=100, d=72, V=1000, strip_V=384),
    WT.with_sizes(N=70, d=8, V=130, strip_V=128, reduction="sum"),
], ids=["f32-ragged", "f32-min-d-sum"])
def test_fp32_reduced(cuda_lib, w):
    parity_case(w)


@pytest.mark.parametrize("cfg", [1, 2], ids=["single-cta", "cta-pair"])
@pytest.mark.parametrize("w", [
    WT.with_sizes(N=300, d=136, V=1000, strip_V=384),      # ragged N, d (K tail), V, strips
    WT.with_sizes(N=517, d=256, V=2048, strip_V=512, ignore_frac=0.1),
    WT.with_sizes(N=129, d=64, V=257, strip_V=128, reduction="sum"),
    WT.with_sizes(N=40, d=8, V=700, strip_V=256),          # N < 128, minimum d
    WT.with_sizes(N=256, d=1024, V=600, strip_V=1024),     # long K loop, one strip wider than V
    WT.with_sizes(N=1000, d=96, V=5000, strip_V=128),      # forward strip by strip, many strips
], ids=["ragged", "ignore10", "tile+1-sum", "N<128-d8", "longK-strip>V", "strip128"])
def test_tf32x3_each_tile_variant(cuda_lib, tile_config, cfg, w):
    """fp32 inputs on the tensor cores (three tf32 products of hi / lo parts): the oracle at the
    fp32 tolerances, with both tile variants, on ragged shapes."""
    tile_config(cfg)
    parity_case(w, f32_mode="tf32x3")


def test_tf32x3_matches_exact_fp32(cuda_lib):
    """The two fp32 paths agree with each other far below the bf16 error level."""
    w = WT.with_sizes(N=700, d=512, V=3000, strip_V=1024)
    H, W, y = make_inputs(w, "cpu")
    a = run_gpu(H, W, y, 1024, "mean", f32_mode="exact")
    b = run_gpu(H, W, y, 1024, "mean", f32_mode="tf32x3")
    assert abs(a["loss"] - b["loss"]) <= 1e-5 * abs(a["loss"])
    assert np.max(np.abs(a["lse"] - b["lse"])) <= 1e-4
    assert rel_fro(b["dH"], a["dH"]) <= 1e-4
    assert rel_fro(b["dW"], a["dW"]) <= 1e-4


@pytest.mark.parametrize("strip", [128, 256, 1024, 4096])
def test_strip_width_invariance(cuda_lib, strip):
    """Only the order changes with the strip width: every width matches one oracle result."""
    w = W4.with_sizes(N=600, d=128, V=3001, strip_V=strip)
    H, W, y = make_inputs(w, "cpu")
    r = run_oracle(H, W, y, "mean")
    g = run_gpu(H, W, y, strip, "mean")
    assert_parity(g, r, "bf16")


@pytest.mark.parametrize("w", [
    W4.with_sizes(N=300, d=64, V=40000, strip_V=128),
    W4.with_sizes(N=1000, d=128, V=70000, strip_V=512),
    WT.with_sizes(N=64, d=32, V=10000, strip_V=128),
], ids=["bf16-strip128", "bf16-strip1024", "f32-strip128"])
def test_forward_strip_by_strip(cuda_lib, w):
    """Strips much narrower than V/64: the per-tile partial states of the whole vocabulary no
    longer fit in the workspace, so the forward runs one launch per strip."""
    bn = 256 if w.dtype == "bf16" else 128
    tiles_all = -(-w.V // bn)
    ws = api.lce_workspace_size(w.N, w.d, w.V, w.strip_V, w.dtype)
    assert 256 + tiles_all * w.N * 8 > ws
    parity_case(w)


@pytest.mark.parametrize("dtype_name", ["bf16", "f32", "tf32x3"])
def test_edge_single_token_and_tiny_vocab(cuda_lib, dtype_name):
    base = W2 if dtype_name == "bf16" else WT
    mode = "tf32x3" if dtype_name == "tf32x3" else "exact"
    for N, d, V in [(1, 8, 1), (1, 16, 2), (3, 8, 5), (130, 24, 1)]:
        w = base.with_sizes(N=N, d=d, V=V, strip_V=128)
        H, W, y = make_inputs(w, "cpu")
        g = run_gpu(H, W, y, 128, "mean", f32_mode=mode)
        r = run_oracle(H, W, y, "mean")
        if V == 1:
            assert abs(g["loss"]) < 1e-6
            assert np.abs(g["dH"]).max() < 1e-6 and np.abs(g["dW"]).max() < 1e-6
            assert np.allclose(g["lse"], r["lse"], rtol=1e-3, atol=1e-3)
        else:
            assert_parity(g, r, dtype_name)


@pytest.mark.parametrize("dtype_name", ["bf16", "tf32x3"])
def test_empty_batch(cuda_lib, dtype_name):
    w = (W2 if dtype_name == "bf16" else WT).with_sizes(N=0, d=64, V=300, strip_V=128)
    H, W, y = make_inputs(w, "cpu")
    mode = "tf32x3" if dtype_name == "tf32x3" else "exact"
    for red in ("mean", "sum"):
        g = run_gpu(H, W, y, 128, red, f32_mode=mode)
        assert g["n_valid"] == 0
        assert np.isnan(g["loss"]) if red == "mean" else g["loss"] == 0.0
        assert g["dH"].shape == (0, 64)
        assert np.all(g["dW"] == 0)


def test_all_rows_ignored(cuda_lib):
    w = W2.with_sizes(N=200, d=64, V=700, strip_V=256)
    H, W, y = make_inputs(w, "cpu")
    y[:] = -100
    g = run_gpu(H, W, y, 256, "mean")
    r = run_oracle(H, W, y, "mean")
    assert np.isnan(g["loss"]) and g["n_valid"] == 0
    assert np.all(g["dH"] == 0) and np.all(g["dW"] == 0)
    assert np.max(np.abs(g["lse"] - r["lse"]) / np.abs(r["lse"])) < 1e-3


# (input format, f32_mode): bf16 on the tensor cores, fp32 exact on the CUDA cores, fp32 as three
# tf32 products on the tensor cores
FORMATS = [("bf16", "exact"), ("f32", "exact"), ("f32", "tf32x3")]
FORMAT_IDS = ["bf16", "f32", "tf32x3"]


def _as_format(w, fmt):
    """The same workload distributions with H and W in the given input format."""
    return w if fmt == w.dtype else w.with_sizes(dtype=fmt)


@pytest.mark.parametrize("fmt,mode", FORMATS, ids=FORMAT_IDS)
def test_custom_ignore_index(cuda_lib, fmt, mode):
    w = _as_format(W3.with_sizes(N=300, d=96, V=900, strip_V=256), fmt)
    H, W, y = make_inputs(w, "cpu")
    y[y == -100] = 7  # the ignored rows now carry label 7, which is the ignore_index below
    g = run_gpu(H, W, y, 256, "mean", ignore_index=7, f32_mode=mode)
    r = run_oracle(H, W, y, "mean", ignore_index=7)
    assert_parity(g, r, "tf32x3" if mode == "tf32x3" else fmt)


@pytest.mark.parametrize("fmt,mode", FORMATS, ids=FORMAT_IDS)
def test_bad_label_is_reported_and_row_excluded(cuda_lib, fmt, mode):
    w = _as_format(W2.with_sizes(N=300, d=64, V=600, strip_V=256), fmt)
    H, W, y = make_inputs(w, "cpu")
    y[5] = 600      # == V
    y[17] = -3      # negative, not ignore_index
    y[290] = 10**9  # far out of range, in the last row tile
    with pytest.raises(LceError) as e:
        run_gpu(H, W, y, 256, "mean", f32_mode=mode)
    assert e.value.name == "LCE_ERR_LABEL_OUT_OF_RANGE"
    g = run_gpu(H, W, y, 256, "mean", check=False, f32_mode=mode)
    r = run_oracle(H, W, y, "mean")
    assert r["n_valid"] == 297
    assert_parity(g, r, "tf32x3" if mode == "tf32x3" else fmt)
    assert np.all(g["dH"][[5, 17, 290]] == 0)


@pytest.mark.parametrize("fmt,mode", FORMATS, ids=FORMAT_IDS)
def test_bitwise_deterministic(cuda_lib, fmt, mode):
    w = _as_format(W5.with_sizes(N=700, d=192, V=3000, strip_V=1024), fmt)
    H, W, y = make_inputs(w, "cpu")
    a = run_gpu(H, W, y, 1024, "sum", f32_mode=mode)
    b = run_gpu(H, W, y, 1024, "sum", f32_mode=mode)
    assert a["loss"] == b["loss"]
    for k in ("lse", "dH", "dW"):
        assert np.array_equal(a[k], b[k]), k


def test_gradient_invariants_on_gpu_output(cuda_lib):
    """sum_v dW_v = 0 (rows of softmax - onehot sum to 0) and <dW, W> = <dH, H> (both equal
    sum_iv G_iv Z_iv), checked on the GPU outputs."""
    w = W2.with_sizes(N=512, d=256, V=4000, strip_V=1024)
    H, W, y = make_inputs(w, "cpu")
    g = run_gpu(H, W, y, 1024, "mean")
    colsum = np.abs(g["dW"].sum(axis=0)).max()
    assert colsum <= 1e-2 * np.abs(g["dW"]).sum(axis=0).max()
    Hn, Wn = H.double().numpy(), W.double().numpy()
    a = float((g["dW"] * Wn).sum())
    b = float((g["dH"] * Hn).sum())
    assert abs(a - b) <= 1e-2 * max(abs(a), abs(b))


def test_autograd_function_matches(cuda_lib):
    w = W3.with_sizes(N=333, d=128, V=1500, strip_V=512)
    H, W, y = make_inputs(w, "cpu")
    Hd = H.cuda().requires_grad_(True)
    Wd = W.cuda().requires_grad_(True)
    loss = api.linear_cross_entropy(Hd, Wd, y.cuda(), strip_V=512)
    loss.backward()
    r = run_oracle(H, W, y, "mean")
    assert abs(loss.item() - r["loss"]) <= 1e-3 * abs(r["loss"])
    assert Hd.grad.dtype == torch.bfloat16 and Wd.grad.dtype == torch.bfloat16
    assert rel_fro(Hd.grad.double().cpu().numpy(), r["dH"]) <= 1.5e-2
    assert rel_fro(Wd.grad.double().cpu().numpy(), r["dW"]) <= 1.5e-2


def test_autograd_function_tf32x3(cuda_lib):
    """fp32 tensors through the autograd function on the tensor-core fp32 path: fp32 gradients at
    the fp32 tolerances."""
    w = WT.with_sizes(N=333, d=128, V=1500, strip_V=512)
    H, W, y = make_inputs(w, "cpu")
    Hd = H.cuda().requires_grad_(True)
    Wd = W.cuda().requires_grad_(True)
    loss = api.linear_cross_entropy(Hd, Wd, y.cuda(), strip_V=512, f32_mode="tf32x3")
    loss.backward()
    r = run_oracle(H, W, y, "mean")
    assert abs(loss.item() - r["loss"]) <= 1e-5 * abs(r["loss"])
    assert Hd.grad.dtype == torch.float32 and Wd.grad.dtype == torch.float32
    assert rel_fro(Hd.grad.double().cpu().numpy(), r["dH"]) <= 1e-4
    assert rel_fro(Wd.grad.double().cpu().numpy(), r["dW"]) <= 1e-4


def test_workspace_bound_and_peak_memory(cuda_lib):
    """The workspace grows with strip_V, not V, and the measured peak of a forward+backward is the
    inputs + outputs + one workspace -- far below the N x V fp32 logits."""
    N, d, V = 4096, 256, 65536
    sizes = [api.lce_workspace_size(N, d, V, s) for s in (1024, 2048, 4096)]
    assert sizes[0] < sizes[1] < sizes[2]
    assert api.lce_workspace_size(N, d, 2 * V, 4096) == sizes[2]
    w = W2.with_sizes(N=N, d=d, V=V, strip_V=2048)
    H, W, y = make_inputs(w, "cuda")
    torch.cuda.synchronize()
    dH = torch.empty(N, d, device="cuda")
    dW = torch.empty(V, d, device="cuda")
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    loss, lse, nv, ws = api.lce_forward(H, W, y, strip_V=2048)
    api.lce_backward(H, W, y, lse, nv, torch.ones((), device="cuda"), strip_V=2048, workspace=ws,
                     dH=dH, dW=dW)
    torch.cuda.synchronize()
    extra = torch.cuda.max_memory_allocated() - base
    assert extra <= sizes[1] + 4 * N * 4 + 4096 + 2 * 1024 * 1024
    assert extra < N * V * 4 / 10


@pytest.mark.parametrize("w,mode", [
    (W2.with_sizes(N=300, d=136, V=1000, strip_V=384), "exact"),     # bf16, overlapped steps
    (W2.with_sizes(N=4352, d=8192, V=700, strip_V=512), "exact"),    # bf16, 17 x 32 dH tiles: 3 launches/strip
    (WT.with_sizes(N=100, d=72, V=1000, strip_V=384), "exact"),      # fp32 CUDA cores
    (WT.with_sizes(N=300, d=136, V=1000, strip_V=384), "tf32x3"),    # fp32 tensor cores
], ids=["bf16-overlap", "bf16-large-step", "f32", "tf32x3"])
def test_backward_parts_match_fused_bitwise(cuda_lib, w, mode):
    """Delayed weight gradient: dH alone and dW alone (lce_backward_parts) are bitwise the dH and
    dW of the fused backward, and the gradient not asked for is not produced."""
    H, W, y = make_inputs(w, "cuda")
    kw = dict(strip_V=w.strip_V, reduction=w.reduction, f32_mode=mode)
    loss, lse, nv, ws = api.lce_forward(H, W, y, **kw)
    one = torch.ones((), device="cuda")
    dH, dW, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws, **kw)
    dH1, no_dW, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws, parts="dh", **kw)
    no_dH, dW2, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws, parts="dw", **kw)
    api.lce_check_error(ws)
    assert no_dW is None and no_dH is None
    assert torch.equal(dH, dH1)
    assert torch.equal(dW, dW2)
    r = run_oracle(H.cpu(), W.cpu(), y.cpu(), w.reduction)
    tol = 1e-2 if w.dtype == "bf16" else 1e-4
    assert rel_fro(dH1.cpu().double().numpy(), r["dH"]) <= tol
    assert rel_fro(dW2.cpu().double().numpy(), r["dW"]) <= tol


@pytest.mark.parametrize("mode", ["exact", "tf32x3"])
def test_backward_parts_empty_batch(cuda_lib, mode):
    """No token: the dW-only call writes dW = 0, the dH-only call has nothing to write."""
    w = (W2 if mode == "exact" else WT).with_sizes(N=0, d=64, V=300, strip_V=128)
    H, W, y = make_inputs(w, "cuda")
    kw = dict(strip_V=128, f32_mode=mode)
    loss, lse, nv, ws = api.lce_forward(H, W, y, **kw)
    one = torch.ones((), device="cuda")
    dW = torch.full((300, 64), 7.0, device="cuda")
    _, dW2, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws, dW=dW, parts="dw", **kw)
    dH1, _, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws, parts="dh", **kw)
    api.lce_check_error(ws)
    assert torch.count_nonzero(dW2).item() == 0
    assert dH1.shape == (0, 64)


def _random_shapes(seed, count, d_mult=8):
    """Seeded random small shapes: odd token counts, hidden sizes of any multiple of d_mult (the
    16-byte row rule: 8 for bf16, 4 for fp32), vocabulary sizes with ragged tails, strip widths of
    128..1024, both reductions."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        N = int(rng.integers(1, 900))
        d = d_mult * int(rng.integers(1, 384 // d_mult))
        V = int(rng.integers(2, 4000))
        strip = 128 * int(rng.integers(1, 9))
        red = "sum" if rng.random() < 0.5 else "mean"
        out.append((N, d, V, strip, red))
    return out


@pytest.mark.parametrize("fmt,mode", FORMATS, ids=FORMAT_IDS)
def test_random_shapes(cuda_lib, fmt, mode):
    """Eight seeded random shapes per input format, each against the oracle at its tolerances."""
    base = W2 if fmt == "bf16" else WT
    seed = 20261202 + {"bf16": 1, "f32": 2}[fmt] + (10 if mode == "tf32x3" else 0)
    for N, d, V, strip, red in _random_shapes(seed, 8, 8 if fmt == "bf16" else 4):
        w = base.with_sizes(N=N, d=d, V=V, strip_V=strip, reduction=red)
        parity_case(w, f32_mode=mode)


@pytest.mark.parametrize("mode", ["exact", "tf32x3"])
@pytest.mark.parametrize("N,d,V,strip", [(37, 4, 300, 128), (129, 12, 1000, 256),
                                         (300, 36, 777, 512), (513, 260, 1500, 1024)])
def test_fp32_hidden_size_multiple_of_four(cuda_lib, mode, N, d, V, strip):
    """fp32 rows need only be 16 bytes a multiple: hidden sizes that are multiples of 4 but not of
    8, down to d = 4 (one float4 a row, a single ragged k-block on either engine)."""
    for red in ("mean", "sum"):
        parity_case(WT.with_sizes(N=N, d=d, V=V, strip_V=strip, reduction=red), f32_mode=mode)


@pytest.mark.parametrize("mode", ["exact", "tf32x3"])
def test_dgrad_and_wgrad_on_two_streams(cuda_lib, mode):
    """The delayed weight gradient in use: dH on one stream and dW on another, in flight together
    (each call with its own workspace), give bitwise the fused backward's dH and dW."""
    w = (W2 if mode == "exact" else WT).with_sizes(N=2048, d=256, V=5000, strip_V=1024)
    H, W, y = make_inputs(w, "cuda")
    kw = dict(strip_V=w.strip_V, reduction=w.reduction, f32_mode=mode)
    loss, lse, nv, ws = api.lce_forward(H, W, y, **kw)
    one = torch.ones((), device="cuda")
    dH_ref, dW_ref, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws, **kw)
    torch.cuda.synchronize()
    ws2 = torch.empty_like(ws)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    dH, _, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws, parts="dh", stream=s1, **kw)
    _, dW, _ = api.lce_backward(H, W, y, lse, nv, one, workspace=ws2, parts="dw", stream=s2, **kw)
    torch.cuda.synchronize()
    api.lce_check_error(ws)
    api.lce_check_error(ws2)
    assert torch.equal(dH, dH_ref)
    assert torch.equal(dW, dW_ref)
