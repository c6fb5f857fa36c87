"""Host-side checks of the C ABI, no GPU needed: the library loads, exports every symbol that
include/lce.h declares, sizes its workspace, and rejects bad arguments before launching anything
(every call below returns from host validation; none reaches the CUDA runtime)."""

import ctypes
import os

import pytest

from memory_bounded_linear_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from memory_bounded_linear_gb300.csrc import build
        build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    declared = _lib.header_symbols()
    assert set(declared) >= {"lce_workspace_size", "lce_forward", "lce_backward",
                             "lce_check_error", "lce_status_string"}
    for name in declared:
        assert hasattr(lib, name), name
    assert set(_lib._SIGNATURES) >= set(declared)


def test_status_strings_and_kernel_names(lib):
    for code, name in _lib.STATUS_NAMES.items():
        s = lib.lce_status_string(code)
        assert s and s != b"unknown status", name
    assert lib.lce_status_string(99) == b"unknown status"
    assert lib.lce_kernel_name(0) == b"tc_fwd_lse"
    assert lib.lce_kernel_name(1) == b"tc_bwd"
    assert lib.lce_kernel_name(8) == b"split_tf32"
    assert lib.lce_kernel_name(9) == b"tc_bwd_grad"
    assert lib.lce_kernel_name(10) == b"tc_dh_dw"
    assert lib.lce_kernel_name(-1) is None and lib.lce_kernel_name(1000) is None


def _ws(lib, N, d, V, s, dt=0):
    return lib.lce_workspace_size(N, d, V, s, dt)


def _strip(V, s, bn):
    """The strip width the header states: ceil(V / s) strips of equal width, rounded up to the
    engine's tile width bn when that stays within s, else to 128; at most V."""
    S = -(-V // s)
    even = -(-V // S)
    w = -(-even // bn) * bn
    if w > s:
        w = -(-even // 128) * 128
    return min(w, V)


@pytest.mark.parametrize("V,s,bn,want", [(151552, 16384, 256, 15360), (151936, 8192, 256, 8192),
                                         (151936, 4096, 256, 4096), (151936, 32768, 256, 30464),
                                         (200000, 16384, 256, 15616), (1000, 384, 256, 384),
                                         (300, 4096, 256, 300), (40000, 128, 256, 128),
                                         (4096, 512, 128, 512), (131072, 16384, 256, 16384)])
def test_strip_columns(lib, V, s, bn, want):
    """Equal strips: the last strip is never a sliver, no strip is wider than strip_V."""
    assert _strip(V, s, bn) == want
    dt = 0 if bn == 256 else 1
    assert lib.lce_strip_columns(V, s, dt) == want
    S = -(-V // want)
    assert want <= s and S == -(-V // s)          # as many strips as strip_V gives
    assert V - (S - 1) * want > 0                  # the last strip is not empty
    assert lib.lce_strip_columns(V, 100, 0) == 0 and lib.lce_strip_columns(0, 128, 0) == 0


def test_workspace_size_formula(lib):
    # bf16, large backward step (128 x 24 dH tiles > 512): header + max(forward state, one strip
    # of bf16 gradient rows padded to 256 columns)
    N, d, V, s = 32768, 6144, 151552, 16384
    g_bytes = N * 15360 * 2   # ten strips of 15360 columns (the last one 13312)
    assert _ws(lib, N, d, V, s) == 256 + g_bytes
    # bf16, small backward step (16 x 8 dH tiles): two gradient strips, consecutive strips overlap
    assert _ws(lib, 4096, 2048, 151936, 8192) == 256 + 2 * 4096 * 8192 * 2
    # fp32 engine: 128-wide tiles, one fp32 gradient strip
    assert _ws(lib, 256, 256, 4096, 512, 1) == 256 + 256 * 512 * 4
    # strip wider than V: the strip is V wide (padded to the tile width)
    assert _ws(lib, 100, 64, 300, 4096) == 256 + max(
        ((100 * 8 + 255) // 256 * 256) + ((100 * 4 + 255) // 256 * 256) + ((2 * 100 * 8 + 255) // 256 * 256),
        2 * ((100 * 512 * 2 + 255) // 256 * 256))


def test_workspace_size_tf32x3(lib):
    # three-product tf32 path: header; hi / lo parts of H and of one W strip; then the larger of
    # the forward region and the backward one (hi / lo parts of H^T, of the W strip transposed,
    # of the gradient strip and of the gradient strip transposed)
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for N, d, V, s in [(16384, 7168, 200000, 16384), (100, 64, 300, 4096), (33, 8, 1000, 128)]:
        w = _strip(V, s, 256)
        ldg = (w + 255) // 256 * 256
        ldt = (N + 31) // 32 * 32
        split = 2 * r(N * d * 4) + 2 * r(w * d * 4)
        fwd = r(N * 8) + r(N * 4) + r((ldg // 256) * N * 8)
        bwd = 2 * (r(d * ldt * 4) + r(d * ldg * 4) + r(N * ldg * 4) + r(ldg * ldt * 4))
        assert _ws(lib, N, d, V, s, 2) == 256 + split + max(fwd, bwd), (N, d, V, s)
    assert _ws(lib, 100, 64, 300, 4096, 3) == 0  # unknown dtype


def test_workspace_is_bounded_by_strip_not_vocab(lib):
    a = _ws(lib, 65536, 2048, 151936, 4096)
    b = _ws(lib, 65536, 2048, 10 * 151936, 4096)
    assert a == b
    sweep = [_ws(lib, 65536, 2048, 151936, s) for s in (4096, 8192, 16384, 32768)]
    assert all(x < y for x, y in zip(sweep, sweep[1:]))
    assert sweep[-1] < 65536 * 151936 * 4 / 4   # well under the N x V fp32 logits


@pytest.mark.parametrize("N,d,V,s", [(-1, 64, 100, 128), (10, 7, 100, 128), (10, 12, 100, 128),
                                     (10, 64, 0, 128), (10, 64, 100, 64), (10, 64, 100, 200),
                                     (1 << 31, 64, 100, 128)])
def test_workspace_size_rejects_bad_shapes(lib, N, d, V, s):
    assert _ws(lib, N, d, V, s) == 0


@pytest.mark.parametrize("d,accepted", [(4, (False, True, True)), (6, (False, False, False)),
                                        (8, (True, True, True)), (12, (False, True, True)),
                                        (20, (False, True, True)), (1028, (False, True, True))])
def test_hidden_size_rule_is_sixteen_bytes_a_row(lib, d, accepted):
    """A row of d elements must be a multiple of 16 bytes: d % 8 == 0 for bf16, d % 4 == 0 for
    both fp32 formats."""
    p = _Buf().addr
    for dt, ok in zip((0, 1, 2), accepted):
        assert (_ws(lib, 100, d, 1000, 256, dt) > 0) == ok, (d, dt)
        # the entry point agrees: an accepted shape gets as far as the workspace-size check
        assert _fwd(lib, p, p, p, N=100, d=d, V=1000, s=256, dt=dt, wsb=100) == (3 if ok else 2)


class _Buf:
    """Host memory that stands in for device pointers; validation fails before any access."""

    def __init__(self, n=1 << 16):
        self.raw = ctypes.create_string_buffer(n + 64)
        self.addr = (ctypes.addressof(self.raw) + 63) // 64 * 64


def _fwd(lib, H, W, y, N=16, d=64, V=300, s=128, red=0, dt=0, ws=None, wsb=1 << 20,
         loss=None, lse=None, nv=None):
    b = _Buf()
    ws = b.addr if ws is None else ws
    return lib.lce_forward(H, W, y, N, d, V, -100, s, red, dt,
                           b.addr if loss is None else loss, b.addr if lse is None else lse,
                           b.addr if nv is None else nv, ws, wsb, None)


def test_forward_validation(lib):
    b = _Buf()
    p = b.addr
    assert _fwd(lib, p, p, p, red=2) == 1                 # unknown reduction
    assert _fwd(lib, p, p, p, dt=5) == 1                  # unknown dtype
    assert _fwd(lib, p, None, p) == 1                     # null W
    assert _fwd(lib, None, p, p) == 1                     # null H with N > 0
    assert _fwd(lib, p + 4, p, p) == 1                    # misaligned H
    assert _fwd(lib, p, p, p, d=12) == 2                  # d % 8 != 0
    assert _fwd(lib, p, p, p, s=100) == 2                 # strip_V % 128 != 0
    assert _fwd(lib, p, p, p, V=0) == 2
    assert _fwd(lib, p, p, p, wsb=100) == 3               # workspace too small
    assert _fwd(lib, p, p, p, lse=p + 8) == 1             # misaligned lse


def test_backward_validation(lib):
    b = _Buf()
    p = b.addr
    args = dict(N=16, d=64, V=300, s=128)

    def bwd(H=p, W=p, y=p, lse=p, nv=p, dl=p, dH=p, dW=p, red=0, dt=0, wsb=1 << 20, **kw):
        a = dict(args, **kw)
        return lib.lce_backward(H, W, y, lse, nv, dl, a["N"], a["d"], a["V"], -100, a["s"], red, dt,
                                dH, dW, p, wsb, None)

    assert bwd(dl=None) == 1
    assert bwd(dW=None) == 1
    assert bwd(dH=p + 4) == 1
    assert bwd(red=7) == 1
    assert bwd(d=4) == 2
    assert bwd(wsb=16) == 3


def test_backward_parts_validation(lib):
    """The one-gradient backward checks its part mask and needs only the requested output."""
    b = _Buf()
    p = b.addr

    def bwd(parts, dH=p, dW=p, dl=p, wsb=1 << 20, N=16):
        return lib.lce_backward_parts(p, p, p, p, p, dl, N, 64, 300, -100, 128, 0, 0, parts,
                                      dH, dW, p, wsb, None)

    assert bwd(0) == 1 and bwd(4) == 1 and bwd(-1) == 1     # unknown part masks
    assert bwd(1, dH=None) == 1                              # dH requested, missing
    assert bwd(2, dW=None) == 1                              # dW requested, missing
    assert bwd(3, dW=None) == 1
    assert bwd(1, dH=p + 4) == 1                             # misaligned requested output
    assert bwd(2, dl=None) == 1
    assert bwd(1, wsb=16) == 3


def test_check_error_and_trace_argument_validation(lib):
    assert lib.lce_check_error(None, None) == 1
    assert lib.lce_trace_begin(None, None, None, 4) == 1
    assert lib.lce_trace_begin(None, None, None, 0) == 0
    assert lib.lce_trace_end() == 0
    assert lib.lce_launch_count() >= 0


def test_host_buffer_size_layout(lib):
    """The host-buffer entry point's device buffer: the workspace, then the device copies of the
    inputs and the results, each 256-byte aligned."""
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for (N, d, V, s, dt, elt) in [(32768, 6144, 151552, 16384, 0, 2), (100, 64, 300, 4096, 0, 2),
                                  (256, 256, 4096, 512, 1, 4), (33, 8, 1000, 128, 2, 4),
                                  (0, 64, 300, 128, 0, 2)]:
        ws = _ws(lib, N, d, V, s, dt)
        want = (r(ws) + r(N * d * elt) + r(V * d * elt) + r(N * 8) + 3 * 256 + r(N * 4)
                + r(N * d * 4) + r(V * d * 4))
        assert lib.lce_host_buffer_size(N, d, V, s, dt) == want, (N, d, V, s, dt)
    assert lib.lce_host_buffer_size(100, 60, 300, 128, 0) == 0   # d % 8 != 0 for bf16
    assert lib.lce_host_buffer_size(100, 64, 300, 100, 0) == 0   # strip not a multiple of 128


def test_host_entry_point_rejects_bad_arguments_on_the_host(lib):
    """Every argument error of lce_forward_backward_host comes back before any CUDA call."""
    f = lib.lce_forward_backward_host
    buf = ctypes.create_string_buffer(1 << 20)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256  # stands in for device memory: never touched
    one = (ctypes.c_float * 1)(1.0)
    H = (ctypes.c_uint16 * 64)()
    W = (ctypes.c_uint16 * (64 * 300))()
    y = (ctypes.c_int64 * 1)()
    ok_args = [H, W, y, one, 1, 64, 300, -100, 128, 0, 0, None, None, None, None, None, None,
               addr, 1 << 19, None, None, None]

    def call(**kw):
        a = list(ok_args)
        names = ["H", "W", "y", "dloss", "N", "d", "V", "ign", "strip", "red", "dt", "loss", "lse",
                 "nv", "dH", "dW", "flags", "buf", "bytes", "stream", "after", "done"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return _lib.STATUS_NAMES[f(*a)]

    assert call(red=7) == "LCE_ERR_INVALID_ARG"
    assert call(dt=9) == "LCE_ERR_INVALID_ARG"
    assert call(W=None) == "LCE_ERR_INVALID_ARG"
    assert call(dloss=None) == "LCE_ERR_INVALID_ARG"
    assert call(buf=None) == "LCE_ERR_INVALID_ARG"
    assert call(buf=addr + 8) == "LCE_ERR_INVALID_ARG"         # not 16-byte aligned
    assert call(H=None) == "LCE_ERR_INVALID_ARG"               # N > 0 needs H and labels
    assert call(d=60) == "LCE_ERR_UNSUPPORTED_SHAPE"
    assert call(strip=100) == "LCE_ERR_UNSUPPORTED_SHAPE"
    need = lib.lce_host_buffer_size(1, 64, 300, 128, 0)
    assert call(bytes=need - 1) == "LCE_ERR_WORKSPACE_TOO_SMALL"
