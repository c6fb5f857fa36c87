"""Memory-bounded fused linear cross-entropy for GB300 (sm_103a).

The vocabulary projection H W^T and the cross-entropy on top of it are computed strip by strip
over the vocabulary, so the N x V logits never exist in device memory.  All arithmetic runs in
the CUDA library ``liblce.so`` (C ABI declared in ``include/lce.h``); this package only marshals
arguments to it.
"""

from .workloads import WORKLOADS, Workload, make_inputs  # noqa: F401


def full_logits_bytes(tokens: int, vocab: int, bytes_per_element: int = 4) -> int:
    """Bytes a materialised fp32 logits tensor would take: tokens x vocab x 4 (the memory this
    operator avoids)."""
    return int(tokens) * int(vocab) * int(bytes_per_element)


def __getattr__(name):
    # The binding is imported lazily so that host-only users (input recipes, sizes) do not need
    # torch.cuda; it never falls back to anything when the library is missing.
    if name in ("lce_workspace_size", "lce_strip_columns", "lce_forward", "lce_backward", "lce_check_error",
                "lce_host_buffer_size", "lce_forward_backward_host", "lce_launch_count",
                "linear_cross_entropy", "LinearCrossEntropy"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
