"""The allocation-free entry point, called through the C ABI.

attn_prefill_fwd_noalloc serves callers that cannot have the library allocate
device memory (a caller-owned memory pool or arena that must account for every
allocation, a framework that owns the allocator): it keeps the kernel's status word in a fixed array
inside the library instead of a cudaMalloc'd buffer. Its results must equal
those of attn_prefill_fwd on the same inputs, call after call (the array is
shared and keeps the previous call's contents).

This file is named so that pytest collects it last; it also passes alone in a
fresh process, where its first call performs the one-time device set-up.
"""

import math

import numpy as np
import pytest

from causal_gqa_prefill_gb300 import ATTN_OK, _abi, attn_prefill_fwd, attn_device_check
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import errors, assert_within, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _noalloc(q, k, v, o, lse, w, stream):
    lib = _abi.load()
    return int(lib.attn_prefill_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
        w.B, w.L, w.n_q, w.n_kv, w.d_h, int(w.causal), w.d_h ** -0.5, int(stream.cuda_stream)))


def test_noalloc_matches_allocating_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    cases = [W.custom(1, 1000, 8, 2, 128), W.custom(2, 333, 4, 1, 64)]
    for n, w in enumerate(cases):          # two calls in a row, different shapes
        q, k, v = W.make_inputs(w, "cuda", seed=500 + n)
        o_ref = torch.empty_like(q)
        l_ref = torch.empty(w.B, w.n_q, w.L, device="cuda")
        st = attn_prefill_fwd(q, k, v, o_ref, l_ref, w.B, w.L, w.n_q, w.n_kv, w.d_h,
                              int(w.causal), w.d_h ** -0.5, stream)
        assert st == ATTN_OK
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.n_q, w.L), float("nan"), device="cuda")
        st = _noalloc(q, k, v, o, lse, w, stream)
        assert st == ATTN_OK
        assert attn_device_check(stream) == ATTN_OK
        err = errors(to_np(o), lse.cpu().numpy().astype(np.float64), to_np(o_ref),
                     l_ref.cpu().numpy().astype(np.float64))
        assert_within(err, f"noalloc call {n}")
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()
