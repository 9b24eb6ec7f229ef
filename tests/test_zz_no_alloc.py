"""The allocation-free entry point, called through the C ABI.

attn_prefill_fwd_noalloc serves callers that cannot have the library allocate
device memory: code whose device memory all comes from its own pool or arena
(a cudaMalloc behind its back would escape that pool's accounting and
limits), or a framework that owns the allocator and forbids libraries to
call it. It keeps the kernel's status word in a fixed array inside the
library instead of a cudaMalloc'd buffer.

Checked here: two calls in a row against the fp64 oracle (and against
attn_prefill_fwd on the same inputs, since the array is shared and keeps the
previous call's contents); a wait that runs out in this variant is reported
by attn_device_check; and, in a fresh process whose first library call is
this entry point, the device's free memory is the same before and after it.

This file is named so that pytest collects it last; it also passes alone in a
fresh process, where its first call performs the one-time device set-up.
"""

import json
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

from causal_gqa_prefill_gb300 import (ATTN_ERR_TIMEOUT, ATTN_OK, _abi, attn_device_check,
                                      attn_prefill_fwd, attn_selftest_wait_timeout_noalloc)
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import assert_within, check_full, errors, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc(q, k, v, o, lse, w, stream):
    lib = _abi.load()
    return int(lib.attn_prefill_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
        w.B, w.L, w.n_q, w.n_kv, w.d_h, int(w.causal), w.d_h ** -0.5, int(stream.cuda_stream)))


def _setup():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    return torch.cuda.current_stream()


def test_noalloc_matches_oracle_twice():
    stream = _setup()
    cases = [W.custom(1, 1000, 8, 2, 128), W.custom(2, 333, 4, 1, 64)]
    for n, w in enumerate(cases):          # two calls in a row, different shapes
        q, k, v = W.make_inputs(w, "cuda", seed=500 + n)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.n_q, w.L), float("nan"), device="cuda")
        assert _noalloc(q, k, v, o, lse, w, stream) == ATTN_OK
        assert attn_device_check(stream) == ATTN_OK
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()
        check_full(q, k, v, o, lse, causal=True, scale=w.scale, what=f"noalloc call {n}")
        # the allocating entry point on the same inputs
        o_ref = torch.empty_like(q)
        l_ref = torch.empty(w.B, w.n_q, w.L, device="cuda")
        assert attn_prefill_fwd(q, k, v, o_ref, l_ref, w.B, w.L, w.n_q, w.n_kv, w.d_h,
                                int(w.causal), w.scale, stream) == ATTN_OK
        assert attn_device_check(stream) == ATTN_OK
        err = errors(to_np(o), lse.cpu().numpy().astype(np.float64), to_np(o_ref),
                     l_ref.cpu().numpy().astype(np.float64))
        assert_within(err, f"noalloc call {n} against attn_prefill_fwd")


def test_noalloc_wait_timeout_is_reported():
    stream = _setup()
    assert attn_device_check(stream) == ATTN_OK                 # nothing pending
    assert attn_selftest_wait_timeout_noalloc(1 << 18, stream) == ATTN_OK
    assert attn_device_check(stream) == ATTN_ERR_TIMEOUT        # the fixed word said so
    assert attn_device_check(stream) == ATTN_OK                 # and reading cleared it
    # the context still runs the allocation-free forward correctly
    w = W.custom(1, 300, 4, 2, 128)
    q, k, v = W.make_inputs(w, "cuda", seed=77)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.n_q, w.L, device="cuda")
    assert _noalloc(q, k, v, o, lse, w, stream) == ATTN_OK
    assert attn_device_check(stream) == ATTN_OK
    check_full(q, k, v, o, lse, causal=True, scale=w.scale, what="noalloc after a timeout")


_CHILD = r"""
import json, os, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from causal_gqa_prefill_gb300 import _abi
lib = _abi.load()                       # loaded before the process's first CUDA call
import torch
from causal_gqa_prefill_gb300 import workloads as W
torch.cuda.set_device(0)
stream = torch.cuda.current_stream()
w = W.custom(1, 1000, 8, 2, 128)
q, k, v = W.make_inputs(w, "cuda", seed=901)
out = []
for _ in range(2):
    out.append((torch.full_like(q, float("nan")),
                torch.full((w.B, w.n_q, w.L), float("nan"), device="cuda")))
torch.cuda.synchronize()
free = [torch.cuda.mem_get_info()[0]]
status = []
for o, lse in out:                      # the library's first call, then a second one
    status.append(int(lib.attn_prefill_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
        w.B, w.L, w.n_q, w.n_kv, w.d_h, 1, w.d_h ** -0.5, int(stream.cuda_stream))))
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
status.append(int(lib.attn_device_check(int(stream.cuda_stream))))
d = sys.argv[2]
for t, name in ((q, "q"), (k, "k"), (v, "v"), (out[0][0], "o0"), (out[1][0], "o1")):
    np.save(os.path.join(d, name + ".npy"), t.float().cpu().numpy())
for t, name in ((out[0][1], "lse0"), (out[1][1], "lse1")):
    np.save(os.path.join(d, name + ".npy"), t.cpu().numpy())
print(json.dumps({"free": free, "status": status}))
"""


def test_noalloc_first_call_in_fresh_process_allocates_nothing():
    _setup()                                # builds the library if needed
    env = dict(os.environ)
    # load every module of the library with the context, so that no module
    # load by the driver lands between the two free-memory readings
    env["CUDA_MODULE_LOADING"] = "EAGER"
    with tempfile.TemporaryDirectory() as d:
        res = subprocess.run([sys.executable, "-c", _CHILD, ROOT, d], env=env,
                             capture_output=True, text=True, timeout=600)
        assert res.returncode == 0, res.stderr[-3000:]
        rec = json.loads(res.stdout.strip().splitlines()[-1])
        assert rec["status"] == [ATTN_OK, ATTN_OK, ATTN_OK], rec
        free = rec["free"]
        # a cudaMalloc of even 256 bytes takes a whole 2 MiB page from the device
        assert free[1] == free[0] and free[2] == free[0], rec
        ld = lambda name: np.load(os.path.join(d, name + ".npy")).astype(np.float64)
        import oracle
        w = W.custom(1, 1000, 8, 2, 128)
        o_ref, lse_ref = oracle.attention(ld("q"), ld("k"), ld("v"), causal=True, scale=w.scale)
        for n in ("0", "1"):
            assert_within(errors(ld("o" + n), ld("lse" + n), o_ref, lse_ref),
                          f"fresh-process noalloc call {n}")
