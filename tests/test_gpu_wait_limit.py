"""Failure detection on the GPU without a fault: a device-side wait that runs
past its limit must end the kernel with an error status the host can read,
and leave the CUDA context usable.

The diagnostic entry point runs the attention kernels' own bounded wait on an
mbarrier that nothing completes (limit 2^20 cycles, about half a millisecond),
so the wait is certain to run out; a second warp waiting on another such
barrier must leave through the abort flag the first one raises.
"""

import numpy as np
import pytest

import oracle
from causal_gqa_prefill_gb300 import (ATTN_ERR_TIMEOUT, ATTN_OK, attn_device_check, attn_prefill,
                                      attn_selftest_wait_timeout)
from causal_gqa_prefill_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_limit_reports_timeout_and_context_survives():
    assert attn_device_check() == ATTN_OK                      # nothing pending
    assert attn_selftest_wait_timeout(1 << 20) == ATTN_OK
    assert attn_device_check() == ATTN_ERR_TIMEOUT             # the wait gave up and said so
    assert attn_device_check() == ATTN_OK                      # reading cleared the word
    # the context still runs the real kernel correctly
    w = W.custom(1, 300, 4, 2, 128, number=1401)
    q, k, v = W.make_inputs(w)
    o, lse = attn_prefill(q, k, v)
    assert attn_device_check() == ATTN_OK
    ref_o, ref_lse = oracle.attention(*(t.float().cpu().numpy().astype(np.float64) for t in (q, k, v)),
                                      causal=True, scale=w.scale)
    assert np.abs(o.float().cpu().numpy() - ref_o).max() <= 1e-2
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3


def test_wait_limit_repeats():
    for _ in range(3):
        assert attn_selftest_wait_timeout(1 << 16) == ATTN_OK
        assert attn_device_check() == ATTN_ERR_TIMEOUT
    assert attn_device_check() == ATTN_OK
