"""attn_prefill_fwd_host: the forward over host buffers (copies in, the
device kernel, copies out on one stream) gives bit-for-bit the results of
the device entry point on the same inputs, from pinned and from pageable
host memory, square and chunked."""

import pytest
import torch

from causal_gqa_prefill_gb300 import (ATTN_OK, attn_device_check, attn_prefill,
                                      attn_prefill_fwd_host, attn_prefill_host_staging_bytes)
from causal_gqa_prefill_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("shape", [(2, 300, 300, 8, 2, 128), (1, 200, 520, 4, 1, 64)],
                         ids=["square", "chunk"])
def test_host_entry_matches_device_entry(shape, pinned):
    B, Lq, Lk, n_q, n_kv, d = shape
    w = W.custom(B, Lq, n_q, n_kv, d, Lk=Lk, number=1500 + Lq)
    q, k, v = W.make_inputs(w)
    o_dev, lse_dev = attn_prefill(q, k, v)
    hq, hk, hv = (t.cpu() for t in (q, k, v))
    ho = torch.empty(q.shape, dtype=torch.bfloat16)
    hl = torch.full((B, n_q, Lq), float("nan"), dtype=torch.float32)
    if pinned:
        hq, hk, hv, ho, hl = (t.pin_memory() for t in (hq, hk, hv, ho, hl))
    need = attn_prefill_host_staging_bytes(B, Lq, Lk, n_q, n_kv, d)
    staging = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    st = attn_prefill_fwd_host(hq, hk, hv, ho, hl, staging, need, B, Lq, Lk, n_q, n_kv, d, 1,
                               w.scale, stream)
    assert st == ATTN_OK
    stream.synchronize()
    assert attn_device_check() == ATTN_OK
    assert torch.equal(ho, o_dev.cpu())
    assert torch.equal(hl, lse_dev.cpu())
