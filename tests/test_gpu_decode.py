"""GPU parity of the decode kernel (one new token per sequence against its
cache) against the fp64 oracle: the chunked definition with Lq = 1."""

import numpy as np
import pytest

from causal_gqa_prefill_gb300 import (ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_OK,
                                      attn_decode, attn_decode_fwd, attn_decode_workspace_bytes,
                                      attn_device_check, attn_prefill)
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import check_full

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _decode(q, k, v, **kw):
    o, lse = attn_decode(q, k, v, **kw)
    assert attn_device_check() == ATTN_OK
    return o, lse


DECODE = [
    # B, Lk, n_q, n_kv
    (2, 1000, 8, 2),
    (1, 1, 4, 1),          # a single cached key
    (3, 300, 6, 2),        # g = 3
    (4, 777, 4, 4),        # g = 1
    (1, 2049, 8, 1),       # g = 8, ragged last tile
    (1, 5000, 32, 8),
    (2, 64, 2, 2),         # a partial first tile only
    (1, 128, 4, 1),        # exactly one whole tile
    (3, 700, 10, 5),       # 90 tiles: fewer tiles than CTAs, one tile per CTA
    (2, 20000, 6, 3),      # 942 tiles over 152 CTAs: ranges cross head boundaries
    (1, 3000, 12, 1),      # g = 12
    (2, 1500, 32, 2),      # g = 16
    (64, 100, 16, 1),      # 64 sequences of one partial tile each: 64 CTAs, g = 16
    (40, 3000, 8, 8),      # g = 1, many sequences
]


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "B%d_Lk%d_q%d_kv%d" % c)
def test_decode_small_shapes(case):
    B, Lk, n_q, n_kv = case
    w = W.custom(B, 1, n_q, n_kv, 128, Lk=Lk)
    q, k, v = W.make_inputs(w, "cuda", seed=hash(case) % 100000)
    o, lse = _decode(q, k, v)
    check_full(q, k, v, o, lse, what=str(case))


def test_decode_matches_last_row_of_prefill():
    """The decode step equals the last row of a causal prefill over the whole
    sequence (same keys, same query)."""
    w = W.custom(2, 3000, 8, 2, 128)
    qf, k, v = W.make_inputs(w, "cuda", seed=11)
    o_full, l_full = attn_prefill(qf, k, v)
    o, lse = _decode(qf[:, -1:].contiguous(), k, v)
    assert (o.float() - o_full[:, -1:].float()).abs().max().item() <= 1e-2
    assert (lse - l_full[:, :, -1:]).abs().max().item() <= 1e-3


def test_decode_workspace_is_reused():
    w1 = W.custom(2, 1, 8, 2, 128, Lk=1500)
    ws = torch.empty(attn_decode_workspace_bytes(2, 1500, 8, 2), dtype=torch.uint8, device="cuda")
    for seed in (1, 2):
        q, k, v = W.make_inputs(w1, "cuda", seed=seed)
        o, lse = _decode(q, k, v, workspace=ws)
        check_full(q, k, v, o, lse, what=f"reuse {seed}")


def test_decode_back_to_back_calls():
    """Calls queued on one stream with one workspace and no host sync between
    them. Each call's kernels are programmatic dependents of the kernel before
    them: the next call's split kernel sets up while this call's combine still
    reads the partial results, and the cache is rewritten by a kernel right
    before each call. Every call must still see its own inputs and partials."""
    B, Lk, n_q, n_kv = 2, 20000, 6, 3          # ranges cross head boundaries
    w = W.custom(B, 1, n_q, n_kv, 128, Lk=Lk)
    ws = torch.empty(attn_decode_workspace_bytes(B, Lk, n_q, n_kv), dtype=torch.uint8,
                     device="cuda")
    inputs = [W.make_inputs(w, "cuda", seed=s) for s in (21, 22, 23, 24)]
    kbuf = torch.empty_like(inputs[0][1])
    vbuf = torch.empty_like(inputs[0][2])
    torch.cuda.synchronize()
    outs = []
    for q, k, v in inputs:
        torch.mul(k, 1.0, out=kbuf)             # an elementwise kernel writes the cache
        torch.mul(v, 1.0, out=vbuf)
        outs.append(attn_decode(q, kbuf, vbuf, workspace=ws))
    torch.cuda.synchronize()
    assert attn_device_check() == ATTN_OK
    for i, ((q, k, v), (o, lse)) in enumerate(zip(inputs, outs)):
        check_full(q, k, v, o, lse, what=f"call {i}")


def test_decode_million_token_cache():
    """One new token against 1,000,003 cached keys (a ragged last tile; 7,813
    key tiles per K/V head spread over every CTA)."""
    w = W.custom(1, 1, 8, 1, 128, Lk=1_000_003)
    q, k, v = W.make_inputs(w, "cuda", seed=1000003)
    o, lse = _decode(q, k, v)
    check_full(q, k, v, o, lse, what="Lk=1000003")


@pytest.mark.parametrize("num", [10, 11])
def test_decode_workloads(num):
    w = W.WORKLOADS[num]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = _decode(q, k, v, scale=w.scale)
    err = check_full(q, k, v, o, lse, scale=w.scale, what=w.name)
    print(f"parity {w.name}: {err}")


def test_decode_argument_errors():
    q = torch.zeros(1, 1, 17, 128, device="cuda", dtype=torch.bfloat16)
    kv = torch.zeros(1, 64, 1, 128, device="cuda", dtype=torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 17, 1, device="cuda")
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    assert attn_decode_fwd(q, kv, kv, o, lse, ws, ws.numel(), 1, 64, 17, 1, 128, 0.1) == \
        ATTN_ERR_UNSUPPORTED                                  # g = 17 > 16
    q = torch.zeros(1, 1, 8, 128, device="cuda", dtype=torch.bfloat16)
    need = attn_decode_workspace_bytes(1, 64, 8, 1)
    assert attn_decode_fwd(q, kv, kv, torch.empty_like(q), lse, ws, need - 1, 1, 64, 8, 1, 128,
                           0.1) == ATTN_ERR_INVALID_ARG        # workspace too small
