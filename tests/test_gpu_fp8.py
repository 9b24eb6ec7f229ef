"""GPU parity of the fp8 (e4m3) forward against the fp64 oracle on the exactly
dequantised inputs, with the bound derived in gpu_common (e4m3 rounding of the
softmax weights, bf16 rounding of O)."""

import math

import numpy as np
import pytest

from causal_gqa_prefill_gb300 import (ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_OK,
                                      attn_device_check, attn_prefill, attn_prefill_fp8,
                                      attn_prefill_fwd_fp8)
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import check_fp8_full, check_fp8_rows, dequant

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _run(q, k, v, **kw):
    o, lse = attn_prefill_fp8(q, k, v, **kw)
    assert attn_device_check() == ATTN_OK
    return o, lse


FP8_CASES = [
    # B, Lq, Lk, n_q, n_kv, causal
    (1, 1000, 1000, 8, 2, True),
    (2, 300, 300, 4, 4, True),       # g = 1
    (1, 129, 129, 2, 1, True),
    (1, 1, 1, 2, 1, True),
    (3, 300, 300, 6, 2, True),       # g = 3
    (1, 500, 500, 4, 2, False),
    (2, 300, 1000, 8, 2, True),      # chunk, unaligned offset
    (1, 256, 1280, 4, 1, True),      # chunk, aligned offset
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "B%d_Lq%d_Lk%d_q%d_kv%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
def test_fp8_small_shapes_full(case):
    B, Lq, Lk, n_q, n_kv, causal = case
    w = W.custom(B, Lq, n_q, n_kv, 128, causal, Lk=Lk, dtype="e4m3")
    q, k, v = W.make_inputs(w, "cuda", seed=hash(case) % 100000)
    o, lse = _run(q, k, v, causal=causal)
    err = check_fp8_full(q, k, v, o, lse, causal=causal, what=str(case))
    print(f"fp8 {case}: {err}")


def test_fp8_descales():
    """Inputs stored at a different scale with the matching descale factors."""
    w = W.custom(1, 600, 4, 2, 128)
    q, k, v = (t.float() for t in W.make_inputs(w, "cuda", seed=77))
    ds = (4.0, 0.5, 8.0)
    q8 = (q / ds[0]).to(torch.float8_e4m3fn)
    k8 = (k / ds[1]).to(torch.float8_e4m3fn)
    v8 = (v / ds[2]).to(torch.float8_e4m3fn)
    o, lse = _run(q8, k8, v8, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    check_fp8_full(q8, k8, v8, o, lse, descales=ds, what="descales")


def test_fp8_agrees_with_bf16_path_on_the_same_values():
    """e4m3 values are exact in bf16: the bf16 kernel on the same numbers is a
    second estimate; the two differ by at most the fp8 bound plus the bf16
    kernel's own error."""
    w = W.custom(1, 2048, 8, 2, 128, dtype="e4m3")
    q, k, v = W.make_inputs(w, "cuda", seed=5)
    o8, l8 = _run(q, k, v)
    o16, l16 = attn_prefill(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16))
    assert attn_device_check() == ATTN_OK
    assert (l8 - l16).abs().max().item() <= 2e-3
    rel = ((o8.float() - o16.float()).norm() / o16.float().norm()).item()
    assert rel <= 2.0 ** -4


@pytest.mark.parametrize("num", [8, 9])
def test_fp8_workload_sampled_rows(num):
    w = W.WORKLOADS[num]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = _run(q, k, v, causal=w.causal, scale=w.scale)
    rows = W.sampled_rows(w)
    err = check_fp8_rows(q, k, v, o, lse, rows, causal=w.causal, scale=w.scale, what=w.name)
    print(f"parity {w.name} ({len(rows)} sampled rows): {err}")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_fp8_argument_errors():
    q = torch.zeros(1, 64, 2, 64, device="cuda", dtype=torch.float8_e4m3fn)
    kv = torch.zeros(1, 64, 1, 64, device="cuda", dtype=torch.float8_e4m3fn)
    o = torch.empty(1, 64, 2, 64, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(1, 2, 64, device="cuda")
    assert attn_prefill_fwd_fp8(q, kv, kv, o, lse, 1, 64, 64, 2, 1, 64, 1, 0.1, 1, 1, 1) == \
        ATTN_ERR_UNSUPPORTED
    q = torch.zeros(1, 64, 2, 128, device="cuda", dtype=torch.float8_e4m3fn)
    kv = torch.zeros(1, 64, 1, 128, device="cuda", dtype=torch.float8_e4m3fn)
    o = torch.empty(1, 64, 2, 128, device="cuda", dtype=torch.bfloat16)
    assert attn_prefill_fwd_fp8(q, kv, kv, o, lse, 1, 64, 64, 2, 1, 128, 1, 0.1, math.inf, 1,
                                1) == ATTN_ERR_INVALID_ARG
