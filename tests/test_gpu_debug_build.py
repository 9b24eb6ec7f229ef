"""The ATTN_DEBUG build of the library on the small parity cases.

The debug library's forward kernels check, before each operation, TMA
coordinates (inside the tensor, 16-byte aligned inner offset, landing inside
the CTA's shared memory), the tensor-memory base and lane quarter, shared
memory operand ranges and the soundness of every mbarrier parity wait; a
failed check ends the launch through the abort path and attn_device_check
returns ATTN_ERR_CHECK. Here every case must pass every check (status OK),
the checks must actually have run (the debug library counts them), and the
outputs must still match the oracle.
"""

import ctypes

import numpy as np
import pytest

import oracle
from causal_gqa_prefill_gb300 import ATTN_OK, _abi, build
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import assert_within, errors, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    torch.cuda.set_device(0)
    return _abi.load(build.build(debug=True))


def _run(lib, q, k, v, Lq, Lk, causal, scale, fp8=False):
    B, _, n_q, d = q.shape
    n_kv = k.shape[2]
    o = torch.full((B, Lq, n_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, n_q, Lq), float("nan"), device="cuda")
    sh = int(torch.cuda.current_stream().cuda_stream)
    if fp8:
        st = lib.attn_prefill_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, Lq, Lk, n_q, n_kv, d, int(causal), scale,
                                      1.0, 1.0, 1.0, sh)
    else:
        st = lib.attn_prefill_fwd_chunk(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), B, Lq, Lk, n_q, n_kv, d, int(causal), scale,
                                        sh)
    assert st == ATTN_OK, st
    assert lib.attn_device_check(sh) == ATTN_OK      # every device-side check passed
    return o, lse


CASES = [(L, d, g) for L in (1, 2, 127, 128, 129, 255, 257) for d in (64, 128)
         for g in (1, 2, 4, 6, 8)]


def test_debug_build_passes_every_check_on_the_small_cases(dbg):
    before = dbg.attn_debug_check_count()
    assert before >= 0, "the debug library must count its checks"
    last = before
    for n, (L, d, g) in enumerate(CASES):
        n_kv = 1 if g >= 4 else 2
        w = W.custom(1, L, g * n_kv, n_kv, d)
        q, k, v = W.make_inputs(w, "cuda", seed=3000 + n)
        o, lse = _run(dbg, q, k, v, L, L, True, w.scale)
        o_ref, lse_ref = oracle.attention(to_np(q), to_np(k), to_np(v), causal=True, scale=w.scale)
        assert_within(errors(to_np(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref),
                      f"debug build L={L} d_h={d} g={g}")
        count = dbg.attn_debug_check_count()
        assert count > last, "no device-side check ran"
        last = count


@pytest.mark.parametrize("Lq,Lk,causal", [(100, 300, True), (128, 1000, True), (257, 257, False),
                                          (33, 513, False)])
def test_debug_build_chunks_and_full_attention(dbg, Lq, Lk, causal):
    w = W.custom(2, Lq, 8, 2, 128, Lk=Lk)
    q, k, v = W.make_inputs(w, "cuda", seed=Lq * 7 + Lk)
    o, lse = _run(dbg, q, k, v, Lq, Lk, causal, w.scale)
    o_ref, lse_ref = oracle.attention(to_np(q), to_np(k), to_np(v), causal=causal, scale=w.scale)
    assert_within(errors(to_np(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref),
                  f"debug build chunk Lq={Lq} Lk={Lk} causal={causal}")


def test_debug_build_fp8_passes_its_checks(dbg):
    w = W.custom(1, 300, 8, 2, 128, dtype="e4m3")
    q, k, v = W.make_inputs(w, "cuda", seed=77)
    before = dbg.attn_debug_check_count()
    o, lse = _run(dbg, q, k, v, 300, 300, True, w.scale, fp8=True)
    assert dbg.attn_debug_check_count() > before
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_release_build_runs_no_checks():
    assert _abi.load().attn_debug_check_count() == -1
