"""GPU parity of the backward pass (dQ, dK, dV) against the fp64 oracle.

The CUDA path: the product's forward (O, LSE) followed by attn_prefill_bwd,
both through the C ABI. The oracle: oracle.attention_backward on the same
bf16 inputs in float64. Large workloads are checked on whole K/V head groups
(the g query heads that share one K/V head and that K/V head), which are
independent of the other groups, so the oracle's output for a group is exact
for that slice.

Acceptance per gradient G (dQ, dK, dV), derived from the arithmetic of the
kernels: P and dS are rounded to bf16 before the products that consume them
(relative error <= 2^-9 each), D comes from the bf16 forward output O, the
products accumulate in fp32, and G is rounded to bf16 at the end
(<= 2^-9 |G| relative). Summed over the terms of a gradient element, the
first three give errors of a few 2^-9 of the RMS of G's terms; the bounds are
  * ||err||_F / ||G_ref||_F <= 1e-2
  * max |err| <= 2^-6 * max |G_ref| + 2^-8 * |G_ref|   (element-wise)
"""

import pytest
import torch

import oracle
from causal_gqa_prefill_gb300 import ATTN_ERR_UNSUPPORTED, AttnError, attn_prefill_backward
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import REL_FRO, assert_grads, grad_errors, run_backward, to_np

pytestmark = pytest.mark.gpu


def inputs(B, L, n_q, n_kv, causal=True, number=0, d_h=128):
    w = W.custom(B, L, n_q, n_kv, d_h, causal=causal, number=number, backward=True)
    q, k, v = W.make_inputs(w)
    return w, q, k, v, W.make_grad(w)


SHAPES = [
    # B, L, n_q, n_kv, causal
    (1, 128, 2, 2, True),        # one tile
    (1, 300, 4, 2, True),        # ragged tail
    (2, 640, 8, 2, True),        # batch, GQA-4, several tiles
    (1, 257, 6, 6, True),        # MHA, one-row tail
    (1, 333, 4, 1, False),       # full attention, MQA, ragged
    (1, 1000, 8, 1, True),       # GQA-8 (one K/V head collects 8 query heads)
    (6, 200, 4, 1, True),        # many short sequences, ragged second tile
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}L{s[1]}h{s[2]}-{s[3]}{'c' if s[4] else 'f'}"
                                               for s in SHAPES])
def test_backward_small_shapes(shape):
    B, L, n_q, n_kv, causal = shape
    w, q, k, v, dout = inputs(B, L, n_q, n_kv, causal, number=1200 + L)
    gpu = run_backward(q, k, v, dout, causal=causal)
    ref = oracle.attention_backward(to_np(q), to_np(k), to_np(v), to_np(dout), causal=causal)
    errs = assert_grads(gpu, ref, str(shape))
    print(shape, errs)


def test_backward_single_row_closed_form():
    # L = 1: the softmax has one entry (P = 1), so dV = dO summed over the group
    # and dS = dP - D = dO.V - dO.O = 0, hence dQ = dK = 0. On the GPU dP (tensor
    # cores) and D (row kernel) are two fp32 sums of the same 128 products in
    # different orders, so dS is zero up to fp32 rounding of a dot product of
    # size |dO||V| ~ 128: |dQ|, |dK| <= scale * 128 * 1e-5 * |K|, well under 1e-3.
    w, q, k, v, dout = inputs(1, 1, 4, 2, True, number=1301)
    dq, dk, dv = run_backward(q, k, v, dout)
    assert dq.float().abs().max().item() <= 1e-3
    assert dk.float().abs().max().item() <= 1e-3
    want = dout.float().view(1, 1, 2, 2, 128).sum(3)
    assert torch.allclose(dv.float(), want, rtol=2 ** -8, atol=0)


@pytest.mark.parametrize("scale", [0.0, -0.05, 0.25])
def test_backward_scales(scale):
    w, q, k, v, dout = inputs(1, 384, 4, 2, True, number=1302)
    gpu = run_backward(q, k, v, dout, scale=scale)
    ref = oracle.attention_backward(to_np(q), to_np(k), to_np(v), to_np(dout), causal=True,
                                    scale=scale)
    if scale == 0.0:
        # uniform weights: dQ = dK = 0 exactly (scale multiplies both)
        assert torch.count_nonzero(gpu[0]).item() == 0
        assert torch.count_nonzero(gpu[1]).item() == 0
        assert grad_errors(to_np(gpu[2]), ref[2])["rel_fro"] <= REL_FRO
    else:
        assert_grads(gpu, ref, f"scale={scale}")


def test_backward_deterministic():
    w, q, k, v, dout = inputs(1, 700, 8, 2, True, number=1303)
    a = run_backward(q, k, v, dout)
    b = run_backward(q, k, v, dout)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


SHAPES_D64 = [
    # B, L, n_q, n_kv, causal; head dimension 64 (one 128-byte swizzle chunk per row)
    (1, 256, 4, 1, True),        # the tiny GQA-4 layer (L = 256, d_h = 64)
    (2, 300, 4, 2, True),        # batch, ragged tail
    (1, 130, 3, 3, False),       # full attention, MHA, two-row tail
    (1, 700, 8, 1, True),        # GQA-8, several tiles
]


@pytest.mark.parametrize("shape", SHAPES_D64,
                         ids=[f"d64-B{s[0]}L{s[1]}h{s[2]}-{s[3]}{'c' if s[4] else 'f'}"
                              for s in SHAPES_D64])
def test_backward_head_dim_64(shape):
    B, L, n_q, n_kv, causal = shape
    w, q, k, v, dout = inputs(B, L, n_q, n_kv, causal, number=1400 + L, d_h=64)
    gpu = run_backward(q, k, v, dout, causal=causal)
    ref = oracle.attention_backward(to_np(q), to_np(k), to_np(v), to_np(dout), causal=causal)
    errs = assert_grads(gpu, ref, str(shape))
    print(shape, errs)


def test_backward_head_dim_32_unsupported():
    q = torch.zeros(1, 128, 2, 32, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 128, 1, 32, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(AttnError) as e:
        attn_prefill_backward(q, k, k, o, lse, torch.zeros_like(q))
    assert e.value.status == ATTN_ERR_UNSUPPORTED


def _group_slice(w, q, k, v, dout, kvh):
    hs = slice(kvh * w.g, (kvh + 1) * w.g)
    return (to_np(q[:, :, hs]), to_np(k[:, :, kvh:kvh + 1]), to_np(v[:, :, kvh:kvh + 1]),
            to_np(dout[:, :, hs]))


@pytest.mark.parametrize("num,groups", [(2, [(0, 0), (3, 31)]), (12, [(0, 0), (0, 7)])])
def test_backward_workload_groups(num, groups):
    """Model-shaped layers at full size; the oracle checks whole head groups
    ((batch, K/V head) pairs listed per workload)."""
    base = W.WORKLOADS[num]
    w = W.custom(base.B, base.L, base.n_q, base.n_kv, base.d_h, number=base.number,
                 backward=True)
    q, k, v = W.make_inputs(w)
    dout = W.make_grad(w)
    dq, dk, dv = run_backward(q, k, v, dout)
    for b, kvh in groups:
        hs = slice(kvh * w.g, (kvh + 1) * w.g)
        qs, ks, vs, ds = _group_slice(w, q[b:b + 1], k[b:b + 1], v[b:b + 1], dout[b:b + 1], kvh)
        ref = oracle.attention_backward(qs, ks, vs, ds, causal=True)
        gpu = (dq[b:b + 1, :, hs], dk[b:b + 1, :, kvh:kvh + 1], dv[b:b + 1, :, kvh:kvh + 1])
        errs = assert_grads(gpu, ref, f"workload {num} group ({b}, {kvh})")
        print(num, b, kvh, errs)
