"""Pins for the fp64 backward oracle, each against something other than itself:

  * PyTorch CPU float64 autograd through scaled_dot_product_attention (GQA by
    repeated K/V heads; autograd sums their gradients);
  * central finite differences of the pinned forward oracle (the directional
    derivative of sum(O * dO) along random directions of Q, K and V);
  * closed forms at scale 0 (uniform causal weights: dQ = dK = 0 and
    dV_j = sum_{i >= j} dO_i / (i + 1));
  * GQA: the K/V gradients equal the MHA gradients of the repeated heads,
    summed over each group.

A mutation test plants plausible mistakes in a copy of the backward oracle.
"""

import math
import os
import types

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(B, L, n_q, n_kv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, L, n_q, d)), rng.standard_normal((B, L, n_kv, d)),
            rng.standard_normal((B, L, n_kv, d)), rng.standard_normal((B, L, n_q, d)))


def pin_autograd(mod):
    torch = pytest.importorskip("torch")
    worst = 0.0
    for (B, L, n_q, n_kv, d, causal) in [(2, 37, 4, 2, 16, True), (1, 50, 6, 3, 8, False),
                                         (1, 64, 2, 2, 32, True)]:
        q, k, v, do = _inputs(B, L, n_q, n_kv, d, seed=L + d)
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv = mod.attention_backward(q, k, v, do, causal=causal, scale=scale)
        g = n_q // n_kv
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        o = torch.nn.functional.scaled_dot_product_attention(
            tq.permute(0, 2, 1, 3), tk.repeat_interleave(g, dim=2).permute(0, 2, 1, 3),
            tv.repeat_interleave(g, dim=2).permute(0, 2, 1, 3), is_causal=causal, scale=scale)
        o.permute(0, 2, 1, 3).backward(torch.tensor(do))
        worst = max(worst, np.abs(dq - tq.grad.numpy()).max(), np.abs(dk - tk.grad.numpy()).max(),
                    np.abs(dv - tv.grad.numpy()).max())
    return worst <= 1e-12, worst


def pin_finite_differences(mod):
    """<dX, E> = d/dt sum(O(X + tE) * dO) at t = 0, by central differences."""
    B, L, n_q, n_kv, d = 1, 9, 4, 2, 6
    q, k, v, do = _inputs(B, L, n_q, n_kv, d, seed=3)
    scale = 0.4
    dq, dk, dv = mod.attention_backward(q, k, v, do, causal=True, scale=scale)
    rng = np.random.default_rng(4)
    eps = 1e-5
    worst = 0.0
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        e = rng.standard_normal(grad.shape)
        args_p = [q, k, v]
        args_m = [q, k, v]
        args_p[which] = args_p[which] + eps * e
        args_m[which] = args_m[which] - eps * e
        fp = (oracle.attention(*args_p, causal=True, scale=scale)[0] * do).sum()
        fm = (oracle.attention(*args_m, causal=True, scale=scale)[0] * do).sum()
        num = (fp - fm) / (2 * eps)
        ana = (grad * e).sum()
        worst = max(worst, abs(num - ana) / max(1.0, abs(ana)))
    return worst <= 1e-7, worst


def pin_scale_zero(mod):
    B, L, n_q, n_kv, d = 2, 11, 2, 1, 5
    q, k, v, do = _inputs(B, L, n_q, n_kv, d, seed=5)
    dq, dk, dv = mod.attention_backward(q, k, v, do, causal=True, scale=0.0)
    ref = np.zeros_like(dv)
    for b in range(B):
        for j in range(L):
            ref[b, j, 0] = sum(do[b, i, h] / (i + 1) for i in range(j, L) for h in range(n_q))
    worst = max(np.abs(dq).max(), np.abs(dk).max(), np.abs(dv - ref).max())
    return worst <= 1e-13, worst


def pin_gqa_sums_heads(mod):
    q, k, v, do = _inputs(2, 13, 6, 2, 8, seed=6)
    dq, dk, dv = mod.attention_backward(q, k, v, do, causal=True)
    dq2, dk2, dv2 = mod.attention_backward(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2), do,
                                           causal=True)
    worst = max(np.abs(dq - dq2).max(),
                np.abs(dk - dk2.reshape(2, 13, 2, 3, 8).sum(axis=3)).max(),
                np.abs(dv - dv2.reshape(2, 13, 2, 3, 8).sum(axis=3)).max())
    return worst <= 1e-13, worst


PINS = [pin_scale_zero, pin_gqa_sums_heads, pin_finite_differences, pin_autograd]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    ok, err = pin(oracle)
    assert ok, f"{pin.__name__}: error {err}"


def test_rowdot_is_dO_dot_O():
    q, k, v, do = _inputs(1, 20, 4, 2, 8, seed=7)
    o, _ = oracle.attention(q, k, v)
    d = oracle.softmax_rowdot(o, do)
    assert np.allclose(d[0, 1, 5], np.dot(o[0, 5, 1], do[0, 5, 1]), rtol=0, atol=1e-14)


MUTANTS = {
    "rowdot_dropped": ("ds = p * (dp - dd)", "ds = p * dp"),
    "ds_transposed_into_dk": ("dk[b, :lv, kvh, :] += scale * (ds.T @ qb)",
                              "dk[b, :lv, kvh, :] += scale * (p.T @ qb)"),
    "dq_scale_dropped": ("dq[b, rows, h, :] = scale * (ds @ kmat[:lv])",
                         "dq[b, rows, h, :] = (ds @ kmat[:lv])"),
    "dv_uses_scores": ("dv[b, :lv, kvh, :] += p.T @ dob", "dv[b, :lv, kvh, :] += ds.T @ dob"),
    "dk_overwrites_group": ("dk[b, :lv, kvh, :] += scale * (ds.T @ qb)",
                            "dk[b, :lv, kvh, :] = scale * (ds.T @ qb)"),
    "dp_uses_keys": ("dp = dob @ vmat[:lv].T", "dp = dob @ kmat[:lv].T"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_backward_mistake(name):
    old, new = MUTANTS[name]
    with open(os.path.join(ROOT, "oracle", "backward.py")) as f:
        src = f.read()
    assert old in src, old
    mod = types.ModuleType("backward_mutant")
    exec(compile(src.replace(old, new), "backward_mutant", "exec"), mod.__dict__)
    for pin in PINS:
        try:
            ok, _ = pin(mod)
        except Exception:
            ok = False
        if not ok:
            return
    pytest.fail(f"mutant {name} passed every pin")
