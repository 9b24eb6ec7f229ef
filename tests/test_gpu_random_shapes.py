"""GPU parity on a seeded sweep of random small shapes, every path against the
fp64 oracle on every output element.

The fixed shape lists of the other files pick the cases the pairing, masking
and scheduling logic distinguishes; this sweep draws further combinations of
them from one fixed seed (so a failure names a reproducible case): batch
sizes, K/V head counts and group sizes g (odd, even, above 8 and up to 16),
query lengths at and around the tile edges or anywhere up to ~900 rows,
chunks whose key range extends past the query rows by aligned and unaligned
offsets, causal and full attention, the default and other (negative,
large) scales, and d_h 64 and 128. fp8, backward and decode draw from the
same generator within what each entry point accepts.
"""

import numpy as np
import pytest

import oracle
from causal_gqa_prefill_gb300 import (ATTN_OK, attn_decode, attn_device_check,
                                      attn_prefill_fp8)
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import assert_grads, check_fp8_full, check_full, run_backward, run_gpu
from gpu_common import to_np as to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SEED = 20261202


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _length(rng):
    kind = rng.integers(0, 3)
    if kind == 0:
        return int(rng.integers(1, 9))                                   # a few rows
    if kind == 1:
        return int(rng.choice([127, 128, 129, 255, 256, 257, 383, 385]))  # tile edges
    return int(rng.integers(9, 900))


def _cases(n, rng, *, fp8=False, square=False, decode=False, d_choices=(64, 128), g_max=16,
           max_flop=6e9):
    """n cases; draws whose oracle work (4 B n_q Lq Lk d flops) exceeds
    max_flop are drawn again, so the whole sweep stays a few seconds of CPU."""
    out = []
    while len(out) < n:
        n_kv = int(rng.choice([1, 2, 3, 5]))
        g = int(rng.choice([g for g in (1, 2, 3, 4, 5, 6, 7, 8, 16) if g <= g_max]))
        B = int(rng.integers(1, 4))
        d = int(rng.choice(d_choices))
        Lq = 1 if decode else _length(rng)
        if decode:
            Lk = int(rng.integers(1, 3000))
        elif square or rng.random() < 0.6:
            Lk = Lq
        else:
            extra = int(rng.choice([128, 256, int(rng.integers(1, 700))]))
            Lk = Lq + extra
        causal = True if decode else bool(rng.random() < 0.8)
        r = rng.random()
        scale = None if r < 0.7 else float(rng.choice([-0.09, 0.03, 0.2]))
        if fp8 and scale is not None and scale > 0.1:
            scale = 0.05                      # e4m3 inputs of magnitude ~1 with large scales
        seed = int(rng.integers(0, 1 << 30))
        if 4.0 * B * g * n_kv * Lq * Lk * d > max_flop:
            continue
        out.append((B, Lq, Lk, g * n_kv, n_kv, d, causal, scale, seed))
    return out


_rng = np.random.default_rng(SEED)
FWD = _cases(160, _rng)
FP8 = _cases(30, _rng, fp8=True, d_choices=(128,))
BWD = _cases(30, _rng, square=True, max_flop=2e9)
DEC = _cases(30, _rng, decode=True, d_choices=(128,))


def _id(c):
    B, Lq, Lk, n_q, n_kv, d, causal, scale, _ = c
    return (f"B{B}_Lq{Lq}_Lk{Lk}_q{n_q}_kv{n_kv}_d{d}_{'c' if causal else 'f'}"
            f"{'' if scale is None else '_s%g' % scale}")


@pytest.mark.parametrize("case", FWD, ids=_id)
def test_random_forward(case):
    B, Lq, Lk, n_q, n_kv, d, causal, scale, seed = case
    w = W.custom(B, Lq, n_q, n_kv, d, causal, Lk=Lk)
    q, k, v = W.make_inputs(w, "cuda", seed=seed)
    o, lse = run_gpu(q, k, v, causal=causal, scale=scale)
    check_full(q, k, v, o, lse, causal=causal, scale=scale, what=_id(case))


@pytest.mark.parametrize("case", FP8, ids=_id)
def test_random_fp8(case):
    B, Lq, Lk, n_q, n_kv, d, causal, scale, seed = case
    w = W.custom(B, Lq, n_q, n_kv, d, causal, Lk=Lk, dtype="e4m3")
    q, k, v = W.make_inputs(w, "cuda", seed=seed)
    o, lse = attn_prefill_fp8(q, k, v, causal=causal, scale=scale)
    assert attn_device_check() == ATTN_OK
    check_fp8_full(q, k, v, o, lse, causal=causal, scale=scale, what=_id(case))


@pytest.mark.parametrize("case", BWD, ids=_id)
def test_random_backward(case):
    B, L, _, n_q, n_kv, d, causal, scale, seed = case
    w = W.custom(B, L, n_q, n_kv, d, causal=causal, backward=True)
    q, k, v = W.make_inputs(w, "cuda", seed=seed)
    dout = W.make_grad(w)
    gpu = run_backward(q, k, v, dout, causal=causal, scale=scale)
    ref = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(dout),
                                    causal=causal, scale=scale)
    assert_grads(gpu, ref, _id(case))


@pytest.mark.parametrize("case", DEC, ids=_id)
def test_random_decode(case):
    B, _, Lk, n_q, n_kv, d, _, scale, seed = case
    w = W.custom(B, 1, n_q, n_kv, d, Lk=Lk)
    q, k, v = W.make_inputs(w, "cuda", seed=seed)
    o, lse = attn_decode(q, k, v, scale=scale)
    assert attn_device_check() == ATTN_OK
    check_full(q, k, v, o, lse, scale=scale, what=_id(case))
