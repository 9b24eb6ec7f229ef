"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

Each pin compares the oracle with something other than itself:
  * brute force on tiny inputs (pure-Python loops, exactly rounded sums via
    math.fsum, softmax without max subtraction, LSE as log of the sum);
  * a library routine: PyTorch's CPU float64 scaled_dot_product_attention
    (the pages report it within 8.9e-16 of a plain implementation, causal);
  * closed forms: causal row 0 returns V[0]; constant V returns that value;
    scale 0 gives the running mean of V and LSE = ln(i+1);
  * invariants: GQA equals MHA with each K/V head repeated g times; adding one
    vector to every key shifts each score row by a constant, which leaves O
    unchanged and moves LSE by exactly that constant (this also drives scores
    far past the 162 at which an unshifted exp overflows in float32);
    one-hot values expose the softmax weights, whose rows sum to 1;
  * the pages' worked example and block-size checks, against an independent
    online-softmax restatement written here from the pages' five steps;
  * the pages' printed cost-model numbers, for the FLOP and intensity model.

A mutation test at the end plants plausible mistakes in a copy of the oracle
(on the CPU) and checks that each one breaks at least one pin.
"""

import json
import math
import os
import types

import numpy as np
import pytest

import oracle
from oracle import flops as oflops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# ----------------------------------------------------------------------------
# helpers (test-side, independent of the oracle's code)

def _bf16_round(x):
    """Round float64 values to the nearest bfloat16 (ties to even), as float64."""
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _inputs(B, L, n_q, n_kv, d, seed=0, bf16=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, L, n_q, d))
    k = rng.standard_normal((B, L, n_kv, d))
    v = rng.standard_normal((B, L, n_kv, d))
    if bf16:
        q, k, v = _bf16_round(q), _bf16_round(k), _bf16_round(v)
    return q, k, v


def brute_force(q, k, v, causal, scale):
    """Pure-Python attention: exact sums, exp of the raw scores, LSE = log Z.

    q may hold fewer rows than k, v: they are the last rows of the sequence."""
    B, L, n_q, d = q.shape
    n_kv = k.shape[2]
    g = n_q // n_kv
    off = k.shape[1] - L
    o = np.zeros(q.shape)
    lse = np.zeros((B, n_q, L))
    for b in range(B):
        for h in range(n_q):
            kvh = h // g
            for i in range(L):
                keys = range(i + off + 1) if causal else range(k.shape[1])
                sc = [scale * math.fsum(float(q[b, i, h, t]) * float(k[b, j, kvh, t])
                                        for t in range(d)) for j in keys]
                w = [math.exp(x) for x in sc]
                z = math.fsum(w)
                for t in range(d):
                    o[b, i, h, t] = math.fsum(w[n] * float(v[b, j, kvh, t])
                                              for n, j in enumerate(keys)) / z
                lse[b, h, i] = math.log(z)
    return o, lse


def online_softmax_single_head(q, k, v, block, causal, scale):
    """One head [N, d], tiled over query and key blocks with running (m, l, acc).

    Follows the pages' online-softmax steps: keep a running max m, a running
    sum l of exp(score - m) and a running weighted sum acc; for each key tile
    take the new max, rescale l and acc by exp(m_old - m_new), add the tile's
    exponentials and their product with V, and divide by l once at the end.
    """
    n, d = q.shape
    out = np.zeros((n, d))
    lse = np.zeros(n)
    for r0 in range(0, n, block):
        qb = q[r0:r0 + block]
        rows = np.arange(r0, r0 + qb.shape[0])
        run_max = np.full(qb.shape[0], -np.inf)
        run_sum = np.zeros(qb.shape[0])
        run_acc = np.zeros((qb.shape[0], d))
        for c0 in range(0, n, block):
            if causal and c0 > rows[-1]:
                break
            cols = np.arange(c0, min(n, c0 + block))
            t = (qb @ k[c0:c0 + block].T) * scale
            if causal:
                t = np.where(cols[None, :] <= rows[:, None], t, -np.inf)
            new_max = np.maximum(run_max, t.max(axis=1))
            shrink = np.exp(run_max - new_max)
            e = np.exp(t - new_max[:, None])
            run_sum = run_sum * shrink + e.sum(axis=1)
            run_acc = run_acc * shrink[:, None] + e @ v[c0:c0 + block]
            run_max = new_max
        out[r0:r0 + qb.shape[0]] = run_acc / run_sum[:, None]
        lse[r0:r0 + qb.shape[0]] = run_max + np.log(run_sum)
    return out, lse


def _load_golden(name):
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# pin suite, parameterised by the module under test so the mutation test can
# run it on planted mistakes

def pin_bruteforce(att):
    worst = 0.0
    for (B, L, n_q, n_kv, d, causal) in [(2, 5, 4, 2, 4, True), (1, 7, 3, 1, 3, False),
                                         (1, 16, 2, 2, 8, True), (1, 1, 2, 1, 4, True)]:
        q, k, v = _inputs(B, L, n_q, n_kv, d, seed=L * 31 + d)
        scale = 1.0 / math.sqrt(d)
        o, lse = att.attention(q, k, v, causal=causal, scale=scale)
        ob, lb = brute_force(q, k, v, causal, scale)
        worst = max(worst, np.abs(o - ob).max(), np.abs(lse - lb).max())
    return worst <= 1e-13, worst


def pin_sdpa(att):
    torch = pytest.importorskip("torch")
    worst = 0.0
    for (B, L, n_q, n_kv, d, causal) in [(2, 37, 8, 2, 16, True), (1, 64, 6, 3, 32, False),
                                         (1, 50, 4, 4, 8, True)]:
        q, k, v = _inputs(B, L, n_q, n_kv, d, seed=L)
        scale = 1.0 / math.sqrt(d)
        o, lse = att.attention(q, k, v, causal=causal, scale=scale)
        g = n_q // n_kv
        tq = torch.from_numpy(q).permute(0, 2, 1, 3)
        tk = torch.from_numpy(np.repeat(k, g, axis=2)).permute(0, 2, 1, 3)
        tv = torch.from_numpy(np.repeat(v, g, axis=2)).permute(0, 2, 1, 3)
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=causal, scale=scale).permute(0, 2, 1, 3).numpy()
        sc = torch.matmul(tq, tk.transpose(-1, -2)) * scale
        if causal:
            keep = torch.ones(L, L, dtype=torch.bool).tril()
            sc = sc.masked_fill(~keep, float("-inf"))
        ref_lse = torch.logsumexp(sc, dim=-1).numpy()
        worst = max(worst, np.abs(o - ref).max(), np.abs(lse - ref_lse).max())
    return worst <= 1e-13, worst


def pin_row0(att):
    q, k, v = _inputs(2, 9, 4, 2, 16, seed=3)
    scale = 0.3
    o, lse = att.attention(q, k, v, causal=True, scale=scale)
    ok = True
    worst = 0.0
    for b in range(2):
        for h in range(4):
            kvh = h // 2
            ok &= bool(np.array_equal(o[b, 0, h], v[b, 0, kvh]))
            s00 = scale * float(np.dot(q[b, 0, h], k[b, 0, kvh]))
            worst = max(worst, abs(lse[b, h, 0] - s00))
    return ok and worst <= 1e-14, worst


def pin_constant_v(att):
    q, k, _ = _inputs(1, 40, 6, 2, 8, seed=4)
    c = np.array([1.75, -0.3125])
    v = np.broadcast_to(c[None, None, :, None], (1, 40, 2, 8)).copy()
    worst = 0.0
    for causal in (True, False):
        o, _ = att.attention(q, k, v, causal=causal)
        for h in range(6):
            worst = max(worst, np.abs(o[0, :, h, :] - c[h // 3]).max() / abs(c[h // 3]))
    return worst <= 8 * 2.0 ** -52, worst


def pin_scale_zero(att):
    q, k, v = _inputs(2, 23, 4, 1, 5, seed=5)
    worst = 0.0
    o, lse = att.attention(q, k, v, causal=True, scale=0.0)
    for b in range(2):
        mean = np.cumsum(v[b, :, 0, :], axis=0) / np.arange(1, 24)[:, None]
        for h in range(4):
            worst = max(worst, np.abs(o[b, :, h, :] - mean).max(),
                        np.abs(lse[b, h] - np.log(np.arange(1, 24))).max())
    o, lse = att.attention(q, k, v, causal=False, scale=0.0)
    worst = max(worst, np.abs(o[0, :, 1, :] - v[0, :, 0, :].mean(axis=0)).max(),
                np.abs(lse - math.log(23)).max())
    return worst <= 1e-14, worst


def pin_gqa_equals_mha(att):
    ok = True
    for causal in (True, False):
        q, k, v = _inputs(2, 19, 8, 2, 8, seed=6)
        o1, l1 = att.attention(q, k, v, causal=causal)
        o2, l2 = att.attention(q, np.repeat(k, 4, axis=2), np.repeat(v, 4, axis=2), causal=causal)
        ok &= bool(np.array_equal(o1, o2) and np.array_equal(l1, l2))
    return ok, 0.0


def pin_shift_invariance(att):
    """K -> K + u shifts row i's scores by scale*q_i.u; O fixed, LSE moves by it."""
    q, k, v = _inputs(1, 33, 4, 2, 16, seed=7)
    scale = 0.25
    u = 200.0 * np.sign(q[0, :, 0, :].mean(axis=0))
    k2 = k + u[None, None, None, :]
    worst_scores = np.abs(scale * np.einsum("lhd,d->lh", q[0], u)).max()
    worst = 0.0
    for causal in (True, False):
        o1, l1 = att.attention(q, k, v, causal=causal, scale=scale)
        o2, l2 = att.attention(q, k2, v, causal=causal, scale=scale)
        shift = scale * np.einsum("blhd,d->bhl", q, u)
        if not (np.isfinite(o2).all() and np.isfinite(l2).all()):
            return False, float("inf")
        worst = max(worst, np.abs(o1 - o2).max(), np.abs(l2 - (l1 + shift)).max() / 100.0)
    return worst_scores >= 200 and worst <= 1e-11, worst


def pin_onehot_weights(att):
    """V = identity exposes the softmax weights P: rows sum to 1, zero above the
    diagonal, and P_ij / P_ik = exp(s_ij - s_ik)."""
    L = 12
    rng = np.random.default_rng(8)
    q = _bf16_round(rng.standard_normal((1, L, 2, L)))
    k = _bf16_round(rng.standard_normal((1, L, 1, L)))
    v = np.eye(L)[None, :, None, :]
    scale = 1.0 / math.sqrt(L)
    o, _ = att.attention(q, k, v, causal=True, scale=scale)
    worst = 0.0
    ok = True
    for h in range(2):
        p = o[0, :, h, :]
        worst = max(worst, np.abs(p.sum(axis=1) - 1.0).max())
        ok &= bool((np.triu(p, 1) == 0).all())
        for i in range(1, L):
            s = [scale * float(np.dot(q[0, i, h], k[0, j, 0])) for j in range(i + 1)]
            worst = max(worst, abs(p[i, i] / p[i, 0] - math.exp(s[i] - s[0])))
    return ok and worst <= 1e-12, worst


def pin_tiled_blocks(att):
    """The pages' harder check: block sizes 1, 7, 32, 64, 128 and 1000 on 1000
    tokens all agree with the plain version within 1.3e-15 (fp64)."""
    gold = _load_golden("long_context_tiling_checks.json")["harder_checks"]
    rng = np.random.default_rng(9)
    n, d = 1000, 64
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    worst = 0.0
    for causal in (False, True):
        o, lse = att.attention(q[None, :, None], k[None, :, None], v[None, :, None], causal=causal)
        for blk in gold["block_sizes_on_1000_tokens"]:
            ot, lt = online_softmax_single_head(q, k, v, blk, causal, 1.0 / math.sqrt(d))
            worst = max(worst, np.abs(o[0, :, 0] - ot).max(), np.abs(lse[0, 0] - lt).max())
    return worst <= 4 * gold["max_abs_difference_bound"], worst


def pin_chunk_bruteforce(att):
    """A query chunk at the end of a longer key range, against brute force."""
    worst = 0.0
    for (B, Lq, Lk, n_q, n_kv, d, causal) in [(2, 3, 7, 4, 2, 4, True), (1, 5, 11, 3, 1, 3, True),
                                               (1, 4, 9, 2, 2, 8, False)]:
        q, _, _ = _inputs(B, Lq, n_q, n_kv, d, seed=Lq * 13 + Lk)
        _, k, v = _inputs(B, Lk, n_q, n_kv, d, seed=Lk * 17 + Lq)
        scale = 1.0 / math.sqrt(d)
        o, lse = att.attention(q, k, v, causal=causal, scale=scale)
        ob, lb = brute_force(q, k, v, causal, scale)
        worst = max(worst, np.abs(o - ob).max(), np.abs(lse - lb).max())
    return worst <= 1e-13, worst


def pin_chunk_is_suffix(att):
    """Chunked prefill reproduces the last rows of one full causal pass: the
    chunk's rows are rows Lk-Lq.. of the square problem on the whole sequence."""
    worst = 0.0
    for (Lq, Lk) in [(37, 100), (64, 64), (1, 50), (50, 51)]:
        qf, k, v = _inputs(2, Lk, 6, 2, 16, seed=Lq + 3 * Lk)
        o_full, l_full = att.attention(qf, k, v, causal=True)
        o, lse = att.attention(qf[:, Lk - Lq:], k, v, causal=True)
        worst = max(worst, np.abs(o - o_full[:, Lk - Lq:]).max(),
                    np.abs(lse - l_full[:, :, Lk - Lq:]).max())
    return worst <= 1e-14, worst


def pin_chunk_sdpa(att):
    """Library check with an explicit bottom-right causal mask."""
    torch = pytest.importorskip("torch")
    B, Lq, Lk, n_q, n_kv, d = 2, 23, 61, 4, 2, 16
    q, _, _ = _inputs(B, Lq, n_q, n_kv, d, seed=41)
    _, k, v = _inputs(B, Lk, n_q, n_kv, d, seed=43)
    o, _ = att.attention(q, k, v, causal=True)
    keep = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(0, 2, 1, 3),
        torch.from_numpy(np.repeat(k, 2, axis=2)).permute(0, 2, 1, 3),
        torch.from_numpy(np.repeat(v, 2, axis=2)).permute(0, 2, 1, 3),
        attn_mask=keep).permute(0, 2, 1, 3).numpy()
    worst = np.abs(o - ref).max()
    return worst <= 1e-13, worst


PINS = [pin_bruteforce, pin_chunk_bruteforce, pin_chunk_is_suffix, pin_chunk_sdpa, pin_sdpa, pin_row0, pin_constant_v, pin_scale_zero,
        pin_gqa_equals_mha, pin_shift_invariance, pin_onehot_weights, pin_tiled_blocks]


# ----------------------------------------------------------------------------
# the pins applied to the oracle

@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    ok, err = pin(oracle)
    assert ok, f"{pin.__name__}: error {err}"


def test_pages_worked_example():
    """The pages' NumPy example: N=1024, d=64, default_rng(0), Q, K, V drawn in
    that order; plain vs tiled (block 64) differ by 3.9e-16 and allclose holds."""
    gold = _load_golden("long_context_tiling_checks.json")["worked_example"]
    rng = np.random.default_rng(0)
    n, d = gold["N"], gold["d"]
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    o, _ = oracle.attention(q[None, :, None], k[None, :, None], v[None, :, None], causal=False)
    ot, _ = online_softmax_single_head(q, k, v, gold["block"], False, 1.0 / math.sqrt(d))
    diff = np.abs(o[0, :, 0] - ot).max()
    assert diff <= 4 * gold["printed_max_abs_difference"]
    assert np.allclose(o[0, :, 0], ot) == gold["printed_allclose"]


def test_rows_mode_matches_full():
    q, k, v = _inputs(2, 300, 6, 3, 16, seed=10)
    o, lse = oracle.attention(q, k, v, causal=True)
    rng = np.random.default_rng(11)
    rows = np.stack([rng.integers(0, 2, 200), rng.integers(0, 6, 200), rng.integers(0, 300, 200)], 1)
    orow, lrow = oracle.attention_rows(q, k, v, rows, causal=True)
    assert np.abs(orow - o[rows[:, 0], rows[:, 2], rows[:, 1]]).max() <= 1e-14
    assert np.abs(lrow - lse[rows[:, 0], rows[:, 1], rows[:, 2]]).max() <= 1e-14


def test_rejects_bad_shapes():
    q, k, v = _inputs(1, 4, 3, 2, 4)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v)


# ----------------------------------------------------------------------------
# cost model pins (values printed on the pages)

def test_flop_record_ridges_and_intensity():
    gold = _load_golden("prefill_attention_flop_record.json")
    for r in gold["ridge"]:
        assert round(oflops.ridge(r["tflops"], r["gbs"]), 1) == r["ridge"]
        for g, lr in r.get("L_ridge", {}).items():
            assert round(oflops.ridge_length(r["tflops"], r["gbs"], int(g))) == lr
    ex = gold["ai_example"]
    ai = oflops.arithmetic_intensity(ex["L"], ex["n_q"], ex["n_kv"])
    assert ai == ex["ai"]
    assert round(ai / oflops.ridge(989.5, 3350)) == ex["times_h100_ridge"]
    # AI is FLOPs over K/V bytes: both sides of the ratio must be the pages' forms
    assert oflops.causal_attention_flops(1, 8192, 32, 128) == 2 * 32 * 128 * 8192 ** 2
    assert oflops.kv_bytes(1, 8192, 8, 128) == 4 * 8192 * 128 * 8


def test_flop_record_attention_share():
    gold = _load_golden("prefill_attention_flop_record.json")
    for m in gold["crossover"]:
        n_q, d_h = m["n_q_times_d_h"] // 128, 128
        assert oflops.flop_crossover(m["p_layer"], n_q, d_h) == m["L_star"]
        for L, pct in m.get("share_pct", {}).items():
            assert round(100 * oflops.attention_share(int(L), m["p_layer"], n_q, d_h), 1) == pct


def test_long_context_shape_costs():
    gold = _load_golden("long_context_36head_shape.json")
    s = gold["shape"]
    layers, n_q, d_h, width = s["layers"], s["n_q"], s["d_h"], s["width"]
    tot = gold["prefill_total_tflop_with_causal_skipping"]

    def attn(L, dense=False):
        f = oflops.dense_attention_flops if dense else oflops.causal_attention_flops
        return layers * f(1, L, n_q, d_h)

    # solve the (unprinted) weight count from the 4K total, then predict the rest
    p_total = (tot["4096"] * 1e12 - attn(4096)) / (2 * 4096)
    pred_128k = (attn(131072) + 2 * p_total * 131072) / 1e12
    assert abs(pred_128k - tot["131072"]) / tot["131072"] < 2e-3
    r = gold["doubling_32k_to_64k"]
    assert attn(65536, True) / attn(32768, True) == r["attention_ratio"]
    total = lambda L: attn(L, True) + 2 * p_total * L
    assert round(total(65536) / total(32768), 2) == r["total_ratio"]
    p_layer = p_total / layers
    c = gold["crossover_tokens"]
    dense_x = 2 * p_layer / (oflops.dense_attention_flops(1, 1, n_q, d_h))
    skip_x = 2 * p_layer / (oflops.causal_attention_flops(1, 1, n_q, d_h))
    assert abs(dense_x - c["dense_count"]) <= c["tolerance_tokens"]
    assert abs(skip_x - c["with_causal_skipping"]) <= c["tolerance_tokens"]
    assert n_q * d_h == width
    sb = gold["score_table_bytes"]
    assert round(n_q * 32768 ** 2 * 2 / 1e9, 1) == sb["32768_all_heads_gb"]
    assert round(n_q * 131072 ** 2 * 2 / 1e9) == sb["131072_all_heads_gb"]
    assert round(131072 ** 2 * 2 / 1e9, 1) == sb["131072_one_head_gb"]
    assert oflops.kv_bytes(1, 1, s["n_kv"], d_h) * layers == gold["kv_cache_bytes_per_token"]


# ----------------------------------------------------------------------------
# mutation test: plausible mistakes planted in a copy of the oracle must each
# break at least one pin

MUTANTS = {
    "mask_excludes_diagonal": ("keys[None, :] <= pos[:, None]", "keys[None, :] < pos[:, None]"),
    "kv_head_modulo": ("return h // (n_q // n_kv)", "return h % n_kv"),
    "scale_dropped": ("s = scale * (qrows @ krows.T)", "s = (qrows @ krows.T)"),
    "lse_without_max": ("lse = m_safe + np.log(l)", "lse = np.log(l)"),
    "no_max_subtraction": ("p = np.exp(s - m_safe[:, None])", "p = np.exp(s)"),
    "values_reversed": ("o = (p @ vrows) / l[:, None]", "o = (p @ vrows[::-1]) / l[:, None]"),
    "prefix_off_by_one": ("lv = int(pos[-1]) + 1 if causal else Lk", "lv = int(pos[-1]) if causal else Lk"),
    "chunk_aligned_top_left": ("offset = Lk - L", "offset = 0"),
    "max_over_keys_axis": ("m = s.max(axis=1)", "m = s.max(axis=0)"),
    "normalise_by_max": ("o = (p @ vrows) / l[:, None]", "o = (p @ vrows) / p.max(axis=1)[:, None]"),
}


def _mutant_module(old, new):
    path = os.path.join(ROOT, "oracle", "attention.py")
    with open(path) as f:
        src = f.read()
    assert old in src, old
    src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    old, new = MUTANTS[name]
    mod = _mutant_module(old, new)
    failed = []
    import warnings
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        for pin in PINS:
            try:
                ok, _ = pin(mod)
            except Exception:
                ok = False
            if not ok:
                failed.append(pin.__name__)
                break
    assert failed, f"mutant {name} passed every pin"
