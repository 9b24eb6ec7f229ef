"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes are compared on every output element; they span several tiles,
ragged tails, every GQA group shape the pairing logic distinguishes (g = 1,
odd g, even g, MQA), d_h 64 and 128, causal and full attention, and the
degenerate cases (L = 1, 2, one tile, scale 0, negative scale, logits far
beyond the float32 overflow point of an unshifted exp). The model-shaped
workloads run at full size in the launch configuration the benchmark times:
the three smaller ones compared in full, the two large ones on sampled rows
covering every head and every position inside a tile.
"""

import math

import numpy as np
import pytest

from causal_gqa_prefill_gb300 import (ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_OK,
                                      attn_prefill, attn_prefill_fwd)
from causal_gqa_prefill_gb300 import workloads as W
from gpu_common import check_full, check_rows, run_gpu, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(0)


SMALL = [
    # B, L, n_q, n_kv, d_h, causal
    (2, 1000, 8, 2, 128, True),
    (1, 129, 2, 1, 128, True),
    (1, 127, 1, 1, 64, True),
    (1, 1, 1, 1, 128, True),
    (1, 2, 4, 4, 64, True),
    (3, 300, 6, 2, 128, True),      # g = 3: pairs cross heads and tiles
    (1, 520, 12, 2, 128, True),     # g = 6
    (1, 384, 8, 1, 128, True),      # g = 8, one K/V head
    (2, 640, 4, 4, 128, True),      # g = 1, even tile count
    (1, 700, 2, 1, 64, True),
    (1, 1537, 4, 2, 64, True),
    (2, 300, 4, 2, 128, False),
    (1, 1000, 2, 2, 64, False),
    (1, 128, 2, 2, 128, False),
    (1, 1, 2, 1, 64, False),
    (48, 200, 8, 2, 128, True),     # many short sequences (B = 48), ragged second tile
    (2, 300, 64, 1, 128, True),     # g = 64: one K/V head for 64 query heads
    (5, 257, 10, 5, 64, True),      # g = 2, d_h = 64, one-row tail
    (16, 128, 4, 1, 64, False),     # full attention over many batches
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B%d_L%d_q%d_kv%d_d%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
def test_small_shapes_full(case):
    B, L, n_q, n_kv, d, causal = case
    w = W.custom(B, L, n_q, n_kv, d, causal)
    q, k, v = W.make_inputs(w, "cuda", seed=hash(case) % 100000)
    o, lse = run_gpu(q, k, v, causal=causal)
    check_full(q, k, v, o, lse, causal=causal, what=str(case))


@pytest.mark.parametrize("num", [1, 2, 3])
def test_workload_full(num):
    w = W.WORKLOADS[num]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_gpu(q, k, v, causal=w.causal, scale=w.scale)
    err = check_full(q, k, v, o, lse, causal=w.causal, scale=w.scale, what=w.name)
    print(f"parity {w.name}: {err}")


@pytest.mark.parametrize("num", [4, 5])
def test_workload_sampled_rows(num):
    w = W.WORKLOADS[num]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_gpu(q, k, v, causal=w.causal, scale=w.scale)
    rows = W.sampled_rows(w)
    err = check_rows(q, k, v, o, lse, rows, causal=w.causal, scale=w.scale, what=w.name)
    print(f"parity {w.name} ({len(rows)} sampled rows): {err}")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_outputs_past_2_31_elements():
    """One MQA layer whose Q and O hold more than 2^31 elements (4.3 GB of
    bf16 each): the output row offsets and the tensor-map row coordinates of
    the last heads' last tiles lie past the 32-bit element range, where an
    index computed in 32 bits would wrap. Checked on rows of five heads at
    the tile edges, the middle and the last rows (the last one past 2^31)."""
    w = W.custom(1, 262500, 64, 1, 128)             # rows >= 262144 lie past 2^31 elements
    assert (w.L - 129) * w.n_q * w.d_h >= 2 ** 31
    q, k, v = W.make_inputs(w, "cuda", seed=4242)
    o, lse = run_gpu(q, k, v, causal=True, scale=w.scale)
    L = w.L
    pos = [0, 1, 127, 128, 129, L // 2, L - 257, L - 129, L - 128, L - 2, L - 1]
    rng = np.random.default_rng(4242)
    rows = [(0, h, i) for h in (0, 1, 31, 62, 63)
            for i in pos + [int(x) for x in rng.integers(0, L, 6)]]
    err = check_rows(q, k, v, o, lse, rows, causal=True, scale=w.scale, what=w.name)
    print(f"parity {w.name} ({len(rows)} rows): {err}")
    del q, k, v, o, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("scale", [0.0, -0.0883883, 0.5, 1e-3])
def test_scale_values(scale):
    w = W.custom(1, 400, 4, 2, 128)
    q, k, v = W.make_inputs(w, "cuda", seed=17)
    for causal in (True, False):
        o, lse = run_gpu(q, k, v, causal=causal, scale=scale)
        check_full(q, k, v, o, lse, causal=causal, scale=scale, what=f"scale={scale}",
                   stress=abs(scale) > 0.1)


def test_logits_past_float32_overflow():
    """Keys scaled by 40: logits reach several hundred (the pages saw NaN from an
    unshifted float32 softmax at 162); output must stay finite and match."""
    w = W.custom(1, 600, 4, 2, 128)
    q, k, v = W.make_inputs(w, "cuda", seed=23)
    k = (k.float() * 40).to(torch.bfloat16)
    s = (q.float()[0, :, 0] @ k.float()[0, :, 0].T) / math.sqrt(128)
    assert s.abs().max().item() > 162
    o, lse = run_gpu(q, k, v)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    check_full(q, k, v, o, lse, what="heavy logits", stress=True)


def test_row0_returns_v0_and_constant_v():
    w = W.custom(2, 300, 4, 2, 128)
    q, k, v = W.make_inputs(w, "cuda", seed=29)
    o, lse = run_gpu(q, k, v)
    for h in range(4):
        assert torch.equal(o[:, 0, h], v[:, 0, h // 2])
    c = torch.tensor([1.5, -0.75], device="cuda", dtype=torch.bfloat16)
    vc = c.view(1, 1, 2, 1).expand(2, 300, 2, 128).contiguous()
    o, _ = run_gpu(q, k, vc)
    for h in range(4):
        err = (o[:, :, h].float() - float(c[h // 2])).abs().max().item()
        assert err <= 2 ** -8 * abs(float(c[h // 2]))


def test_deterministic():
    w = W.custom(1, 2048, 8, 2, 128)
    q, k, v = W.make_inputs(w, "cuda", seed=31)
    o1, l1 = run_gpu(q, k, v)
    o2, l2 = run_gpu(q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_argument_errors_on_device():
    q = torch.zeros(1, 64, 2, 96, device="cuda", dtype=torch.bfloat16)
    kv = torch.zeros(1, 64, 1, 96, device="cuda", dtype=torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 64, device="cuda")
    st = attn_prefill_fwd(q, kv, kv, o, lse, 1, 64, 2, 1, 96, 1, 0.1)
    assert st == ATTN_ERR_UNSUPPORTED
    q = torch.zeros(1, 64, 3, 64, device="cuda", dtype=torch.bfloat16)
    kv = torch.zeros(1, 64, 2, 64, device="cuda", dtype=torch.bfloat16)
    st = attn_prefill_fwd(q, kv, kv, torch.empty_like(q), torch.empty(1, 3, 64, device="cuda"),
                          1, 64, 3, 2, 64, 1, 0.1)
    assert st == ATTN_ERR_INVALID_ARG


def test_explicit_stream_and_preallocated_outputs():
    w = W.custom(1, 333, 4, 1, 64)
    q, k, v = W.make_inputs(w, "cuda", seed=37)
    s = torch.cuda.Stream()
    o = torch.empty_like(q)
    lse = torch.empty(1, 4, 333, device="cuda")
    torch.cuda.current_stream().synchronize()
    with torch.cuda.stream(s):
        attn_prefill(q, k, v, out=o, lse=lse, stream=s)
    s.synchronize()
    check_full(q, k, v, o, lse, what="side stream")


# ----------------------------------------------------------------------------
# chunked prefill: the query is the last Lq of Lk positions

CHUNKS = [
    # B, Lq, Lk, n_q, n_kv, d_h, causal
    (2, 300, 1000, 8, 2, 128, True),     # offset 700: diagonal spans two key tiles
    (1, 128, 256, 4, 4, 64, True),       # aligned offset
    (1, 1, 777, 2, 1, 128, True),        # a single new token
    (2, 129, 1000, 6, 2, 128, True),     # g = 3, ragged chunk
    (1, 250, 250, 4, 2, 128, True),      # Lq = Lk through the chunk entry point
    (1, 300, 500, 4, 2, 128, False),     # full attention over the prefix
    (1, 640, 1664, 2, 1, 64, True),      # g = 1, aligned offset 1024
]


@pytest.mark.parametrize("case", CHUNKS, ids=lambda c: "B%d_Lq%d_Lk%d_q%d_kv%d_d%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full"))
def test_chunk_full(case):
    B, Lq, Lk, n_q, n_kv, d, causal = case
    w = W.custom(B, Lq, n_q, n_kv, d, causal, Lk=Lk)
    q, k, v = W.make_inputs(w, "cuda", seed=hash(case) % 100000)
    o, lse = run_gpu(q, k, v, causal=causal)
    check_full(q, k, v, o, lse, causal=causal, what=str(case))


@pytest.mark.parametrize("Lq,Lk", [(256, 1024), (640, 2048), (100, 1100)])
def test_chunk_matches_suffix_of_full_pass(Lq, Lk):
    """A chunk's rows are the last rows of one full causal pass over the whole
    sequence; with a tile-aligned offset every query tile sees the same key
    tiles in the same order, so the outputs are bit-identical."""
    w = W.custom(1, Lk, 8, 2, 128)
    qf, k, v = W.make_inputs(w, "cuda", seed=Lq + Lk)
    o_full, l_full = run_gpu(qf, k, v)
    q = qf[:, Lk - Lq:].contiguous()
    o, lse = run_gpu(q, k, v)
    if (Lk - Lq) % 128 == 0:
        assert torch.equal(o, o_full[:, Lk - Lq:]) and torch.equal(lse, l_full[:, :, Lk - Lq:])
    else:
        d = (o.float() - o_full[:, Lk - Lq:].float()).abs().max().item()
        assert d <= 1e-2
        assert (lse - l_full[:, :, Lk - Lq:]).abs().max().item() <= 1e-3


def test_chunked_prefill_in_pieces_equals_one_pass():
    """Prefilling a prompt as four chunks, each attending to everything before
    it, reproduces the single causal pass."""
    w = W.custom(2, 1536, 4, 2, 128)
    qf, k, v = W.make_inputs(w, "cuda", seed=91)
    o_full, l_full = run_gpu(qf, k, v)
    for c0, c1 in [(0, 384), (384, 768), (768, 1152), (1152, 1536)]:
        o, lse = run_gpu(qf[:, c0:c1].contiguous(), k[:, :c1].contiguous(), v[:, :c1].contiguous())
        assert torch.equal(o, o_full[:, c0:c1]) and torch.equal(lse, l_full[:, :, c0:c1])


def test_chunk_workload_full():
    w = W.WORKLOADS[6]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_gpu(q, k, v, causal=w.causal, scale=w.scale)
    err = check_full(q, k, v, o, lse, causal=w.causal, scale=w.scale, what=w.name)
    print(f"parity {w.name}: {err}")


def test_chunk_workload_sampled_rows():
    w = W.WORKLOADS[7]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_gpu(q, k, v, causal=w.causal, scale=w.scale)
    rows = W.sampled_rows(w)
    err = check_rows(q, k, v, o, lse, rows, causal=w.causal, scale=w.scale, what=w.name)
    print(f"parity {w.name} ({len(rows)} sampled rows): {err}")
