"""Host-side checks of the C ABI (no GPU needed, no compute call).

The library is built here if needed (nvcc cross-compiles sm_103a without a
GPU), loaded, and checked to export every function the public header
declares. Argument validation is exercised only with calls that the library
rejects before its first CUDA call.
"""

import ctypes
import math
import os
import re

import numpy as np
import pytest

import causal_gqa_prefill_gb300 as cg
from causal_gqa_prefill_gb300 import build, workloads
from oracle import flops as oflops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return cg.load_library()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("attn_prefill_fwd", "attn_status_string", "attn_device_check"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_debug_library_builds_and_exports_every_declared_symbol():
    dbg = cg.load_library(build.build(debug=True))
    for name in _declared_functions():
        assert hasattr(dbg, name), name
    assert cg.status_string(cg.ATTN_ERR_CHECK).startswith("ATTN_ERR_CHECK")


def test_status_strings(lib):
    for code in range(5):
        s = cg.status_string(code)
        assert s.startswith("ATTN_")
    assert "UNKNOWN" in cg.status_string(99)


FAKE = 1 << 20   # 16-byte aligned, never dereferenced: each call fails validation first


@pytest.mark.parametrize("args,expect", [
    (dict(q=0), cg.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), cg.ATTN_ERR_INVALID_ARG),
    (dict(B=0), cg.ATTN_ERR_INVALID_ARG),
    (dict(L=0), cg.ATTN_ERR_INVALID_ARG),
    (dict(L=-5), cg.ATTN_ERR_INVALID_ARG),
    (dict(n_q=6, n_kv=4), cg.ATTN_ERR_INVALID_ARG),
    (dict(n_kv=0), cg.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), cg.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.nan), cg.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.inf), cg.ATTN_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), cg.ATTN_ERR_INVALID_ARG),
    (dict(o=FAKE + 2), cg.ATTN_ERR_INVALID_ARG),
    (dict(lse=FAKE + 2), cg.ATTN_ERR_INVALID_ARG),
    (dict(d_h=96), cg.ATTN_ERR_UNSUPPORTED),
    (dict(d_h=256), cg.ATTN_ERR_UNSUPPORTED),
    (dict(L=1 << 31), cg.ATTN_ERR_UNSUPPORTED),
])
def test_validation_rejects_before_any_cuda_call(lib, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, L=128, n_q=4, n_kv=2, d_h=128,
             causal=1, scale=0.125)
    a.update(args)
    st = cg.attn_prefill_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"], a["n_q"],
                             a["n_kv"], a["d_h"], a["causal"], a["scale"], stream=0)
    assert st == expect


@pytest.mark.parametrize("Lq,Lk,expect", [(0, 10, cg.ATTN_ERR_INVALID_ARG),
                                           (11, 10, cg.ATTN_ERR_INVALID_ARG),
                                           (10, 1 << 31, cg.ATTN_ERR_UNSUPPORTED)])
def test_chunk_validation(lib, Lq, Lk, expect):
    st = cg.attn_prefill_fwd_chunk(FAKE, FAKE, FAKE, FAKE, FAKE, 1, Lq, Lk, 4, 2, 128, 1, 0.125,
                                   stream=0)
    assert st == expect


@pytest.mark.parametrize("args,expect", [
    (dict(d_h=64), cg.ATTN_ERR_UNSUPPORTED),
    (dict(qd=math.nan), cg.ATTN_ERR_INVALID_ARG),
    (dict(vd=math.inf), cg.ATTN_ERR_INVALID_ARG),
    (dict(q=0), cg.ATTN_ERR_INVALID_ARG),
])
def test_fp8_validation(lib, args, expect):
    a = dict(q=FAKE, d_h=128, qd=1.0, vd=1.0)
    a.update(args)
    st = cg.attn_prefill_fwd_fp8(a["q"], FAKE, FAKE, FAKE, FAKE, 1, 128, 128, 4, 2, a["d_h"], 1,
                                 0.125, a["qd"], 1.0, a["vd"], stream=0)
    assert st == expect


def test_decode_workspace_and_validation(lib):
    assert cg.attn_decode_workspace_bytes(1, 1000, 8, 2) > 0
    assert cg.attn_decode_workspace_bytes(1, 1000, 8, 2, 64) == -1
    assert cg.attn_decode_workspace_bytes(0, 1000, 8, 2) == -1
    need = cg.attn_decode_workspace_bytes(1, 1000, 8, 2)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, 1, 1000, 8, 2, 128, 0.1]
    bad = list(args); bad[5] = 0                       # no workspace
    assert cg.attn_decode_fwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[6] = need - 16               # workspace too small
    assert cg.attn_decode_fwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[11] = 64                     # head dim
    assert cg.attn_decode_fwd(*bad, stream=0) == cg.ATTN_ERR_UNSUPPORTED
    bad = list(args); bad[9], bad[10] = 34, 2          # g = 17
    assert cg.attn_decode_fwd(*bad, stream=0) == cg.ATTN_ERR_UNSUPPORTED
    assert cg.attn_decode_workspace_bytes(1, 1000, 32, 2) > 0     # g = 16
    assert cg.attn_decode_workspace_bytes(1, 1000, 34, 2) == -1   # g = 17


def test_backward_workspace_and_validation(lib):
    need = cg.attn_prefill_bwd_workspace_bytes(2, 300, 8, 2)
    assert need == 2 * 2 * 8 * 384 * 4        # LSE*log2(e) and D, padded to 128-row tiles
    assert cg.attn_prefill_bwd_workspace_bytes(2, 300, 8, 2, 64) == need   # independent of d_h
    assert cg.attn_prefill_bwd_workspace_bytes(2, 300, 8, 2, 32) == -1
    assert cg.attn_prefill_bwd_workspace_bytes(2, 300, 8, 3) == -1
    assert cg.attn_prefill_bwd_workspace_bytes(0, 300, 8, 2) == -1
    args = [FAKE] * 10 + [need, 2, 300, 8, 2, 128, 1, 0.1]
    for idx in range(10):                                # every pointer is required
        bad = list(args); bad[idx] = 0
        assert cg.attn_prefill_bwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG, idx
    bad = list(args); bad[5] = FAKE + 2                  # dout misaligned
    assert cg.attn_prefill_bwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[10] = need - 16                # workspace too small
    assert cg.attn_prefill_bwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[16] = 2                        # causal not 0/1
    assert cg.attn_prefill_bwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[17] = math.inf
    assert cg.attn_prefill_bwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[14] = 3                        # n_q % n_kv
    assert cg.attn_prefill_bwd(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[15] = 96                       # head dim
    assert cg.attn_prefill_bwd(*bad, stream=0) == cg.ATTN_ERR_UNSUPPORTED


def test_host_entry_staging_and_validation(lib):
    need = cg.attn_prefill_host_staging_bytes(2, 300, 500, 8, 2, 128)
    r = lambda x: (x + 255) // 256 * 256
    q, kv, ls = 2 * 300 * 8 * 128 * 2, 2 * 500 * 2 * 128 * 2, 2 * 8 * 300 * 4
    assert need == r(q) + 2 * r(kv) + r(q) + r(ls)
    assert cg.attn_prefill_host_staging_bytes(2, 500, 300, 8, 2, 128) == -1     # Lk < Lq
    assert cg.attn_prefill_host_staging_bytes(2, 300, 500, 8, 3, 128) == -1
    assert cg.attn_prefill_host_staging_bytes(2, 300, 500, 8, 2, 96) == -1
    args = [FAKE] * 6 + [need, 2, 300, 500, 8, 2, 128, 1, 0.1]
    for idx in range(6):                                   # every pointer is required
        bad = list(args); bad[idx] = 0
        assert cg.attn_prefill_fwd_host(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG, idx
    bad = list(args); bad[5] = FAKE + 128                  # staging not 256-byte aligned
    assert cg.attn_prefill_fwd_host(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[6] = need - 256                  # staging too small
    assert cg.attn_prefill_fwd_host(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[13] = 2                          # causal
    assert cg.attn_prefill_fwd_host(*bad, stream=0) == cg.ATTN_ERR_INVALID_ARG
    bad = list(args); bad[12] = 96                         # head dim
    assert cg.attn_prefill_fwd_host(*bad, stream=0) == cg.ATTN_ERR_UNSUPPORTED


def test_selftest_rejects_bad_limits(lib):
    assert cg.attn_selftest_wait_timeout(0, stream=0) == cg.ATTN_ERR_INVALID_ARG
    assert cg.attn_selftest_wait_timeout(-5, stream=0) == cg.ATTN_ERR_INVALID_ARG
    assert cg.attn_selftest_wait_timeout((1 << 31) + 1, stream=0) == cg.ATTN_ERR_INVALID_ARG
    for bad in (0, -5, (1 << 31) + 1):
        assert cg.attn_selftest_wait_timeout_noalloc(bad, stream=0) == cg.ATTN_ERR_INVALID_ARG


def test_chunk_workload_flops_reduce_to_square():
    w = workloads.custom(1, 300, 4, 2, 64, Lk=300)
    assert w.metric_flops() == oflops.causal_attention_flops(1, 300, 4, 64)
    c = workloads.WORKLOADS[6]
    # rows at positions offset..offset+L-1 see offset+i+1 keys: sum of 4*d*(offset+i) in L^2/2 form
    assert c.metric_flops() == 2 * c.n_q * c.d_h * (2 * c.L * c.offset + c.L ** 2)


def test_grid_size_argument_errors(lib):
    assert cg.attn_prefill_grid_size(0, 128, 4, 2, 128) == -1
    assert cg.attn_prefill_grid_size(1, 128, 4, 3, 128) == -1
    assert cg.attn_prefill_grid_size(1, 128, 4, 2, 80) == -1


def test_wrapper_rejects_host_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        cg.attn_prefill(x, x, x)


def test_metric_flops_match_the_oracle_cost_model():
    for w in workloads.WORKLOADS.values():
        if w.keys == w.L:
            fwd = oflops.causal_attention_flops(w.B, w.L, w.n_q, w.d_h)
            # backward: five products of the forward's size against its two
            assert w.metric_flops() == (fwd * 5 // 2 if w.backward else fwd)


def test_sampled_rows_cover_every_head_tile_and_tile_position():
    # the sampled-row workloads (the L=32768 and L=131072 layers and the
    # 16384-row chunk): every query tile, every head and every position inside
    # a tile is checked, plus rows 0 and L-1 of every head
    for num in (4, 5, 7, 8, 9):
        w = workloads.WORKLOADS[num]
        rows = workloads.sampled_rows(w)
        assert rows.shape[1] == 3 and len(rows) >= 4000
        assert set(rows[:, 1]) == set(range(w.n_q))
        assert set(rows[:, 2] % 128) == set(range(128))
        T = (w.L + 127) // 128
        assert T <= 4096
        assert set(rows[:, 2] // 128) == set(range(T)), num
        for h in range(w.n_q):
            sel = rows[rows[:, 1] == h, 2]
            assert 0 in sel and w.L - 1 in sel
        assert (rows[:, 2] < w.L).all() and (rows[:, 2] >= 0).all()
        assert (rows[:, 0] == 0).all()
        # every tile meets more than one head where there are samples to spare
        if 4096 >= 2 * T:
            heads_per_tile = [len(set(rows[rows[:, 2] // 128 == t, 1])) for t in range(T)]
            assert min(heads_per_tile) >= 2, num


def test_sampled_rows_ragged_tail_and_batches():
    w = workloads.custom(3, 1000, 6, 2, 128)      # 8 tiles, the last one ragged
    rows = workloads.sampled_rows(w, count=512)
    assert set(rows[:, 2] // 128) == set(range(8))
    assert (rows[:, 2] <= 999).all() and 999 in rows[:, 2]
    assert set(rows[:, 0]) == {0, 1, 2} and set(rows[:, 1]) == set(range(6))
