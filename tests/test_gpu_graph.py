"""The library's calls inside CUDA graphs: after the one-time set-up, forward,
chunked forward, decode and backward calls captured into one graph replay to
the same bits as the eager calls, and follow new values written into the
captured input buffers. A first call made during a capture is refused
without setting anything up."""

import json
import os
import subprocess
import sys

import pytest

from causal_gqa_prefill_gb300 import (ATTN_ERR_UNSUPPORTED, ATTN_OK, attn_decode,
                                      attn_decode_workspace_bytes, attn_device_check,
                                      attn_prefill, attn_prefill_backward,
                                      attn_prefill_bwd_workspace_bytes, attn_prefill_fwd_chunk)
from causal_gqa_prefill_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from causal_gqa_prefill_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _chunk(q, k, v, o, lse):
    B, Lq, n_q, d = q.shape
    Lk, n_kv = k.shape[1], k.shape[2]
    st = attn_prefill_fwd_chunk(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d, 1, d ** -0.5)
    assert st == ATTN_OK, st


def _all_calls(x, outs):
    """Every captured call, writing into the preallocated `outs`."""
    q, k, v, qc, qd, do, o_f, l_f = x
    attn_prefill(q, k, v, out=outs["o"], lse=outs["lse"])
    _chunk(qc, k, v, outs["oc"], outs["lc"])
    attn_decode(qd, k, v, out=outs["od"], lse=outs["ld"], workspace=outs["ws_dec"])
    attn_prefill_backward(q, k, v, o_f, l_f, do, workspace=outs["ws_bwd"], dq=outs["dq"],
                          dk=outs["dk"], dv=outs["dv"])


def _make(seed):
    w = W.custom(2, 700, 8, 2, 128)
    q, k, v = W.make_inputs(w, "cuda", seed=seed)
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    qc = torch.randn(2, 300, 8, 128, device="cuda", generator=g).to(torch.bfloat16)
    qd = torch.randn(2, 1, 8, 128, device="cuda", generator=g).to(torch.bfloat16)
    do = torch.randn(2, 700, 8, 128, device="cuda", generator=g).to(torch.bfloat16)
    return q, k, v, qc, qd, do


def test_graph_replay_matches_eager_calls():
    q, k, v, qc, qd, do = _make(31)
    o_f, l_f = attn_prefill(q, k, v)              # the backward's saved forward
    x = (q, k, v, qc, qd, do, o_f, l_f)
    outs = {
        "o": torch.empty_like(q), "lse": torch.empty(2, 8, 700, device="cuda"),
        "oc": torch.empty_like(qc), "lc": torch.empty(2, 8, 300, device="cuda"),
        "od": torch.empty_like(qd), "ld": torch.empty(2, 8, 1, device="cuda"),
        "dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
        "ws_dec": torch.empty(attn_decode_workspace_bytes(2, 700, 8, 2), dtype=torch.uint8,
                              device="cuda"),
        "ws_bwd": torch.empty(attn_prefill_bwd_workspace_bytes(2, 700, 8, 2), dtype=torch.uint8,
                              device="cuda"),
    }
    # eager: the one-time set-up of every family happens here
    _all_calls(x, outs)
    torch.cuda.synchronize()
    assert attn_device_check() == ATTN_OK
    eager = {n: t.clone() for n, t in outs.items() if not n.startswith("ws")}

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _all_calls(x, outs)                         # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        _all_calls(x, outs)
    for n in eager:
        outs[n].zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert attn_device_check() == ATTN_OK
    for n, t in eager.items():
        assert torch.equal(outs[n], t), n

    # new values in the captured input buffers: the replay follows them
    q2, k2, v2, qc2, qd2, do2 = _make(32)
    for dst, src in zip((q, k, v, qc, qd, do), (q2, k2, v2, qc2, qd2, do2)):
        dst.copy_(src)
    ref = {n: torch.empty_like(t) for n, t in eager.items()}
    ref.update({n: outs[n] for n in ("ws_dec", "ws_bwd")})
    _all_calls(x, ref)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert attn_device_check() == ATTN_OK
    for n in eager:
        assert torch.equal(outs[n], ref[n]), n
        assert not torch.equal(outs[n], eager[n]), n


_FIRST_CALL = r"""
import json, torch
import causal_gqa_prefill_gb300 as cg
torch.cuda.set_device(0)
q = torch.randn(1, 256, 4, 128, device="cuda").to(torch.bfloat16)
k = torch.randn(1, 256, 2, 128, device="cuda").to(torch.bfloat16)
v = torch.randn_like(k)
qd = q[:, -1:].contiguous()
torch.cuda.synchronize()
res = {}
def in_capture(name, fn):
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            fn()
        res[name + "_capture"] = "ok"
    except cg.AttnError as e:
        res[name + "_capture"] = e.status
    out = fn()
    torch.cuda.synchronize()
    res[name + "_eager"] = cg.attn_device_check()
    return out
o, lse = in_capture("fwd", lambda: cg.attn_prefill(q, k, v))
in_capture("dec", lambda: cg.attn_decode(qd, k, v))
in_capture("bwd", lambda: cg.attn_prefill_backward(q, k, v, o, lse, torch.randn_like(o)))
print(json.dumps(res))
"""


def test_first_call_during_capture_is_refused():
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    for fam in ("fwd", "dec", "bwd"):
        assert res[fam + "_capture"] == ATTN_ERR_UNSUPPORTED, res
        assert res[fam + "_eager"] == ATTN_OK, res


def test_concurrent_streams_match_sequential_calls():
    """The same calls issued on two streams with no ordering between them
    (each stream with its own workspaces and outputs) give the bits they give
    one after another: no state of one call leaks into the other."""
    a, b = _make(41), _make(42)
    o_a, l_a = attn_prefill(a[0], a[1], a[2])
    o_b, l_b = attn_prefill(b[0], b[1], b[2])
    torch.cuda.synchronize()

    def calls(x, o_f, l_f):
        q, k, v, qc, qd, do = x
        o, lse = attn_prefill(q, k, v)
        od, ld = attn_decode(qd, k, v)
        grads = attn_prefill_backward(q, k, v, o_f, l_f, do)
        return (o, lse, od, ld) + tuple(grads)

    seq = [calls(a, o_a, l_a), calls(b, o_b, l_b)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    par = []
    for _ in range(3):                     # several rounds so the calls overlap on the GPU
        par = []
        for s, (x, o_f, l_f) in zip(streams, ((a, o_a, l_a), (b, o_b, l_b))):
            with torch.cuda.stream(s):
                par.append(calls(x, o_f, l_f))
    torch.cuda.synchronize()
    assert attn_device_check() == ATTN_OK
    for got, want in zip(par, seq):
        for g, w in zip(got, want):
            assert torch.equal(g, w)


def test_programmatic_successor_sees_complete_backward_outputs():
    """A kernel launched as a programmatic dependent right after the backward
    must find dK and dV complete. The shape makes the dQ kernel (the call's
    last) short and dK/dV long (full attention, 64 query heads on one K/V
    head: 8 dK/dV CTAs of 512 steps against ~3 dQ units per CTA). The decode
    step, whose kernels are programmatic dependents, reads dK and dV as its
    cache straight after the backward; it must equal the same decode step run
    after a synchronize."""
    w = W.custom(1, 1024, 64, 1, 128, causal=False)
    q, k, v = W.make_inputs(w, "cuda", seed=51)
    do = W.make_grad(w, "cuda", seed=51)
    o, lse = attn_prefill(q, k, v, causal=False)
    g = torch.Generator(device="cuda").manual_seed(52)
    qd = torch.randn(1, 1, 16, 128, device="cuda", generator=g).to(torch.bfloat16)
    torch.cuda.synchronize()
    dq, dk, dv = attn_prefill_backward(q, k, v, o, lse, do, causal=False)
    od, ld = attn_decode(qd, dk, dv)                 # no host sync in between
    torch.cuda.synchronize()
    assert attn_device_check() == ATTN_OK
    od2, ld2 = attn_decode(qd, dk, dv)
    torch.cuda.synchronize()
    assert torch.equal(od, od2) and torch.equal(ld, ld2)
