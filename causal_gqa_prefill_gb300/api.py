"""Python entry points over the C ABI (torch supplies device memory and streams).

``attn_prefill_fwd`` mirrors the C function argument for argument; the
convenience wrapper ``attn_prefill`` allocates the outputs and derives the
sizes from the tensors. Both only marshal arguments: the attention forward
runs entirely in the CUDA library, and a status other than ATTN_OK raises.
"""

from __future__ import annotations

import math

from . import _abi


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {_abi.status_string(status)}")


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def attn_prefill_fwd(q, k, v, o, lse, B, L, n_q, n_kv, d_h, causal, scale, stream=None) -> int:
    """Direct call of the C entry point; returns the raw status code.

    q, k, v, o, lse are CUDA tensors or integer device addresses with the
    layouts of the C header; ``stream`` is a torch.cuda.Stream, a raw
    cudaStream_t as int, or None for torch's current stream.
    """
    lib = _abi.load()
    return int(lib.attn_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(L),
                                    int(n_q), int(n_kv), int(d_h), int(causal), float(scale),
                                    _stream_handle(stream)))


def attn_prefill_fwd_chunk(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d_h, causal, scale,
                           stream=None) -> int:
    """Direct call of the chunked-prefill C entry point (query = last Lq of Lk
    positions); returns the raw status code."""
    lib = _abi.load()
    return int(lib.attn_prefill_fwd_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                          int(Lq), int(Lk), int(n_q), int(n_kv), int(d_h),
                                          int(causal), float(scale), _stream_handle(stream)))


def attn_prefill_fwd_fp8(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d_h, causal, scale, q_descale,
                         k_descale, v_descale, stream=None) -> int:
    """Direct call of the e4m3 C entry point; returns the raw status code."""
    lib = _abi.load()
    return int(lib.attn_prefill_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                        int(Lq), int(Lk), int(n_q), int(n_kv), int(d_h),
                                        int(causal), float(scale), float(q_descale),
                                        float(k_descale), float(v_descale),
                                        _stream_handle(stream)))


def attn_prefill_fp8(q, k, v, *, q_descale=1.0, k_descale=1.0, v_descale=1.0, causal=True,
                     scale=None, out=None, lse=None, stream=None):
    """Attention over e4m3 CUDA tensors (torch.float8_e4m3fn) q [B,Lq,n_q,128],
    k/v [B,Lk,n_kv,128], real values = stored * descale. Returns (o bf16
    [B, Lq, n_q, 128], lse fp32 [B, n_q, Lq])."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.float8_e4m3fn:
            raise TypeError(f"{name} must be float8_e4m3fn")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, L, H, d_h] tensor")
    B, L, n_q, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] < L or k.shape[3] != d:
        raise ValueError("k and v must be [B, Lk, n_kv, d_h] with Lk >= Lq, matching q")
    Lk, n_kv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, L, n_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, n_q, L), dtype=torch.float32, device=q.device)
    st = attn_prefill_fwd_fp8(q, k, v, out, lse, B, L, Lk, n_q, n_kv, d, int(bool(causal)),
                              scale, q_descale, k_descale, v_descale, stream)
    if st != _abi.ATTN_OK:
        raise AttnError(st, "attn_prefill_fwd_fp8")
    return out, lse


def attn_decode_workspace_bytes(B, Lk, n_q, n_kv, d_h=128) -> int:
    return int(_abi.load().attn_decode_workspace_bytes(int(B), int(Lk), int(n_q), int(n_kv),
                                                       int(d_h)))


def attn_decode_fwd(q, k, v, o, lse, workspace, workspace_bytes, B, Lk, n_q, n_kv, d_h, scale,
                    stream=None) -> int:
    """Direct call of the decode C entry point; returns the raw status code."""
    lib = _abi.load()
    return int(lib.attn_decode_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                   int(workspace_bytes), int(B), int(Lk), int(n_q), int(n_kv),
                                   int(d_h), float(scale), _stream_handle(stream)))


def attn_decode(q, k, v, *, scale=None, workspace=None, out=None, lse=None, stream=None):
    """One decode step: q bf16 [B, 1, n_q, 128] against the cache k/v bf16
    [B, Lk, n_kv, 128]. Returns (o bf16 [B, 1, n_q, 128], lse fp32 [B, n_q, 1]).
    ``workspace`` (a CUDA tensor of at least attn_decode_workspace_bytes
    bytes) is allocated with torch when not given."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be a bfloat16 CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, L, H, d_h] tensor")
    B, one, n_q, d = q.shape
    if one != 1 or k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("q must be [B, 1, n_q, d_h] and k, v [B, Lk, n_kv, d_h]")
    Lk, n_kv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_decode_workspace_bytes(B, Lk, n_q, n_kv, d)
    if need < 0:
        raise AttnError(_abi.ATTN_ERR_UNSUPPORTED, "attn_decode_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, n_q, 1), dtype=torch.float32, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    st = attn_decode_fwd(q, k, v, out, lse, workspace, nbytes, B, Lk, n_q, n_kv, d, scale, stream)
    if st != _abi.ATTN_OK:
        raise AttnError(st, "attn_decode_fwd")
    return out, lse


def attn_prefill_bwd_workspace_bytes(B, L, n_q, n_kv, d_h=128) -> int:
    return int(_abi.load().attn_prefill_bwd_workspace_bytes(int(B), int(L), int(n_q), int(n_kv),
                                                            int(d_h)))


def attn_prefill_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, L, n_q,
                     n_kv, d_h, causal, scale, stream=None) -> int:
    """Direct call of the backward C entry point; returns the raw status code."""
    lib = _abi.load()
    return int(lib.attn_prefill_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                    int(workspace_bytes), int(B), int(L), int(n_q), int(n_kv),
                                    int(d_h), int(causal), float(scale), _stream_handle(stream)))


def attn_prefill_backward(q, k, v, o, lse, dout, *, causal=True, scale=None, workspace=None,
                          dq=None, dk=None, dv=None, stream=None):
    """Gradients (dq, dk, dv) of attn_prefill for the upstream gradient ``dout``.

    q, o, dout: bf16 CUDA tensors [B, L, n_q, d_h]; k, v: [B, L, n_kv, d_h], d_h 64 or 128;
    lse: the forward's fp32 [B, n_q, L]. Outputs are allocated unless passed
    in; ``workspace`` (at least attn_prefill_bwd_workspace_bytes bytes) is
    allocated with torch when not given."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be a bfloat16 CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, L, H, d_h] tensor")
    B, L, n_q, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != L or k.shape[3] != d:
        raise ValueError("k and v must be [B, L, n_kv, d_h] matching q")
    if o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("o and dout must be shaped like q")
    n_kv = k.shape[2]
    if (not isinstance(lse, torch.Tensor) or lse.dtype != torch.float32 or not lse.is_cuda
            or tuple(lse.shape) != (B, n_q, L) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, n_q, L]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_prefill_bwd_workspace_bytes(B, L, n_q, n_kv, d)
    if need < 0:
        raise AttnError(_abi.ATTN_ERR_UNSUPPORTED, "attn_prefill_bwd_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = workspace.numel() * workspace.element_size()
    st = attn_prefill_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, nbytes, B, L, n_q, n_kv,
                          d, int(bool(causal)), scale, stream)
    if st != _abi.ATTN_OK:
        raise AttnError(st, "attn_prefill_bwd")
    return dq, dk, dv


def attn_device_check(stream=None) -> int:
    """Synchronise the stream and report device-side timeouts (raw status)."""
    return int(_abi.load().attn_device_check(_stream_handle(stream)))


def attn_prefill_host_staging_bytes(B, Lq, Lk, n_q, n_kv, d_h=128) -> int:
    return int(_abi.load().attn_prefill_host_staging_bytes(int(B), int(Lq), int(Lk), int(n_q),
                                                           int(n_kv), int(d_h)))


def attn_prefill_fwd_host(q, k, v, o, lse, staging, staging_bytes, B, Lq, Lk, n_q, n_kv, d_h,
                          causal, scale, stream=None) -> int:
    """Direct call of the host-buffer C entry point (q, k, v, o, lse host
    tensors or addresses; staging a device buffer); returns the raw status."""
    lib = _abi.load()
    return int(lib.attn_prefill_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                         _ptr(staging), int(staging_bytes), int(B), int(Lq),
                                         int(Lk), int(n_q), int(n_kv), int(d_h), int(causal),
                                         float(scale), _stream_handle(stream)))


def attn_selftest_wait_timeout(spin_cycles: int, stream=None) -> int:
    """Enqueue the wait-limit diagnostic kernel (raw status of the launch)."""
    return int(_abi.load().attn_selftest_wait_timeout(int(spin_cycles), _stream_handle(stream)))


def attn_selftest_wait_timeout_noalloc(spin_cycles: int, stream=None) -> int:
    """The wait-limit diagnostic reporting into the allocation-free entry
    point's fixed status word (raw status of the launch)."""
    return int(_abi.load().attn_selftest_wait_timeout_noalloc(int(spin_cycles),
                                                             _stream_handle(stream)))


def attn_prefill_grid_size(B, L, n_q, n_kv, d_h, causal=True) -> int:
    return int(_abi.load().attn_prefill_grid_size(int(B), int(L), int(n_q), int(n_kv), int(d_h),
                                                  int(bool(causal))))


def attn_prefill(q, k, v, *, causal: bool = True, scale: float | None = None, out=None, lse=None,
                 stream=None):
    """O, LSE = attention(q, k, v) for bf16 CUDA tensors q [B,Lq,n_q,d], k/v [B,Lk,n_kv,d].

    Lk = Lq is ordinary prefill; Lk > Lq is a chunk whose rows are the last Lq
    positions of the key range (chunked prefill). Returns (o bf16
    [B, Lq, n_q, d], lse fp32 [B, n_q, Lq]). ``scale`` defaults to 1/sqrt(d).
    Outputs may be passed in (``out``, ``lse``) to avoid allocation. The call
    is asynchronous on ``stream`` (default: current).
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, L, H, d_h] tensor")
    B, L, n_q, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] < L or k.shape[3] != d:
        raise ValueError("k and v must be [B, Lk, n_kv, d_h] with Lk >= Lq, matching q")
    Lk, n_kv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse is None:
        lse = torch.empty((B, n_q, L), dtype=torch.float32, device=q.device)
    elif tuple(lse.shape) != (B, n_q, L) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, n_q, L] tensor")
    if Lk == L:
        st = attn_prefill_fwd(q, k, v, out, lse, B, L, n_q, n_kv, d, int(bool(causal)), scale,
                              stream)
    else:
        st = attn_prefill_fwd_chunk(q, k, v, out, lse, B, L, Lk, n_q, n_kv, d,
                                    int(bool(causal)), scale, stream)
    if st != _abi.ATTN_OK:
        raise AttnError(st, "attn_prefill_fwd" if Lk == L else "attn_prefill_fwd_chunk")
    return out, lse
