"""The pages' cost model for prefill attention, as plain functions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
  * "prefill-attention" flop record (phantomic12), section "Arithmetic
    intensity": causal FLOPs = 2*n_q*d_h*L^2 (Q K^T and P V each
    2*L^2*d_h*n_q, both halved by the mask); K/V bytes = 2 tensors *
    L*d_h*n_kv elements * 2 bytes; AI = g*L/2; ridge = 1000*TFLOP/s / (GB/s);
    L_ridge = 2*ridge/g; flop crossover L* = P_layer/(n_q*d_h).
  * "Long-Context Attention Explained" (sevydevy), quadratic-cost section:
    the dense count 4*N^2*width per layer (the FlashAttention-2 paper's
    4*seq^2*head_size*heads).
"""

from __future__ import annotations


def causal_attention_flops(B: int, L: int, n_q: int, d_h: int) -> int:
    """Causal prefill attention FLOPs, 2*n_q*d_h*L^2 per sequence, times B."""
    return 2 * n_q * d_h * L * L * B


def dense_attention_flops(B: int, L: int, n_q: int, d_h: int) -> int:
    """Unmasked attention FLOPs, 4*L^2*d_h*n_q per sequence, times B."""
    return 4 * L * L * d_h * n_q * B


def kv_bytes(B: int, L: int, n_kv: int, d_h: int, elem_bytes: int = 2) -> int:
    """Bytes of K and V read once: 2 tensors * L*d_h*n_kv elements."""
    return 2 * L * d_h * n_kv * elem_bytes * B


def arithmetic_intensity(L: int, n_q: int, n_kv: int) -> float:
    """Causal FLOPs per K/V byte for bf16 K/V: (n_q/n_kv) * L / 2."""
    return causal_attention_flops(1, L, n_q, 1) / kv_bytes(1, L, n_kv, 1)


def ridge(tflops: float, gbs: float) -> float:
    """Dense balance point in FLOP/byte: 1000 * TFLOP/s / (GB/s)."""
    return 1000.0 * tflops / gbs


def ridge_length(tflops: float, gbs: float, g: float) -> float:
    """Sequence length where causal attention reaches the ridge: 2*ridge/g."""
    return 2.0 * ridge(tflops, gbs) / g


def flop_crossover(p_layer: float, n_q: int, d_h: int) -> float:
    """Length where attention FLOPs equal the layer's weight-matmul FLOPs.

    Weight matmuls cost 2*P_layer FLOPs per token; causal attention costs
    2*n_q*d_h*L per token at length L, so the two meet at P_layer/(n_q*d_h).
    """
    return p_layer / (n_q * d_h)


def attention_share(L: int, p_layer: float, n_q: int, d_h: int) -> float:
    """Fraction of one layer's prefill FLOPs spent in causal attention."""
    attn = causal_attention_flops(1, L, n_q, d_h)
    gemm = 2.0 * p_layer * L
    return attn / (attn + gemm)
