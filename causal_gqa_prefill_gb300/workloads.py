"""Seeded synthetic workloads shaped like the pages' models (no attention math here).

Both the CUDA path's tests/benchmark and the oracle's checks draw their inputs
from this module; it holds only shapes, seeds, random draws and the
sampled-row selector.

Recipe: seed = 1000 + config number; a torch.Generator on the target device
draws Q, K, V in that order as float32 N(0, 1), each rounded to bf16 (round to
nearest even). The 70B-shaped workload multiplies K channels 0..3 of every
K/V head by 8 (N(0, 8^2) there), which pushes single logits far above the
rest and exercises the online-softmax rescaling. Backward workloads draw
the upstream gradient dO after Q, K, V from a second generator seeded with
seed + 500000, float32 N(0, 1) rounded to bf16.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    number: int
    name: str
    B: int
    L: int
    n_q: int
    n_kv: int
    d_h: int
    causal: bool = True
    heavy_k_channels: int = 0       # leading K channels drawn with std 8
    full_check: bool = True         # oracle over every row (else sampled rows)
    Lk: int = 0                     # keys (0: = L); L < Lk makes Q the last L positions
    dtype: str = "bf16"             # "bf16" or "e4m3" (Q, K, V stored as fp8, descale 1)
    decode: bool = False            # one query token per sequence against Lk cached keys
    backward: bool = False          # gradients (dQ, dK, dV) for a seeded upstream dO

    @property
    def keys(self) -> int:
        return self.Lk or self.L

    @property
    def offset(self) -> int:
        return self.keys - self.L

    @property
    def g(self) -> int:
        return self.n_q // self.n_kv

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def scale(self) -> float:
        return self.d_h ** -0.5

    def metric_flops(self) -> int:
        """Causal prefill FLOPs as the metric counts them: 2*n_q*d_h*L^2*B.

        A chunk of L rows after `offset` earlier positions counts the same
        way, 4*d_h*(offset + i) per row i summed in the L^2/2 form:
        2*n_q*d_h*(2*L*offset + L^2)*B (equal to the square count at offset 0).
        """
        if self.decode or not self.causal:
            f = 4 * self.n_q * self.d_h * self.L * self.keys * self.B
        else:
            f = 2 * self.n_q * self.d_h * (2 * self.L * self.offset + self.L * self.L) * self.B
        # backward: five products of the forward's size (S, dP, dV, dK, dQ) against
        # the forward's two, i.e. 2.5x the forward count
        return f * 5 // 2 if self.backward else f

    def io_bytes(self) -> int:
        """Bytes read and written once: Q, K, V, O in bf16 and LSE in fp32 (the
        backward adds dO read and dQ, dK, dV written)."""
        e = self.B * self.d_h * 2
        if self.backward:
            return (e * (4 * self.n_q * self.L + 4 * self.n_kv * self.keys)
                    + self.B * self.n_q * self.L * 4)
        return (e * (2 * self.n_q * self.L + 2 * self.n_kv * self.keys)
                + self.B * self.n_q * self.L * 4)

    def describe(self) -> dict:
        d = {"workload": self.name, "B": self.B, "L": self.L, "n_q": self.n_q,
             "n_kv": self.n_kv, "d_h": self.d_h, "causal": self.causal}
        if self.keys != self.L:
            d["Lk"] = self.keys
        if self.dtype != "bf16":
            d["inputs"] = self.dtype
        if self.decode:
            d["step"] = "decode"
        if self.backward:
            d["step"] = "backward"
        return d


WORKLOADS = {
    1: Workload(1, "tiny GQA-4 (B=1, L=256, n_q=4, n_kv=1, d_h=64)", 1, 256, 4, 1, 64),
    2: Workload(2, "Llama-2-7B-shaped layer, MHA (B=4, L=2048, n_q=n_kv=32, d_h=128)",
                4, 2048, 32, 32, 128),
    3: Workload(3, "Llama-3-8B-shaped layer, GQA-4 (B=1, L=8192, n_q=32, n_kv=8, d_h=128)",
                1, 8192, 32, 8, 128),
    4: Workload(4, "Llama-2-70B-shaped layer, GQA-8, heavy K channels "
                   "(B=1, L=32768, n_q=64, n_kv=8, d_h=128)",
                1, 32768, 64, 8, 128, heavy_k_channels=4, full_check=False),
    5: Workload(5, "long-context 36-head shape, GQA-6 (B=1, L=131072, n_q=36, n_kv=6, d_h=128)",
                1, 131072, 36, 6, 128, full_check=False),
    # chunked prefill: the last chunk of a prompt, attending to its whole prefix
    6: Workload(6, "chunked prefill, Llama-3-8B-shaped layer: last 2048-token chunk of an "
                   "8192-token prompt (B=1, Lq=2048, Lk=8192, n_q=32, n_kv=8, d_h=128)",
                1, 2048, 32, 8, 128, Lk=8192),
    7: Workload(7, "chunked prefill, 36-head shape: last 16384-token chunk of a 131072-token "
                   "prompt (B=1, Lq=16384, Lk=131072, n_q=36, n_kv=6, d_h=128)",
                1, 16384, 36, 6, 128, Lk=131072, full_check=False),
    # fp8 (e4m3) inputs on the model-shaped layers
    8: Workload(8, "fp8 e4m3, Llama-3-8B-shaped layer, GQA-4 (B=1, L=8192, n_q=32, n_kv=8, "
                   "d_h=128)", 1, 8192, 32, 8, 128, dtype="e4m3", full_check=False),
    9: Workload(9, "fp8 e4m3, long-context 36-head shape, GQA-6 (B=1, L=131072, n_q=36, n_kv=6, "
                   "d_h=128)", 1, 131072, 36, 6, 128, dtype="e4m3", full_check=False),
    # decode: one new token per sequence against its cache
    10: Workload(10, "decode, Llama-3-8B-shaped layer: 16 sequences with 8192 cached tokens "
                     "(B=16, Lk=8192, n_q=32, n_kv=8, d_h=128)", 16, 1, 32, 8, 128, Lk=8192,
                 decode=True),
    11: Workload(11, "decode, 36-head shape after a 131072-token prompt (B=1, Lk=131072, n_q=36, "
                     "n_kv=6, d_h=128)", 1, 1, 36, 6, 128, Lk=131072, decode=True),
    # backward: gradients of the Llama-3-8B-shaped layer
    12: Workload(12, "backward, Llama-3-8B-shaped layer, GQA-4 (B=1, L=8192, n_q=32, n_kv=8, "
                     "d_h=128)", 1, 8192, 32, 8, 128, full_check=False, backward=True),
}


def make_inputs(w: Workload, device="cuda", seed: int | None = None):
    """Seeded bf16 (q, k, v) for workload ``w`` on ``device``."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    shape_q = (w.B, w.L, w.n_q, w.d_h)
    shape_kv = (w.B, w.keys, w.n_kv, w.d_h)
    dt = torch.float8_e4m3fn if w.dtype == "e4m3" else torch.bfloat16
    q = torch.randn(shape_q, generator=gen, device=device, dtype=torch.float32).to(dt)
    k = torch.randn(shape_kv, generator=gen, device=device, dtype=torch.float32)
    if w.heavy_k_channels:
        k[..., :w.heavy_k_channels] *= 8.0
    k = k.to(dt)
    v = torch.randn(shape_kv, generator=gen, device=device, dtype=torch.float32).to(dt)
    return q, k, v


def make_grad(w: Workload, device="cuda", seed: int | None = None):
    """Seeded bf16 upstream gradient dO [B, L, n_q, d_h] for a backward workload."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed((w.seed if seed is None else seed) + 500000)
    shape = (w.B, w.L, w.n_q, w.d_h)
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def custom(B, L, n_q, n_kv, d_h, causal=True, number=0, name=None, Lk=0,
           dtype="bf16", backward=False) -> Workload:
    return Workload(number, name or f"B={B} L={L} Lk={Lk or L} n_q={n_q} n_kv={n_kv} d_h={d_h}",
                    B, L, n_q, n_kv, d_h, causal, Lk=Lk, dtype=dtype, backward=backward)


def sampled_rows(w: Workload, count: int = 4096, tile: int = 128):
    """Rows (b, h, i) to check on large workloads.

    For s = 0..count-1: position in tile = s mod 128, head =
    (s + 7 (s div 128)) mod n_q and query tile = perm[(s + s div T) mod T],
    perm a permutation of the T tiles drawn from numpy's default_rng(seed).
    So every head and every intra-tile position is covered, every tile is hit
    whenever count >= T (the tail tile's positions past L-1 fall on row L-1),
    and the shifts by s div 128 and s div T keep head, tile and position from
    locking together when T and n_q share factors with 128 (each tile meets
    several heads and positions). The batch index is drawn from the same
    generator. Rows 0 and L-1 of every (b, head) are added.
    Returns a sorted, de-duplicated int64 array [R, 3].
    """
    import numpy as np

    T = (w.L + tile - 1) // tile
    rng = np.random.default_rng(w.seed)
    s = np.arange(count, dtype=np.int64)
    perm = rng.permutation(T).astype(np.int64)
    i = perm[(s + s // T) % T] * tile + (s % tile)
    i = np.minimum(i, w.L - 1)
    b = rng.integers(0, w.B, count)
    rows = [np.stack([b, (s + 7 * (s // tile)) % w.n_q, i], axis=1)]
    for bb in range(w.B):
        for h in range(w.n_q):
            rows.append(np.array([[bb, h, 0], [bb, h, w.L - 1]], dtype=np.int64))
    return np.unique(np.concatenate(rows, axis=0), axis=0)
