"""Seeded synthetic inputs for the attention KL divergence.

Shared by the tests, the benchmark and the smoke check; it holds none of the
method's arithmetic (no scores, softmax or KL), only the recipe that draws the
teacher and student query/key tensors:

    Q1, K1 ~ N(0, 1) i.i.d. (times ``teacher_scale`` for peaked attention)
    Q2 = Q1 + sigma * eps_Q,  K2 = K1 + sigma * eps_K,  eps ~ N(0, 1)

drawn in float32 in the order Q1, K1, eps_Q, eps_K from one seeded generator
and rounded to bf16 (round-to-nearest-even) after the student is formed.  The
shapes follow the workloads the StreamKL pages evaluate (contexts 4K-512K,
32 heads, BF16; "Experimental Results").
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    sigma: float
    causal: bool
    teacher_scale: float = 1.0
    seed: int = 0
    fwd_only: bool = False  # the decode (Split-K) workloads run the forward only
    H_kv: int = 0           # key heads when keys are shared by groups of query heads (0 = H)

    @property
    def g_value(self) -> float:
        """Upstream gradient per row: 1 for the tiny case, 1/(H*Nq) otherwise."""
        return 1.0 if self.name == "tiny" else 1.0 / (self.H * self.Nq)

    def fwd_bytes(self) -> int:
        """Algorithmic HBM bytes of one forward: every Q and K element read once
        (bf16) and KL, LSE1, LSE2 written once (float32)."""
        hk = self.H_kv or self.H
        return 2 * 2 * self.B * (self.H * self.Nq + hk * self.Nk) * self.d + 12 * self.B * self.H * self.Nq

    def bwd_bytes(self) -> int:
        """Algorithmic HBM bytes of one backward with float32 gradients: every Q
        and K element read once (bf16), LSE1, LSE2, KL and g read (16 B per row),
        dQ and dK of the trainable side written once (float32)."""
        hk = self.H_kv or self.H
        rows_q, rows_k = self.B * self.H * self.Nq, self.B * hk * self.Nk
        return 2 * 2 * (rows_q + rows_k) * self.d + 16 * rows_q + 4 * (rows_q + rows_k) * self.d

    def visible_pairs(self) -> int:
        """Query/key pairs inside the mask, per head.  Causal rows are aligned
        bottom-right (row i sees keys j <= i + Nk - Nq), so row i sees
        i + Nk - Nq + 1 keys."""
        if not self.causal:
            return self.Nq * self.Nk
        off = self.Nk - self.Nq
        return self.Nq * (off + 1) + self.Nq * (self.Nq - 1) // 2


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 256, 256, 64, 0.5, False, seed=0),
    "8k_causal": Workload("8k_causal", 1, 32, 8192, 8192, 128, 0.3, True, seed=1),
    "64k_causal": Workload("64k_causal", 1, 32, 65536, 65536, 128, 0.3, True, seed=2),
    "64k": Workload("64k", 1, 32, 65536, 65536, 128, 0.3, False, seed=2),
    "decode_q1_k128k": Workload("decode_q1_k128k", 4, 32, 1, 131072, 128, 0.3, False, seed=3, fwd_only=True),
    "decode_q16_k128k": Workload("decode_q16_k128k", 4, 32, 16, 131072, 128, 0.3, False, seed=3, fwd_only=True),
    "decode_q1_k512k": Workload("decode_q1_k512k", 4, 32, 1, 524288, 128, 0.3, False, seed=3, fwd_only=True),
    "decode_q16_k512k": Workload("decode_q16_k512k", 4, 32, 16, 524288, 128, 0.3, False, seed=3, fwd_only=True),
    # causal (bottom-right) Split-K: 16 new queries against a 128K-key prefix (chunked prefill)
    "decode_causal_q16_k128k": Workload("decode_causal_q16_k128k", 4, 32, 16, 131072, 128, 0.3, True, seed=5,
                                        fwd_only=True),
    # decode with keys shared by groups of 4 query heads (32 query heads, 8 key heads)
    "decode_gqa_q1_k128k": Workload("decode_gqa_q1_k128k", 4, 32, 1, 131072, 128, 0.3, False, seed=7,
                                    fwd_only=True, H_kv=8),
    # backward of a decode-shaped problem: 16 query rows against 128K keys, both settings; each
    # 128-key tile is its own CTA, so the key range is split across the whole grid
    "decode_bwd_q16_k128k": Workload("decode_bwd_q16_k128k", 4, 32, 16, 131072, 128, 0.3, False, seed=8),
    # one batch of it, small enough for a full ncu capture (2 GiB of keys)
    "decode_bwd_q16_k128k_b1": Workload("decode_bwd_q16_k128k_b1", 1, 32, 16, 131072, 128, 0.3, False, seed=8),
    # one batch of the 128K decode: small enough for a full ncu capture (2 GiB of keys)
    "decode_q1_k128k_b1": Workload("decode_q1_k128k_b1", 1, 32, 1, 131072, 128, 0.3, False, seed=3,
                                   fwd_only=True),
    # head dimension 64 (the tiny case's d) at 8K and 64K context
    "8k_causal_d64": Workload("8k_causal_d64", 1, 32, 8192, 8192, 64, 0.3, True, seed=6),
    "64k_causal_d64": Workload("64k_causal_d64", 1, 32, 65536, 65536, 64, 0.3, True, seed=6),
    "512k_causal": Workload("512k_causal", 1, 8, 524288, 524288, 128, 0.3, True, teacher_scale=1.5, seed=4),
    # 4 heads of the 64K causal workload (same seed and per-head shape; 0.5 GiB of inputs, more
    # than L2): a DRAM-counter capture of it, times 8, gives the 32-head figure
    "64k_causal_h4": Workload("64k_causal_h4", 1, 4, 65536, 65536, 128, 0.3, True, seed=2),
    # 64K causal with keys shared by groups of 4 query heads (32 query heads, 8 key heads)
    "64k_causal_gqa": Workload("64k_causal_gqa", 1, 32, 65536, 65536, 128, 0.3, True, seed=9, H_kv=8),
}


def make_qk(B, H, Nq, Nk, d, sigma, teacher_scale=1.0, seed=0, device="cpu", H_kv=0):
    """(Q1, K1, Q2, K2) as contiguous bf16 [B, H, N, d] tensors on ``device``
    (K1, K2 with H_kv heads when H_kv is given)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    hk = H_kv or H

    def draw(heads, n):
        return torch.randn((B, heads, n, d), generator=gen, device=device, dtype=torch.float32)

    Q1 = draw(H, Nq)
    K1 = draw(hk, Nk)
    if teacher_scale != 1.0:
        Q1.mul_(teacher_scale)
        K1.mul_(teacher_scale)
    Q2 = draw(H, Nq).mul_(sigma).add_(Q1)
    K2 = draw(hk, Nk).mul_(sigma).add_(K1)
    return tuple(t.to(torch.bfloat16).contiguous() for t in (Q1, K1, Q2, K2))


def make_workload(w: Workload, device="cpu"):
    return make_qk(w.B, w.H, w.Nq, w.Nk, w.d, w.sigma, w.teacher_scale, w.seed, device, H_kv=w.H_kv)


def make_g(B, H, Nq, value, device="cpu"):
    """Upstream gradient dL/dKL per row: a constant fill, float32 [B, H, Nq]."""
    return torch.full((B, H, Nq), float(value), dtype=torch.float32, device=device)
