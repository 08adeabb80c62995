"""Seeded synthetic workloads shared by the tests, ``bench.py`` and ``smoke()``.

This module holds input shapes and random draws only: no attention arithmetic.
Both the CUDA path and the CPU oracle consume the tensors made here.

Recipe (one per workload): a CPU ``torch.Generator`` seeded with
``1000 + index`` draws Q, K, V, dO in that order as fp32 standard normals of
shape ``[B, H, N, d]``; each is rounded once to bf16 (round to nearest even).
The GPU receives those bf16 tensors; the oracle receives the same values
upcast to float64, so parity measures kernel error, not input quantisation.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int          # seed = 1000 + index
    B: int
    H: int
    N: int
    d: int
    causal: bool
    backward: bool = True
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "N": self.N, "d": self.d,
                "causal": self.causal, "scale": "1/sqrt(d)", "backward": self.backward}


# The five workloads the method is measured and checked on.
TINY = Workload("tiny_b1_h2_n256_d64", 0, 1, 2, 256, 64, False, True,
                "fwd+bwd, no mask; small enough for a full oracle in seconds")
GPT2_MEDIUM = Workload("gpt2_medium_b64_h16_n1024_d64_causal", 1, 64, 16, 1024, 64, True, True,
                       "GPT-2 medium attention shape (blog.teqners.com opening benchmark), fwd+bwd")
LLAMA7B_LAYER = Workload("7b_layer_b1_h32_n4096_d128_causal", 2, 1, 32, 4096, 128, True, False,
                         "7B-layer attention shape, forward only")
LLAMA7B_LAYER_NC = Workload("7b_layer_b1_h32_n4096_d128", 2, 1, 32, 4096, 128, False, False,
                            "7B-layer attention shape, forward only, no mask")
LONG_SEQ = Workload("long_b1_h16_n16384_d128", 3, 1, 16, 16384, 128, False, True,
                    "long sequence, small batch: work is split along the sequence")


def sweep() -> list[Workload]:
    """B*N fixed at 16384 tokens, H = 16, N in 512..16384, d in {64, 128}, both masks."""
    out = []
    for d in (64, 128):
        for causal in (False, True):
            for n in (512, 1024, 2048, 4096, 8192, 16384):
                out.append(Workload(f"sweep_b{16384 // n}_h16_n{n}_d{d}{'_causal' if causal else ''}",
                                    4, 16384 // n, 16, n, d, causal, True))
    return out


ALL = [TINY, GPT2_MEDIUM, LLAMA7B_LAYER, LLAMA7B_LAYER_NC, LONG_SEQ]
BY_NAME = {w.name: w for w in ALL + sweep()}


def make_inputs(B, H, N, d, seed, stress=None):
    """Seeded bf16 Q, K, V, dO of shape [B, H, N, d] on the CPU.

    ``stress``: ``None`` for plain N(0, 1); ``"wide"`` multiplies Q by 8 so score
    rows span dozens of units (exercises running-max growth and rescaling);
    ``"spike"`` additionally plants one large key per query block; ``"sorted"``
    sorts keys so each row's maximum keeps growing along the sequence.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if stress in ("wide", "spike", "sorted"):
        q = q * 8.0
    if stress == "spike":
        idx = torch.randint(0, N, (B, H), generator=g)
        for b in range(B):
            for h in range(H):
                k[b, h, idx[b, h]] *= 6.0
    if stress == "sorted":
        k, _ = torch.sort(k, dim=2)
    return tuple(t.to(torch.bfloat16) for t in (q, k, v, do))


def make_fp8_inputs(B, H, N, d, seed, stress=None):
    """Seeded E4M3 codes for Q and K, their descale factors, and bf16 V, on the CPU.

    Q, K, V are drawn as in :func:`make_inputs` (same seed, same stress); Q and K
    are then stored per tensor as E4M3 codes: descale = max|x| / 448 (so the
    largest element lands on the largest finite code) and code = the
    round-to-nearest E4M3 of x / descale (PyTorch's float8_e4m3fn conversion),
    returned as uint8.  Both the CUDA path and the oracle consume these codes.
    """
    q, k, v, _ = make_inputs(B, H, N, d, seed, stress)
    out = []
    for t in (q, k):
        x = t.float()
        descale = max(float(x.abs().max()), 1e-30) / 448.0
        out.append(((x / descale).to(torch.float8_e4m3fn).view(torch.uint8), descale))
    (q8, q_descale), (k8, k_descale) = out
    return q8, k8, q_descale, k_descale, v


def replica_seed(w: Workload, rank: int = 0) -> int:
    """Seed of rank ``rank``'s batch: rank 0 draws the workload's own inputs,
    every other rank an independent batch of the same shape."""
    return w.seed + 100003 * rank


def workload_inputs(w: Workload, stress=None, rank: int = 0):
    return make_inputs(w.B, w.H, w.N, w.d, replica_seed(w, rank), stress)


# ------------------------------------------------------------- decoding ----
@dataclass(frozen=True)
class DecodeWorkload:
    """Nq new queries per head (the last Nq positions) against an Nk-long K/V cache."""
    name: str
    index: int          # seed = 2000 + index
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool = True
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def seed(self) -> int:
        return 2000 + self.index

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "Nq": self.Nq, "Nk": self.Nk, "d": self.d,
                "causal": self.causal, "scale": "1/sqrt(d)"}


# Decode steps on the shapes of the measured workloads: the long-sequence head
# shape with its whole 16384-key cache, and the GPT-2 medium batch with its
# 1024-key cache; one query per sequence, and eight (a speculative step).
DECODE_LONG = DecodeWorkload("decode_b1_h16_q1_k16384_d128", 0, 1, 16, 1, 16384, 128, True,
                             "long-sequence shape at decode time: one query against a 16384-key cache")
DECODE_GPT2 = DecodeWorkload("decode_b64_h16_q1_k1024_d64", 1, 64, 16, 1, 1024, 64, True,
                             "GPT-2 medium batch at decode time: one query per sequence, 1024-key cache")
DECODE_LONG_Q8 = DecodeWorkload("decode_b1_h16_q8_k16384_d128", 2, 1, 16, 8, 16384, 128, True,
                                "long-sequence shape, eight new queries (speculative step)")
DECODE_ALL = [DECODE_LONG, DECODE_GPT2, DECODE_LONG_Q8]
DECODE_BY_NAME = {w.name: w for w in DECODE_ALL}


def make_decode_inputs(B, H, Nq, Nk, d, seed, stress=None):
    """Seeded bf16 Q [B, H, Nq, d] and K, V [B, H, Nk, d] on the CPU (drawn in that order,
    fp32 standard normals rounded once to bf16; ``stress="wide"`` multiplies Q by 8)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    if stress == "wide":
        q = q * 8.0
    return tuple(t.to(torch.bfloat16) for t in (q, k, v))
