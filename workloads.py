"""Seeded synthetic workloads for the SDPA backward.

This module holds shapes, mask settings and random draws only: none of the
attention arithmetic. Both the fp64 oracle side (tests, CPU baseline) and the
GPU side (tests, benchmark) read the same tensors from here.

Recipe (the same for every workload):
  g = torch.Generator("cpu").manual_seed(seed)
  if the workload is padded: lens = randint(lo, hi + 1, (B,)) (seq_q_lens = seq_kv_lens)
  Q, K, V, dO = randn(shape, float32, generator=g) in that order, rounded to bf16 (RNE).
O and LSE are not drawn: they come from the oracle forward on these inputs
(O rounded to bf16, LSE kept in fp32).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    Dqk: int
    Dv: int
    causal: bool = False
    bottom_right: bool = False
    window_left: int = -1
    window_right: int = -1
    deterministic: bool = False
    padded: Optional[Tuple[int, int]] = None  # inclusive length range when padded
    seed: int = 0
    scale: Optional[float] = None  # None -> 1/sqrt(Dqk)

    @property
    def resolved_scale(self) -> float:
        return 1.0 / math.sqrt(self.Dqk) if self.scale is None else float(self.scale)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the benchmark and parity tests use.
WORKLOADS: Dict[str, Workload] = {
    "tiny_dense": Workload("tiny_dense", B=1, Hq=2, Hkv=2, Sq=128, Skv=128, Dqk=64, Dv=64,
                           seed=0),
    "causal_mha": Workload("causal_mha", B=2, Hq=16, Hkv=16, Sq=2048, Skv=2048, Dqk=128,
                           Dv=128, causal=True, seed=1),
    "causal_gqa_det": Workload("causal_gqa_det", B=1, Hq=32, Hkv=8, Sq=4096, Skv=4096,
                               Dqk=128, Dv=128, causal=True, deterministic=True, seed=2),
    "swa_causal_padded": Workload("swa_causal_padded", B=4, Hq=16, Hkv=16, Sq=4096, Skv=4096,
                                  Dqk=128, Dv=128, causal=True, window_left=1024,
                                  padded=(512, 4096), seed=3),
    "mla_br_causal": Workload("mla_br_causal", B=1, Hq=16, Hkv=16, Sq=4096, Skv=4096, Dqk=192,
                              Dv=128, causal=True, bottom_right=True, seed=4),
    # The NVFP4 QAT backward page's example shape (BHSD (1, 16, 4096, 128),
    # non-causal), for the QAT path; not one of the five above.
    "qat_dense": Workload("qat_dense", B=1, Hq=16, Hkv=16, Sq=4096, Skv=4096, Dqk=128, Dv=128,
                          seed=5),
    # Head dim 256 (listed among the pages' head sizes), a causal shape of the
    # same visible-pair count as the S = 4096 workloads above; not one of the five.
    "d256_causal": Workload("d256_causal", B=1, Hq=16, Hkv=16, Sq=4096, Skv=4096, Dqk=256, Dv=256,
                            causal=True, seed=6),
}

ORDER = ["tiny_dense", "causal_mha", "causal_gqa_det", "swa_causal_padded", "mla_br_causal"]


def generate(w: Workload, dtype=torch.bfloat16) -> Dict[str, Optional[torch.Tensor]]:
    """Seeded CPU tensors: q, k, v, do (bf16, or ``dtype``: the same fp32 draws
    rounded to fp16 for fp16 io) and seq_q_lens/seq_kv_lens (int32 or None)."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    lens = None
    if w.padded is not None:
        lo, hi = w.padded
        lens = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)

    def draw(*shape):
        return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)

    q = draw(w.B, w.Hq, w.Sq, w.Dqk)
    k = draw(w.B, w.Hkv, w.Skv, w.Dqk)
    v = draw(w.B, w.Hkv, w.Skv, w.Dv)
    do = draw(w.B, w.Hq, w.Sq, w.Dv)
    return {"q": q, "k": k, "v": v, "do": do,
            "seq_q_lens": lens, "seq_kv_lens": None if lens is None else lens.clone()}


def bias_tensor(w: Workload, batch: int, dtype=torch.bfloat16) -> torch.Tensor:
    """Seeded additive bias (batch, Hq, Sq, Skv), batch 1 or B, N(0, 1) rounded to
    ``dtype``, from a stream of its own."""
    if batch not in (1, w.B):
        raise ValueError("the bias batch is 1 or B")
    g = torch.Generator("cpu").manual_seed(w.seed + 2_000_003)
    return torch.randn(batch, w.Hq, w.Sq, w.Skv, generator=g, dtype=torch.float32).to(dtype)


def sink_logits(w: Workload) -> torch.Tensor:
    """Seeded fp32 (Hq,) sink-token logits, N(0, 1), from a stream of their own."""
    g = torch.Generator("cpu").manual_seed(w.seed + 1_000_003)
    return torch.randn(w.Hq, generator=g, dtype=torch.float32)
