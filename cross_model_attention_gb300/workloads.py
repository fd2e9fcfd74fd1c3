"""The five synthetic sender/receiver workloads, described by shape only.

Each workload names the sender model shape (layers, q-heads, KV heads), the
receiver model shapes (layers, q-heads, KV heads, recomputed prefix r), the
head dimension, block size B, top-p threshold(s), sequence lengths and seed.
Nothing here computes any part of the method; the seeded tensors themselves
come from :mod:`cross_model_attention_gb300.synth`.

Layer mapping follows the partial-recomputation design of "Accelerating
Cross-Model LLM Inference via Attention Map Reuse" (section "MapFlow System
Design", items 1 and 2): receiver layers 1..r run normally and each later
layer j reuses sender layer m(j).  The pages do not give m(j); the plainest
depth-proportional reading m(j) = round(j * L_s / L_r) is used (1-based on
both sides).  No workload here hits a .5 tie.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Receiver:
    name: str
    layers: int          # L_r
    heads: int           # H_r
    kv_heads: int        # H_kv
    recompute: int       # r: layers 1..r are recomputed, r+1..L_r reuse maps
    w_var: float         # variance of the i.i.d. normal head-mapping weights
    w_identity: bool = False  # add the identity (H_r == H_s only)

    def layer_map(self, sender_layers: int) -> List[Tuple[int, int]]:
        """[(receiver layer j, sender layer m(j))] for j = r+1..L_r, 1-based."""
        out = []
        for j in range(self.recompute + 1, self.layers + 1):
            x = j * sender_layers / self.layers
            m = int(np.floor(x + 0.5))
            if abs(x - np.floor(x) - 0.5) < 1e-12:
                raise ValueError("layer map hits a .5 tie; state a tie rule first")
            out.append((j, max(1, min(sender_layers, m))))
        return out


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    seed: int
    sender_layers: int   # L_s
    sender_heads: int    # H_s
    sender_kv_heads: int  # H_ks
    d: int
    B: int
    p: Tuple[float, ...]
    seqlens: Tuple[int, ...]
    receivers: Tuple[Receiver, ...]
    dtype: str           # "f32" or "bf16"
    retrieval_blocks: int = 0     # structured +3.0 key blocks per KV head
    temperature: Optional[Tuple[float, float]] = (0.8, 2.0)
    causal: bool = True

    @property
    def T(self) -> int:
        return int(sum(self.seqlens))

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens)]).astype(np.int32)

    def sender_layers_used(self) -> List[int]:
        used = set()
        for rcv in self.receivers:
            used.update(m for _, m in rcv.layer_map(self.sender_layers))
        return sorted(used)


def _varlen_lengths(seed: int) -> Tuple[int, ...]:
    # 16 sequences with lengths uniform on [1024, 8192] (inclusive).
    rng = np.random.default_rng([seed, 7001])
    return tuple(int(x) for x in rng.integers(1024, 8193, 16))


WORKLOADS: Tuple[Workload, ...] = (
    Workload(
        index=0, name="tiny-fp32-N512", seed=0, sender_layers=1, sender_heads=4,
        sender_kv_heads=4, d=64, B=64, p=(0.95,), seqlens=(512,),
        receivers=(Receiver("r0", layers=1, heads=4, kv_heads=4, recompute=0,
                            w_var=0.25, w_identity=True),),
        dtype="f32", temperature=None),
    Workload(
        index=1, name="40Lx40H-to-36Lx32q8kv-N4096", seed=1, sender_layers=40,
        sender_heads=40, sender_kv_heads=40, d=128, B=64, p=(0.95,),
        seqlens=(4096,),
        receivers=(Receiver("r36", layers=36, heads=32, kv_heads=8, recompute=4,
                            w_var=1.0 / 40),),
        dtype="bf16"),
    Workload(
        index=2, name="32Lx32q8kv-to-26Lx24q8kv-N16384", seed=2, sender_layers=32,
        sender_heads=32, sender_kv_heads=8, d=128, B=64, p=(0.90,),
        seqlens=(16384,),
        receivers=(Receiver("r26", layers=26, heads=24, kv_heads=8, recompute=3,
                            w_var=1.0 / 32),),
        dtype="bf16", retrieval_blocks=8),
    Workload(
        index=3, name="1Lx40H-to-32q8kv-N32768-B128", seed=3, sender_layers=1,
        sender_heads=40, sender_kv_heads=40, d=128, B=128,
        p=(0.80, 0.90, 0.95, 0.99), seqlens=(32768,),
        receivers=(Receiver("r1", layers=1, heads=32, kv_heads=8, recompute=0,
                            w_var=1.0 / 40),),
        dtype="bf16"),
    Workload(
        index=4, name="varlen16-40Lx40H-to-two-receivers", seed=4, sender_layers=40,
        sender_heads=40, sender_kv_heads=40, d=128, B=64, p=(0.95,),
        seqlens=_varlen_lengths(4),
        receivers=(Receiver("a36", layers=36, heads=32, kv_heads=8, recompute=4,
                            w_var=1.0 / 40),
                   Receiver("b26", layers=26, heads=24, kv_heads=8, recompute=3,
                            w_var=1.0 / 40)),
        dtype="bf16"),
)


def get(index: int) -> Workload:
    return WORKLOADS[index]


def scaled(w: Workload, seqlens: Sequence[int], **kw) -> Workload:
    """A copy of workload *w* with other sequence lengths (and overrides)."""
    return dataclasses.replace(w, seqlens=tuple(int(x) for x in seqlens), **kw)
