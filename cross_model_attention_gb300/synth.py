"""Seeded synthetic inputs shared by the GPU path's tests/bench and the oracle.

This module only draws random numbers and lays out the structured logit
biases of the workloads inside Q and K; it computes no step of the method
(no softmax, no block statistics, no selection, no head mixing).

Recipe (the pages give the biases as logit offsets but the method has no bias
input, so they are realised inside Q and K, in dimensions that carry no noise):

* noise dims: Q, K ~ N(0, 1) * 1.5 (standard deviation 1.5);
* sink: one dim with Q = 1 and K_j = 4*sqrt(d) for the first four keys of each
  sequence, so q.k/sqrt(d) gains exactly +4.0 on those keys;
* local band: R = 16 rotary pairs with frequencies w_r ~ U(0, pi/32); Q gets
  c*(cos w_r i, sin w_r i), K gets c*sqrt(d)*(cos w_r j, sin w_r j) with
  c^2 = 2/R, so the logit gains (2/R) * sum_r cos(w_r (i-j)): +2.0 at i = j,
  on average 2*sinc((i-j)/32), first zero at |i-j| = 32 (a rank-32 stand-in
  for a +2.0 box on |i-j| < 32, which no low-rank Q/K can realise exactly);
* retrieval blocks (when asked): one dim with Q = 1 and K_j = 3*sqrt(d) on the
  keys of n random key blocks per KV head (block indices >= 1, no
  replacement), i.e. an exact +3.0;
* temperature (when asked): tau_h ~ U(lo, hi) per sender q-head, applied last
  as Q_h <- Q_h / tau_h.

All positions are relative to the start of each packed sequence.  Values are
rounded once to the workload dtype (bf16 round-to-nearest-even, or fp32) and
the same arrays feed both the GPU path and the oracle.
"""
from __future__ import annotations

import math
import zlib
from typing import Dict, Optional, Tuple

import numpy as np

from .workloads import Receiver, Workload

BAND_PAIRS = 16
SINK_KEYS = 4


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    # finite inputs only: b + 0x8000 never wraps a 32-bit word
    r = (b >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += b
    r >>= 16
    return r.astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rng(w: Workload, *key: int) -> np.random.Generator:
    return np.random.default_rng([w.seed] + [int(k) for k in key])


def _name_key(name: str) -> int:
    # deterministic across processes (unlike hash())
    return zlib.crc32(name.encode()) % 100003


def _structure_dims(w: Workload) -> int:
    return 1 + 2 * BAND_PAIRS + (1 if w.retrieval_blocks else 0)


def sender_qk_f32(w: Workload, layer: int) -> Tuple[np.ndarray, np.ndarray]:
    """Unrounded fp32 Q [T, H_s, d] and K [T, H_ks, d] of sender layer (1-based)."""
    d, T = w.d, w.T
    Hs, Hks = w.sender_heads, w.sender_kv_heads
    ns = _structure_dims(w)
    if d < ns + 1:
        raise ValueError("head dim too small for the structure dims")
    rng = _rng(w, 11, layer)
    q = np.zeros((T, Hs, d), np.float32)
    k = np.zeros((T, Hks, d), np.float32)
    q[:, :, ns:] = rng.standard_normal((T, Hs, d - ns), dtype=np.float32) * 1.5
    k[:, :, ns:] = rng.standard_normal((T, Hks, d - ns), dtype=np.float32) * 1.5
    sd = math.sqrt(d)
    omega = rng.uniform(0.0, math.pi / 32.0, size=BAND_PAIRS)
    c = math.sqrt(2.0 / BAND_PAIRS)
    cu = w.cu_seqlens
    for s in range(len(w.seqlens)):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        pos = np.arange(L, dtype=np.float64)
        # sink
        q[a:b, :, 0] = 1.0
        k[a:a + min(SINK_KEYS, L), :, 0] = 4.0 * sd
        # band (computed in fp64, rounded once)
        ang = pos[:, None] * omega[None, :]
        cs, sn = np.cos(ang), np.sin(ang)
        qb = np.empty((L, 2 * BAND_PAIRS))
        qb[:, 0::2], qb[:, 1::2] = c * cs, c * sn
        q[a:b, :, 1:1 + 2 * BAND_PAIRS] = qb[:, None, :].astype(np.float32)
        k[a:b, :, 1:1 + 2 * BAND_PAIRS] = (qb * sd)[:, None, :].astype(np.float32)
        if w.retrieval_blocks:
            col = 1 + 2 * BAND_PAIRS
            q[a:b, :, col] = 1.0
            nb = (L + w.B - 1) // w.B
            for hk in range(Hks):
                pick = rng.choice(np.arange(1, nb), size=min(w.retrieval_blocks, nb - 1),
                                  replace=False)
                for bj in pick:
                    k[a + bj * w.B:a + min(L, (bj + 1) * w.B), hk, col] = 3.0 * sd
    if w.temperature is not None:
        lo, hi = w.temperature
        tau = rng.uniform(lo, hi, size=Hs).astype(np.float32)
        q /= tau[None, :, None]
    return q, k


def sender_qk(w: Workload, layer: int) -> Dict[str, np.ndarray]:
    """Rounded sender Q/K: 'q','k' as stored (uint16 bf16 bits or fp32) plus
    'q64','k64' (the same values widened exactly to fp64)."""
    q, k = sender_qk_f32(w, layer)
    if w.dtype == "bf16":
        qb, kb = bf16_round(q), bf16_round(k)
        return {"q": qb, "k": kb, "q64": bf16_to_f64(qb), "k64": bf16_to_f64(kb)}
    return {"q": q, "k": k, "q64": q.astype(np.float64), "k64": k.astype(np.float64)}


def receiver_v(w: Workload, rcv: Receiver, layer: int) -> Dict[str, np.ndarray]:
    """Receiver V [T, H_kv, d] ~ N(0, 1) for receiver layer j (1-based)."""
    rng = _rng(w, 23, _name_key(rcv.name), layer)
    v = rng.standard_normal((w.T, rcv.kv_heads, w.d), dtype=np.float32)
    if w.dtype == "bf16":
        vb = bf16_round(v)
        return {"v": vb, "v64": bf16_to_f64(vb)}
    return {"v": v, "v64": v.astype(np.float64)}


def head_map_weights(w: Workload, rcv: Receiver, layer: int) -> np.ndarray:
    """W_j [H_r, H_s] in fp32: i.i.d. N(0, w_var) (plus I when asked)."""
    rng = _rng(w, 37, _name_key(rcv.name), layer)
    W = rng.standard_normal((rcv.heads, w.sender_heads)) * math.sqrt(rcv.w_var)
    if rcv.w_identity:
        if rcv.heads != w.sender_heads:
            raise ValueError("identity head map needs H_r == H_s")
        W = W + np.eye(rcv.heads)
    return W.astype(np.float32)


def random_qk(T: int, Hs: int, Hks: int, d: int, seed: int, scale: float = 1.5,
              dtype: str = "bf16") -> Dict[str, np.ndarray]:
    """Unstructured Q/K (plain N(0,1)*scale) for edge-case tests."""
    rng = np.random.default_rng([seed, 91])
    q = rng.standard_normal((T, Hs, d), dtype=np.float32) * scale
    k = rng.standard_normal((T, Hks, d), dtype=np.float32) * scale
    if dtype == "bf16":
        qb, kb = bf16_round(q), bf16_round(k)
        return {"q": qb, "k": kb, "q64": bf16_to_f64(qb), "k64": bf16_to_f64(kb)}
    return {"q": q, "k": k, "q64": q.astype(np.float64), "k64": k.astype(np.float64)}


def random_v(T: int, Hkv: int, d: int, seed: int, dtype: str = "bf16") -> Dict[str, np.ndarray]:
    rng = np.random.default_rng([seed, 92])
    v = rng.standard_normal((T, Hkv, d), dtype=np.float32)
    if dtype == "bf16":
        vb = bf16_round(v)
        return {"v": vb, "v64": bf16_to_f64(vb)}
    return {"v": v, "v64": v.astype(np.float64)}


def random_w(Hr: int, Hs: int, seed: int, var: Optional[float] = None) -> np.ndarray:
    rng = np.random.default_rng([seed, 93])
    var = (1.0 / Hs) if var is None else var
    return (rng.standard_normal((Hr, Hs)) * math.sqrt(var)).astype(np.float32)


# --------------------------------------------------- device-side drawing ----
# Full-size benchmark inputs (tens of GB over all layers) would take the host
# minutes to draw and to hold; these functions draw the same recipe on a CUDA
# device with torch's generator.  The random numbers differ from the numpy
# draw above (the distribution and the structure are the same), so parity
# tests, which compare with the oracle, use the numpy functions.

def _torch_seed(*key: int) -> int:
    return int(np.random.SeedSequence([int(x) for x in key]).generate_state(1, np.uint64)[0] >> 1)


def sender_qk_device(w: Workload, layer: int, device):
    """Sender Q [T, H_s, d] and K [T, H_ks, d] of sender layer `layer`
    (1-based), drawn on `device` by the recipe of sender_qk_f32 and rounded
    once to the workload dtype (torch's fp32 -> bf16 conversion rounds to
    nearest even)."""
    import torch
    d, T = w.d, w.T
    Hs, Hks = w.sender_heads, w.sender_kv_heads
    ns = _structure_dims(w)
    if d < ns + 1:
        raise ValueError("head dim too small for the structure dims")
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(w.seed, 11, layer))
    rng = _rng(w, 11, layer, 1)  # the small per-layer draws (frequencies, blocks, tau)
    q = torch.zeros((T, Hs, d), dtype=torch.float32, device=device)
    k = torch.zeros((T, Hks, d), dtype=torch.float32, device=device)
    q[:, :, ns:] = torch.randn((T, Hs, d - ns), generator=g, device=device) * 1.5
    k[:, :, ns:] = torch.randn((T, Hks, d - ns), generator=g, device=device) * 1.5
    sd = math.sqrt(d)
    omega = torch.from_numpy(rng.uniform(0.0, math.pi / 32.0, size=BAND_PAIRS)).to(device)
    c = math.sqrt(2.0 / BAND_PAIRS)
    cu = w.cu_seqlens
    pos = torch.cat([torch.arange(int(cu[s + 1] - cu[s]), dtype=torch.float64, device=device)
                     for s in range(len(w.seqlens))])
    ang = pos[:, None] * omega[None, :]
    qb = torch.empty((T, 2 * BAND_PAIRS), dtype=torch.float64, device=device)
    qb[:, 0::2], qb[:, 1::2] = c * torch.cos(ang), c * torch.sin(ang)
    q[:, :, 1:1 + 2 * BAND_PAIRS] = qb[:, None, :].float()
    k[:, :, 1:1 + 2 * BAND_PAIRS] = (qb * sd)[:, None, :].float()
    q[:, :, 0] = 1.0
    for s in range(len(w.seqlens)):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        k[a:a + min(SINK_KEYS, L), :, 0] = 4.0 * sd
        if w.retrieval_blocks:
            col = 1 + 2 * BAND_PAIRS
            nb = (L + w.B - 1) // w.B
            for hk in range(Hks):
                pick = rng.choice(np.arange(1, nb), size=min(w.retrieval_blocks, nb - 1),
                                  replace=False)
                for bj in pick:
                    k[a + bj * w.B:a + min(L, (bj + 1) * w.B), hk, col] = 3.0 * sd
    if w.retrieval_blocks:
        q[:, :, 1 + 2 * BAND_PAIRS] = 1.0
    if w.temperature is not None:
        lo, hi = w.temperature
        tau = torch.from_numpy(rng.uniform(lo, hi, size=Hs).astype(np.float32)).to(device)
        q /= tau[None, :, None]
    if w.dtype == "bf16":
        return q.to(torch.bfloat16), k.to(torch.bfloat16)
    return q, k


def receiver_v_device(w: Workload, rcv: Receiver, layer: int, device):
    """Receiver V [T, H_kv, d] ~ N(0, 1) of receiver layer j (1-based), drawn
    on `device`, rounded once to the workload dtype."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(w.seed, 23, _name_key(rcv.name), layer))
    v = torch.randn((w.T, rcv.kv_heads, w.d), generator=g, device=device)
    return v.to(torch.bfloat16) if w.dtype == "bf16" else v
