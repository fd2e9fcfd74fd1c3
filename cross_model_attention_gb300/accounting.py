"""Algorithmic work of the hot path (bytes, flops, exp2 count) for the
bench and the profiling case: the roofline denominators' numerators."""
from __future__ import annotations

import numpy as np


def qk_flops(w) -> float:
    """Q.K^T flops of one causal pass over one sender layer."""
    return float(sum(2.0 * w.d * w.sender_heads * L * (L + 1) / 2 for L in w.seqlens))


def retrieval_bytes(w, rcv, nnz: int) -> float:
    """Algorithmic HBM bytes of one retrieval launch (one reuse layer)."""
    R = sum((L + w.B - 1) // w.B for L in w.seqlens)
    return float(nnz * 2 * w.B * w.B + 4 * nnz + 4 * (w.sender_heads * R + 1)
                 + 4 * rcv.heads * w.sender_heads + 2 * w.T * rcv.kv_heads * w.d
                 + 2 * w.T * rcv.heads * w.d)


def pack_bytes(w, nnz: int) -> float:
    """Algorithmic HBM bytes of one pack launch: Q and K read once, kept tiles
    and col_idx written."""
    return float(2 * w.T * (w.sender_heads + w.sender_kv_heads) * w.d + nnz * 2 * w.B * w.B
                 + 4 * nnz)


def union_blocks(row_ptr: np.ndarray, col_idx: np.ndarray, H_s: int, R: int) -> int:
    """Sum over block-rows of the number of block columns kept by at least one
    sender head (the blocks the retrieval multiplies by V)."""
    rows = np.repeat(np.arange(H_s * R), np.diff(row_ptr))
    if rows.size == 0:
        return 0
    mark = np.zeros((R, int(col_idx.max()) + 1), dtype=bool)
    mark[rows % R, col_idx] = True
    return int(mark.sum())


def candidate_blocks(w) -> int:
    """Candidate blocks of one head: causal block-rows bi keep bj = 0..bi."""
    return sum((L + w.B - 1) // w.B * ((L + w.B - 1) // w.B + 1) // 2 for L in w.seqlens)
