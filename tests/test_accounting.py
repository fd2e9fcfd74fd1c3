"""The bench's work accounting (no GPU): the union-of-kept-blocks count
against a brute-force set union, and the candidate and flop formulas against
direct counts."""
import numpy as np

from cross_model_attention_gb300 import accounting, workloads


def test_union_blocks_matches_set_union():
    rng = np.random.default_rng(3)
    H_s, R, nb = 5, 7, 9
    rows = []
    for h in range(H_s):
        for rb in range(R):
            k = int(rng.integers(0, nb + 1))
            rows.append(sorted(rng.choice(nb, size=k, replace=False).tolist()))
    row_ptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int64)
    col_idx = np.array([c for r in rows for c in r], dtype=np.int64)
    want = sum(len(set().union(*[rows[h * R + rb] for h in range(H_s)])) for rb in range(R))
    assert accounting.union_blocks(row_ptr, col_idx, H_s, R) == want


def test_union_blocks_empty():
    assert accounting.union_blocks(np.zeros(7, np.int64), np.zeros(0, np.int64), 2, 3) == 0


def test_candidate_blocks_and_qk_flops_count_directly():
    w = workloads.scaled(workloads.get(1), [200, 64, 1], sender_heads=3, sender_kv_heads=3)
    cand = 0
    flops = 0.0
    for L in w.seqlens:
        nb = -(-L // w.B)
        cand += sum(bi + 1 for bi in range(nb))
        flops += 2.0 * w.d * w.sender_heads * sum(i + 1 for i in range(L))
    assert accounting.candidate_blocks(w) == cand
    assert accounting.qk_flops(w) == flops
