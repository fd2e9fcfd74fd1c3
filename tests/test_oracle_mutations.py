"""Planted mistakes in the oracle (on the CPU) must be caught by the pins.

Each test swaps one oracle function for a subtly wrong copy and checks that a
pin from tests/test_oracle_pins.py now fails.  This is how we know the pins
would notice a dropped term, a wrong sign or index, or a transposed operand.
"""
import math

import numpy as np
import pytest

from oracle import mapflow_oracle as orc
from tests import test_oracle_pins as pins


def _attention_rows_factory(scale_fn=None, causal_strict=False, sign=1.0):
    def attention_rows(q_rows, k_seq, row_pos, causal):
        d = q_rows.shape[1]
        L = k_seq.shape[0]
        S = sign * (q_rows @ k_seq.T) / (scale_fn(d) if scale_fn else math.sqrt(d))
        if causal:
            if causal_strict:
                allowed = np.arange(L)[None, :] < row_pos[:, None]
                allowed[:, 0] = True
            else:
                allowed = np.arange(L)[None, :] <= row_pos[:, None]
        else:
            allowed = np.ones((len(row_pos), L), dtype=bool)
        S = np.where(allowed, S, -np.inf)
        m = S.max(axis=1)
        E = np.exp(S - m[:, None])
        l = E.sum(axis=1)
        return E / l[:, None], m, l
    return attention_rows


@pytest.mark.parametrize("mut", [
    dict(scale_fn=lambda d: 1.0),            # dropped 1/sqrt(d)
    dict(scale_fn=lambda d: float(d)),       # 1/d instead of 1/sqrt(d)
    dict(causal_strict=True),                # mask excludes the diagonal
    dict(sign=-1.0),                         # sign flip of the logits
])
def test_sdpa_pin_catches_softmax_mistakes(monkeypatch, mut):
    monkeypatch.setattr(orc, "attention_rows", _attention_rows_factory(**mut))
    assert pins.check_sdpa_closed_form(o=orc) > 1e-3


def test_onehot_pin_catches_transposed_head_map(monkeypatch):
    real = orc.retrieve_rows

    def transposed(P, W, v, H_kv):
        # plausible mistake: contract W over its first index
        Wt = np.zeros_like(W)
        n = min(W.shape)
        Wt[:n, :n] = W[:n, :n].T
        return real(P, Wt, v, H_kv)
    monkeypatch.setattr(orc, "retrieve_rows", transposed)
    assert pins.check_onehot_head_map(o=orc) > 1e-3


def test_onehot_pin_catches_wrong_gqa_grouping(monkeypatch):
    def wrong_group(P_kept_rows, W, v_seq, H_kv):
        Hs, n, L = P_kept_rows.shape
        Hr = W.shape[0]
        A_hat = np.tensordot(W, P_kept_rows, axes=([1], [0]))
        out = np.zeros((n, Hr, v_seq.shape[2]))
        for i in range(Hr):
            out[:, i, :] = A_hat[i] @ v_seq[:, i % H_kv, :]  # interleaved, not contiguous
        return out
    monkeypatch.setattr(orc, "retrieve_rows", wrong_group)
    assert pins.check_onehot_head_map(o=orc) > 1e-3


def test_no_renorm_pin_catches_renormalisation(monkeypatch):
    real = orc.kept_mask_rows

    def renorm_mask(grid, kept, bi, s, n_rows):
        mk = real(grid, kept, bi, s, n_rows)
        return mk * 1.05  # e.g. dividing by the kept fraction
    monkeypatch.setattr(orc, "kept_mask_rows", renorm_mask)
    assert pins.check_no_renormalisation(o=orc) > 1e-3


def _select_factory(tie_high=False, strict=False, frac_bits=20):
    def select_topp(mass, p):
        mass = np.asarray(mass, dtype=np.float64)
        n = len(mass)
        key = (lambda b: (-mass[b], -b)) if tie_high else (lambda b: (-mass[b], b))
        order = sorted(range(n), key=key)
        q = [int(np.rint(mass[b] * 2.0 ** 32)) for b in range(n)]
        tot = sum(q)
        pq = int(np.rint(p * 2 ** frac_bits))
        acc, k = 0, 0
        while k < n and ((acc << frac_bits) <= pq * tot if strict else (acc << frac_bits) < pq * tot):
            acc += q[order[k]]
            k += 1
        return sorted(order[:k])
    return select_topp


@pytest.mark.parametrize("mut", [dict(tie_high=True), dict(strict=True)])
def test_bruteforce_pin_catches_selection_mistakes(mut):
    bad = _select_factory(**mut)
    caught = False
    for seed in range(40):
        rng = np.random.default_rng(seed)
        n = int(rng.integers(2, 9))
        mass = rng.random(n)
        mass[1] = mass[0]
        mass[-1] = mass[0]
        mass = mass.astype(np.float32).astype(np.float64)
        for p in (0.5, 0.8, 0.95, 1.0):
            kept = bad(mass, p)
            size, subsets = pins.selection_bruteforce(mass, p)
            dropped = [b for b in range(n) if b not in kept]
            ok = len(kept) == size and tuple(kept) in subsets and all(
                mass[a] > mass[b] or (mass[a] == mass[b] and a < b)
                for a in kept for b in dropped)
            caught |= not ok
    assert caught


def test_mass_pin_catches_block_offset(monkeypatch):
    """Summing the wrong column range (off by one block edge) is caught by the
    uniform-attention closed form."""
    def off_by_one(P_rows, B, n_cand):
        L = P_rows.shape[1]
        out = np.zeros(n_cand)
        for bj in range(n_cand):
            out[bj] = P_rows[:, bj * B:min(L, (bj + 1) * B + 1)].sum()
        return out
    monkeypatch.setattr(orc, "block_masses", off_by_one)
    with pytest.raises(AssertionError):
        pins.test_uniform_causal_closed_form(64, 8)


# ------------------------------------------------------- head-map calibration
def _calibrate_factory(mode):
    def calibrate_head_map(sender, receiver, ridge=0.0):
        S = np.asarray(sender, np.float64)
        R = np.asarray(receiver, np.float64)
        G = S @ S.T
        if mode == "ridge_dropped":
            pass
        elif mode == "ridge_everywhere":
            G = G + ridge  # added to every entry instead of the diagonal
        else:
            G = G + ridge * np.eye(S.shape[0])
        if mode == "receiver_gram":
            return np.linalg.solve(G, S @ R.T).T @ (R @ R.T) / max(np.trace(R @ R.T), 1.0)
        return np.linalg.solve(G, S @ R.T).T
    return calibrate_head_map


@pytest.mark.parametrize("mode,pin", [
    ("ridge_dropped", pins.test_calibration_is_the_least_squares_solution),
    ("ridge_everywhere", pins.test_calibration_is_the_least_squares_solution),
    ("receiver_gram", pins.test_calibration_recovers_a_planted_map_exactly),
])
def test_calibration_pins_catch_mistakes(monkeypatch, mode, pin):
    monkeypatch.setattr(orc, "calibrate_head_map", _calibrate_factory(mode))
    with pytest.raises((AssertionError, ValueError)):
        pin()


def test_map_entries_pin_catches_an_off_by_one_block_mask(monkeypatch):
    def shifted_mask(grid, kept, bi, s, n_rows):
        # plausible mistake: kept block bj marks the columns of block bj + 1
        L = int(grid.lens[s])
        mk = np.zeros((n_rows, L))
        for bj in kept:
            mk[:, min(L, (bj + 1) * grid.B):min(L, (bj + 2) * grid.B)] = 1.0
        return mk
    monkeypatch.setattr(orc, "kept_mask_rows", shifted_mask)
    with pytest.raises(AssertionError):
        pins.test_map_entries_masks_dropped_blocks_and_rows_sum_to_one()


# ------------------------------------------- full-size per-block-row helpers

def _shifted_span(grid, rb):
    """Row range of a block-row shifted down by one row (a plausible slip in
    the offset arithmetic), clipped to the sequence."""
    s, bi = int(grid.rb_seq[rb]), int(grid.rb_local[rb])
    a, L = int(grid.cu[s]), int(grid.lens[s])
    r0, r1 = min(L - 1, bi * grid.B + 1), min(L, (bi + 1) * grid.B + 1)
    return s, bi, a, L, r0, r1


def test_helper_pin_catches_an_off_by_one_row_slice_in_block_row_reference(monkeypatch):
    def shifted(q64, k64, grid, h, rb):
        Hs, Hks = q64.shape[1], k64.shape[1]
        s, bi, a, L, r0, r1 = _shifted_span(grid, rb)
        P, m, l = orc.attention_rows(q64[a + r0:a + r1, h], k64[a:a + L, h // (Hs // Hks)],
                                     np.arange(r0, r1), grid.causal)
        return {"P": P, "m": m, "l": l, "mass": orc.block_masses(P, grid.B, int(grid.ncand[rb])),
                "rows": np.arange(a + r0, a + r1)}
    monkeypatch.setattr(orc, "block_row_reference", shifted)
    assert pins.check_block_row_helpers(o=orc) > 1e-3


def test_helper_pin_catches_an_off_by_one_row_slice_in_retrieve_block_row(monkeypatch):
    def shifted(q64, k64, grid, kept_of, W, v64, H_kv, rb):
        Hs, Hks = q64.shape[1], k64.shape[1]
        s, bi, a, L, r0, r1 = _shifted_span(grid, rb)
        Pk = np.zeros((Hs, r1 - r0, L))
        for h in range(Hs):
            P, _, _ = orc.attention_rows(q64[a + r0:a + r1, h], k64[a:a + L, h // (Hs // Hks)],
                                         np.arange(r0, r1), grid.causal)
            Pk[h] = P * orc.kept_mask_rows(grid, kept_of(h, rb), bi, s, r1 - r0)
        # the rows reported are the block-row's own, the values are not
        return orc.retrieve_rows(Pk, W, v64[a:a + L], H_kv), np.arange(a + bi * grid.B,
                                                                        a + bi * grid.B + r1 - r0)
    monkeypatch.setattr(orc, "retrieve_block_row", shifted)
    assert pins.check_block_row_helpers(o=orc) > 1e-3


def test_helper_pin_catches_a_wrong_gqa_head_in_block_row_reference(monkeypatch):
    real = orc.block_row_reference

    def wrong_kv(q64, k64, grid, h, rb):
        # a wrong sender KV index: the KV heads taken in reverse order
        return real(q64, k64[:, ::-1], grid, h, rb)
    monkeypatch.setattr(orc, "block_row_reference", wrong_kv)
    assert pins.check_block_row_helpers(o=orc) > 1e-3
