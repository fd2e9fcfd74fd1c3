"""Pins of the fp64 oracle against facts fixed by mathematics, by an
independent library routine, by brute force, or by hand-derived closed forms.

Each pin is written so that a plausible mistake in the oracle (a dropped
scale, a wrong mask, a transposed operand, a flipped tie rule, a
renormalisation) fails at least one test; tests/test_oracle_mutations.py
plants such mistakes and checks that the pins catch them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mapflow_oracle as orc
from cross_model_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers --

def rand_case(T_list, Hs, Hks, d, seed, scale=1.5):
    rng = np.random.default_rng(seed)
    T = sum(T_list)
    q = rng.standard_normal((T, Hs, d)) * scale
    k = rng.standard_normal((T, Hks, d)) * scale
    cu = np.concatenate([[0], np.cumsum(T_list)])
    return q, k, cu


def sdpa_reference(q, k, v, cu, causal=True):
    """torch scaled_dot_product_attention in fp64 per sequence (an
    independent library routine)."""
    T, H, d = q.shape
    out = np.zeros((T, H, v.shape[2]))
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        Q = torch.from_numpy(q[a:b]).permute(1, 0, 2)[None]
        K = torch.from_numpy(k[a:b]).permute(1, 0, 2)[None]
        V = torch.from_numpy(v[a:b]).permute(1, 0, 2)[None]
        O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=causal)
        out[a:b] = O[0].permute(1, 0, 2).numpy()
    return out


def check_sdpa_closed_form(o=orc, seed=0, T_list=(70, 33, 128), H=3, d=16, B=16,
                           causal=True):
    """p = 1, W = I, H_r = H_s = H_kv: the method reduces to plain softmax
    attention of the sender's Q, K with the receiver's V.  Returns max err."""
    q, k, cu = rand_case(T_list, H, H, d, seed)
    v = np.random.default_rng(seed + 1).standard_normal((sum(T_list), H, d))
    bsr = o.compress(q, k, cu, B, 1.0, causal)
    W = np.eye(H)
    O, done = o.retrieve(q, k, bsr, W, v, H)
    ref = sdpa_reference(q, k, v, cu, causal)
    assert done.all()
    return float(np.abs(O - ref).max())


# -------------------------------------------------------------------- pins --

def test_rows_sum_to_one_and_block_row_totals():
    q, k, cu = rand_case((100, 64, 7), 2, 1, 32, 3, scale=2.0)
    g = orc.BlockGrid(cu, 16, True)
    for h in range(2):
        for rb in range(g.R):
            ref = orc.block_row_reference(q, k, g, h, rb)
            assert np.allclose(ref["P"].sum(1), 1.0, atol=1e-12, rtol=0)
            # each valid row contributes exactly 1 to its block-row's masses
            assert abs(ref["mass"].sum() - len(ref["rows"])) < 1e-11


def test_python_loop_bruteforce_tiny():
    """Everything re-derived with scalar Python loops (math.exp, math.fsum)
    for N <= 64: logits, causal softmax, row statistics, block masses."""
    rng = np.random.default_rng(11)
    L, d, B = 37, 5, 8
    q = rng.standard_normal((L, 1, d)) * 2
    k = rng.standard_normal((L, 1, d)) * 2
    bsr = orc.compress(q, k, [0, L], B, 0.9, True)
    nb = (L + B - 1) // B
    for i in range(L):
        s = [math.fsum(q[i, 0, t] * k[j, 0, t] for t in range(d)) / math.sqrt(d)
             for j in range(i + 1)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        l = math.fsum(e)
        assert abs(bsr.m[0, i] - m) < 1e-12
        assert abs(bsr.l[0, i] - l) < 1e-12 * l
    g = bsr.grid
    for bi in range(nb):
        for bj in range(bi + 1):
            tot = []
            for i in range(bi * B, min(L, (bi + 1) * B)):
                s = [math.fsum(q[i, 0, t] * k[j, 0, t] for t in range(d)) / math.sqrt(d)
                     for j in range(i + 1)]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                l = math.fsum(e)
                tot.extend(e[j] / l for j in range(bj * B, min(i + 1, (bj + 1) * B)))
            assert abs(bsr.mass[0, g.cand_ptr[bi] + bj] - math.fsum(tot)) < 1e-12


def test_golden_uniform_causal():
    fx = json.load(open(os.path.join(GOLDEN, "uniform_causal_N4_B2.json")))
    N, B, d = fx["N"], fx["B"], fx["d"]
    q = np.zeros((N, 1, d))
    k = np.random.default_rng(0).standard_normal((N, 1, d))
    for pstr, kept in fx["kept"].items():
        bsr = orc.compress(q, k, [0, N], B, float(pstr), True)
        g = bsr.grid
        for rb in range(g.R):
            want = [a / b for a, b in fx["masses"][rb]]
            got = bsr.mass[0, g.cand_ptr[rb]:g.cand_ptr[rb + 1]]
            assert np.allclose(got, want, atol=1e-15, rtol=0)
            assert bsr.kept(0, rb) == kept[rb]
    assert np.allclose(bsr.m[0], fx["row_max"]) and np.allclose(bsr.l[0], fx["row_sum"])


@pytest.mark.parametrize("N,B", [(64, 8), (50, 16), (128, 32)])
def test_uniform_causal_closed_form(N, B):
    """q = 0: P[i][j] = 1/(i+1); masses are exact harmonic-type sums."""
    q = np.zeros((N, 1, 4))
    k = np.random.default_rng(1).standard_normal((N, 1, 4))
    bsr = orc.compress(q, k, [0, N], B, 0.95, True)
    g = bsr.grid
    for rb in range(g.R):
        for bj in range(int(g.ncand[rb])):
            exact = sum(Fraction(len([j for j in range(bj * B, min(N, (bj + 1) * B)) if j <= i]),
                                 i + 1) for i in range(rb * B, min(N, (rb + 1) * B)))
            assert abs(bsr.mass[0, g.cand_ptr[rb] + bj] - float(exact)) < 1e-12


def test_uniform_noncausal_closed_form():
    N, B = 96, 32
    q = np.zeros((N, 1, 4))
    k = np.ones((N, 1, 4))
    bsr = orc.compress(q, k, [0, N], B, 0.5, causal=False)
    assert np.allclose(bsr.mass, B * B / N, atol=1e-13)
    # all masses equal: the tie rule keeps the lowest columns; 2^20 k >= P_q * 3
    for rb in range(3):
        assert bsr.kept(0, rb) == [0, 1]


def test_identity_attention():
    """Dominant diagonal logits: P ~ I, only diagonal blocks carry mass."""
    N, d, B = 48, 48, 16
    q = np.eye(N)[:, None, :] * 40.0
    k = np.eye(N)[:, None, :] * 40.0
    bsr = orc.compress(q, k, [0, N], B, 0.99, True)
    for rb in range(3):
        assert bsr.kept(0, rb) == [rb]
    v = np.random.default_rng(2).standard_normal((N, 1, 8))
    O, _ = orc.retrieve(q, k, bsr, np.eye(1), v, 1)
    assert np.abs(O - v).max() < 1e-12


def selection_bruteforce(mass, p):
    """All subsets of the candidates: the minimal-cardinality subsets whose
    fixed-point sum reaches the threshold, and the one the tie rule picks."""
    n = len(mass)
    q = [int(np.rint(x * 2.0 ** 32)) for x in mass]
    tot = sum(q)
    # the threshold as the library receives it: a 32-bit float
    pq = int(np.rint(float(np.float32(p)) * 2 ** 20))
    for size in range(n + 1):
        ok = [S for S in itertools.combinations(range(n), size)
              if (sum(q[b] for b in S) << 20) >= pq * tot]
        if ok:
            return size, ok
    raise AssertionError


@pytest.mark.parametrize("seed", range(40))
def test_selection_bruteforce(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 9))
    mass = rng.random(n) * rng.choice([1.0, 1e-3, 64.0])
    if seed % 3 == 0 and n > 2:  # plant exact ties
        mass[1] = mass[0]
        mass[-1] = mass[0]
    mass = mass.astype(np.float32).astype(np.float64)
    for p in (0.5, 0.8, 0.9, 0.95, 0.99, 1.0, float(rng.random())):
        kept = orc.select_topp(mass, p)
        size, subsets = selection_bruteforce(mass, p)
        assert len(kept) == size
        assert tuple(kept) in subsets
        dropped = [b for b in range(n) if b not in kept]
        for a in kept:
            for b in dropped:
                assert mass[a] > mass[b] or (mass[a] == mass[b] and a < b)


def test_selection_fixed_point_constants():
    assert [orc.threshold_fixed(p) for p in (0.80, 0.90, 0.95, 0.99, 1.0)] == \
        [838861, 943718, 996147, 1038090, 1048576]


def test_threshold_is_taken_from_the_float32_the_abi_receives():
    """The compressor's entry point takes p as a 32-bit float, so P_q comes
    from float32(p).  For p = 838860.51 / 2^20 the double gives
    rint(838860.51) = 838861, but float32 keeps 24 significant bits (steps of
    2^-24 here, i.e. 1/16 of a 2^-20 unit), so float32(p) * 2^20 = 838860.5
    exactly and the half-even rint gives 838860."""
    p = 838860.51 / 2 ** 20
    assert float(np.float32(p)) * 2 ** 20 == 838860.5
    assert orc.threshold_fixed(p) == 838860
    for x in np.random.default_rng(3).random(200):
        assert orc.threshold_fixed(float(x)) == orc.threshold_fixed(float(np.float32(x)))


def test_selection_uniform_closed_form():
    for n in range(1, 40):
        for p in (0.8, 0.95):
            k = orc.select_topp([0.25] * n, p)
            pq = orc.threshold_fixed(p)
            want = -(-(pq * n) // (1 << 20))  # ceil(P_q * n / 2^20)
            assert k == list(range(want))


@pytest.mark.parametrize("causal", [True, False])
def test_sdpa_closed_form(causal):
    """The whole path at p = 1, W = I, H_r = H_s = H_kv equals torch's
    scaled_dot_product_attention (fp64), over a packed varlen batch."""
    assert check_sdpa_closed_form(causal=causal) < 1e-12


def test_p1_equals_dense_head_mapped():
    q, k, cu = rand_case((45, 80), 4, 2, 16, 5)
    v = np.random.default_rng(6).standard_normal((125, 2, 16))
    W = np.random.default_rng(7).standard_normal((6, 4))
    bsr = orc.compress(q, k, cu, 16, 1.0, True)
    O, _ = orc.retrieve(q, k, bsr, W, v, 2)
    ref = orc.dense_head_mapped(q, k, cu, W, v, 2)
    assert np.abs(O - ref).max() < 1e-12


def torch_probs(q, k, cu, h, hk, causal=True):
    """Independent softmax rows via torch (fp64) for one head."""
    out = []
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        S = torch.from_numpy(q[a:b, h]) @ torch.from_numpy(k[a:b, hk]).T / math.sqrt(q.shape[2])
        if causal:
            S = S.masked_fill(torch.triu(torch.ones(b - a, b - a, dtype=torch.bool), 1), -math.inf)
        out.append(torch.softmax(S, dim=1).numpy())
    return out


def kept_dense_mask(bsr, h, s):
    g = bsr.grid
    L = int(g.lens[s])
    mk = np.zeros((L, L))
    for bi in range(int(g.nblocks[s])):
        rb = int(g.rb_base[s]) + bi
        for bj in bsr.kept(h, rb):
            mk[bi * g.B:(bi + 1) * g.B, bj * g.B:(bj + 1) * g.B] = 1
    return mk


def check_onehot_head_map(o=orc, seed=8):
    """W = e_h (one-hot row i -> sender head h) returns sender head h's kept
    map times V of receiver head i's KV group.  Non-square, GQA."""
    q, k, cu = rand_case((40, 57), 6, 3, 8, seed)
    Hr, Hkv = 4, 2
    v = np.random.default_rng(seed + 1).standard_normal((97, Hkv, 8))
    bsr = o.compress(q, k, cu, 16, 0.8, True)
    W = np.zeros((Hr, 6))
    pick = [5, 0, 3, 1]
    for i, h in enumerate(pick):
        W[i, h] = 1.0
    O, _ = o.retrieve(q, k, bsr, W, v, Hkv)
    err = 0.0
    for i, h in enumerate(pick):
        Ps = torch_probs(q, k, cu, h, h // 2)
        for s in range(2):
            a, b = int(cu[s]), int(cu[s + 1])
            ref = (Ps[s] * kept_dense_mask(bsr, h, s)) @ v[a:b, i // (Hr // Hkv)]
            err = max(err, float(np.abs(O[a:b, i] - ref).max()))
    return err


def test_onehot_head_map():
    assert check_onehot_head_map() < 1e-12


def test_linearity_in_W():
    q, k, cu = rand_case((64,), 3, 3, 8, 9)
    v = np.random.default_rng(10).standard_normal((64, 1, 8))
    bsr = orc.compress(q, k, cu, 16, 0.7, True)
    W1 = np.random.default_rng(1).standard_normal((2, 3))
    W2 = np.random.default_rng(2).standard_normal((2, 3))
    O1, _ = orc.retrieve(q, k, bsr, W1, v, 1)
    O2, _ = orc.retrieve(q, k, bsr, W2, v, 1)
    O3, _ = orc.retrieve(q, k, bsr, W1 - 2.5 * W2, v, 1)
    assert np.abs(O3 - (O1 - 2.5 * O2)).max() < 1e-12


def check_no_renormalisation(o=orc, seed=12):
    """With V = 1, O_i(row) = sum_h W[i,h] * (kept probability of that row
    in head h): dropped blocks are zero and nothing is rescaled."""
    q, k, cu = rand_case((90,), 3, 3, 8, seed)
    v = np.ones((90, 1, 4))
    bsr = o.compress(q, k, cu, 16, 0.6, True)
    W = np.random.default_rng(seed).standard_normal((2, 3))
    O, _ = o.retrieve(q, k, bsr, W, v, 1)
    kept_mass = np.stack([(torch_probs(q, k, cu, h, h)[0] * kept_dense_mask(bsr, h, 0)).sum(1)
                          for h in range(3)])  # [H_s, T]
    ref = W @ kept_mass  # [H_r, T]
    assert (kept_mass < 1 - 1e-6).any()  # something was actually dropped
    return float(np.abs(O[:, :, 0].T - ref).max())


def test_no_renormalisation():
    assert check_no_renormalisation() < 1e-12


def test_selection_invariants_on_structured_workload():
    """On the structured synthetic recipe (sink + band), each kept row reaches
    the threshold and dropping its smallest kept block falls below it."""
    from cross_model_attention_gb300 import workloads
    w = workloads.scaled(workloads.get(1), [512], sender_heads=4, sender_kv_heads=4)
    x = synth.sender_qk(w, 1)
    bsr = orc.compress(x["q64"], x["k64"], w.cu_seqlens, w.B, 0.95, True, keep_tiles=False)
    g = bsr.grid
    pq = orc.threshold_fixed(0.95)
    for h in range(4):
        for rb in range(g.R):
            ms = bsr.mass[h, g.cand_ptr[rb]:g.cand_ptr[rb + 1]]
            q = np.rint(ms * 2.0 ** 32).astype(np.int64)
            kept = bsr.kept(h, rb)
            tot = int(q.sum())
            s = int(q[kept].sum())
            assert (s << 20) >= pq * tot
            smallest = min(kept, key=lambda b: (ms[b], -b))
            assert ((s - int(q[smallest])) << 20) < pq * tot


def test_tiles_are_probabilities():
    q, k, cu = rand_case((70, 20), 2, 2, 8, 13)
    bsr = orc.compress(q, k, cu, 16, 0.9, True)
    g = bsr.grid
    for h in range(2):
        Ps = torch_probs(q, k, cu, h, h)
        for rb in range(g.R):
            s, bi = int(g.rb_seq[rb]), int(g.rb_local[rb])
            L = int(g.lens[s])
            for t, bj in enumerate(bsr.kept(h, rb)):
                tile = bsr.tiles[bsr.row_ptr[h * g.R + rb] + t]
                ref = np.zeros((16, 16))
                blk = Ps[s][bi * 16:(bi + 1) * 16, bj * 16:(bj + 1) * 16]
                ref[:blk.shape[0], :blk.shape[1]] = blk
                assert np.abs(tile - ref).max() < 1e-14
                # the tile's sum is the candidate's mass
                assert abs(tile.sum() - bsr.mass[h, g.cand_ptr[rb] + bj]) < 1e-12


# ------------------------------------------------------- head-map calibration

def test_calibration_recovers_a_planted_map_exactly():
    """Receiver maps that are exactly W_true times the sender maps give back
    W_true (signed, non-square)."""
    rng = np.random.default_rng(5)
    S = rng.random((5, 400))
    W_true = rng.standard_normal((3, 5))
    W = orc.calibrate_head_map(S, W_true @ S)
    assert np.allclose(W, W_true, atol=1e-10)


def test_calibration_is_the_least_squares_solution():
    """Against numpy's least-squares routine on the stacked system, with and
    without the ridge (the ridge as sqrt(ridge) * I rows appended)."""
    rng = np.random.default_rng(6)
    S = rng.random((4, 300))
    R = rng.random((6, 300))
    W = orc.calibrate_head_map(S, R)
    ref = np.linalg.lstsq(S.T, R.T, rcond=None)[0].T
    assert np.allclose(W, ref, atol=1e-10)
    lam = 0.37
    Wr = orc.calibrate_head_map(S, R, ridge=lam)
    A = np.concatenate([S.T, np.sqrt(lam) * np.eye(4)])
    Bm = np.concatenate([R.T, np.zeros((4, 6))])
    assert np.allclose(Wr, np.linalg.lstsq(A, Bm, rcond=None)[0].T, atol=1e-10)


def test_map_entries_masks_dropped_blocks_and_rows_sum_to_one():
    rng = np.random.default_rng(7)
    cu = np.array([0, 100, 164])
    q = rng.standard_normal((164, 2, 16))
    k = rng.standard_normal((164, 2, 16))
    g = orc.BlockGrid(cu, 32, True)
    full = orc.map_entries(q, k, g)
    # each sequence's L x L map has rows summing to one
    assert np.allclose(full[:, :100 * 100].reshape(2, 100, 100).sum(-1), 1.0)
    assert np.allclose(full[:, 100 * 100:].reshape(2, 64, 64).sum(-1), 1.0)
    # dropping block column 0 of block-row 1 of sequence 0 (head 1) zeroes
    # exactly rows 32..63, columns 0..31 of that head's map
    kept = lambda h, rb: [bj for bj in range(int(g.ncand[rb])) if not (h == 1 and rb == 1 and bj == 0)]
    part = orc.map_entries(q, k, g, kept)
    m0 = part[1, :100 * 100].reshape(100, 100)
    f0 = full[1, :100 * 100].reshape(100, 100)
    assert np.all(m0[32:64, 0:32] == 0)
    diff = (m0 != f0)
    assert diff[32:64, 0:32].all() and diff.sum() == 32 * 32
    assert np.array_equal(part[0], full[0])


# ------------------------------------------- prefix sharing (block manager)

def test_prefix_block_rows_do_not_depend_on_the_continuation():
    """Reading behind the prefix-hash cache: with a causal mask, block-row bi
    (masses, kept set, tiles, row statistics) depends only on the tokens of
    blocks 0..bi, so two sequences that share three full blocks share the
    states of those block-rows; without the mask they do not."""
    rng = np.random.default_rng(21)
    B, d, H, P = 16, 16, 2, 48
    qa, ka = rng.standard_normal((P + 20, H, d)), rng.standard_normal((P + 20, H, d))
    qb, kb = rng.standard_normal((P + 37, H, d)), rng.standard_normal((P + 37, H, d))
    qb[:P], kb[:P] = qa[:P], ka[:P]
    for causal in (True, False):
        A = orc.compress(qa, ka, [0, P + 20], B, 0.9, causal)
        Bq = orc.compress(qb, kb, [0, P + 37], B, 0.9, causal)
        same = True
        for h in range(H):
            for rb in range(P // B):
                ka_, kb_ = A.kept(h, rb), Bq.kept(h, rb)
                ca, cb = A.grid.cand_ptr[rb], Bq.grid.cand_ptr[rb]
                na = A.grid.cand_ptr[rb + 1] - ca
                nb_ = Bq.grid.cand_ptr[rb + 1] - cb
                ma, mb = A.mass[h, ca:ca + na], Bq.mass[h, cb:cb + nb_]
                if na != nb_ or not np.allclose(ma, mb, rtol=1e-13, atol=0):
                    same = False
                    continue
                assert ka_ == kb_
                ta = A.tiles[A.row_ptr[h * A.grid.R + rb]:A.row_ptr[h * A.grid.R + rb + 1]]
                tb = Bq.tiles[Bq.row_ptr[h * Bq.grid.R + rb]:Bq.row_ptr[h * Bq.grid.R + rb + 1]]
                assert np.allclose(ta, tb, rtol=1e-13, atol=1e-300)
            for key in ("m", "l"):
                if not np.allclose(getattr(A, key)[h, :P], getattr(Bq, key)[h, :P], rtol=1e-13):
                    same = False
        assert same == causal


# ------------------------------------------- full-size per-block-row helpers

def dense_rows_torch(q, k, cu, h, hk, s, causal):
    """Scaled logits, their row max and exp-sum, and the softmax of sequence
    s for one head, all via torch (fp64) over the whole L x L map."""
    a, b = int(cu[s]), int(cu[s + 1])
    d = q.shape[2]
    S = torch.from_numpy(q[a:b, h]) @ torch.from_numpy(k[a:b, hk]).T / math.sqrt(d)
    if causal:
        S = S.masked_fill(torch.triu(torch.ones(b - a, b - a, dtype=torch.bool), 1), -math.inf)
    m = S.max(dim=1).values
    l = torch.exp(S - m[:, None]).sum(dim=1)
    return torch.softmax(S, dim=1).numpy(), m.numpy(), l.numpy()


def check_block_row_helpers(o=orc, B=16, causal=True, seed=31):
    """block_row_reference and retrieve_block_row, which the GPU parity tests
    use at full size one block-row at a time, against (i) whole-sequence
    softmax maps from torch, sliced at the block-row's rows, and (ii) the
    oracle's own compress / retrieve.  Packed sequences with ragged tails
    (and one full-block sequence), a GQA sender (4 q-heads on 2 KV heads) and
    a receiver with H_r = 6 != H_s on 3 KV groups.  Returns the largest
    deviation found."""
    T_list = (45, 70, 2 * B, 33)
    Hs, Hks, d, Hr, Hkv = 4, 2, 16, 6, 3
    q, k, cu = rand_case(T_list, Hs, Hks, d, seed)
    rng = np.random.default_rng(seed + 1)
    v = rng.standard_normal((sum(T_list), Hkv, d))
    W = rng.standard_normal((Hr, Hs))
    bsr = orc.compress(q, k, cu, B, 0.8, causal)
    O_full, _ = orc.retrieve(q, k, bsr, W, v, Hkv)
    g = bsr.grid
    err = 0.0
    dense = {(h, s): dense_rows_torch(q, k, cu, h, h // (Hs // Hks), s, causal)
             for h in range(Hs) for s in range(g.n_seqs)}
    for rb in range(g.R):
        s, bi = int(g.rb_seq[rb]), int(g.rb_local[rb])
        a, L = int(cu[s]), int(cu[s + 1] - cu[s])
        r0, r1 = bi * B, min(L, (bi + 1) * B)
        want_rows = np.arange(a + r0, a + r1)
        for h in range(Hs):
            ref = o.block_row_reference(q, k, g, h, rb)
            P, m, l = dense[(h, s)]
            if not np.array_equal(ref["rows"], want_rows) or ref["P"].shape != (r1 - r0, L):
                return math.inf
            err = max(err, float(np.abs(ref["P"] - P[r0:r1]).max()),
                      float(np.abs(ref["m"] - m[r0:r1]).max()),
                      float(np.abs(ref["l"] / l[r0:r1] - 1).max()))
            c0, c1 = int(g.cand_ptr[rb]), int(g.cand_ptr[rb + 1])
            err = max(err, float(np.abs(ref["mass"] - bsr.mass[h, c0:c1]).max()))
        got, rows = o.retrieve_block_row(q, k, g, bsr.kept, W, v, Hkv, rb)
        if not np.array_equal(rows, want_rows):
            return math.inf
        err = max(err, float(np.abs(got - O_full[want_rows]).max()))
        # the same rows from the torch maps: sum_h W[i,h] (P_h * kept_h) V_g(i)
        for i in range(Hr):
            Ahat = sum(W[i, h] * dense[(h, s)][0][r0:r1] *
                       orc.kept_mask_rows(g, bsr.kept(h, rb), bi, s, r1 - r0) for h in range(Hs))
            want = Ahat @ v[a:a + L, i // (Hr // Hkv)]
            err = max(err, float(np.abs(got[:, i] - want).max()))
    return err


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("causal", [True, False])
def test_block_row_helpers(B, causal):
    assert check_block_row_helpers(B=B, causal=causal) < 1e-13
