"""Plain fp64 CPU oracle of the cross-model attention-map reuse hot path.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline / reference leg may import this module.  The GPU
library never calls it, and it shares no code, constants or helpers with the
CUDA path.

What it follows (the two pages on the method; neither prints pseudo-code):

* "Accelerating Cross-Model LLM Inference via Attention Map Reuse"
  (paper summary page; cited below as [Summary]):
  - "MapFlow System Design", items 1-3: partial recomputation, layer mapping
    m(j), head mapping by a linear transformation of the sender's maps;
  - "Practical Implementation Details": the Attention State Compressor keeps
    blocks by block-level top-p and stores them in Block Sparse Row form; the
    Attention Retrieval fuses the reconstruction of the receiver map with the
    multiplication by the receiver's V and never materialises it densely;
  - bold headers 2-4: linear translation across heads, the cumulative
    probability threshold p, the fused retrieval kernel.
* "北大MapFlow：注意力图跨模型复用，prefill延迟降15%–20%" (news article; cited
  below as [Article]): the paragraphs "其一" (block statistics first, then
  block selection, with no dense map), "其三" (heads combined on chip, then
  multiplied by the receiver's Value and accumulated), and the section on
  reusing token-dependency structure (the receiver keeps its own V).

Readings where the pages are silent:

1. Head mapping: A_hat_i = sum_h W[i, h] * A_h of the mapped sender layer,
   W real and signed, no renormalisation; missing blocks count as zero.
2. A block's mass is the sum of the normalised probabilities inside it; the
   block-row total is the sum of its candidate masses.
3. Selection order: mass descending, ties to the lower block column.  The
   cumulative sum and the threshold are evaluated exactly in fixed point:
   q_b = rint(mass_b * 2**32), Tot = sum q_b, P_q = rint(p * 2**20); keep the
   shortest sorted prefix with 2**20 * (prefix sum) >= P_q * Tot.  p is the
   32-bit float the library's entry point receives, so P_q is taken from
   float32(p), widened exactly.
4. Causal candidates are the blocks bj <= bi; non-causal: all blocks.
5. Kept tiles hold the normalised probabilities P_ij, zero above the diagonal
   and outside the sequence; tiles never straddle packed sequences; block
   grids start at each sequence's first token.
6. col_idx ascending within a row and relative to the sequence's first block.
   BSR rows are ordered head-major, then global block-row.
7. GQA: query head h uses KV head h // (H_q / H_kv) (contiguous groups), for
   the sender's K and for the receiver's V alike.

The oracle works block-row by block-row: every quantity of the method is
defined per row (softmax) or per block-row (mass, selection, BSR row), so
this is the method's own granularity, not an optimisation.  Library
primitives used as steps: numpy matmul, exp, sort.

Parity pins for every function live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

# --------------------------------------------------------------------------
# Layout helpers (host-side bookkeeping of the block grid; plain definitions)
# --------------------------------------------------------------------------


@dataclasses.dataclass
class BlockGrid:
    """Block grid of a packed batch: one grid per sequence, starting at its
    first token ([Summary] "Practical Implementation Details": regular 2-D
    blocks; reading 5)."""

    cu_seqlens: np.ndarray
    B: int
    causal: bool

    def __post_init__(self):
        cu = np.asarray(self.cu_seqlens, dtype=np.int64)
        self.cu = cu
        self.n_seqs = len(cu) - 1
        self.lens = np.diff(cu)
        self.nblocks = (self.lens + self.B - 1) // self.B
        self.rb_base = np.concatenate([[0], np.cumsum(self.nblocks)])
        self.R = int(self.rb_base[-1])
        # candidate list per global block-row
        ncand = []
        self.rb_seq = np.zeros(self.R, np.int64)
        self.rb_local = np.zeros(self.R, np.int64)
        for s in range(self.n_seqs):
            for bi in range(int(self.nblocks[s])):
                rb = int(self.rb_base[s]) + bi
                self.rb_seq[rb] = s
                self.rb_local[rb] = bi
                ncand.append(bi + 1 if self.causal else int(self.nblocks[s]))
        self.ncand = np.asarray(ncand, np.int64)
        self.cand_ptr = np.concatenate([[0], np.cumsum(self.ncand)]).astype(np.int64)
        self.C = int(self.cand_ptr[-1])


# --------------------------------------------------------------------------
# Step a1/a2: attention probabilities, row statistics, block masses
# --------------------------------------------------------------------------


def attention_rows(q_rows: np.ndarray, k_seq: np.ndarray, row_pos: np.ndarray,
                   causal: bool) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Softmax attention of some query rows of one head over one sequence.

    q_rows [n, d], k_seq [L, d] (fp64), row_pos [n] = positions of the rows in
    the sequence.  Returns P [n, L] (the normalised attention map rows,
    [Summary] "Attention Maps as Reuse States"), the row maxima m [n] of the
    scaled logits s_ij = q_i . k_j / sqrt(d), and the row sums
    l [n] = sum_j exp(s_ij - m_i), over the keys a causal row may see.
    """
    d = q_rows.shape[1]
    L = k_seq.shape[0]
    S = (q_rows @ k_seq.T) / math.sqrt(d)
    if causal:
        allowed = np.arange(L)[None, :] <= row_pos[:, None]
    else:
        allowed = np.ones((len(row_pos), L), dtype=bool)
    S = np.where(allowed, S, -np.inf)
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    P = E / l[:, None]
    return P, m, l


def block_masses(P_rows: np.ndarray, B: int, n_cand: int) -> np.ndarray:
    """Mass of each candidate block of one block-row: the sum of the
    probabilities of P_rows [<=B, L] that fall in key block bj
    ([Article] "其一": block-level statistics; reading 2)."""
    L = P_rows.shape[1]
    out = np.zeros(n_cand)
    for bj in range(n_cand):
        out[bj] = P_rows[:, bj * B:min(L, (bj + 1) * B)].sum()
    return out


# --------------------------------------------------------------------------
# Step a3: block-level top-p
# --------------------------------------------------------------------------

P_FRAC_BITS = 20
MASS_FRAC_BITS = 32


def threshold_fixed(p: float) -> int:
    """P_q = rint(p * 2**20) of the threshold as the compressor receives it:
    a 32-bit float (reading 3).  float32(p) widens to fp64 exactly and its
    product with 2**20 is exact, so the only rounding is the rint."""
    return int(np.rint(np.float64(np.float32(p)) * (1 << P_FRAC_BITS)))


def select_topp(mass: Sequence[float], p: float) -> List[int]:
    """Block-level top-p of one block-row ([Summary] "Practical Implementation
    Details" and bold header 3; [Article] "其一": keep the blocks needed to
    reach cumulative probability p of the row).

    mass: candidate masses in block-column order (fp64, or fp32 values
    widened exactly).  Sort by mass descending, ties to the smaller column;
    keep the shortest prefix whose cumulative mass reaches p of the row total,
    both sides evaluated exactly in fixed point (reading 3).  Returns the kept
    block columns in ascending order.
    """
    mass = np.asarray(mass, dtype=np.float64)
    n = len(mass)
    if n == 0:
        return []
    order = sorted(range(n), key=lambda b: (-mass[b], b))
    q = [int(np.rint(mass[b] * float(1 << MASS_FRAC_BITS))) for b in range(n)]
    tot = sum(q)
    pq = threshold_fixed(p)
    acc, k = 0, 0
    while k < n and (acc << P_FRAC_BITS) < pq * tot:
        acc += q[order[k]]
        k += 1
    return sorted(order[:k])


# --------------------------------------------------------------------------
# Step a4: BSR
# --------------------------------------------------------------------------


@dataclasses.dataclass
class OracleBSR:
    """Block Sparse Row form of one sender layer ([Summary] "Practical
    Implementation Details"): rows are (head, global block-row) head-major;
    row_ptr [H_s*R+1], col_idx [nnz] (sequence-relative block column),
    tiles [nnz, B, B] fp64 probabilities.  Also the candidate masses
    mass [H_s, C] and row statistics m, l [H_s, T]."""

    grid: BlockGrid
    H_s: int
    row_ptr: np.ndarray
    col_idx: np.ndarray
    tiles: Optional[np.ndarray]
    mass: np.ndarray
    m: np.ndarray
    l: np.ndarray

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    def kept(self, h: int, rb: int) -> List[int]:
        r = h * self.grid.R + rb
        return [int(x) for x in self.col_idx[self.row_ptr[r]:self.row_ptr[r + 1]]]


def _tile(P_rows: np.ndarray, B: int, bj: int) -> np.ndarray:
    t = np.zeros((B, B))
    L = P_rows.shape[1]
    c0, c1 = bj * B, min(L, (bj + 1) * B)
    t[:P_rows.shape[0], :c1 - c0] = P_rows[:, c0:c1]
    return t


def compress(q64: np.ndarray, k64: np.ndarray, cu_seqlens: Sequence[int], B: int,
             p: float, causal: bool = True, keep_tiles: bool = True,
             mass_for_selection: Optional[np.ndarray] = None) -> OracleBSR:
    """The Attention State Compressor on one sender layer.

    q64 [T, H_s, d], k64 [T, H_ks, d] (fp64).  For every head and block-row:
    softmax rows (a1), candidate block masses (a2), block top-p (a3), kept
    probability tiles packed as BSR (a4).  ([Summary] "Practical
    Implementation Details"; [Article] "其一".)

    mass_for_selection [H_s, C], when given, replaces the oracle's own masses
    as the input of the selection step only (the selection rule is then
    evaluated on another implementation's mass tensor, bit for bit).
    """
    T, Hs, d = q64.shape
    Hks = k64.shape[1]
    g = BlockGrid(np.asarray(cu_seqlens), B, causal)
    mass = np.zeros((Hs, g.C))
    m_all = np.full((Hs, T), np.nan)
    l_all = np.full((Hs, T), np.nan)
    kept_rows: List[List[int]] = []
    tiles: List[np.ndarray] = []
    for h in range(Hs):
        hk = h // (Hs // Hks)
        for rb in range(g.R):
            s, bi = int(g.rb_seq[rb]), int(g.rb_local[rb])
            a, L = int(g.cu[s]), int(g.lens[s])
            r0, r1 = bi * B, min(L, (bi + 1) * B)
            pos = np.arange(r0, r1)
            P, m, l = attention_rows(q64[a + r0:a + r1, h], k64[a:a + L, hk], pos, causal)
            m_all[h, a + r0:a + r1] = m
            l_all[h, a + r0:a + r1] = l
            nc = int(g.ncand[rb])
            ms = block_masses(P, B, nc)
            c0 = int(g.cand_ptr[rb])
            mass[h, c0:c0 + nc] = ms
            sel_in = ms if mass_for_selection is None else mass_for_selection[h, c0:c0 + nc]
            kept = select_topp(sel_in, p)
            kept_rows.append(kept)
            if keep_tiles:
                tiles.extend(_tile(P, B, bj) for bj in kept)
    counts = np.array([len(k) for k in kept_rows], np.int64)
    row_ptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    col_idx = np.array([bj for k in kept_rows for bj in k], np.int64)
    tl = np.stack(tiles) if (keep_tiles and tiles) else (np.zeros((0, B, B)) if keep_tiles else None)
    return OracleBSR(g, Hs, row_ptr, col_idx, tl, mass, m_all, l_all)


# --------------------------------------------------------------------------
# Step a5: head-mapped retrieval
# --------------------------------------------------------------------------


def retrieve_rows(P_kept_rows: np.ndarray, W: np.ndarray, v_seq: np.ndarray,
                  H_kv: int) -> np.ndarray:
    """Receiver output rows from sender probabilities.

    P_kept_rows [H_s, n, L]: the sender map rows of every sender head with the
    dropped blocks already zeroed (missing blocks count as zero, no
    renormalisation).  W [H_r, H_s]; v_seq [L, H_kv, d].
    A_hat_i = sum_h W[i,h] * P_h ([Summary] "MapFlow System Design" item 3 and
    bold header 2), then O_i = A_hat_i @ V_{g(i)} ([Summary] "Practical
    Implementation Details": the reconstruction is multiplied by the
    receiver's value vectors; [Article] "其三").  Returns O [n, H_r, d].
    """
    Hs, n, L = P_kept_rows.shape
    Hr = W.shape[0]
    A_hat = np.tensordot(W.astype(np.float64), P_kept_rows, axes=([1], [0]))  # [H_r, n, L]
    out = np.zeros((n, Hr, v_seq.shape[2]))
    for i in range(Hr):
        gi = i // (Hr // H_kv)
        out[:, i, :] = A_hat[i] @ v_seq[:, gi, :]
    return out


def kept_mask_rows(grid: BlockGrid, kept: Sequence[int], bi: int, s: int,
                   n_rows: int) -> np.ndarray:
    """[n_rows, L] 0/1 mask of the kept blocks of one block-row."""
    L = int(grid.lens[s])
    mk = np.zeros((n_rows, L))
    for bj in kept:
        mk[:, bj * grid.B:min(L, (bj + 1) * grid.B)] = 1.0
    return mk


def retrieve(q64: np.ndarray, k64: np.ndarray, bsr: OracleBSR, W: np.ndarray,
             v64: np.ndarray, H_kv: int, block_rows: Optional[Iterable[int]] = None
             ) -> Tuple[np.ndarray, np.ndarray]:
    """Dense-reconstruction reference of the fused retrieval for one receiver
    layer: for each block-row, rebuild every sender head's map rows, keep
    only that head's kept blocks, combine heads with W, multiply by V.

    Returns (O [T, H_r, d] with NaN for rows not computed, row_done [T]).
    """
    g = bsr.grid
    T, Hs, d = q64.shape
    Hks = k64.shape[1]
    Hr = W.shape[0]
    O = np.full((T, Hr, v64.shape[2]), np.nan)
    done = np.zeros(T, bool)
    rbs = range(g.R) if block_rows is None else block_rows
    for rb in rbs:
        s, bi = int(g.rb_seq[rb]), int(g.rb_local[rb])
        a, L = int(g.cu[s]), int(g.lens[s])
        r0, r1 = bi * g.B, min(L, (bi + 1) * g.B)
        pos = np.arange(r0, r1)
        Pk = np.zeros((Hs, r1 - r0, L))
        for h in range(Hs):
            hk = h // (Hs // Hks)
            P, _, _ = attention_rows(q64[a + r0:a + r1, h], k64[a:a + L, hk], pos, g.causal)
            Pk[h] = P * kept_mask_rows(g, bsr.kept(h, rb), bi, s, r1 - r0)
        O[a + r0:a + r1] = retrieve_rows(Pk, W, v64[a:a + L], H_kv)
        done[a + r0:a + r1] = True
    return O, done


def dense_head_mapped(q64: np.ndarray, k64: np.ndarray, cu_seqlens: Sequence[int],
                      W: np.ndarray, v64: np.ndarray, H_kv: int,
                      causal: bool = True) -> np.ndarray:
    """The unsparsified head-mapped output sum_h W[i,h] softmax_h @ V_g(i):
    the retrieval with every block kept (what the BSR path must equal at
    p = 1)."""
    T, Hs, d = q64.shape
    Hks = k64.shape[1]
    Hr = W.shape[0]
    O = np.zeros((T, Hr, v64.shape[2]))
    cu = np.asarray(cu_seqlens)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        Ps = np.stack([attention_rows(q64[a:b, h], k64[a:b, h // (Hs // Hks)],
                                      np.arange(L), causal)[0] for h in range(Hs)])
        O[a:b] = retrieve_rows(Ps, W, v64[a:b], H_kv)
    return O


# --------------------------------------------------------------------------
# Head-map calibration ([Summary] "MapFlow System Design" item 3: the head
# map is a linear transformation of the sender's maps, fitted offline)
# --------------------------------------------------------------------------


def map_entries(q64: np.ndarray, k64: np.ndarray, grid: BlockGrid,
                kept_of=None, causal: bool = True) -> np.ndarray:
    """Every head's attention map over every packed sequence, flattened to
    [H, sum_s L_s^2]; when kept_of(h, rb) is given, the blocks it does not
    list are zero (the map as the BSR stores it)."""
    T, H, d = q64.shape
    Hk = k64.shape[1]
    out = [[] for _ in range(H)]
    cu = grid.cu
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        for h in range(H):
            P = attention_rows(q64[a:b, h], k64[a:b, h // (H // Hk)], np.arange(L), causal)[0]
            if kept_of is not None:
                for bi in range(int(grid.nblocks[s])):
                    r0, r1 = bi * grid.B, min(L, (bi + 1) * grid.B)
                    P[r0:r1] *= kept_mask_rows(grid, kept_of(h, int(grid.rb_base[s]) + bi), bi, s, r1 - r0)
            out[h].append(P.reshape(-1))
    return np.stack([np.concatenate(x) for x in out])


def calibrate_head_map(sender: np.ndarray, receiver: np.ndarray, ridge: float = 0.0) -> np.ndarray:
    """W [H_r, H_s] minimising sum_i sum_m (receiver[i, m] - sum_h W[i, h]
    sender[h, m])^2 + ridge * |W|^2 over the map entries m (reading: least
    squares of the receiver's map against the sender heads' kept maps):
    the normal equations (S S^T + ridge I) W^T = S R^T."""
    S = np.asarray(sender, np.float64)
    R = np.asarray(receiver, np.float64)
    G = S @ S.T + ridge * np.eye(S.shape[0])
    return np.linalg.solve(G, S @ R.T).T


# --------------------------------------------------------------------------
# Full-size helpers: sampled checks that stay exact per block-row
# --------------------------------------------------------------------------


def block_row_reference(q64: np.ndarray, k64: np.ndarray, grid: BlockGrid, h: int,
                        rb: int) -> Dict[str, np.ndarray]:
    """Row statistics, candidate masses and P rows of one (head, block-row)."""
    Hs, Hks = q64.shape[1], k64.shape[1]
    hk = h // (Hs // Hks)
    s, bi = int(grid.rb_seq[rb]), int(grid.rb_local[rb])
    a, L = int(grid.cu[s]), int(grid.lens[s])
    r0, r1 = bi * grid.B, min(L, (bi + 1) * grid.B)
    P, m, l = attention_rows(q64[a + r0:a + r1, h], k64[a:a + L, hk], np.arange(r0, r1),
                             grid.causal)
    return {"P": P, "m": m, "l": l,
            "mass": block_masses(P, grid.B, int(grid.ncand[rb])),
            "rows": np.arange(a + r0, a + r1)}


def retrieve_block_row(q64: np.ndarray, k64: np.ndarray, grid: BlockGrid,
                       kept_of: "callable", W: np.ndarray, v64: np.ndarray, H_kv: int,
                       rb: int) -> Tuple[np.ndarray, np.ndarray]:
    """O rows of one block-row given kept_of(h, rb) -> kept block columns."""
    Hs, Hks = q64.shape[1], k64.shape[1]
    s, bi = int(grid.rb_seq[rb]), int(grid.rb_local[rb])
    a, L = int(grid.cu[s]), int(grid.lens[s])
    r0, r1 = bi * grid.B, min(L, (bi + 1) * grid.B)
    Pk = np.zeros((Hs, r1 - r0, L))
    for h in range(Hs):
        P, _, _ = attention_rows(q64[a + r0:a + r1, h], k64[a:a + L, h // (Hs // Hks)],
                                 np.arange(r0, r1), grid.causal)
        Pk[h] = P * kept_mask_rows(grid, kept_of(h, rb), bi, s, r1 - r0)
    return retrieve_rows(Pk, W, v64[a:a + L], H_kv), np.arange(a + r0, a + r1)
