"""Shared runner of the GPU parity tests: run the CUDA path through the C-ABI
binding on seeded inputs and compare with the fp64 oracle.

Tolerances:
  * row_ptr / col_idx: bit-exact, with the selection evaluated by the oracle
    on the GPU's own block-mass tensor;
  * block masses: relative 1e-4, with an absolute floor of B^2 * 2^-126: the
    kernels take exp2 with flush-to-zero, so each of a block's B^2
    probabilities (or a row's partial sum, of which a block has fewer) that
    falls below fp32's smallest normal 2^-126 may come out as zero;
  * bf16 tiles: within one bf16 ulp of the oracle's probability;
  * row statistics: m within 1e-5 (absolute, natural-log units), l within
    1e-5 relative;
  * O: max |O - O_oracle| <= 1e-2 * max |O_oracle|.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence

import numpy as np
import torch

from cross_model_attention_gb300 import mapflow
from oracle import mapflow_oracle as orc

MASS_RTOL = 1e-4
O_TOL = 1e-2


def dev():
    assert torch.cuda.is_available(), "GPU test selected on a machine without a GPU"
    return torch.device("cuda", 0)


def to_dev(a: np.ndarray, dtype: str):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev()).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def export_np(bsr: mapflow.BSR, layer: int) -> Dict[str, np.ndarray]:
    """Small arrays as numpy; the tiles stay on the device ("values_dev") and
    are fetched on demand with tiles()."""
    ex = bsr.export(layer)
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in ex.items() if k != "values"}
    out["values_dev"] = ex["values"]
    return out


def tiles(ex, idx) -> np.ndarray:
    """bf16 bit patterns of the tiles with the given indices."""
    idx_t = torch.as_tensor(np.asarray(idx, np.int64), device=ex["values_dev"].device)
    sel = ex["values_dev"].index_select(0, idx_t).cpu()
    return sel.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_structure(ex, grid: orc.BlockGrid, H_s: int, p: float) -> None:
    """Selection rule re-evaluated by the oracle on the GPU's own masses."""
    mass = ex["mass"].reshape(H_s, grid.C).astype(np.float64)
    rp = [0]
    cols: List[int] = []
    for h in range(H_s):
        for rb in range(grid.R):
            kept = orc.select_topp(mass[h, grid.cand_ptr[rb]:grid.cand_ptr[rb + 1]], p)
            rp.append(rp[-1] + len(kept))
            cols.extend(kept)
    assert np.array_equal(ex["row_ptr"].astype(np.int64), np.asarray(rp)), "row_ptr differs"
    assert np.array_equal(ex["col_idx"].astype(np.int64), np.asarray(cols, np.int64)), \
        "col_idx differs"


def check_block_rows(ex, q64, k64, grid: orc.BlockGrid, H_s: int, pairs: Iterable) -> int:
    """Masses, row statistics and kept tiles of the sampled (head, block-row)
    pairs against the oracle.  Returns the number of tiles checked."""
    mass = ex["mass"].reshape(H_s, grid.C).astype(np.float64)
    T = q64.shape[0]
    rmax = ex["row_max"].reshape(H_s, T)
    rsum = ex["row_sum"].reshape(H_s, T)
    n_tiles = 0
    for h, rb in pairs:
        ref = orc.block_row_reference(q64, k64, grid, h, rb)
        got = mass[h, grid.cand_ptr[rb]:grid.cand_ptr[rb + 1]]
        err = np.abs(got - ref["mass"])
        bad = err > MASS_RTOL * np.abs(ref["mass"]) + grid.B ** 2 * 2.0 ** -126
        assert not bad.any(), f"mass (h={h}, rb={rb}) rel err {np.max(err / np.abs(ref['mass']))}"
        rows = ref["rows"]
        # m_i in fp32 carries three roundings (score, scale to log2 units,
        # back to natural units): 1e-5 absolute plus 1e-6 relative
        assert (np.abs(rmax[h, rows] - ref["m"]) <= 1e-5 + 1e-6 * np.abs(ref["m"])).all(), "row max differs"
        assert (np.abs(rsum[h, rows] - ref["l"]) <= 1e-5 * ref["l"]).all(), "row sum differs"
        r = h * grid.R + rb
        B = grid.B
        t0, t1 = int(ex["row_ptr"][r]), int(ex["row_ptr"][r + 1])
        got_tiles = tiles(ex, range(t0, t1)) if t1 > t0 else None
        for t in range(t0, t1):
            bj = int(ex["col_idx"][t])
            tile = bf16_bits_to_f64(got_tiles[t - t0])
            want = np.zeros((B, B))
            blk = ref["P"][:, bj * B:(bj + 1) * B]
            want[:blk.shape[0], :blk.shape[1]] = blk
            ulp = np.where(want > 0, 2.0 ** (np.floor(np.log2(np.maximum(want, 1e-300))) - 7), 0)
            assert (np.abs(tile - want) <= ulp + 1e-37).all(), f"tile (h={h}, rb={rb}, bj={bj})"
            n_tiles += 1
    return n_tiles


def check_output(O_gpu: np.ndarray, q64, k64, grid: orc.BlockGrid, ex, H_s: int, W: np.ndarray,
                 v64: np.ndarray, H_kv: int, block_rows: Iterable[int]) -> float:
    """O of the sampled block-rows against the oracle's dense reconstruction
    with the kept sets of the (verified) BSR.  Returns max |err| / max |O|."""
    def kept_of(h, rb):
        r = h * grid.R + rb
        return [int(x) for x in ex["col_idx"][ex["row_ptr"][r]:ex["row_ptr"][r + 1]]]
    worst = 0.0
    refs, gots = [], []
    for rb in block_rows:
        ref, rows = orc.retrieve_block_row(q64, k64, grid, kept_of, W.astype(np.float64), v64,
                                           H_kv, rb)
        refs.append(ref)
        gots.append(O_gpu[rows].astype(np.float64))
    ref = np.concatenate(refs)
    got = np.concatenate(gots)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    assert np.isfinite(got).all()
    assert err <= O_TOL * scale, f"O err {err} > {O_TOL} * {scale}"
    return err / max(scale, 1e-300)


def run_compress(bsr: mapflow.BSR, layer: int, x: Dict[str, np.ndarray], dtype: str, p: float):
    q = to_dev(x["q"], dtype)
    k = to_dev(x["k"], dtype)
    bsr.compress(layer, q, k, p)
    return q, k


def run_retrieve(bsr: mapflow.BSR, W: np.ndarray, v: np.ndarray, H_r: int, dtype: str,
                 layer_map: Sequence[int]) -> np.ndarray:
    """v: [n, T, H_kv, d] stored values, W: [n, H_r, H_s]."""
    n, T, H_kv, d = v.shape
    vt = torch.stack([to_dev(v[i], dtype) for i in range(n)])
    Wt = torch.from_numpy(np.ascontiguousarray(W, np.float32)).to(dev())
    o = torch.full((n, T, H_r, d), float("nan"), dtype=vt.dtype, device=dev())
    bsr.retrieve(Wt, vt, o, layer_map)
    bsr.device_status()
    return o.float().cpu().numpy()


def sample_block_rows(grid: orc.BlockGrid, n: int, seed: int) -> List[int]:
    rng = np.random.default_rng(seed)
    pick = {0, grid.R - 1}
    # the last block-row of every sequence (ragged tails) and a few random ones
    for s in range(grid.n_seqs):
        pick.add(int(grid.rb_base[s + 1]) - 1)
    pick.update(int(x) for x in rng.choice(grid.R, size=min(n, grid.R), replace=False))
    return sorted(pick)
