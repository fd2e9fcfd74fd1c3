"""GPU parity: the CUDA path (through the C-ABI) against the fp64 oracle.

Small cases span several tiles, ragged tails, packed sequences, GQA, odd
heads-per-group, both block sizes and head dims, non-causal attention, p = 1
and a p so small that no block is kept.  Full-size cases run each workload at
its real sequence length and head counts (one sender layer) and compare
sampled block-rows with the oracle; the selection is always checked on every
row.
"""
import math

import numpy as np
import pytest
import torch

from cross_model_attention_gb300 import mapflow, synth, workloads
from oracle import mapflow_oracle as orc
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    gc.dev()


def small_case(seqlens, Hs, Hks, d, B, p, Hr, Hkv, dtype="bf16", causal=True, seed=0,
               structured=True, n_rlayers=1):
    T = int(sum(seqlens))
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    if structured:
        w = workloads.scaled(workloads.get(1), seqlens, sender_heads=Hs, sender_kv_heads=Hks,
                             d=d, B=B, dtype=dtype, causal=causal, seed=seed)
        x = synth.sender_qk(w, 1)
    else:
        x = synth.random_qk(T, Hs, Hks, d, seed, dtype=dtype)
    vs = [synth.random_v(T, Hkv, d, seed + 10 + j, dtype=dtype) for j in range(n_rlayers)]
    W = np.stack([synth.random_w(Hr, Hs, seed + 20 + j) for j in range(n_rlayers)])
    bsr = mapflow.BSR(1, T, Hs, B, cu, causal=causal)
    gc.run_compress(bsr, 0, x, dtype, p)
    ex = gc.export_np(bsr, 0)
    grid = orc.BlockGrid(cu, B, causal)
    gc.check_structure(ex, grid, Hs, p)
    pairs = [(h, rb) for h in range(Hs) for rb in range(grid.R)]
    gc.check_block_rows(ex, x["q64"], x["k64"], grid, Hs, pairs)
    O = gc.run_retrieve(bsr, W, np.stack([v["v"] for v in vs]), Hr, dtype, [0] * n_rlayers)
    for j in range(n_rlayers):
        gc.check_output(O[j], x["q64"], x["k64"], grid, ex, Hs, W[j], vs[j]["v64"], Hkv,
                        range(grid.R))
    bsr.close()
    return ex


@pytest.mark.parametrize("seqlens,Hs,Hks,d,B,Hr,Hkv", [
    ((512,), 4, 4, 128, 64, 8, 2),            # several tiles, hpg 4
    ((200, 137, 64, 1, 130), 4, 2, 128, 64, 6, 2),  # varlen, ragged, GQA, hpg 3
    ((300, 129), 3, 3, 128, 128, 8, 2),       # B = 128, ragged
    ((333,), 2, 1, 64, 64, 4, 4),             # d = 64, hpg 1
    ((257, 64), 2, 2, 64, 128, 16, 2),        # d = 64, B = 128, hpg 8
    # 8 receiver KV heads: the cluster retrieval
    ((512,), 8, 8, 128, 64, 32, 8),           # 4 heads per group
    ((200, 137, 64, 1, 130), 8, 4, 128, 64, 24, 8),  # varlen, ragged, GQA sender, 3 per group
    ((300, 129), 6, 6, 128, 128, 16, 8),      # B = 128, 2 per group
    ((333,), 3, 3, 64, 64, 8, 8),             # d = 64, 1 per group
    ((257, 64), 20, 20, 64, 128, 32, 8),      # d = 64, B = 128, padded sender heads
    ((256,), 64, 64, 128, 64, 32, 8),         # 64 sender heads (one V stage)
])
def test_small_bf16(seqlens, Hs, Hks, d, B, Hr, Hkv):
    small_case(seqlens, Hs, Hks, d, B, 0.95, Hr, Hkv)


def test_noncausal():
    small_case((190, 70), 2, 2, 128, 64, 0.9, 4, 2, causal=False, structured=False)
    small_case((190, 70), 4, 4, 128, 64, 0.9, 16, 8, causal=False, structured=False)


def test_p1_keeps_every_block_with_mass():
    ex = small_case((384,), 2, 2, 128, 64, 1.0, 4, 2)
    # every causal candidate with non-zero fixed-point mass is kept
    assert ex["row_ptr"][-1] > 0


def test_nothing_kept_gives_zero_output():
    # p * 2^20 rounds to 0: the threshold is 0, no block is needed
    seqlens = (256,)
    T = 256
    x = synth.random_qk(T, 2, 2, 128, 3)
    v = synth.random_v(T, 2, 128, 4)
    W = synth.random_w(4, 2, 5)[None]
    bsr = mapflow.BSR(1, T, 2, 64, [0, T])
    gc.run_compress(bsr, 0, x, "bf16", 2e-7)
    ex = gc.export_np(bsr, 0)
    assert ex["row_ptr"][-1] == 0
    O = gc.run_retrieve(bsr, W, v["v"][None], 4, "bf16", [0])
    assert np.all(O == 0.0)
    bsr.close()


def test_unstructured_random_logits():
    small_case((448,), 3, 3, 128, 64, 0.9, 6, 3, structured=False, seed=7)


def test_extreme_logits():
    """Scores far outside the usual range: a row's first key block sits near
    -90 (natural units, about -130 in log2 units) and, for rows past it, the
    next block near +90, so the statistics kernels must take a row's first
    block against its own max and later re-reference across a gap no sum of
    exp2 terms could span.  Every product and sum of q.k is an exact fp32
    integer (one large dimension, one of small integers), so the oracle's
    fp64 scores are the kernel's scores."""
    T, Hs, d, B, p = 384, 2, 64, 64, 0.9
    rng = np.random.default_rng(11)
    q = np.zeros((T, Hs, d), np.float32)
    k = np.zeros((T, Hs, d), np.float32)
    q[:, :, 0] = 8.0
    q[:, :, 1] = 1.0
    k[:64, :, 0] = -90.0
    k[64:128, :, 0] = 90.0
    k[:, :, 1] = rng.integers(-8, 9, size=(T, Hs)).astype(np.float32)
    qb, kb = synth.bf16_round(q), synth.bf16_round(k)
    x = {"q": qb, "k": kb, "q64": synth.bf16_to_f64(qb), "k64": synth.bf16_to_f64(kb)}
    cu = np.array([0, T], np.int32)
    bsr = mapflow.BSR(1, T, Hs, B, cu)
    gc.run_compress(bsr, 0, x, "bf16", p)
    ex = gc.export_np(bsr, 0)
    grid = orc.BlockGrid(cu, B, True)
    gc.check_structure(ex, grid, Hs, p)
    gc.check_block_rows(ex, x["q64"], x["k64"], grid, Hs, [(h, rb) for h in range(Hs) for rb in range(grid.R)])
    v = synth.random_v(T, 2, d, 5)
    W = synth.random_w(4, Hs, 6)
    O = gc.run_retrieve(bsr, W[None], v["v"][None], 4, "bf16", [0])
    gc.check_output(O[0], x["q64"], x["k64"], grid, ex, Hs, W, v["v64"], 2, range(grid.R))
    bsr.close()


@pytest.mark.parametrize("L", [8192, 8193])
def test_statistics_kernel_boundary(L):
    """8192 tokens at B = 64 give rows of 128 candidate blocks (the statistics
    kernel with two CTAs per SM); 8193 give 129 (the one-CTA kernel).  Sampled
    block-rows, the full selection and the retrieval against the oracle."""
    Hs, d, B, p = 2, 64, 64, 0.95
    x = synth.random_qk(L, Hs, Hs, d, 3)
    cu = np.array([0, L], np.int32)
    bsr = mapflow.BSR(1, L, Hs, B, cu)
    gc.run_compress(bsr, 0, x, "bf16", p)
    ex = gc.export_np(bsr, 0)
    grid = orc.BlockGrid(cu, B, True)
    gc.check_structure(ex, grid, Hs, p)
    rows = [0, 1, grid.R // 2, grid.R - 2, grid.R - 1]
    gc.check_block_rows(ex, x["q64"], x["k64"], grid, Hs, [(h, rb) for h in range(Hs) for rb in rows])
    v = synth.random_v(L, 8, d, 4)
    W = synth.random_w(16, Hs, 5)
    O = gc.run_retrieve(bsr, W[None], v["v"][None], 16, "bf16", [0])
    gc.check_output(O[0], x["q64"], x["k64"], grid, ex, Hs, W, v["v64"], 8, rows)
    bsr.close()


def test_fp32_workload0():
    """The fp32 workload exactly: N=512, H_s=4, d=64, B=64, p=0.95, W = I + N(0,1/4)."""
    w = workloads.get(0)
    x = synth.sender_qk(w, 1)
    rcv = w.receivers[0]
    v = synth.receiver_v(w, rcv, 1)
    W = synth.head_map_weights(w, rcv, 1)
    bsr = mapflow.BSR(1, w.T, w.sender_heads, w.B, w.cu_seqlens)
    gc.run_compress(bsr, 0, x, "f32", w.p[0])
    ex = gc.export_np(bsr, 0)
    grid = orc.BlockGrid(w.cu_seqlens, w.B, True)
    gc.check_structure(ex, grid, w.sender_heads, w.p[0])
    gc.check_block_rows(ex, x["q64"], x["k64"], grid, w.sender_heads,
                        [(h, rb) for h in range(4) for rb in range(grid.R)])
    O = gc.run_retrieve(bsr, W[None], v["v"][None], rcv.heads, "f32", [0])
    gc.check_output(O[0], x["q64"], x["k64"], grid, ex, 4, W, v["v64"], rcv.kv_heads,
                    range(grid.R))
    bsr.close()


def test_multi_layer_map_and_determinism():
    seqlens = (320, 200)
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    w = workloads.scaled(workloads.get(1), seqlens, sender_heads=4, sender_kv_heads=4)
    xs = [synth.sender_qk(w, l) for l in (1, 2)]
    bsr = mapflow.BSR(2, T, 4, 64, cu)
    for l in range(2):
        gc.run_compress(bsr, l, xs[l], "bf16", 0.9)
    ex0 = gc.export_np(bsr, 0)
    # recompress layer 0: bit-identical BSR
    gc.run_compress(bsr, 0, xs[0], "bf16", 0.9)
    ex0b = gc.export_np(bsr, 0)
    for key in ("row_ptr", "col_idx", "mass", "row_max", "row_sum"):
        assert np.array_equal(ex0[key], ex0b[key]), key
    assert torch.equal(ex0["values_dev"].view(torch.int16), ex0b["values_dev"].view(torch.int16))
    ex1 = gc.export_np(bsr, 1)
    vs = [synth.random_v(T, 2, 128, 40 + j) for j in range(3)]
    W = np.stack([synth.random_w(8, 4, 50 + j) for j in range(3)])
    lm = [1, 0, 1]
    O = gc.run_retrieve(bsr, W, np.stack([v["v"] for v in vs]), 8, "bf16", lm)
    grid = orc.BlockGrid(cu, 64, True)
    for j, l in enumerate(lm):
        gc.check_output(O[j], xs[l]["q64"], xs[l]["k64"], grid, (ex0, ex1)[l], 4, W[j],
                        vs[j]["v64"], 2, range(grid.R))
    bsr.close()


def test_device_wait_timeout_is_reported():
    """A bounded device wait that nothing completes returns MF_ERR_TIMEOUT
    through the error word; the context stays usable."""
    bsr = mapflow.BSR(1, 64, 1, 64, [0, 64])
    mapflow.mf_selftest_wait(bsr.handle, 50)
    with pytest.raises(mapflow.MapFlowError) as ei:
        bsr.device_status()
    assert ei.value.code == mapflow.MF_ERR_TIMEOUT
    bsr.device_status()  # cleared
    small_case((128,), 1, 1, 64, 64, 0.9, 1, 1)  # the context still works
    bsr.close()


def test_retrieve_before_compress_is_rejected():
    bsr = mapflow.BSR(1, 64, 1, 64, [0, 64])
    W = torch.zeros((1, 1, 1), device=gc.dev())
    v = torch.zeros((1, 64, 1, 64), dtype=torch.bfloat16, device=gc.dev())
    o = torch.zeros((1, 64, 1, 64), dtype=torch.bfloat16, device=gc.dev())
    with pytest.raises(mapflow.MapFlowError) as ei:
        bsr.retrieve(W, v, o, [0])
    assert ei.value.code == mapflow.MF_ERR_STATE
    bsr.close()


# ---------------------------------------------------------------- full size --

def full_size(idx, p=None, sender_layer=None, n_rows=4, receivers=None):
    """One sender layer of workload idx at its full size: the selection on
    every row; masses, row statistics and tiles of one random head on the
    sampled block-rows; and O of every receiver on all the sampled
    block-rows (block-row 0, the last block-row of every sequence, which is
    the longest row of its sequence, and n_rows random ones)."""
    w = workloads.get(idx)
    p = w.p[0] if p is None else p
    rcvs = w.receivers if receivers is None else receivers
    layer = sender_layer or rcvs[0].layer_map(w.sender_layers)[0][1]
    x = synth.sender_qk(w, layer)
    bsr = mapflow.BSR(1, w.T, w.sender_heads, w.B, w.cu_seqlens)
    gc.run_compress(bsr, 0, x, w.dtype, p)
    ex = gc.export_np(bsr, 0)
    grid = orc.BlockGrid(w.cu_seqlens, w.B, True)
    gc.check_structure(ex, grid, w.sender_heads, p)
    rbs = gc.sample_block_rows(grid, n_rows, 100 + idx)
    rng = np.random.default_rng(idx)
    pairs = [(int(rng.integers(w.sender_heads)), rb) for rb in rbs]
    gc.check_block_rows(ex, x["q64"], x["k64"], grid, w.sender_heads, pairs)
    res = {"kept_frac": ex["row_ptr"][-1] / (w.sender_heads * grid.C)}
    for rcv in rcvs:
        j = next(jj for jj, m in rcv.layer_map(w.sender_layers) if m == layer) \
            if any(m == layer for _, m in rcv.layer_map(w.sender_layers)) else rcv.recompute + 1
        v = synth.receiver_v(w, rcv, j)
        W = synth.head_map_weights(w, rcv, j)
        O = gc.run_retrieve(bsr, W[None], v["v"][None], rcv.heads, w.dtype, [0])
        res[rcv.name] = gc.check_output(O[0], x["q64"], x["k64"], grid, ex, w.sender_heads, W,
                                        v["v64"], rcv.kv_heads, rbs)
        del O
    bsr.close()
    torch.cuda.empty_cache()
    return res


def test_full_workload1():
    full_size(1)


def test_full_workload2():
    full_size(2)


@pytest.mark.parametrize("p", [0.80, 0.90, 0.95, 0.99])
def test_full_workload3(p):
    full_size(3, p=p, n_rows=2)


def test_full_workload4_two_receivers():
    full_size(4)


def test_offload_and_prefetch_roundtrip():
    """A layer moved to host memory and brought back on another stream gives
    the same BSR and the same retrieval output; while offloaded the
    retrieval rejects it.  The prefetch shrinks the tile buffer to the kept
    tiles (the zero tile moves to index nnz), which the retrieval must follow."""
    seqlens = (700, 333)
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    w = workloads.scaled(workloads.get(1), seqlens, sender_heads=8, sender_kv_heads=8)
    x = synth.sender_qk(w, 1)
    v = synth.random_v(T, 8, 128, 3)["v"][None]
    W = synth.random_w(32, 8, 4)[None]
    bsr = mapflow.BSR(2, T, 8, 64, cu)
    gc.run_compress(bsr, 0, x, "bf16", 0.95)
    gc.run_compress(bsr, 1, x, "bf16", 0.80)
    before = gc.export_np(bsr, 0)
    O_before = gc.run_retrieve(bsr, W, v, 32, "bf16", [0])
    bsr.offload(0)
    with pytest.raises(mapflow.MapFlowError) as ei:
        gc.run_retrieve(bsr, W, v, 32, "bf16", [0])
    assert ei.value.code == mapflow.MF_ERR_STATE
    O_other = gc.run_retrieve(bsr, W, v, 32, "bf16", [1])  # the other layer is untouched
    side = torch.cuda.Stream()
    bsr.prefetch(0, stream=side)
    O_after = gc.run_retrieve(bsr, W, v, 32, "bf16", [0])  # waits for the prefetch itself
    after = gc.export_np(bsr, 0)
    for key in ("row_ptr", "col_idx", "mass", "row_max", "row_sum"):
        assert np.array_equal(before[key], after[key]), key
    assert torch.equal(before["values_dev"], after["values_dev"])
    assert np.array_equal(O_before, O_after)
    # and the layer that came back is the oracle's: structure, masses, row
    # statistics and tiles of every (head, block-row), O of every block-row
    grid = orc.BlockGrid(cu, 64, True)
    gc.check_structure(after, grid, 8, 0.95)
    gc.check_block_rows(after, x["q64"], x["k64"], grid, 8,
                        [(h, rb) for h in range(8) for rb in range(grid.R)])
    gc.check_output(O_after[0], x["q64"], x["k64"], grid, after, 8, W[0].astype(np.float64),
                    synth.bf16_to_f64(v[0]), 8, range(grid.R))
    assert not np.array_equal(O_other, O_after)
    bsr.offload(0)
    bsr.offload(0)  # a no-op when already offloaded
    gc.run_compress(bsr, 0, x, "bf16", 0.95)  # recompressing an offloaded layer replaces it
    assert np.array_equal(gc.run_retrieve(bsr, W, v, 32, "bf16", [0]), O_before)
    bsr.close()


def test_exact_and_bound_allocation_agree():
    """mf_compress sized exactly (one sync) and at the upper bound (no sync)
    produce the same BSR and the same retrieval output."""
    seqlens = (700, 333)
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    w = workloads.scaled(workloads.get(1), seqlens, sender_heads=8, sender_kv_heads=8)
    x = synth.sender_qk(w, 1)
    v = synth.random_v(T, 8, 128, 3)["v"][None]
    W = synth.random_w(32, 8, 4)[None]
    outs = []
    for exact in (True, False):
        bsr = mapflow.BSR(1, T, 8, 64, cu)
        bsr.set_exact(exact)
        gc.run_compress(bsr, 0, x, "bf16", 0.9)
        ex = gc.export_np(bsr, 0)
        O = gc.run_retrieve(bsr, W, v, 32, "bf16", [0])
        outs.append((ex, O))
        bsr.close()
    (a, Oa), (b, Ob) = outs
    for key in ("row_ptr", "col_idx", "mass", "row_max", "row_sum"):
        assert np.array_equal(a[key], b[key]), key
    assert torch.equal(a["values_dev"].view(torch.int16), b["values_dev"].view(torch.int16))
    assert np.array_equal(Oa, Ob)


def _kept_of(ex, R):
    rp, ci = ex["row_ptr"], ex["col_idx"]
    return lambda h, rb: ci[rp[h * R + rb]:rp[h * R + rb + 1]]


def _calib_bound(W_gpu, W_or, S, Rm, ridge):
    """Both sides minimise J(W) = |R - W S|^2 + ridge |W|^2, the GPU on the
    maps as stored (each entry within 2^-9 relative of the exact one after
    the bf16 rounding; eps = 2^-8 leaves room for the fp32 softmax and Gram
    sums).  sqrt(J) moves by at most eps (|R| + |W|_2 |S|) under that
    perturbation, so the GPU's W can exceed the exact minimum by at most
    eps (2 |R| + (|W_gpu|_2 + |W_or|_2) |S|)."""
    eps = 2.0 ** -8

    def sqrtJ(W):
        return math.sqrt(np.sum((Rm - W @ S) ** 2) + ridge * np.sum(W ** 2))

    slack = eps * (2 * np.linalg.norm(Rm) + (np.linalg.norm(W_gpu, 2) + np.linalg.norm(W_or, 2))
                   * np.linalg.norm(S))
    assert sqrtJ(W_or) <= sqrtJ(W_gpu) * (1 + 1e-9) + 1e-12, "the oracle is not the minimum"
    assert sqrtJ(W_gpu) <= sqrtJ(W_or) + slack, (sqrtJ(W_gpu), sqrtJ(W_or), slack)
    return sqrtJ(W_gpu), sqrtJ(W_or), slack


@pytest.mark.parametrize("ridge", [0.0, 2.0])
def test_calibrate_head_map_against_oracle(ridge):
    """W fitted from a sender layer (p = 0.9) and another layer's maps
    compressed with p = 1 against the oracle's fp64 least squares on the same
    kept blocks."""
    seqlens, B, Hs, Hr = (300, 129, 64), 64, 6, 5
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    grid = orc.BlockGrid(cu, B, True)
    ws = workloads.scaled(workloads.get(1), seqlens, sender_heads=Hs, sender_kv_heads=3)
    wr = workloads.scaled(workloads.get(1), seqlens, sender_heads=Hr, sender_kv_heads=Hr, seed=7)
    xs, xr = synth.sender_qk(ws, 1), synth.sender_qk(wr, 2)
    sb, rbh = mapflow.BSR(1, T, Hs, B, cu), mapflow.BSR(1, T, Hr, B, cu)
    gc.run_compress(sb, 0, xs, "bf16", 0.9)
    gc.run_compress(rbh, 0, xr, "bf16", 1.0)
    es, er = gc.export_np(sb, 0), gc.export_np(rbh, 0)
    gc.check_structure(es, grid, Hs, 0.9)
    gc.check_structure(er, grid, Hr, 1.0)
    W_gpu = mapflow.calibrate_head_map(sb, 0, rbh, 0, ridge=ridge).astype(np.float64)
    S = orc.map_entries(xs["q64"], xs["k64"], grid, _kept_of(es, grid.R))
    Rm = orc.map_entries(xr["q64"], xr["k64"], grid, _kept_of(er, grid.R))
    W_or = orc.calibrate_head_map(S, Rm, ridge)
    assert W_gpu.shape == (Hr, Hs)
    _calib_bound(W_gpu, W_or, S, Rm, ridge)
    sb.close()
    rbh.close()


def test_calibrate_head_map_recovers_a_head_selection():
    """Receiver heads that are copies of sender heads (same Q/K, same p, so
    bitwise the same stored maps): W is the 0/1 selection matrix, which pins
    the [H_r][H_s] layout and the head indexing.  The sender against itself
    gives the identity."""
    seqlens, B, Hs = (257, 64, 130), 64, 6
    pick = [4, 0, 5, 2]
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    ws = workloads.scaled(workloads.get(1), seqlens, sender_heads=Hs, sender_kv_heads=Hs)
    xs = synth.sender_qk(ws, 3)
    xr = {k: np.ascontiguousarray(v[:, pick]) for k, v in xs.items()}
    sb, rbh = mapflow.BSR(1, T, Hs, B, cu), mapflow.BSR(1, T, len(pick), B, cu)
    gc.run_compress(sb, 0, xs, "bf16", 0.9)
    gc.run_compress(rbh, 0, xr, "bf16", 0.9)
    sel = np.zeros((len(pick), Hs))
    sel[np.arange(len(pick)), pick] = 1.0
    W = mapflow.calibrate_head_map(sb, 0, rbh, 0)
    assert np.abs(W - sel).max() < 1e-4, W
    I = mapflow.calibrate_head_map(sb, 0, sb, 0)
    assert np.abs(I - np.eye(Hs)).max() < 1e-4, I
    sb.close()
    rbh.close()


def test_calibrate_head_map_rejects_bad_arguments():
    cu = np.array([0, 200], np.int32)
    a = mapflow.BSR(1, 200, 64, 64, cu)
    b = mapflow.BSR(1, 200, 64, 64, cu)
    c = mapflow.BSR(1, 200, 4, 64, np.array([0, 100, 200], np.int32))
    d = mapflow.BSR(1, 200, 4, 64, cu)
    with pytest.raises(mapflow.MapFlowError) as ei:
        mapflow.calibrate_head_map(a, 0, b, 0)  # 128 rows
    assert ei.value.code == mapflow.MF_ERR_UNSUPPORTED
    with pytest.raises(mapflow.MapFlowError) as ei:
        mapflow.calibrate_head_map(c, 0, d, 0)  # other sequences
    assert ei.value.code == mapflow.MF_ERR_ARG
    with pytest.raises(mapflow.MapFlowError) as ei:
        mapflow.calibrate_head_map(d, 0, d, 0)  # not compressed
    assert ei.value.code == mapflow.MF_ERR_STATE
    for h in (a, b, c, d):
        h.close()
