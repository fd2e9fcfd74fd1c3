"""The no-allocation selection entry point (mf_select_noalloc).

It serves callers that cannot allocate device memory when they select: an
engine that has reserved nearly all memory up front, or a latency-critical
loop that cannot pay for cudaFree's device synchronisation.  Its
intermediates live in one static device array shared by every call, so the
test calls it twice in a row (with outputs poisoned in between) and checks
both results, bit for bit, against the structure that the allocating entry
point mf_compress produced for the same masses, and against the oracle's
selection rule evaluated on those masses.

This file is named so that pytest collects it last.
"""
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
    assert torch.cuda.is_available(), "GPU test selected on a machine without a GPU"


def _compressed(seqlens, Hs, B, p, seed, causal):
    dev = torch.device("cuda", 0)
    w = workloads.scaled(workloads.get(1), seqlens, sender_heads=Hs, sender_kv_heads=Hs, B=B,
                         seed=seed, causal=causal)
    x = synth.sender_qk(w, 1)
    bf = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    bsr = mapflow.BSR(1, w.T, Hs, B, w.cu_seqlens, causal=causal)
    bsr.compress(0, bf(x["q"]), bf(x["k"]), p)
    ex = bsr.export(0)
    torch.cuda.synchronize()
    bsr.close()
    return w, ex


@pytest.mark.parametrize("seqlens,Hs,B,p,causal", [
    ((1024, 333, 700), 8, 64, 0.95, True),
    ((2048, 129), 4, 128, 0.8, True),
    ((1024, 333), 4, 64, 0.9, False),
])
def test_noalloc_matches_compress_twice(seqlens, Hs, B, p, causal):
    w, ex = _compressed(seqlens, Hs, B, p, 11, causal)
    dev = ex["mass"].device
    n_rows = ex["row_ptr"].numel() - 1
    cap = ex["mass"].numel()
    for call in range(2):
        row_ptr = torch.full((n_rows + 1,), -7, dtype=torch.int32, device=dev)
        col_idx = torch.full((cap,), -7, dtype=torch.int32, device=dev)
        nnz = torch.full((1,), -7, dtype=torch.int64, device=dev)
        mapflow.mf_select_noalloc(ex["mass"], w.cu_seqlens, Hs, B, causal, p, row_ptr, col_idx,
                                  nnz)
        torch.cuda.synchronize()
        n = int(nnz.item())
        assert n == ex["col_idx"].numel(), f"call {call}: nnz {n}"
        assert torch.equal(row_ptr, ex["row_ptr"]), f"call {call}: row_ptr differs"
        assert torch.equal(col_idx[:n], ex["col_idx"]), f"call {call}: col_idx differs"
        # the oracle's selection rule on the same masses, row by row
        got = {"mass": ex["mass"].cpu().numpy(), "row_ptr": row_ptr.cpu().numpy(),
               "col_idx": col_idx[:n].cpu().numpy()}
        gc.check_structure(got, orc.BlockGrid(w.cu_seqlens, B, causal), Hs, p)


def test_noalloc_rejects_oversized_problem():
    dev = torch.device("cuda", 0)
    cu = [0, 16384]
    Hs = 128  # 128 heads x 32896 candidates x 4 B > 16 MiB of scratch
    mass = torch.zeros(Hs * 32896, dtype=torch.float32, device=dev)
    row_ptr = torch.zeros(Hs * 256 + 1, dtype=torch.int32, device=dev)
    col_idx = torch.zeros(Hs * 32896, dtype=torch.int32, device=dev)
    nnz = torch.zeros(1, dtype=torch.int64, device=dev)
    with pytest.raises(mapflow.MapFlowError) as ei:
        mapflow.mf_select_noalloc(mass, cu, Hs, 64, True, 0.9, row_ptr, col_idx, nnz)
    assert ei.value.code == mapflow.MF_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)


def test_noalloc_wrapper_rejects_short_buffers():
    """The binding checks every buffer against the sizes the call implies
    (H_s*C masses, H_s*R+1 row offsets, one nnz word) before the library
    sees a pointer, so no kernel can run past a caller's buffer."""
    dev = torch.device("cuda", 0)
    cu, Hs, B = [0, 200], 2, 64  # R = 4 block-rows, C = 10 causal candidates
    ok = dict(mass=torch.zeros(Hs * 10, device=dev),
              row_ptr=torch.zeros(Hs * 4 + 1, dtype=torch.int32, device=dev),
              col_idx=torch.zeros(Hs * 10, dtype=torch.int32, device=dev),
              nnz=torch.zeros(1, dtype=torch.int64, device=dev))
    bad = [("mass", torch.zeros(Hs * 10 - 1, device=dev)),
           ("row_ptr", torch.zeros(Hs * 4, dtype=torch.int32, device=dev)),
           ("nnz", torch.zeros(0, dtype=torch.int64, device=dev)),
           ("mass", torch.zeros(Hs * 10, dtype=torch.float64, device=dev)),
           ("row_ptr", torch.zeros(Hs * 4 + 1, dtype=torch.int32))]
    for name, t in bad:
        args = dict(ok, **{name: t})
        with pytest.raises(mapflow.MapFlowError) as ei:
            mapflow.mf_select_noalloc(args["mass"], cu, Hs, B, True, 0.9, args["row_ptr"],
                                      args["col_idx"], args["nnz"])
        assert ei.value.code == mapflow.MF_ERR_ARG, name
