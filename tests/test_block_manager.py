"""Block manager and chunked prefill: prefix hashes (host, no GPU), block-row
states cached under them and assembled into BSR views that the retrieval
reads, and handles whose query rows are a chunk over a prefix (GPU).

Reading tested here: under a causal mask block-row bi of a sequence depends
only on the tokens of blocks 0..bi, so two requests that share a prefix share
the compressed states of its full blocks, a view assembled from cached
block-rows retrieves exactly what the request's own compressed BSR does, and
a chunk's block-rows are exactly the full sequence's block-rows from the
chunk's start on."""
import numpy as np
import pytest

from cross_model_attention_gb300 import build as build_mod
from cross_model_attention_gb300 import mapflow, synth, workloads
from oracle import mapflow_oracle as orc
from tests import gpu_cases as gc

B = 64


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return mapflow.load_library()


def _tokens(n, seed):
    return np.random.default_rng([seed, 5150]).integers(0, 32000, size=n).astype(np.int32)


# ------------------------------------------------------------ host only --
def test_prefix_hashes_follow_the_prefix(lib):
    P = _tokens(3 * B, 1)
    a = np.concatenate([P, _tokens(100, 2)])
    b = np.concatenate([P, _tokens(2 * B, 3)])
    ha = mapflow.mf_prefix_hashes(a, [0, len(a)], B)
    hb = mapflow.mf_prefix_hashes(b, [0, len(b)], B)
    assert len(ha) == 5 and len(hb) == 5
    assert np.array_equal(ha[:3], hb[:3])          # shared full blocks
    assert not np.isin(ha[3:], hb).any()           # different continuations
    # a change in block 1 changes every later hash (the chain), not block 0
    c = a.copy()
    c[B + 5] += 1
    hc = mapflow.mf_prefix_hashes(c, [0, len(c)], B)
    assert hc[0] == ha[0] and not np.isin(hc[1:], ha).any()
    # packing: a sequence's hashes do not depend on its place in the batch
    packed = np.concatenate([b, a])
    hp = mapflow.mf_prefix_hashes(packed, [0, len(b), len(b) + len(a)], B)
    assert np.array_equal(hp, np.concatenate([hb, ha]))
    # seeds separate namespaces
    assert not np.isin(mapflow.mf_prefix_hashes(a, [0, len(a)], B, seed=7), ha).any()


def test_prefix_hashes_ragged_block_is_not_a_full_block(lib):
    a = _tokens(2 * B, 4)
    short = a[:B + 10]
    ha = mapflow.mf_prefix_hashes(a, [0, len(a)], B)
    hs = mapflow.mf_prefix_hashes(short, [0, len(short)], B)
    assert hs[0] == ha[0]
    assert hs[1] != ha[1]  # 10 tokens of block 1 vs all 64
    # and the same 10 tokens as a separate ragged block match themselves
    assert mapflow.mf_prefix_hashes(short, [0, len(short)], B)[1] == hs[1]
    # empty sequences have no block-rows; the size query answers alone
    h = mapflow.mf_prefix_hashes(a, [0, 0, len(a), len(a)], B)
    assert np.array_equal(h, ha)


def test_prefix_hashes_of_a_chunk_continue_the_chain(lib):
    a, b = _tokens(700, 6), _tokens(333, 7)
    cu = [0, 700, 1033]
    full = mapflow.mf_prefix_hashes(np.concatenate([a, b]), cu, B)
    chunk = mapflow.mf_prefix_hashes(np.concatenate([a, b]), cu, B, q_begin=[384, 128])
    nb_a = (700 + B - 1) // B
    assert np.array_equal(chunk, np.concatenate([full[384 // B:nb_a], full[nb_a + 128 // B:]]))
    with pytest.raises(mapflow.MapFlowError):
        mapflow.mf_prefix_hashes(a, [0, 700], B, q_begin=[100])  # not a block start
    # a chunk that starts at a ragged end is empty
    assert len(mapflow.mf_prefix_hashes(np.concatenate([a, b]), cu, B, q_begin=[700, 0])) == 6


def test_chunked_handle_rejects_bad_chunks(lib):
    cu = [0, 700, 1033]
    for qb, causal in (([100, 0], True), ([768, 0], True), ([700, 333], True), ([128, 0], False)):
        with pytest.raises(mapflow.MapFlowError) as ei:
            mapflow.BSR(1, 1033, 8, B, cu, causal=causal, q_begin=qb)
        assert ei.value.code in (mapflow.MF_ERR_ARG, mapflow.MF_ERR_UNSUPPORTED)


# ------------------------------------------------------------------ GPU --
def _request(prefix_len, suffix_len, seed, x_prefix=None, tok_prefix=None, Hs=8):
    """Synthetic sender Q/K and token ids of one request; the prefix rows are
    taken from another request's when given (the shared context)."""
    T = prefix_len + suffix_len
    w = workloads.scaled(workloads.get(1), (T,), sender_heads=Hs, sender_kv_heads=Hs, seed=seed)
    x = synth.sender_qk(w, 1)
    tok = _tokens(T, seed)
    if x_prefix is not None:
        for key in x:
            x[key][:prefix_len] = x_prefix[key][:prefix_len]
        tok[:prefix_len] = tok_prefix[:prefix_len]
    return x, tok


def _retrieve_both(bsr, T, Hs, seed):
    """Retrieval through the team kernel (8 KV groups) and the per-group
    kernel (2 KV groups)."""
    outs = []
    for Hr, Hkv in ((32, 8), (8, 2)):
        v = synth.random_v(T, Hkv, 128, seed + Hkv)["v"][None]
        W = synth.random_w(Hr, Hs, seed + Hr)[None]
        outs.append(gc.run_retrieve(bsr, W, v, Hr, "bf16", [0]))
    return outs


@pytest.mark.gpu
def test_shared_prefix_view_equals_own_compression(lib):
    gc.dev()
    Hs, LP = 8, 4 * B
    xa, ta = _request(LP, 200, 11)
    xb, tb = _request(LP, 150, 12, xa, ta)
    Ta, Tb = len(ta), len(tb)
    ha = mapflow.mf_prefix_hashes(ta, [0, Ta], B)
    hb = mapflow.mf_prefix_hashes(tb, [0, Tb], B)
    A = mapflow.BSR(1, Ta, Hs, B, [0, Ta])
    Bh = mapflow.BSR(1, Tb, Hs, B, [0, Tb])
    gc.run_compress(A, 0, xa, "bf16", 0.9)
    gc.run_compress(Bh, 0, xb, "bf16", 0.9)
    bm = mapflow.BlockManager(Hs, B, 4096)
    assert bm.insert(0, A, 0, ha) == (len(ha), 0, 0)
    assert bm.match(0, hb) == LP // B
    assert bm.match(1, hb) == 0  # another layer key
    ins, found, ev = bm.insert(0, Bh, 0, hb)
    assert (ins, found, ev) == (len(hb) - LP // B, LP // B, 0)
    st = bm.stats()
    assert st["entries"] == len(ha) + len(hb) - LP // B
    # B's view: its prefix block-rows come from A's compression
    V = mapflow.BSR(1, Tb, Hs, B, [0, Tb])
    bm.assemble(0, hb, V, 0)
    assert bm.stats()["pinned"] == len(hb)
    own = _retrieve_both(Bh, Tb, Hs, 3)
    view = _retrieve_both(V, Tb, Hs, 3)
    for o, v in zip(own, view):
        assert np.array_equal(o, v)
    # and against the oracle on B's verified kept sets
    ex = gc.export_np(Bh, 0)
    grid = orc.BlockGrid(np.array([0, Tb], np.int32), B, True)
    gc.check_structure(ex, grid, Hs, 0.9)
    v64 = synth.random_v(Tb, 8, 128, 3 + 8)["v64"]
    W = synth.random_w(32, Hs, 3 + 32)
    gc.check_output(view[0][0], xb["q64"], xb["k64"], grid, ex, Hs, W, v64, 8, range(grid.R))
    # a packed view of both requests gives each its own rows
    P = mapflow.BSR(1, Tb + Ta, Hs, B, [0, Tb, Tb + Ta])
    hp = mapflow.mf_prefix_hashes(np.concatenate([tb, ta]), [0, Tb, Tb + Ta], B)
    bm.assemble(0, hp, P, 0)
    v = synth.random_v(Tb + Ta, 8, 128, 21)["v"]
    W = synth.random_w(32, Hs, 22)[None]
    Op = gc.run_retrieve(P, W, v[None], 32, "bf16", [0])[0]
    Oa = gc.run_retrieve(A, W, v[None, Tb:], 32, "bf16", [0])[0]
    Ob = gc.run_retrieve(Bh, W, v[None, :Tb], 32, "bf16", [0])[0]
    assert np.array_equal(Op[:Tb], Ob) and np.array_equal(Op[Tb:], Oa)
    # views refuse export; the manager refuses to go while views pin it
    with pytest.raises(mapflow.MapFlowError) as ei:
        V.export(0)
    assert ei.value.code == mapflow.MF_ERR_STATE
    with pytest.raises(mapflow.MapFlowError) as ei:
        bm.close()
    assert ei.value.code == mapflow.MF_ERR_STATE
    V.close()
    P.close()
    assert bm.stats()["pinned"] == 0
    bm.close()
    for h in (A, Bh):
        h.close()


@pytest.mark.gpu
def test_eviction_spares_pinned_and_current_entries(lib):
    gc.dev()
    Hs, LP = 8, 3 * B
    xa, ta = _request(LP, 190, 31)
    xb, tb = _request(LP, 170, 32, xa, ta)
    Ta, Tb = len(ta), len(tb)
    ha = mapflow.mf_prefix_hashes(ta, [0, Ta], B)
    hb = mapflow.mf_prefix_hashes(tb, [0, Tb], B)
    A = mapflow.BSR(1, Ta, Hs, B, [0, Ta])
    Bh = mapflow.BSR(1, Tb, Hs, B, [0, Tb])
    gc.run_compress(A, 0, xa, "bf16", 0.9)
    gc.run_compress(Bh, 0, xb, "bf16", 0.9)
    nnz_a, nnz_b = A.info(0)[0], Bh.info(0)[0]
    # room for either request, not for both
    bm = mapflow.BlockManager(Hs, B, max(nnz_a, nnz_b))
    bm.insert(0, A, 0, ha)
    VA = mapflow.BSR(1, Ta, Hs, B, [0, Ta])
    bm.assemble(0, ha, VA, 0)  # pins all of A
    with pytest.raises(mapflow.MapFlowError) as ei:
        bm.insert(0, Bh, 0, hb)
    assert ei.value.code == mapflow.MF_ERR_OOM
    assert bm.stats()["entries"] == len(ha)  # nothing inserted
    VA.release_layer(0)
    ins, found, ev = bm.insert(0, Bh, 0, hb)
    assert ins == len(hb) - LP // B and found == LP // B and ev >= 1
    # the evicted entries were A's oldest unshared block-rows
    assert bm.match(0, ha) == LP // B
    V = mapflow.BSR(1, Tb, Hs, B, [0, Tb])
    bm.assemble(0, hb, V, 0)
    for o, v in zip(_retrieve_both(Bh, Tb, Hs, 5), _retrieve_both(V, Tb, Hs, 5)):
        assert np.array_equal(o, v)
    with pytest.raises(mapflow.MapFlowError) as ei:
        bm.assemble(0, ha, VA, 0)  # A's suffix is gone
    assert ei.value.code == mapflow.MF_ERR_ARG
    V.close()
    VA.close()
    bm.close()
    A.close()
    Bh.close()


@pytest.mark.gpu
def test_chunk_rows_equal_the_full_sequence_rows(lib):
    """A chunked handle (query rows from q_begin, keys from 0) compresses and
    retrieves exactly the full handle's block-rows from q_begin on, and writes
    no output row before it; one sequence's chunk is empty."""
    gc.dev()
    seqlens, qb, Hs = (700, 333, 200), (384, 128, 200), 8
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    w = workloads.scaled(workloads.get(1), seqlens, sender_heads=Hs, sender_kv_heads=4)
    x = synth.sender_qk(w, 1)
    F = mapflow.BSR(1, T, Hs, B, cu)
    Cn = mapflow.BSR(1, T, Hs, B, cu, q_begin=qb)
    gc.run_compress(F, 0, x, "bf16", 0.9)
    gc.run_compress(Cn, 0, x, "bf16", 0.9)
    grid = orc.BlockGrid(cu, B, True)
    exF, exC = gc.export_np(F, 0), gc.export_np(Cn, 0)
    gc.check_structure(exF, grid, Hs, 0.9)
    rows_f = [int(grid.rb_base[s]) + bi for s in range(3) if qb[s] < seqlens[s]
              for bi in range(qb[s] // B, (seqlens[s] + B - 1) // B)]
    RC = len(rows_f)
    assert Cn.info(0)[1] == Hs * RC
    cand_c = np.concatenate([[0], np.cumsum([grid.cand_ptr[r + 1] - grid.cand_ptr[r] for r in rows_f])])
    massF = exF["mass"].reshape(Hs, grid.C)
    massC = exC["mass"].reshape(Hs, int(cand_c[-1]))
    for h in range(Hs):
        for j, rf in enumerate(rows_f):
            rc_, rf_ = h * RC + j, h * grid.R + rf
            a0, a1 = exC["row_ptr"][rc_], exC["row_ptr"][rc_ + 1]
            b0, b1 = exF["row_ptr"][rf_], exF["row_ptr"][rf_ + 1]
            assert np.array_equal(exC["col_idx"][a0:a1], exF["col_idx"][b0:b1])
            assert np.array_equal(gc.tiles(exC, range(a0, a1)), gc.tiles(exF, range(b0, b1)))
            assert np.array_equal(massC[h, cand_c[j]:cand_c[j + 1]],
                                  massF[h, grid.cand_ptr[rf]:grid.cand_ptr[rf + 1]])
    chunk_rows = np.concatenate([np.arange(cu[s] + qb[s], cu[s + 1]) for s in range(3)])
    other = np.setdiff1d(np.arange(T), chunk_rows)
    for key in ("row_max", "row_sum"):
        assert np.array_equal(exC[key][:, chunk_rows], exF[key][:, chunk_rows])
    # the chunk's own rows against the oracle: masses, row statistics and
    # tiles of every head, and O of every chunk block-row
    exCg = _chunk_on_full_grid(exC, grid, Hs, rows_f, cand_c)
    gc.check_block_rows(exCg, x["q64"], x["k64"], grid, Hs,
                        [(h, rf) for h in range(Hs) for rf in rows_f])
    for Hr, Hkv in ((32, 8), (8, 2)):
        vv = synth.random_v(T, Hkv, 128, 50 + Hkv)
        v = vv["v"][None]
        W = synth.random_w(Hr, Hs, 60 + Hr)[None]
        OF = gc.run_retrieve(F, W, v, Hr, "bf16", [0])[0]
        OC = gc.run_retrieve(Cn, W, v, Hr, "bf16", [0])[0]
        assert np.array_equal(OC[chunk_rows], OF[chunk_rows])
        assert np.isnan(OC[other]).all()
        gc.check_output(OC, x["q64"], x["k64"], grid, exCg, Hs, W[0].astype(np.float64),
                        vv["v64"], Hkv, rows_f)
    F.close()
    Cn.close()


def _chunk_on_full_grid(exC, grid, Hs, rows_f, cand_c):
    """A chunked handle's export re-indexed on the full sequence's block grid:
    the chunk's block-rows keep their masses and kept tiles (the tile indices
    still point into the chunk's own value buffer, in the same head-major
    order), every other block-row is empty."""
    RC = len(rows_f)
    mass = np.zeros((Hs, grid.C), np.float32)
    massC = exC["mass"].reshape(Hs, int(cand_c[-1]))
    rp = np.zeros(Hs * grid.R + 1, np.int64)
    pos = {rf: j for j, rf in enumerate(rows_f)}
    nxt = 0
    for h in range(Hs):
        for rb in range(grid.R):
            rp[h * grid.R + rb] = nxt
            if rb in pos:
                j = pos[rb]
                mass[h, grid.cand_ptr[rb]:grid.cand_ptr[rb + 1]] = massC[h, cand_c[j]:cand_c[j + 1]]
                assert exC["row_ptr"][h * RC + j] == nxt
                nxt = int(exC["row_ptr"][h * RC + j + 1])
    rp[-1] = nxt
    return {"mass": mass.reshape(-1), "row_ptr": rp, "col_idx": exC["col_idx"],
            "row_max": exC["row_max"], "row_sum": exC["row_sum"], "values_dev": exC["values_dev"]}


@pytest.mark.gpu
def test_cached_prefix_then_chunk(lib):
    """The serving flow: request 1 is compressed and cached; request 2 finds
    its 6-block prefix cached, compresses only the chunk after it, caches
    that, and a view of all its block-rows retrieves exactly what a full
    compression of request 2 does; a receiver chunk over the cached prefix
    gets exactly those rows."""
    gc.dev()
    Hs, LP = 8, 6 * B
    xa, ta = _request(LP, 116, 41)
    xb, tb = _request(LP, 316, 42, xa, ta)
    Ta, Tb = len(ta), len(tb)
    ha = mapflow.mf_prefix_hashes(ta, [0, Ta], B)
    hb = mapflow.mf_prefix_hashes(tb, [0, Tb], B)
    A = mapflow.BSR(1, Ta, Hs, B, [0, Ta])
    gc.run_compress(A, 0, xa, "bf16", 0.9)
    bm = mapflow.BlockManager(Hs, B, 4096)
    bm.insert(0, A, 0, ha)
    k = bm.match(0, hb)
    assert k == LP // B
    q0 = (k * B) // 128 * 128
    Cn = mapflow.BSR(1, Tb, Hs, B, [0, Tb], q_begin=[q0])
    gc.run_compress(Cn, 0, xb, "bf16", 0.9)
    hc = mapflow.mf_prefix_hashes(tb, [0, Tb], B, q_begin=[q0])
    assert np.array_equal(hc, hb[q0 // B:])
    assert bm.insert(0, Cn, 0, hc) == (len(hc), 0, 0)
    V = mapflow.BSR(1, Tb, Hs, B, [0, Tb])
    bm.assemble(0, hb, V, 0)
    F = mapflow.BSR(1, Tb, Hs, B, [0, Tb])
    gc.run_compress(F, 0, xb, "bf16", 0.9)
    own, view = _retrieve_both(F, Tb, Hs, 7), _retrieve_both(V, Tb, Hs, 7)
    for o, v in zip(own, view):
        assert np.array_equal(o, v)
    VC = mapflow.BSR(1, Tb, Hs, B, [0, Tb], q_begin=[q0])
    bm.assemble(0, hc, VC, 0)
    for o, c in zip(own, _retrieve_both(VC, Tb, Hs, 7)):
        assert np.array_equal(c[:, q0:], o[:, q0:]) and np.isnan(c[:, :q0]).all()
    for h in (V, VC):
        h.close()
    bm.close()
    for h in (A, Cn, F):
        h.close()

