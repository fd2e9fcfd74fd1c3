"""The C-ABI library loads and exports every symbol include/mapflow.h
declares; host-side argument validation answers without touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

from cross_model_attention_gb300 import build as build_mod
from cross_model_attention_gb300 import mapflow

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return mapflow.load_library()


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(mf_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mf_compress" in names and "mf_retrieve" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(mapflow.EXPORTED) <= set(names)


def test_version_and_supported(lib):
    assert lib.mf_version() >= 100
    assert mapflow.mf_supported(mapflow.MF_DTYPE_BF16, 128, 64)
    assert mapflow.mf_supported(mapflow.MF_DTYPE_BF16, 64, 128)
    assert not mapflow.mf_supported(mapflow.MF_DTYPE_BF16, 96, 64)
    assert not mapflow.mf_supported(mapflow.MF_DTYPE_BF16, 128, 32)
    assert not mapflow.mf_supported(mapflow.MF_DTYPE_F32, 128, 128)


def _create(cu, **kw):
    args = dict(n_layers=1, T=int(cu[-1]), H_s=4, B=64, causal=True)
    args.update(kw)
    return mapflow.mf_bsr_create(args["n_layers"], args["T"], args["H_s"], args["B"],
                                 args["causal"], cu, use_torch_allocator=False)


@pytest.mark.parametrize("cu,kw,code", [
    ([0, 100], dict(B=32), mapflow.MF_ERR_UNSUPPORTED),
    ([0, 100], dict(B=96), mapflow.MF_ERR_UNSUPPORTED),
    ([0, 100, 50], {}, mapflow.MF_ERR_ARG),                 # non-monotone
    ([1, 100], {}, mapflow.MF_ERR_ARG),                     # cu[0] != 0
    ([0, 100], dict(T=99), mapflow.MF_ERR_ARG),             # cu[n] != T
    ([0, 100], dict(n_layers=0), mapflow.MF_ERR_ARG),
    ([0, 100], dict(H_s=0), mapflow.MF_ERR_ARG),
    ([0, 100], dict(H_s=129), mapflow.MF_ERR_UNSUPPORTED),
    ([0, 64 * 256 + 1], dict(B=64), mapflow.MF_ERR_UNSUPPORTED),  # > 256 blocks per row
])
def test_create_rejects_bad_arguments(lib, cu, kw, code):
    with pytest.raises(mapflow.MapFlowError) as ei:
        _create(np.array(cu), **kw)
    assert ei.value.code == code
    assert lib.mf_last_error().decode()


def test_null_handle_and_pointers(lib):
    assert lib.mf_compress(None, 0, None, None, 1, 1, 1, 1, 64, 64, ctypes.c_float(0.9), 1, None) \
        == mapflow.MF_ERR_ARG
    assert lib.mf_retrieve(None, None, None, None, 1, 1, 1, 64, None, 1, None) == mapflow.MF_ERR_ARG
    assert lib.mf_bsr_info(None, 0, None, None, None) == mapflow.MF_ERR_ARG
    assert lib.mf_device_status(None, None) == mapflow.MF_ERR_ARG
    lib.mf_bsr_destroy(None)


def test_later_entry_points_validate_on_the_host(lib):
    E = mapflow
    vp = ctypes.c_void_p
    h = vp()
    A, F = mapflow.ALLOC_FN(), mapflow.FREE_FN()
    assert lib.mf_bm_create(None, 8, 64, 16, A, F, None, None) == E.MF_ERR_ARG
    assert lib.mf_bm_create(ctypes.byref(h), 0, 64, 16, A, F, None, None) == E.MF_ERR_ARG
    assert lib.mf_bm_create(ctypes.byref(h), 8, 32, 16, A, F, None, None) == E.MF_ERR_UNSUPPORTED
    assert lib.mf_bm_create(ctypes.byref(h), 8, 64, 0, A, F, None, None) == E.MF_ERR_ARG
    assert lib.mf_bm_create(ctypes.byref(h), 8, 64, 16,
                            mapflow.ALLOC_FN(lambda n, c, s: None), F, None, None) == E.MF_ERR_ARG
    assert lib.mf_bm_insert(None, 0, None, 0, None, None, None) == E.MF_ERR_ARG
    n = ctypes.c_int()
    assert lib.mf_bm_match(None, 0, None, 0, ctypes.byref(n)) == E.MF_ERR_ARG
    assert lib.mf_bm_assemble(None, 0, None, None, 0, None) == E.MF_ERR_ARG
    assert lib.mf_bm_stats(None, None) == E.MF_ERR_ARG
    assert lib.mf_bm_destroy(None) == E.MF_OK
    assert lib.mf_calibrate_head_map(None, 0, None, 0, ctypes.c_float(0.0), None, None) == E.MF_ERR_ARG
    assert lib.mf_bsr_offload(None, 0, None) == E.MF_ERR_ARG
    assert lib.mf_bsr_prefetch(None, 0, None) == E.MF_ERR_ARG
    assert lib.mf_last_error().decode()


def test_allocator_pair_must_match(lib):
    cu = np.array([0, 64], np.int32)
    h = ctypes.c_void_p()
    alloc = mapflow.ALLOC_FN(lambda n, c, s: None)
    rc = lib.mf_bsr_create(ctypes.byref(h), 1, 64, 4, 64, 1,
                           cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), 1, alloc,
                           mapflow.FREE_FN(), None)
    assert rc == mapflow.MF_ERR_ARG


def test_library_has_no_driver_link(lib):
    """The library reaches the driver through the runtime's entry-point query,
    so it loads on machines without libcuda (CPU-only build hosts): no NEEDED
    entry names libcuda."""
    import shutil
    import subprocess
    if not shutil.which("readelf"):
        pytest.skip("readelf not available")
    out = subprocess.run(["readelf", "-d", mapflow.LIB_PATH], capture_output=True, text=True).stdout
    needed = [l for l in out.splitlines() if "NEEDED" in l]
    assert needed and not any("libcuda" in l for l in needed)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without the built library every entry point raises."""
    monkeypatch.setattr(mapflow, "_lib", None)
    missing = str(tmp_path / "libmapflow.so")
    with pytest.raises(ImportError):
        mapflow.load_library(missing)
    monkeypatch.setattr(mapflow, "LIB_PATH", missing)
    monkeypatch.setattr(mapflow.load_library, "__defaults__", (missing,))
    with pytest.raises(ImportError):
        mapflow.mf_version()
    with pytest.raises(ImportError):
        mapflow.mf_prefix_hashes(np.zeros(4, np.int32), [0, 4], 64)
