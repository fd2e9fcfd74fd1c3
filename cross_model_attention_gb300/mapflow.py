"""Thin ctypes binding of libmapflow (include/mapflow.h).

Argument marshalling only: every step of the method runs in the CUDA
library.  PyTorch supplies device memory (its caching allocator is handed to
the library as the BSR allocator) and streams.  If the shared library is
missing, importing this module raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmapflow.so")

MF_OK, MF_ERR_ARG, MF_ERR_UNSUPPORTED, MF_ERR_CUDA, MF_ERR_OOM, MF_ERR_TIMEOUT, MF_ERR_STATE = range(7)
MF_DTYPE_F32, MF_DTYPE_BF16 = 0, 1

EXPORTED = ("mf_version", "mf_last_error", "mf_supported", "mf_bsr_create", "mf_bsr_destroy",
            "mf_compress", "mf_retrieve", "mf_bsr_info", "mf_bsr_export", "mf_bsr_copy",
            "mf_bsr_release_layer", "mf_bsr_offload", "mf_bsr_prefetch", "mf_calibrate_head_map",
            "mf_device_status", "mf_selftest_wait", "mf_profile",
            "mf_profile_read", "mf_profile_kinds", "mf_select_noalloc", "mf_bsr_set_exact",
            "mf_bsr_create_chunked", "mf_prefix_hashes", "mf_bm_create", "mf_bm_destroy",
            "mf_bm_insert", "mf_bm_match", "mf_bm_assemble", "mf_bm_stats")
KERNELS = ("stats", "select", "scan", "pack", "union", "retrieve")


class MapFlowError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"mapflow error {code}: {msg}")
        self.code = code


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmapflow.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, i64p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)
    lib.mf_version.restype = i32
    lib.mf_last_error.restype = ctypes.c_char_p
    lib.mf_supported.argtypes = [i32, i32, i32]
    lib.mf_bsr_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32,
                                  ctypes.POINTER(ctypes.c_int32), i32, ALLOC_FN, FREE_FN, vp]
    lib.mf_bsr_destroy.argtypes = [vp]
    lib.mf_bsr_destroy.restype = None
    lib.mf_compress.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, ctypes.c_float,
                                i32, vp]
    lib.mf_retrieve.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32,
                                ctypes.POINTER(ctypes.c_int32), i32, vp]
    lib.mf_bsr_info.argtypes = [vp, i32, i64p, i64p, i64p]
    lib.mf_bsr_export.argtypes = [vp, i32] + [ctypes.POINTER(vp)] * 6
    lib.mf_bsr_copy.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.mf_bsr_release_layer.argtypes = [vp, i32]
    lib.mf_bsr_offload.argtypes = [vp, i32, vp]
    lib.mf_calibrate_head_map.argtypes = [vp, i32, vp, i32, ctypes.c_float, vp, vp]
    lib.mf_bsr_prefetch.argtypes = [vp, i32, vp]
    lib.mf_bsr_set_exact.argtypes = [vp, i32]
    lib.mf_device_status.argtypes = [vp, vp]
    lib.mf_selftest_wait.argtypes = [vp, i32, vp]
    lib.mf_select_noalloc.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), i32, i32, i32, i32,
                                      ctypes.c_float, vp, vp, ctypes.c_int64, vp, vp]
    lib.mf_profile.argtypes = [vp, i32]
    lib.mf_profile_kinds.argtypes = [vp, i32]
    lib.mf_profile_read.argtypes = [vp, i32, i64p, ctypes.POINTER(ctypes.c_double)]
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.mf_prefix_hashes.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                     vp, i32, i32, ctypes.c_uint64, u64p, ctypes.c_int64, i64p]
    lib.mf_bsr_create_chunked.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32,
                                          ctypes.POINTER(ctypes.c_int32), vp, i32, ALLOC_FN,
                                          FREE_FN, vp]
    lib.mf_bm_create.argtypes = [ctypes.POINTER(vp), i32, i32, ctypes.c_int64, ALLOC_FN, FREE_FN,
                                 vp, vp]
    lib.mf_bm_destroy.argtypes = [vp]
    lib.mf_bm_insert.argtypes = [vp, i32, vp, i32, u64p, i64p, vp]
    lib.mf_bm_match.argtypes = [vp, i32, u64p, i32, ctypes.POINTER(i32)]
    lib.mf_bm_assemble.argtypes = [vp, i32, u64p, vp, i32, vp]
    lib.mf_bm_stats.argtypes = [vp, i64p]
    for name in EXPORTED:
        getattr(lib, name)
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != MF_OK:
        raise MapFlowError(rc, load_library().mf_last_error().decode(errors="replace"))


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return MF_DTYPE_BF16
    if t.dtype == torch.float32:
        return MF_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


# ------------------------------------------------------ torch allocator ----
def _torch_allocator():
    import torch

    def _alloc(nbytes, ctx, stream):
        try:
            return torch.cuda.caching_allocator_alloc(int(nbytes), device=torch.cuda.current_device(),
                                                      stream=stream or 0)
        except Exception:  # noqa: BLE001 - signalled to the library as NULL
            return None

    def _free(ptr, ctx, stream):
        if ptr:
            torch.cuda.caching_allocator_delete(ptr)
    return ALLOC_FN(_alloc), FREE_FN(_free)


# --------------------------------------------- same names as the C ABI -----
def mf_version() -> int:
    return load_library().mf_version()


def mf_supported(dtype: int, d: int, B: int) -> bool:
    return bool(load_library().mf_supported(dtype, d, B))


def mf_bsr_create(n_layers: int, T: int, H_s: int, B: int, causal: bool,
                  cu_seqlens: Sequence[int], use_torch_allocator: bool = True,
                  q_begin: Optional[Sequence[int]] = None):
    """Returns (handle, keepalive); keepalive holds the allocator callbacks.
    With q_begin the handle covers query chunks (mf_bsr_create_chunked)."""
    lib = load_library()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    h = ctypes.c_void_p()
    if use_torch_allocator:
        a, f = _torch_allocator()
    else:
        a, f = ALLOC_FN(), FREE_FN()
    i32p = ctypes.POINTER(ctypes.c_int32)
    if q_begin is None:
        rc = lib.mf_bsr_create(ctypes.byref(h), n_layers, T, H_s, B, int(causal),
                               cu.ctypes.data_as(i32p), len(cu) - 1, a, f, None)
    else:
        qb = np.ascontiguousarray(np.asarray(q_begin, dtype=np.int32))
        rc = lib.mf_bsr_create_chunked(ctypes.byref(h), n_layers, T, H_s, B, int(causal),
                                       cu.ctypes.data_as(i32p), qb.ctypes.data_as(ctypes.c_void_p),
                                       len(cu) - 1, a, f, None)
    _check(rc)
    return h, (a, f)


def mf_bsr_destroy(h) -> None:
    load_library().mf_bsr_destroy(h)


def mf_compress(h, layer: int, q, k, T: int, H_s: int, H_ks: int, d: int, B: int, p: float,
                causal: bool, stream=None) -> None:
    _check(load_library().mf_compress(h, layer, _ptr(q), _ptr(k), _dtype_code(q), T, H_s, H_ks,
                                      d, B, float(p), int(causal), _stream(stream)))


def mf_retrieve(h, W, v, o, H_r: int, H_kv: int, d: int, layer_map: Sequence[int],
                stream=None) -> None:
    lm = np.ascontiguousarray(np.asarray(layer_map, dtype=np.int32))
    _check(load_library().mf_retrieve(h, _ptr(W), _ptr(v), _ptr(o), _dtype_code(v), H_r, H_kv, d,
                                       lm.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(lm),
                                       _stream(stream)))


def mf_bsr_set_exact(h, exact: bool) -> None:
    _check(load_library().mf_bsr_set_exact(h, int(exact)))


def mf_bsr_info(h, layer: int):
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(load_library().mf_bsr_info(h, layer, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def mf_bsr_copy(h, layer: int, row_ptr=None, col_idx=None, values=None, mass=None,
                row_max=None, row_sum=None, stream=None) -> None:
    _check(load_library().mf_bsr_copy(h, layer, _ptr(row_ptr), _ptr(col_idx), _ptr(values),
                                      _ptr(mass), _ptr(row_max), _ptr(row_sum), _stream(stream)))


def mf_bsr_release_layer(h, layer: int) -> None:
    _check(load_library().mf_bsr_release_layer(h, layer))


def mf_bsr_offload(h, layer: int, stream=None) -> None:
    _check(load_library().mf_bsr_offload(h, layer, _stream(stream)))


def mf_bsr_prefetch(h, layer: int, stream=None) -> None:
    _check(load_library().mf_bsr_prefetch(h, layer, _stream(stream)))


def calibrate_head_map(sender: "BSR", sender_layer: int, receiver: "BSR", receiver_layer: int,
                       ridge: float = 0.0, stream=None) -> np.ndarray:
    """Least-squares head map W [H_r, H_s] from two compressed layers over the
    same sequences (see mf_calibrate_head_map)."""
    W = np.zeros((receiver.H_s, sender.H_s), np.float32)
    _check(load_library().mf_calibrate_head_map(
        sender.handle, sender_layer, receiver.handle, receiver_layer, float(ridge),
        W.ctypes.data_as(ctypes.c_void_p), _stream(stream)))
    return W


def mf_device_status(h, stream=None) -> None:
    _check(load_library().mf_device_status(h, _stream(stream)))


def mf_selftest_wait(h, limit_ms: int, stream=None) -> None:
    _check(load_library().mf_selftest_wait(h, int(limit_ms), _stream(stream)))


def mf_select_noalloc(mass, cu_seqlens: Sequence[int], H_s: int, B: int, causal: bool,
                      p: float, row_ptr, col_idx, nnz, stream=None) -> None:
    """Selection into caller buffers with no device allocation (see mapflow.h).

    The library sees only pointers, so the buffer sizes, dtypes and devices
    are checked here, before any kernel could read or write past them."""
    import torch
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    lens = np.diff(cu.astype(np.int64))
    if len(cu) < 2 or cu[0] != 0 or (lens < 0).any() or B <= 0 or H_s <= 0:
        raise MapFlowError(MF_ERR_ARG, "cu_seqlens must start at 0 and be non-decreasing; "
                                       "B and H_s positive")
    nb = (lens + B - 1) // B
    R = int(nb.sum())
    C = int((nb * (nb + 1) // 2).sum()) if causal else int((nb * nb).sum())
    need = (("mass", mass, torch.float32, H_s * C), ("row_ptr", row_ptr, torch.int32, H_s * R + 1),
            ("col_idx", col_idx, torch.int32, 0), ("nnz", nnz, torch.int64, 1))
    for name, t, dt, n in need:
        if t.device.type != "cuda" or t.dtype != dt or not t.is_contiguous():
            raise MapFlowError(MF_ERR_ARG, f"{name} must be a contiguous CUDA {dt} tensor")
        if t.numel() < n:
            raise MapFlowError(MF_ERR_ARG, f"{name} holds {t.numel()} elements, needs {n}")
    _check(load_library().mf_select_noalloc(
        _ptr(mass), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(cu) - 1, H_s, B,
        int(causal), float(p), _ptr(row_ptr), _ptr(col_idx), int(col_idx.numel()), _ptr(nnz),
        _stream(stream)))


def mf_profile(h, enable: bool) -> None:
    _check(load_library().mf_profile(h, int(enable)))


def mf_profile_kinds(h, mask: int) -> None:
    _check(load_library().mf_profile_kinds(h, int(mask)))


def mf_profile_read(h, kernel: int):
    n, ms = ctypes.c_int64(), ctypes.c_double()
    _check(load_library().mf_profile_read(h, kernel, ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def mf_prefix_hashes(tokens, cu_seqlens: Sequence[int], B: int, seed: int = 0,
                     q_begin: Optional[Sequence[int]] = None) -> np.ndarray:
    """Chained prefix hashes of the B-token blocks of each packed sequence
    (uint64 [R], the block-row order of a BSR handle with these cu_seqlens and
    q_begin)."""
    lib = load_library()
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    if len(cu) < 2 or cu[-1] != len(tok):
        raise ValueError("cu_seqlens must end at len(tokens)")
    qb = None if q_begin is None else np.ascontiguousarray(np.asarray(q_begin, dtype=np.int32))
    qb_ptr = None if qb is None else qb.ctypes.data_as(ctypes.c_void_p)
    i32p = ctypes.POINTER(ctypes.c_int32)
    n = ctypes.c_int64()
    _check(lib.mf_prefix_hashes(tok.ctypes.data_as(i32p), cu.ctypes.data_as(i32p), qb_ptr, len(cu) - 1,
                                B, ctypes.c_uint64(seed), None, 0, ctypes.byref(n)))
    out = np.zeros(n.value, np.uint64)
    _check(lib.mf_prefix_hashes(tok.ctypes.data_as(i32p), cu.ctypes.data_as(i32p), qb_ptr, len(cu) - 1,
                                B, ctypes.c_uint64(seed),
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), n.value,
                                ctypes.byref(n)))
    return out


def _u64(hashes) -> Tuple[np.ndarray, "ctypes._Pointer"]:
    a = np.ascontiguousarray(np.asarray(hashes, dtype=np.uint64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))


class BlockManager:
    """Owner of one mf_bm_t: block-rows of compressed layers cached under
    prefix hashes in a device tile pool (see mf_bm_* in mapflow.h)."""

    def __init__(self, H_s: int, B: int, tile_capacity: int, use_torch_allocator: bool = True,
                 stream=None):
        lib = load_library()
        self.H_s, self.B, self.tile_capacity = H_s, B, int(tile_capacity)
        h = ctypes.c_void_p()
        if use_torch_allocator:
            a, f = _torch_allocator()
        else:
            a, f = ALLOC_FN(), FREE_FN()
        self._keep = (a, f)
        _check(lib.mf_bm_create(ctypes.byref(h), H_s, B, self.tile_capacity, a, f, None,
                                _stream(stream)))
        self.handle = h

    def insert(self, key_layer: int, bsr: "BSR", layer: int, hashes, stream=None) -> Tuple[int, int, int]:
        """Caches the layer's block-rows; returns (inserted, already cached, evicted)."""
        arr, ptr = _u64(hashes)
        counts = (ctypes.c_int64 * 3)()
        _check(load_library().mf_bm_insert(self.handle, key_layer, bsr.handle, layer, ptr, counts,
                                           _stream(stream)))
        return int(counts[0]), int(counts[1]), int(counts[2])

    def match(self, key_layer: int, hashes) -> int:
        arr, ptr = _u64(hashes)
        n = ctypes.c_int()
        _check(load_library().mf_bm_match(self.handle, key_layer, ptr, len(arr), ctypes.byref(n)))
        return int(n.value)

    def assemble(self, key_layer: int, hashes, bsr: "BSR", layer: int, stream=None) -> None:
        """Makes `layer` of `bsr` a view of the cached block-rows `hashes`."""
        arr, ptr = _u64(hashes)
        _check(load_library().mf_bm_assemble(self.handle, key_layer, ptr, bsr.handle, layer,
                                             _stream(stream)))

    def stats(self) -> Dict[str, int]:
        out = (ctypes.c_int64 * 7)()
        _check(load_library().mf_bm_stats(self.handle, out))
        keys = ("entries", "tiles_used", "tile_capacity", "hits", "misses", "evictions", "pinned")
        return {k: int(v) for k, v in zip(keys, out)}

    def close(self) -> None:
        if self.handle is not None:
            _check(load_library().mf_bm_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001
            pass


# ------------------------------------------------------ convenience class --
class BSR:
    """Owner of one mf_bsr_t (compressed sender state of several layers)."""

    def __init__(self, n_layers: int, T: int, H_s: int, B: int, cu_seqlens: Sequence[int],
                 causal: bool = True, use_torch_allocator: bool = True,
                 q_begin: Optional[Sequence[int]] = None):
        self.n_layers, self.T, self.H_s, self.B, self.causal = n_layers, T, H_s, B, causal
        self.cu_seqlens = [int(x) for x in cu_seqlens]
        self.q_begin = None if q_begin is None else [int(x) for x in q_begin]
        self.handle, self._keep = mf_bsr_create(n_layers, T, H_s, B, causal, self.cu_seqlens,
                                                use_torch_allocator, self.q_begin)
        self.d: Optional[int] = None

    def compress(self, layer: int, q, k, p: float, stream=None) -> None:
        T, H_s, d = q.shape
        self.d = d
        mf_compress(self.handle, layer, q, k, T, H_s, k.shape[1], d, self.B, p, self.causal,
                    stream)

    def retrieve(self, W, v, o, layer_map: Sequence[int], stream=None) -> None:
        n, T, H_kv, d = v.shape
        H_r = o.shape[2]
        mf_retrieve(self.handle, W, v, o, H_r, H_kv, d, layer_map, stream)

    def set_exact(self, exact: bool) -> None:
        mf_bsr_set_exact(self.handle, exact)

    def info(self, layer: int):
        return mf_bsr_info(self.handle, layer)

    def export(self, layer: int, stream=None) -> Dict[str, "object"]:
        """Copies of the layer's BSR arrays as torch tensors on the device."""
        import torch
        nnz, n_rows, n_cand = self.info(layer)
        dev = torch.device("cuda", torch.cuda.current_device())
        out = {
            "row_ptr": torch.empty(n_rows + 1, dtype=torch.int32, device=dev),
            "col_idx": torch.empty(max(nnz, 1), dtype=torch.int32, device=dev)[:nnz],
            "values": torch.empty((max(nnz, 1), self.B, self.B), dtype=torch.bfloat16,
                                  device=dev)[:nnz],
            "mass": torch.empty(n_cand, dtype=torch.float32, device=dev),
            "row_max": torch.empty((self.H_s, self.T), dtype=torch.float32, device=dev),
            "row_sum": torch.empty((self.H_s, self.T), dtype=torch.float32, device=dev),
        }
        mf_bsr_copy(self.handle, layer, out["row_ptr"], out["col_idx"] if nnz else None,
                    out["values"] if nnz else None, out["mass"], out["row_max"],
                    out["row_sum"], stream)
        return out

    def structure(self, layer: int):
        """(row_ptr, col_idx) of a compressed layer as host numpy arrays."""
        import torch
        nnz, n_rows, _ = self.info(layer)
        dev = torch.device("cuda", torch.cuda.current_device())
        rp = torch.empty(n_rows + 1, dtype=torch.int32, device=dev)
        ci = torch.empty(max(nnz, 1), dtype=torch.int32, device=dev)
        mf_bsr_copy(self.handle, layer, rp, ci if nnz else None, None, None, None, None, None)
        torch.cuda.synchronize()
        return rp.cpu().numpy(), ci[:nnz].cpu().numpy().astype(np.int64)

    def release_layer(self, layer: int) -> None:
        mf_bsr_release_layer(self.handle, layer)

    def offload(self, layer: int, stream=None) -> None:
        """Move the layer's BSR to pinned host memory (see mf_bsr_offload)."""
        mf_bsr_offload(self.handle, layer, stream)

    def prefetch(self, layer: int, stream=None) -> None:
        """Bring an offloaded layer back to the device on `stream`."""
        mf_bsr_prefetch(self.handle, layer, stream)

    def device_status(self, stream=None) -> None:
        mf_device_status(self.handle, stream)

    def profile(self, enable: bool) -> None:
        mf_profile(self.handle, enable)

    def profile_kinds(self, names) -> None:
        """Time only the named kernel kinds (e.g. ("stats", "pack"))."""
        mf_profile_kinds(self.handle, sum(1 << KERNELS.index(n) for n in names))

    def profile_read(self) -> Dict[str, tuple]:
        """{kernel: (launches, total device ms)} since profiling was enabled."""
        return {name: mf_profile_read(self.handle, i) for i, name in enumerate(KERNELS)}

    def close(self) -> None:
        if self.handle is not None:
            mf_bsr_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001
            pass
