"""Thin ctypes binding of the C ABI in ``include/moe.h``.

Argument marshalling only: every function here takes torch tensors (or raw
device pointers as ints, or None) and forwards their addresses to the function
of the same name in ``_moe_gb300.so``.  All arithmetic happens in the CUDA
kernels.  There is no CPU fallback: if the library is missing, every call
raises.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_EBIT_TIMEOUT = 0x1
MOE_EBIT_NAN = 0x2
MOE_EBIT_BAD_SLOT = 0x4
MOE_MODE_DECODE = 0
MOE_MODE_PREFILL = 1
MOE_MODE_DEBUG_GU = 0x100
MOE_SLOT_GATE_UP = 1
MOE_SLOT_DOWN = 2
MOE_SLOT_READY = 3
MOE_MODE_SHARED_ONLY = 0x200
MOE_MODE_ROUTED_ONLY = 0x400
MOE_MODE_AFTER_SHARED = 0x800
MOE_MODE_ORDERED = 0x1000
MOE_FMT_MXFP4 = 0
MOE_FMT_Q8_0 = 1
MOE_EPI_NONE = 0
MOE_EPI_ACCUM = 1
MOE_EPI_SWIGLU = 2
MOE_DTYPE_BF16 = 0
MOE_DTYPE_F32 = 1
MOE_CACHE_LRU = 0
MOE_CACHE_KEEP_MULTI_ROW = 1

EXPORTED = [
    "moe_slab_bytes", "moe_workspace_size", "moe_workspace_offsets", "moe_route", "moe_expert_block",
    "moe_combine", "q8_0_workspace_size", "q8_0_block_matmul", "moe_get_error", "moe_device_sm_count",
    "q8_0_block_matmul_noalloc", "q8_0_noalloc_get_error", "moe_shared_experts", "moe_shared_experts_after_route",
    "moe_cache_create", "moe_cache_request", "moe_cache_stats_get", "moe_cache_sync", "moe_cache_destroy",
    "moe_cache_request_staged", "moe_cache_lookup", "moe_nvme_open", "moe_nvme_read", "moe_nvme_wait", "moe_nvme_stats_get",
    "moe_nvme_close",
]


class MoeDesc(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("group", ctypes.c_int32)]


class MoePool(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("slot_bytes", ctypes.c_int64), ("n_slots", ctypes.c_int32),
                ("format", ctypes.c_int32)]


class MoeWsOffsets(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("error_word", "n_unique", "uexp", "uorder", "off", "pair", "dbg_g", "dbg_u", "h", "shared_y",
                 "timeline")]


class MoeNvmeStats(ctypes.Structure):
    _fields_ = [("reads", ctypes.c_int64), ("bytes", ctypes.c_int64), ("failures", ctypes.c_int64),
                ("pending_bytes", ctypes.c_int64), ("bandwidth", ctypes.c_double), ("busy_seconds", ctypes.c_double),
                ("direct", ctypes.c_int32)]


class MoeCacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("requests", "hits", "misses", "evictions", "bytes_uploaded")]


class MoeError(RuntimeError):
    pass


_LIB = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise MoeError("CUDA library not built: call __graft_entry__.build() or "
                           "python -m mxfp4_mixture_experts_router_gb300.build")
        L = ctypes.CDLL(_build.LIB)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(MoeDesc)
        PL = ctypes.POINTER(MoePool)
        L.moe_slab_bytes.argtypes = [D, I32]
        L.moe_slab_bytes.restype = SZ
        L.moe_workspace_size.argtypes = [D, I32, I32]
        L.moe_workspace_size.restype = SZ
        L.moe_workspace_offsets.argtypes = [D, I32, I32, ctypes.POINTER(MoeWsOffsets)]
        L.moe_route.argtypes = [D, I32, P, P, P, P, P, P, P, I32, I32, P]
        L.moe_expert_block.argtypes = [D, I32, I32, PL, P, P, PL, I32, P, I32, P, P]
        L.moe_shared_experts.argtypes = [D, I32, P, PL, I32, P, I32, P]
        L.moe_shared_experts_after_route.argtypes = [D, I32, P, PL, I32, P, I32, P]
        L.moe_cache_create.argtypes = [D, P, ctypes.c_int64, I32, P, I32, I32, ctypes.POINTER(P)]
        L.moe_cache_request.argtypes = [P, I32, I32, P, P, P, P, P, P]
        L.moe_cache_stats_get.argtypes = [P, ctypes.POINTER(MoeCacheStats)]
        L.moe_cache_sync.argtypes = [P]
        L.moe_cache_destroy.argtypes = [P]
        L.moe_cache_request_staged.argtypes = [P, I32, I32, P, P, P, P, P, P, P]
        L.moe_cache_lookup.argtypes = [P, I32, I32, P, P]
        L.moe_nvme_open.argtypes = [P, I32, I64, I64, I32, I32, ctypes.POINTER(P)]
        L.moe_nvme_read.argtypes = [P, I32, P, I64, P, P]
        L.moe_nvme_wait.argtypes = [P, ctypes.c_uint32, I64]
        L.moe_nvme_stats_get.argtypes = [P, I32, ctypes.POINTER(MoeNvmeStats)]
        L.moe_nvme_close.argtypes = [P]
        L.moe_combine.argtypes = [D, I32, P, P, P, P, I32, P, P]
        L.q8_0_workspace_size.argtypes = [I32, I32, I32]
        L.q8_0_workspace_size.restype = SZ
        L.q8_0_block_matmul.argtypes = [I32, I32, I32, P, I32, P, P, P, P, I32, P, P, P]
        L.q8_0_block_matmul_noalloc.argtypes = [I32, I32, I32, P, I32, P, P, P, P, I32, P, P]
        L.q8_0_noalloc_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        L.moe_get_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
        L.moe_device_sm_count.restype = I32
        _LIB = L
    return _LIB


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(f"{what} failed with status {status}")


def desc(d_model: int, d_ff: int, n_experts: int, top_k: int, group: int = 32) -> MoeDesc:
    return MoeDesc(d_model, d_ff, n_experts, top_k, group)


def pool(base, slot_bytes: int, n_slots: int, fmt: int) -> MoePool:
    return MoePool(_ptr(base), slot_bytes, n_slots, fmt)


def moe_slab_bytes(d: MoeDesc, fmt: int) -> int:
    return lib().moe_slab_bytes(ctypes.byref(d), fmt)


def moe_workspace_size(d: MoeDesc, n_rows_max: int, n_shared: int) -> int:
    return lib().moe_workspace_size(ctypes.byref(d), n_rows_max, n_shared)


def moe_workspace_offsets(d: MoeDesc, n_rows_max: int, n_shared: int) -> MoeWsOffsets:
    o = MoeWsOffsets()
    _check(lib().moe_workspace_offsets(ctypes.byref(d), n_rows_max, n_shared, ctypes.byref(o)),
           "moe_workspace_offsets")
    return o


def moe_route(d: MoeDesc, n_rows: int, x, w_router, logits_in, logits_out, topk_idx, topk_w, ws,
              n_rows_max: int, n_shared: int, stream=None):
    _check(lib().moe_route(ctypes.byref(d), n_rows, _ptr(x), _ptr(w_router), _ptr(logits_in),
                           _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(ws), n_rows_max,
                           n_shared, _stream(stream)), "moe_route")


def moe_shared_experts(d: MoeDesc, n_rows: int, x, shared: MoePool, n_shared: int, ws, n_rows_max: int,
                       stream=None):
    _check(lib().moe_shared_experts(ctypes.byref(d), n_rows, _ptr(x), ctypes.byref(shared), n_shared, _ptr(ws),
                                    n_rows_max, _stream(stream)), "moe_shared_experts")


def moe_shared_experts_after_route(d: MoeDesc, n_rows: int, x, shared: MoePool, n_shared: int, ws,
                                   n_rows_max: int, stream=None):
    _check(lib().moe_shared_experts_after_route(ctypes.byref(d), n_rows, _ptr(x), ctypes.byref(shared), n_shared,
                                                _ptr(ws), n_rows_max, _stream(stream)),
           "moe_shared_experts_after_route")


def moe_expert_block(d: MoeDesc, n_rows: int, mode: int, routed: MoePool, expert_slot, slot_ready,
                     shared: MoePool | None, n_shared: int, ws, n_rows_max: int, y_part, stream=None):
    _check(lib().moe_expert_block(ctypes.byref(d), n_rows, mode, ctypes.byref(routed), _ptr(expert_slot),
                                  _ptr(slot_ready), ctypes.byref(shared) if shared is not None else None,
                                  n_shared, _ptr(ws), n_rows_max, _ptr(y_part), _stream(stream)),
           "moe_expert_block")


def moe_combine(d: MoeDesc, n_rows: int, residual, y_part, topk_w, shared_y, n_shared: int, out,
                stream=None):
    _check(lib().moe_combine(ctypes.byref(d), n_rows, _ptr(residual), _ptr(y_part), _ptr(topk_w),
                             _ptr(shared_y), n_shared, _ptr(out), _stream(stream)), "moe_combine")


def q8_0_workspace_size(n_rows: int, k_in: int, n_out: int) -> int:
    return lib().q8_0_workspace_size(n_rows, k_in, n_out)


def q8_0_block_matmul(n_rows: int, k_in: int, n_out: int, x, x_dtype: int, q, dq, q2, d2, epilogue: int,
                      y, ws, stream=None):
    _check(lib().q8_0_block_matmul(n_rows, k_in, n_out, _ptr(x), x_dtype, _ptr(q), _ptr(dq), _ptr(q2),
                                   _ptr(d2), epilogue, _ptr(y), _ptr(ws), _stream(stream)),
           "q8_0_block_matmul")


def q8_0_block_matmul_noalloc(n_rows: int, k_in: int, n_out: int, x, x_dtype: int, q, dq, q2, d2,
                              epilogue: int, y, stream=None):
    """q8_0_block_matmul with the library's own static device scratch (no workspace
    argument, nothing allocated); calls that overlap on the GPU must be serialised."""
    _check(lib().q8_0_block_matmul_noalloc(n_rows, k_in, n_out, _ptr(x), x_dtype, _ptr(q), _ptr(dq), _ptr(q2),
                                           _ptr(d2), epilogue, _ptr(y), _stream(stream)),
           "q8_0_block_matmul_noalloc")


def q8_0_noalloc_get_error(stream=None) -> int:
    """Device error bits collected by q8_0_block_matmul_noalloc calls on the current
    device since the last read (read and cleared)."""
    bits = ctypes.c_uint32(0)
    _check(lib().q8_0_noalloc_get_error(_stream(stream), ctypes.byref(bits)), "q8_0_noalloc_get_error")
    return bits.value


def moe_get_error(ws, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().moe_get_error(_ptr(ws), _stream(stream), ctypes.byref(bits)), "moe_get_error")
    return bits.value


def moe_device_sm_count() -> int:
    return lib().moe_device_sm_count()


# --- device expert cache -----------------------------------------------------

def moe_cache_create(d: MoeDesc, slot_base, slot_bytes: int, n_slots: int, slot_ready, n_streams: int,
                     policy: int) -> int:
    """Opaque cache handle (an int).  n_streams = 0: planning only (no CUDA calls)."""
    h = ctypes.c_void_p(0)
    _check(lib().moe_cache_create(ctypes.byref(d), _ptr(slot_base), slot_bytes, n_slots, _ptr(slot_ready),
                                  n_streams, policy, ctypes.byref(h)), "moe_cache_create")
    return h.value


def moe_cache_request(handle: int, layer: int, experts, rows=None, host_src=None, stream=None):
    """experts, rows: int32 numpy arrays; host_src: numpy uint64 array of pinned host
    addresses, or None.  Returns (slots, uploaded) int32 numpy arrays."""
    import numpy as np
    e = np.ascontiguousarray(experts, dtype=np.int32)
    n = int(e.shape[0])
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    src = None if host_src is None else np.ascontiguousarray(host_src, dtype=np.uint64)
    slots = np.empty(n, dtype=np.int32)
    miss = np.empty(n, dtype=np.int32)
    _check(lib().moe_cache_request(ctypes.c_void_p(handle), layer, n, e.ctypes.data,
                                   None if r is None else r.ctypes.data,
                                   None if src is None else src.ctypes.data, slots.ctypes.data,
                                   miss.ctypes.data, _cache_stream(stream)), "moe_cache_request")
    return slots, miss


def _cache_stream(stream):
    """The caller's stream; with none given, the current one when a GPU is present (a
    planning-only cache makes no CUDA call and ignores it)."""
    if stream is not None:
        return _stream(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None


def moe_cache_stats(handle: int) -> dict:
    st = MoeCacheStats()
    _check(lib().moe_cache_stats_get(ctypes.c_void_p(handle), ctypes.byref(st)), "moe_cache_stats_get")
    return {n: getattr(st, n) for n, _ in MoeCacheStats._fields_}


def moe_cache_sync(handle: int):
    _check(lib().moe_cache_sync(ctypes.c_void_p(handle)), "moe_cache_sync")


def moe_cache_destroy(handle: int):
    _check(lib().moe_cache_destroy(ctypes.c_void_p(handle)), "moe_cache_destroy")


# --- NVMe expert tier ------------------------------------------------------------

MOE_NVME_FAILED = 0x80000000
MOE_ERR_IO = 6


def moe_nvme_open(paths, slab_bytes: int, slab_stride: int, n_bodies: int, depth: int) -> int:
    """Opaque handle (an int) of an expert store replicated over the given files."""
    arr = (ctypes.c_char_p * len(paths))(*[p.encode() for p in paths])
    h = ctypes.c_void_p()
    _check(lib().moe_nvme_open(ctypes.cast(arr, ctypes.c_void_p), len(paths), slab_bytes, slab_stride, n_bodies,
                               depth, ctypes.byref(h)), "moe_nvme_open")
    return h.value


def moe_nvme_read(handle: int, body: int, dst_addr: int, first_bytes: int, flag_addr: int) -> int:
    """Queue one slab read into host memory at dst_addr; returns the replica chosen."""
    rep = ctypes.c_int32(-1)
    _check(lib().moe_nvme_read(ctypes.c_void_p(handle), body, ctypes.c_void_p(dst_addr), first_bytes,
                               ctypes.c_void_p(flag_addr), ctypes.byref(rep)), "moe_nvme_read")
    return rep.value


def moe_nvme_wait(flag_addr: int, bits: int, timeout_ns: int = 10_000_000_000) -> int:
    """MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_IO (returned, not raised)."""
    return lib().moe_nvme_wait(ctypes.c_void_p(flag_addr), bits, timeout_ns)


def moe_nvme_stats(handle: int, replica: int) -> dict:
    st = MoeNvmeStats()
    _check(lib().moe_nvme_stats_get(ctypes.c_void_p(handle), replica, ctypes.byref(st)), "moe_nvme_stats_get")
    return {f: getattr(st, f) for f, _ in MoeNvmeStats._fields_}


def moe_nvme_close(handle: int):
    _check(lib().moe_nvme_close(ctypes.c_void_p(handle)), "moe_nvme_close")


def moe_cache_request_staged(handle: int, layer: int, experts, rows, host_src, host_ready, stream=None):
    """moe_cache_request whose slabs may still be landing in host memory: host_ready is a
    numpy uint64 array of the addresses of their pinned uint32 ready flags."""
    import numpy as np
    e = np.ascontiguousarray(experts, dtype=np.int32)
    n = int(e.shape[0])
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    src = np.ascontiguousarray(host_src, dtype=np.uint64)
    rdy = np.ascontiguousarray(host_ready, dtype=np.uint64)
    slots = np.empty(n, dtype=np.int32)
    miss = np.empty(n, dtype=np.int32)
    _check(lib().moe_cache_request_staged(ctypes.c_void_p(handle), layer, n, e.ctypes.data,
                                          None if r is None else r.ctypes.data, src.ctypes.data, rdy.ctypes.data,
                                          slots.ctypes.data, miss.ctypes.data, _cache_stream(stream)),
           "moe_cache_request_staged")
    return slots, miss


def moe_cache_lookup(handle: int, layer: int, experts):
    """1 where the (layer, expert) slab holds a device slot now, else 0 (no side effects)."""
    import numpy as np
    e = np.ascontiguousarray(experts, dtype=np.int32)
    out = np.empty(e.shape[0], dtype=np.int32)
    _check(lib().moe_cache_lookup(ctypes.c_void_p(handle), layer, int(e.shape[0]), e.ctypes.data, out.ctypes.data),
           "moe_cache_lookup")
    return out
