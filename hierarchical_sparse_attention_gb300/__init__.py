"""Python binding of libhs, the HiSparse decode-step resolver / swap-in for GB300.

Argument marshalling only: every call goes straight to the C ABI declared in
``include/hs.h`` (same names), and every step of the path runs in the library's CUDA
kernels. Arguments that are device arrays accept a torch CUDA tensor (its
``data_ptr()``) or a raw address; host pools accept a numpy array or a raw address;
``stream`` accepts a ``torch.cuda.Stream``, a raw ``cudaStream_t`` or None (the legacy
default stream). A non-OK status raises :class:`HsError` carrying the status code.

The in-tree ``libhs.so`` is loaded on first use; every entry point raises ImportError
if it has not been built (``python -m hierarchical_sparse_attention_gb300.build``).
There is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhs.so")

HS_OK, HS_ERR_INVALID_ARG, HS_ERR_INVALID_CONFIG, HS_ERR_CUDA, HS_ERR_DEVICE_FLAGGED, HS_ERR_TIMEOUT = range(6)
HS_FLAG_TOKEN, HS_FLAG_DUP, HS_FLAG_STATE, HS_FLAG_HOSTROW, HS_FLAG_DEVROW, HS_FLAG_SEQLEN = 1, 2, 4, 8, 16, 32
HS_FLAG_ORDER = 64
HS_FLAG_TIMEOUT = 128
HS_MAX_MLA_SPLITS = 16
HS_MAX_TOP_K, HS_MAX_HOT_SLOTS, HS_MAX_LAYERS = 4096, 16384, 8

# Every symbol include/hs.h declares (checked against the library by the tests).
EXPORTS = ("hs_workspace_bytes", "hs_create", "hs_resolve", "hs_backup", "hs_get_error", "hs_destroy",
           "hs_status_str", "hs_host_register", "hs_host_unregister", "hs_resolve_noalloc",
           "hs_invalidate_tokens", "hs_invalidate_host_rows", "hs_resolve_layers", "hs_gather",
           "hs_resolve_spec", "hs_backup_spec", "hs_reset_hints", "hs_sparse_mla_workspace_bytes",
           "hs_sparse_mla_decode", "hs_launch_shape", "hs_resolve_spec_layers", "hs_gather_spec",
           "hs_host_numa_node", "hs_host_bind_node", "hs_sparse_mla_launches")
HS_MAX_SPEC_QUERIES = 8
HS_NOALLOC_MAX_LAYERS = 8


class hs_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("max_requests", "top_k", "hot_slots", "row_bytes", "num_layers",
                                              "page_size", "max_context", "max_pages", "host_row_stride")]


class HsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {hs_status_str(status)} (status {status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m hierarchical_sparse_attention_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(hs_config)
    lib.hs_workspace_bytes.argtypes = [cfgp]
    lib.hs_workspace_bytes.restype = sz
    lib.hs_create.argtypes = [cfgp, P, P, i64, i64, P, ctypes.POINTER(P)]
    lib.hs_create.restype = ctypes.c_int
    lib.hs_resolve.argtypes = [P, i32] + [P] * 10 + [P]
    lib.hs_resolve.restype = ctypes.c_int
    lib.hs_backup.argtypes = [P, i32, P, P, P, P, P]
    lib.hs_backup.restype = ctypes.c_int
    lib.hs_resolve_layers.argtypes = [P, i32] + [P] * 10 + [i32, P]
    lib.hs_resolve_layers.restype = ctypes.c_int
    lib.hs_gather.argtypes = [P, i32, P, i32, i32, P]
    lib.hs_sparse_mla_workspace_bytes.argtypes = [i32, i32, i32]
    lib.hs_sparse_mla_workspace_bytes.restype = sz
    lib.hs_sparse_mla_launches.argtypes = [i32, i32, i32]
    lib.hs_sparse_mla_launches.restype = i32
    lib.hs_sparse_mla_decode.argtypes = [i32, i32, i32, i32, P, P, i64, P, ctypes.c_float, P, P, P, sz, P, P]
    lib.hs_sparse_mla_decode.restype = ctypes.c_int
    lib.hs_reset_hints.argtypes = [P, P]
    lib.hs_reset_hints.restype = ctypes.c_int
    lib.hs_launch_shape.argtypes = [P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    lib.hs_launch_shape.restype = ctypes.c_int
    lib.hs_resolve_spec.argtypes = [P, i32, i32] + [P] * 10 + [P]
    lib.hs_resolve_spec.restype = ctypes.c_int
    lib.hs_resolve_spec_layers.argtypes = [P, i32, i32] + [P] * 10 + [i32, P]
    lib.hs_resolve_spec_layers.restype = ctypes.c_int
    lib.hs_gather_spec.argtypes = [P, i32, P, i32, i32, i32, P]
    lib.hs_gather_spec.restype = ctypes.c_int
    lib.hs_backup_spec.argtypes = [P, i32, i32] + [P] * 5 + [P]
    lib.hs_backup_spec.restype = ctypes.c_int
    lib.hs_gather.restype = ctypes.c_int
    lib.hs_invalidate_tokens.argtypes = [P, i32] + [P] * 5 + [P]
    lib.hs_invalidate_tokens.restype = ctypes.c_int
    lib.hs_invalidate_host_rows.argtypes = [P, i32, P, P, P, i32, P, P, P]
    lib.hs_invalidate_host_rows.restype = ctypes.c_int
    lib.hs_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    lib.hs_get_error.restype = ctypes.c_int
    lib.hs_destroy.argtypes = [P]
    lib.hs_destroy.restype = ctypes.c_int
    lib.hs_status_str.argtypes = [ctypes.c_int]
    lib.hs_status_str.restype = ctypes.c_char_p
    lib.hs_host_register.argtypes = [P, sz, ctypes.POINTER(P)]
    lib.hs_host_register.restype = ctypes.c_int
    lib.hs_host_unregister.argtypes = [P]
    lib.hs_host_unregister.restype = ctypes.c_int
    lib.hs_host_numa_node.argtypes = [i32, ctypes.POINTER(i32)]
    lib.hs_host_numa_node.restype = ctypes.c_int
    lib.hs_host_bind_node.argtypes = [P, sz, i32]
    lib.hs_host_bind_node.restype = ctypes.c_int
    lib.hs_resolve_noalloc.argtypes = [cfgp, P, P, i64, i64, i32] + [P] * 11 + [P]
    lib.hs_resolve_noalloc.restype = ctypes.c_int
    return lib


class _Lazy:
    """Loads libhs.so on first attribute access (so the build module imports without it)."""

    _cdll = None

    def __getattr__(self, name):
        if _Lazy._cdll is None:
            _Lazy._cdll = _load()
        return getattr(_Lazy._cdll, name)


_lib = _Lazy()


def _addr(x) -> Optional[int]:
    """Raw address of a torch tensor, numpy array or int; None stays None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("arrays passed to libhs must be contiguous")
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        if not x.flags.c_contiguous:
            raise ValueError("arrays passed to libhs must be contiguous")
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, what: str) -> None:
    if status != HS_OK:
        raise HsError(status, what)


def hs_status_str(status: int) -> str:
    return _lib.hs_status_str(status).decode()


def make_config(max_requests: int, top_k: int, hot_slots: int, row_bytes: int, num_layers: int = 1,
                page_size: int = 0, max_context: int = 0, max_pages: int = 0, host_row_stride: int = 0) -> hs_config:
    """host_row_stride: bytes between host rows of one layer (0: row_bytes, one pool per layer;
    num_layers * row_bytes with pools base + l * row_bytes: every layer of a token in one row)."""
    return hs_config(max_requests, top_k, hot_slots, row_bytes, num_layers, page_size, max_context, max_pages,
                     host_row_stride)


def hs_workspace_bytes(cfg: hs_config) -> int:
    return int(_lib.hs_workspace_bytes(ctypes.byref(cfg)))


class Handle:
    """Owns the C handle; the pools, tables and workspace stay the caller's."""

    def __init__(self, ptr: int, cfg: hs_config):
        self.ptr = ptr
        self.cfg = cfg

    def __del__(self):
        if getattr(self, "ptr", None):
            _lib.hs_destroy(self.ptr)
            self.ptr = None


def hs_create(cfg: hs_config, host_pools: Sequence, device_pools: Sequence, host_rows: int, device_rows: int,
              workspace) -> Handle:
    hp = (ctypes.c_void_p * len(host_pools))(*[_addr(p) for p in host_pools])
    dp = (ctypes.c_void_p * len(device_pools))(*[_addr(p) for p in device_pools])
    out = ctypes.c_void_p()
    _check(_lib.hs_create(ctypes.byref(cfg), hp if len(host_pools) else None, dp if len(device_pools) else None,
                          host_rows, device_rows, _addr(workspace), ctypes.byref(out)), "hs_create")
    return Handle(out.value, cfg)


def hs_resolve(h: Handle, num_requests: int, top_k_tokens, seq_lens, host_cache_locs, device_buffer_locs,
               device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows, miss_counts,
               stream=None) -> None:
    _check(_lib.hs_resolve(h.ptr if h else None, num_requests, _addr(top_k_tokens), _addr(seq_lens),
                           _addr(host_cache_locs), _addr(device_buffer_locs), _addr(device_buffer_tokens),
                           _addr(lru_slots), _addr(lru_clock), _addr(resident_pages), _addr(out_rows),
                           _addr(miss_counts), _stream(stream)), "hs_resolve")


def hs_resolve_layers(h: Handle, num_requests: int, top_k_tokens, seq_lens, host_cache_locs, device_buffer_locs,
                      device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows, miss_counts,
                      copy_layers: int, stream=None) -> None:
    _check(_lib.hs_resolve_layers(h.ptr if h else None, num_requests, _addr(top_k_tokens), _addr(seq_lens),
                                  _addr(host_cache_locs), _addr(device_buffer_locs), _addr(device_buffer_tokens),
                                  _addr(lru_slots), _addr(lru_clock), _addr(resident_pages), _addr(out_rows),
                                  _addr(miss_counts), copy_layers, _stream(stream)), "hs_resolve_layers")


def hs_resolve_spec(h: Handle, num_requests: int, num_queries: int, top_k_tokens, committed_lens, host_cache_locs,
                    device_buffer_locs, device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows,
                    miss_counts, stream=None) -> None:
    _check(_lib.hs_resolve_spec(h.ptr if h else None, num_requests, num_queries, _addr(top_k_tokens),
                                _addr(committed_lens), _addr(host_cache_locs), _addr(device_buffer_locs),
                                _addr(device_buffer_tokens), _addr(lru_slots), _addr(lru_clock),
                                _addr(resident_pages), _addr(out_rows), _addr(miss_counts), _stream(stream)),
           "hs_resolve_spec")


def hs_resolve_spec_layers(h: Handle, num_requests: int, num_queries: int, top_k_tokens, committed_lens,
                           host_cache_locs, device_buffer_locs, device_buffer_tokens, lru_slots, lru_clock,
                           resident_pages, out_rows, miss_counts, copy_layers: int, stream=None) -> None:
    _check(_lib.hs_resolve_spec_layers(h.ptr if h else None, num_requests, num_queries, _addr(top_k_tokens),
                                       _addr(committed_lens), _addr(host_cache_locs), _addr(device_buffer_locs),
                                       _addr(device_buffer_tokens), _addr(lru_slots), _addr(lru_clock),
                                       _addr(resident_pages), _addr(out_rows), _addr(miss_counts), copy_layers,
                                       _stream(stream)), "hs_resolve_spec_layers")


def hs_gather_spec(h: Handle, num_requests: int, host_cache_locs, query: int, first_layer: int, num_layers: int,
                   stream=None) -> None:
    _check(_lib.hs_gather_spec(h.ptr if h else None, num_requests, _addr(host_cache_locs), query, first_layer,
                               num_layers, _stream(stream)), "hs_gather_spec")


def hs_backup_spec(h: Handle, num_requests: int, num_queries: int, committed_lens, accepted, host_cache_locs,
                   device_buffer_locs, resident_pages, stream=None) -> None:
    _check(_lib.hs_backup_spec(h.ptr if h else None, num_requests, num_queries, _addr(committed_lens),
                               _addr(accepted), _addr(host_cache_locs), _addr(device_buffer_locs),
                               _addr(resident_pages), _stream(stream)), "hs_backup_spec")


def hs_gather(h: Handle, num_requests: int, host_cache_locs, first_layer: int, num_layers: int,
              stream=None) -> None:
    _check(_lib.hs_gather(h.ptr if h else None, num_requests, _addr(host_cache_locs), first_layer, num_layers,
                          _stream(stream)), "hs_gather")


def hs_backup(h: Handle, num_requests: int, seq_lens, host_cache_locs, device_buffer_locs, resident_pages,
              stream=None) -> None:
    _check(_lib.hs_backup(h.ptr if h else None, num_requests, _addr(seq_lens), _addr(host_cache_locs),
                          _addr(device_buffer_locs), _addr(resident_pages), _stream(stream)), "hs_backup")


def hs_invalidate_tokens(h: Handle, num_requests: int, seq_lens, token_offsets, tokens, device_buffer_tokens,
                         lru_slots, stream=None) -> None:
    _check(_lib.hs_invalidate_tokens(h.ptr if h else None, num_requests, _addr(seq_lens), _addr(token_offsets),
                                     _addr(tokens), _addr(device_buffer_tokens), _addr(lru_slots),
                                     _stream(stream)), "hs_invalidate_tokens")


def hs_invalidate_host_rows(h: Handle, num_requests: int, seq_lens, host_cache_locs, rows, n: int,
                            device_buffer_tokens, lru_slots, stream=None) -> None:
    _check(_lib.hs_invalidate_host_rows(h.ptr if h else None, num_requests, _addr(seq_lens), _addr(host_cache_locs),
                                        _addr(rows), n, _addr(device_buffer_tokens), _addr(lru_slots),
                                        _stream(stream)), "hs_invalidate_host_rows")


def hs_sparse_mla_workspace_bytes(num_requests: int, num_heads: int, splits: int) -> int:
    return int(_lib.hs_sparse_mla_workspace_bytes(num_requests, num_heads, splits))


def hs_sparse_mla_launches(num_requests: int, num_heads: int, splits: int) -> int:
    """Kernel launches of one hs_sparse_mla_decode call of this shape on the current device."""
    return int(_lib.hs_sparse_mla_launches(num_requests, num_heads, splits))


def hs_sparse_mla_decode(num_requests: int, num_heads: int, top_k: int, splits: int, q, kv_pool, pool_rows: int,
                         out_rows, sm_scale: float, o, lse, workspace, workspace_bytes: int, error_flags,
                         stream=None) -> None:
    _check(_lib.hs_sparse_mla_decode(num_requests, num_heads, top_k, splits, _addr(q), _addr(kv_pool), pool_rows,
                                     _addr(out_rows), float(sm_scale), _addr(o), _addr(lse), _addr(workspace),
                                     workspace_bytes, _addr(error_flags), _stream(stream)), "hs_sparse_mla_decode")


def hs_reset_hints(h: Handle, stream=None) -> None:
    _check(_lib.hs_reset_hints(h.ptr if h else None, _stream(stream)), "hs_reset_hints")


def hs_launch_shape(h: Handle):
    """(copy CTAs per request, kernel launches per hs_resolve) chosen by hs_create."""
    c, n = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(_lib.hs_launch_shape(h.ptr if h else None, ctypes.byref(c), ctypes.byref(n)), "hs_launch_shape")
    return int(c.value), int(n.value)


def hs_get_error(h: Handle, clear: bool = False) -> int:
    """The sticky HS_FLAG_* word (synchronises the device)."""
    flags = ctypes.c_uint32(0)
    st = _lib.hs_get_error(h.ptr, ctypes.byref(flags), 1 if clear else 0)
    if st not in (HS_OK, HS_ERR_DEVICE_FLAGGED):
        raise HsError(st, "hs_get_error")
    return int(flags.value)


def hs_destroy(h: Handle) -> None:
    if h and h.ptr:
        _check(_lib.hs_destroy(h.ptr), "hs_destroy")
        h.ptr = None


def hs_host_register(host_array, nbytes: Optional[int] = None) -> int:
    """Pin and map a host range for the kernels; returns its device-side address."""
    ptr = _addr(host_array)
    if nbytes is None:
        nbytes = host_array.nbytes
    dev = ctypes.c_void_p()
    _check(_lib.hs_host_register(ptr, nbytes, ctypes.byref(dev)), "hs_host_register")
    return int(dev.value)


def hs_host_unregister(host_array) -> None:
    _check(_lib.hs_host_unregister(_addr(host_array)), "hs_host_unregister")


def hs_host_numa_node(device: int) -> int:
    """The host memory node nearest `device`, or -1 when the platform does not say."""
    n = ctypes.c_int32(-1)
    _check(_lib.hs_host_numa_node(device, ctypes.byref(n)), "hs_host_numa_node")
    return int(n.value)


def hs_host_bind_node(addr, nbytes: int, node: int) -> None:
    """Prefer memory node `node` for the untouched pages of [addr, addr + nbytes)."""
    _check(_lib.hs_host_bind_node(_addr(addr), nbytes, node), "hs_host_bind_node")


def hs_resolve_noalloc(cfg: hs_config, host_pools: Sequence, device_pools: Sequence, host_rows: int,
                       device_rows: int, num_requests: int, top_k_tokens, seq_lens, host_cache_locs,
                       device_buffer_locs, device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows,
                       miss_counts, error_flags=None, stream=None) -> None:
    """hs_resolve without a handle or workspace, for callers that cannot allocate device
    memory: the library keeps the scratch in its own device array (see include/hs.h)."""
    hp = (ctypes.c_void_p * len(host_pools))(*[_addr(p) for p in host_pools])
    dp = (ctypes.c_void_p * len(device_pools))(*[_addr(p) for p in device_pools])
    _check(_lib.hs_resolve_noalloc(ctypes.byref(cfg), hp if len(host_pools) else None,
                                   dp if len(device_pools) else None, host_rows, device_rows, num_requests,
                                   _addr(top_k_tokens), _addr(seq_lens), _addr(host_cache_locs),
                                   _addr(device_buffer_locs), _addr(device_buffer_tokens), _addr(lru_slots),
                                   _addr(lru_clock), _addr(resident_pages), _addr(out_rows), _addr(miss_counts),
                                   _addr(error_flags), _stream(stream)), "hs_resolve_noalloc")
