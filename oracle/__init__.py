"""CPU oracle of the HiSparse decode-step resolver -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. The library (``hierarchical_sparse_attention_gb300``) never
does, and the two share no code: the oracle is plain single-threaded C
(``hs_oracle.c``) that follows the pages' steps in order, built with gcc, wrapped
here with ctypes.

Every function here is pinned by the CPU tests (brute force, textbook LRU,
invariants, special cases); see ``hs_oracle.c`` for the sources and readings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

ERR_TOKEN, ERR_DUP, ERR_STATE, ERR_HOSTROW, ERR_DEVROW, ERR_SEQLEN = 1, 2, 4, 8, 16, 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


class Geom(ctypes.Structure):
    _fields_ = [("top_k", ctypes.c_int32), ("hot_slots", ctypes.c_int32),
                ("row_bytes", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_context", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("host_rows", ctypes.c_int64),
                ("device_rows", ctypes.c_int64), ("host_row_stride", ctypes.c_int64)]


def build(force: bool = False) -> str:
    """Compile hs_oracle.c into liboracle.so next to it."""
    src = os.path.join(_HERE, "hs_oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        path = os.environ.get("HS_ORACLE_LIB")  # tests load deliberately broken builds this way
        if not path:
            path = build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.oracle_resolve.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32] + [P] * 13
        lib.oracle_resolve.restype = None
        lib.oracle_resolve_plan.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32] + [P] * 13 + [ctypes.c_int32,
                                                                                                P, P, P]
        lib.oracle_resolve_plan.restype = None
        lib.oracle_resolve_spec.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32, ctypes.c_int32] + [P] * 13
        lib.oracle_resolve_spec.restype = None
        lib.oracle_resolve_spec_plan.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32, ctypes.c_int32] + [P] * 13 + \
            [ctypes.c_int32, P, P, P]
        lib.oracle_resolve_spec_plan.restype = None
        lib.oracle_backup_spec.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32, ctypes.c_int32] + [P] * 8
        lib.oracle_backup_spec.restype = None
        lib.oracle_gather.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32, P, P, P, P, ctypes.c_int32,
                                      ctypes.c_int32, P, P, P]
        lib.oracle_gather.restype = None
        lib.oracle_backup.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32] + [P] * 7
        lib.oracle_backup.restype = None
        lib.oracle_invalidate_tokens.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32] + [P] * 6
        lib.oracle_invalidate_tokens.restype = None
        lib.oracle_invalidate_host_rows.argtypes = [ctypes.POINTER(Geom), ctypes.c_int32, P, P, P,
                                                    ctypes.c_int32, P, P, P]
        lib.oracle_invalidate_host_rows.restype = None
        lib.oracle_hot_bytes_per_request.argtypes = [ctypes.c_int32] * 4
        lib.oracle_hot_bytes_per_request.restype = ctypes.c_int64
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]) -> Optional[int]:
    return None if a is None else a.ctypes.data


def _i32(a: np.ndarray, shape=None) -> np.ndarray:
    assert a.dtype == np.int32 and a.flags.c_contiguous, "int32 C-contiguous array expected"
    if shape is not None:
        assert a.shape == tuple(shape), (a.shape, shape)
    return a


def hot_bytes_per_request(top_k: int, n_spec: int, row_bytes: int, layers: int) -> int:
    return int(_load().oracle_hot_bytes_per_request(top_k, n_spec, row_bytes, layers))


class Plan:
    """A recorded miss plan: per request `count` misses, miss j = (tokens[j], dst[j])."""

    def __init__(self, tokens: np.ndarray, dst: np.ndarray, count: np.ndarray):
        self.tokens, self.dst, self.count = tokens, dst, count


class Oracle:
    """State-free wrapper: the caller owns every array (as with the library)."""

    def __init__(self, top_k: int, hot_slots: int, row_bytes: int, num_layers: int,
                 max_context: int, host_rows: int, device_rows: int, page_size: int = 0,
                 max_pages: int = 0, host_row_stride: int = 0):
        """host_row_stride: bytes between host rows of one layer's pool (0: row_bytes). With
        num_layers * row_bytes the host pools are views base[l * row_bytes:] of one array."""
        assert host_row_stride == 0 or host_row_stride >= row_bytes
        self.g = Geom(top_k, hot_slots, row_bytes, num_layers, page_size, max_context, max_pages,
                      host_rows, device_rows, host_row_stride)
        self.lib = _load()

    def _pools(self, pools: Sequence[np.ndarray], rows: int, stride: int = 0):
        assert len(pools) == self.g.num_layers
        stride = stride or self.g.row_bytes
        for p in pools:
            assert p.dtype == np.uint8 and p.flags.c_contiguous and p.size >= (rows - 1) * stride + self.g.row_bytes
        return (ctypes.c_void_p * len(pools))(*[p.ctypes.data for p in pools])

    def _host(self, pools: Sequence[np.ndarray]):
        return self._pools(pools, self.g.host_rows, self.g.host_row_stride)

    def resolve(self, top_k_tokens, seq_lens, host_cache_locs, device_buffer_locs,
                device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows,
                miss_counts, host_pools, device_pools, copy_layers: Optional[int] = None,
                plan: Optional["Plan"] = None) -> int:
        """One decode step. With copy_layers < num_layers only the leader layers [0,
        copy_layers) get their miss rows; with a Plan the miss plan is recorded for gather()."""
        g = self.g
        R = seq_lens.shape[0]
        _i32(top_k_tokens, (R, g.top_k)); _i32(seq_lens); _i32(host_cache_locs, (R, g.max_context))
        _i32(device_buffer_locs, (R, g.hot_slots + 1)); _i32(device_buffer_tokens, (R, g.hot_slots))
        _i32(lru_slots, (R, g.hot_slots)); _i32(lru_clock, (R,)); _i32(out_rows, (R, g.top_k))
        if resident_pages is not None:
            _i32(resident_pages, (R, g.max_pages))
        if miss_counts is not None:
            _i32(miss_counts, (R,))
        err = ctypes.c_uint32(0)
        hp = self._host(host_pools)
        dp = self._pools(device_pools, g.device_rows)
        args = (ctypes.byref(g), R, _p(top_k_tokens), _p(seq_lens), _p(host_cache_locs),
                _p(device_buffer_locs), _p(device_buffer_tokens), _p(lru_slots), _p(lru_clock),
                _p(resident_pages), _p(out_rows), _p(miss_counts), hp, dp, ctypes.byref(err))
        if copy_layers is None and plan is None:
            self.lib.oracle_resolve(*args)
        else:
            cl = g.num_layers if copy_layers is None else int(copy_layers)
            assert 0 <= cl <= g.num_layers
            if plan is not None:
                _i32(plan.tokens, (R, g.top_k)); _i32(plan.dst, (R, g.top_k)); _i32(plan.count, (R,))
            self.lib.oracle_resolve_plan(*args, cl, _p(plan.tokens) if plan else None,
                                         _p(plan.dst) if plan else None, _p(plan.count) if plan else None)
        return int(err.value)

    def new_plan(self, R: int) -> "Plan":
        return Plan(np.zeros((R, self.g.top_k), np.int32), np.zeros((R, self.g.top_k), np.int32),
                    np.zeros(R, np.int32))

    def gather(self, plan: "Plan", host_cache_locs, first_layer: int, num_layers: int, host_pools,
               device_pools) -> int:
        """Copy the plan's rows for layers [first_layer, first_layer + num_layers)."""
        g = self.g
        R = plan.count.shape[0]
        _i32(host_cache_locs, (R, g.max_context))
        assert 0 <= first_layer and first_layer + num_layers <= g.num_layers
        err = ctypes.c_uint32(0)
        hp = self._host(host_pools)
        dp = self._pools(device_pools, g.device_rows)
        self.lib.oracle_gather(ctypes.byref(g), R, _p(plan.count), _p(plan.tokens), _p(plan.dst),
                               _p(host_cache_locs), first_layer, num_layers, hp, dp, ctypes.byref(err))
        return int(err.value)

    def backup(self, seq_lens, host_cache_locs, device_buffer_locs, resident_pages, host_pools,
               device_pools) -> int:
        g = self.g
        R = seq_lens.shape[0]
        _i32(seq_lens); _i32(host_cache_locs, (R, g.max_context)); _i32(device_buffer_locs, (R, g.hot_slots + 1))
        if resident_pages is not None:
            _i32(resident_pages, (R, g.max_pages))
        err = ctypes.c_uint32(0)
        hp = self._host(host_pools)
        dp = self._pools(device_pools, g.device_rows)
        self.lib.oracle_backup(ctypes.byref(g), R, _p(seq_lens), _p(host_cache_locs),
                               _p(device_buffer_locs), _p(resident_pages), hp, dp, ctypes.byref(err))
        return int(err.value)

    def invalidate_tokens(self, seq_lens, offsets, tokens, device_buffer_tokens, lru_slots) -> int:
        """Request r's tokens tokens[offsets[r]:offsets[r+1]] leave its hot set."""
        g = self.g
        R = seq_lens.shape[0]
        _i32(seq_lens); _i32(offsets, (R + 1,)); _i32(tokens)
        _i32(device_buffer_tokens, (R, g.hot_slots)); _i32(lru_slots, (R, g.hot_slots))
        assert int(offsets[0]) == 0 and int(offsets[-1]) <= tokens.size and np.all(np.diff(offsets) >= 0)
        err = ctypes.c_uint32(0)
        self.lib.oracle_invalidate_tokens(ctypes.byref(g), R, _p(seq_lens), _p(offsets), _p(tokens),
                                          _p(device_buffer_tokens), _p(lru_slots), ctypes.byref(err))
        return int(err.value)

    def invalidate_host_rows(self, seq_lens, host_cache_locs, rows, device_buffer_tokens, lru_slots) -> int:
        """Every slot whose token's host row is in `rows` leaves its request's hot set."""
        g = self.g
        R = seq_lens.shape[0]
        _i32(seq_lens); _i32(host_cache_locs, (R, g.max_context)); _i32(rows)
        _i32(device_buffer_tokens, (R, g.hot_slots)); _i32(lru_slots, (R, g.hot_slots))
        err = ctypes.c_uint32(0)
        self.lib.oracle_invalidate_host_rows(ctypes.byref(g), R, _p(seq_lens), _p(host_cache_locs), _p(rows),
                                             int(rows.size), _p(device_buffer_tokens), _p(lru_slots),
                                             ctypes.byref(err))
        return int(err.value)

    def new_spec_plan(self, Q: int, R: int) -> "Plan":
        """Room for a speculative batch's plans: slice q (tokens[q], dst[q], count[q]) is
        verify step q's miss plan; step_plan(plan, q) views it as a one-step Plan."""
        return Plan(np.zeros((Q, R, self.g.top_k), np.int32), np.zeros((Q, R, self.g.top_k), np.int32),
                    np.zeros((Q, R), np.int32))

    @staticmethod
    def step_plan(plan: "Plan", q: int) -> "Plan":
        return Plan(plan.tokens[q], plan.dst[q], plan.count[q])

    def resolve_spec(self, top_k_tokens, committed_lens, host_cache_locs, device_buffer_locs,
                     device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows, miss_counts,
                     host_pools, device_pools, copy_layers: Optional[int] = None,
                     plan: Optional["Plan"] = None) -> int:
        """A speculative batch of Q = top_k_tokens.shape[0] verify steps, in order: step q
        resolves top_k_tokens[q] for committed_lens + q + 1 tokens into out_rows[q];
        device_buffer_locs is [R, H + Q] (H slots, then Q reserved rows). With copy_layers <
        num_layers each step copies only the leader layers; with a plan (new_spec_plan) each
        step records its miss plan in its slice, for gather(step_plan(plan, q), ...)."""
        g = self.g
        Q, R = top_k_tokens.shape[0], committed_lens.shape[0]
        _i32(top_k_tokens, (Q, R, g.top_k)); _i32(committed_lens); _i32(host_cache_locs, (R, g.max_context))
        _i32(device_buffer_locs, (R, g.hot_slots + Q)); _i32(device_buffer_tokens, (R, g.hot_slots))
        _i32(lru_slots, (R, g.hot_slots)); _i32(lru_clock, (R,)); _i32(out_rows, (Q, R, g.top_k))
        if resident_pages is not None:
            _i32(resident_pages, (R, g.max_pages))
        if miss_counts is not None:
            _i32(miss_counts, (Q, R))
        err = ctypes.c_uint32(0)
        hp = self._host(host_pools)
        dp = self._pools(device_pools, g.device_rows)
        args = (ctypes.byref(g), R, Q, _p(top_k_tokens), _p(committed_lens), _p(host_cache_locs),
                _p(device_buffer_locs), _p(device_buffer_tokens), _p(lru_slots), _p(lru_clock),
                _p(resident_pages), _p(out_rows), _p(miss_counts), hp, dp, ctypes.byref(err))
        if copy_layers is None and plan is None:
            self.lib.oracle_resolve_spec(*args)
        else:
            cl = g.num_layers if copy_layers is None else int(copy_layers)
            assert 0 <= cl <= g.num_layers
            if plan is not None:
                _i32(plan.tokens, (Q, R, g.top_k)); _i32(plan.dst, (Q, R, g.top_k)); _i32(plan.count, (Q, R))
            self.lib.oracle_resolve_spec_plan(*args, cl, _p(plan.tokens) if plan else None,
                                              _p(plan.dst) if plan else None, _p(plan.count) if plan else None)
        return int(err.value)

    def backup_spec(self, num_queries: int, committed_lens, accepted, host_cache_locs, device_buffer_locs,
                    resident_pages, host_pools, device_pools) -> int:
        """Back up the first accepted[r] positions of a speculative batch of num_queries."""
        g = self.g
        R = committed_lens.shape[0]
        _i32(committed_lens); _i32(accepted, (R,)); _i32(host_cache_locs, (R, g.max_context))
        _i32(device_buffer_locs, (R, g.hot_slots + num_queries))
        if resident_pages is not None:
            _i32(resident_pages, (R, g.max_pages))
        err = ctypes.c_uint32(0)
        hp = self._host(host_pools)
        dp = self._pools(device_pools, g.device_rows)
        self.lib.oracle_backup_spec(ctypes.byref(g), R, num_queries, _p(committed_lens), _p(accepted),
                                    _p(host_cache_locs), _p(device_buffer_locs), _p(resident_pages), hp, dp,
                                    ctypes.byref(err))
        return int(err.value)
