"""Step driver shared by the CPU and GPU tests.

It plays the caller around the resolver: it owns the host pools, the device pool
(a numpy model for the oracle, a torch tensor for the library), the slot map,
stamps and clock, and before every step it does what the forward pass does --
writes the newest token's row into its device location and overwrites that
token's host row with poison, which the step's eager backup must restore.
"""
from __future__ import annotations

import numpy as np

import workloads as W


def host_pools_for(wl: W.Workload, nthreads: int = 0, with_bases: bool = False):
    """Plain (unpinned) host pools holding every token's row: one array per layer, or for a
    page-first layout per-layer views of one array. with_bases: also return the distinct
    arrays behind the views."""
    if wl.cfg.host_layout == "page_first":
        base = np.zeros(wl.host_pool_bytes, dtype=np.uint8)
        views = wl.host_layer_views(base)
        for layer, v in enumerate(views):
            wl.fill_host_pool(layer, v, nthreads)
        return (views, [base]) if with_bases else views
    pools = []
    for layer in range(wl.L):
        p = np.zeros(wl.host_rows * wl.B, dtype=np.uint8)
        wl.fill_host_pool(layer, p, nthreads)
        pools.append(p)
    return (pools, list(pools)) if with_bases else pools


def device_pool_model(wl: W.Workload):
    pools = []
    rq, tk, rows = wl.initial_device_writes()
    for layer in range(wl.L):
        p = np.full(wl.device_rows * wl.B, W.POISON_DEVICE, dtype=np.uint8)
        wl.scatter_rows(layer, rq, tk, rows, p)
        pools.append(p)
    return pools


def newest_writes(wl: W.Workload, step: int):
    """(requests, tokens, device rows) of the rows the forward pass writes before `step`."""
    S = wl.seq_lens(step)
    rq = np.arange(wl.R, dtype=np.int32)
    tk = (S - 1).astype(np.int32)
    rows = np.array([wl.newest_device_row(r, int(S[r])) for r in range(wl.R)], dtype=np.int64)
    return rq, tk, rows


def poison_host_newest(wl: W.Workload, step: int, host_pools):
    S = wl.seq_lens(step)
    for r in range(wl.R):
        h = int(wl.host_cache_locs[r, int(S[r]) - 1])
        for p in host_pools:
            wl.host_row_bytes_of(p, h)[:] = W.POISON_HOST


def host_newest_ok(wl: W.Workload, step: int, host_pools) -> bool:
    S = wl.seq_lens(step)
    for r in range(wl.R):
        t = int(S[r]) - 1
        h = int(wl.host_cache_locs[r, t])
        for layer, p in enumerate(host_pools):
            if not np.array_equal(wl.host_row_bytes_of(p, h), wl.rows(layer, r, [t])[0]):
                return False
    return True


class OracleSim:
    """The oracle run over a workload, step by step (all arrays numpy)."""

    def __init__(self, wl: W.Workload, host_pools=None, nthreads: int = 0):
        """host_pools: per-layer host pools to use; by default the run fills its own, so no
        other party (the GPU run in particular) ever writes the bytes it reads."""
        import oracle
        self.wl = wl
        if host_pools is not None:
            self.host, self.host_bases = host_pools, list(host_pools)
        else:
            self.host, self.host_bases = host_pools_for(wl, nthreads, with_bases=True)
        self.dev = device_pool_model(wl)
        self.tokens, self.stamps, self.clock = wl.initial_state()
        stride = wl.host_row_stride if wl.cfg.host_layout == "page_first" else 0
        self.orc = oracle.Oracle(wl.K, wl.H, wl.B, wl.L, wl.max_context, wl.host_rows, wl.device_rows,
                                 wl.ps, wl.max_pages, stride)
        self.out = np.full((wl.R, wl.K), -1, dtype=np.int32)
        self.miss = np.zeros(wl.R, dtype=np.int32)

    def write_newest(self, step: int):
        rq, tk, rows = newest_writes(self.wl, step)
        for layer, p in enumerate(self.dev):
            self.wl.scatter_rows(layer, rq, tk, rows, p)

    def resolve(self, step: int, top_k=None, seq_lens=None, host_cache_locs=None,
                device_buffer_locs=None, resident_pages="default") -> int:
        wl = self.wl
        tk = wl.top_k_tokens(step) if top_k is None else top_k
        S = wl.seq_lens(step) if seq_lens is None else seq_lens
        hcl = wl.host_cache_locs if host_cache_locs is None else host_cache_locs
        dbl = wl.device_buffer_locs if device_buffer_locs is None else device_buffer_locs
        rp = wl.resident_pages if isinstance(resident_pages, str) else resident_pages
        return self.orc.resolve(tk, S, hcl, dbl, self.tokens, self.stamps, self.clock, rp, self.out,
                                self.miss, self.host, self.dev)

    def backup(self, step: int, seq_lens=None) -> int:
        wl = self.wl
        S = wl.seq_lens(step) if seq_lens is None else seq_lens
        return self.orc.backup(S, wl.host_cache_locs, wl.device_buffer_locs, wl.resident_pages,
                               self.host, self.dev)

    def step(self, step: int, poison: bool = True) -> int:
        self.write_newest(step)
        if poison:
            poison_host_newest(self.wl, step, self.host)
        err = self.resolve(step)
        if self.wl.cfg.backup:
            err |= self.backup(step)
        return err

    def dev_row(self, layer: int, row: int) -> np.ndarray:
        B = self.wl.B
        return self.dev[layer][row * B:(row + 1) * B]
