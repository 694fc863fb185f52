"""GPU side of the step driver: the library called through its C ABI binding.

Host pools are page-aligned anonymous mappings, registered (pinned + mapped) with
hs_host_register. The oracle run never reads them: it keeps its own plain copies
(harness.OracleSim), so a stray GPU write into host memory shows up as a difference.

Every pool carries guard rows: GUARD_ROWS rows of CANARY bytes before and after each host
pool and each device pool, and a CANARY tail after the workspace. The library is given only
the inner rows; check_guards() proves that nothing was written outside them.
"""
from __future__ import annotations

import numpy as np
import torch

import hierarchical_sparse_attention_gb300 as hs
import workloads as W
from harness import newest_writes

GUARD_ROWS = 16  # a multiple of 16 bytes for every row size, so inner pools stay 16-byte aligned
CANARY = 0xC3    # differs from the host and device poison bytes
WS_GUARD = 4096

_POOLS = {}  # inner data address -> (workloads.HostPool, guard bytes)


def alloc_host(nbytes: int, guard: int = 0) -> np.ndarray:
    """Host bytes for a KV pool (huge pages when the host gives the whole pool, else
    driver-pinned memory; see workloads.HostPool), with `guard` CANARY bytes on each side.
    Returns the inner `nbytes` bytes."""
    pool = W.HostPool(nbytes + 2 * guard)
    full = pool.array
    if not pool.needs_register:
        full[:] = 0  # driver-pinned memory is not zeroed; an anonymous mapping is
    if guard:
        full[:guard] = CANARY
        full[guard + nbytes:] = CANARY
    inner = full[guard:guard + nbytes]
    _POOLS[inner.ctypes.data] = (pool, guard)
    return inner


def _entry(arr: np.ndarray):
    return _POOLS.get(arr.ctypes.data)


def needs_register(arr: np.ndarray) -> bool:
    e = _entry(arr)
    return True if e is None else e[0].needs_register


def registration_span(arr: np.ndarray):
    """(array, nbytes) to register for a host pool made here: the whole mapping, guards included."""
    e = _entry(arr)
    if e is None:
        return arr, arr.nbytes
    return e[0].array, e[0].array.nbytes


def guards_intact(arr: np.ndarray) -> bool:
    e = _entry(arr)
    if e is None or not e[1]:
        return True
    full, g = e[0].array, e[1]
    return bool(np.all(full[:g] == CANARY) and np.all(full[full.size - g:] == CANARY))


def free_host(arrays) -> None:
    """Release host pools made by alloc_host (after every GpuSim using them is closed)."""
    for a in arrays:
        e = _POOLS.pop(a.ctypes.data, None)
        if e is not None:
            e[0].free()


def host_pools(wl: W.Workload, nthreads: int = 0):
    """The workload's host pools for the GPU: one guarded pool per layer, or for a page-first
    layout one guarded pool and its per-layer views. Returns (per-layer pools, base arrays)."""
    guard = GUARD_ROWS * wl.host_row_stride
    if wl.cfg.host_layout == "page_first":
        base = alloc_host(wl.host_pool_bytes, guard)
        views = wl.host_layer_views(base)
        for layer, v in enumerate(views):
            wl.fill_host_pool(layer, v, nthreads)
        return views, [base]
    pools = []
    for layer in range(wl.L):
        p = alloc_host(wl.host_rows * wl.B, guard)
        wl.fill_host_pool(layer, p, nthreads)
        pools.append(p)
    return pools, list(pools)


class GpuSim:
    def __init__(self, wl: W.Workload, host, dev_init, device: str = "cuda", host_io: bool = False,
                 host_bases=None):
        """host: per-layer host pools (views of one array for a page-first layout);
        host_bases: the distinct arrays behind them (default: host itself).
        host_io: the step's top-k, seq_lens, row table and miss counts live in pinned host
        memory, which the kernels read and write directly (zero-copy step I/O)."""
        self.wl = wl
        self.host = host
        self.host_bases = list(host_bases) if host_bases is not None else list(host)
        self.registered = []
        for p in self.host_bases:
            if needs_register(p):
                arr, n = registration_span(p)
                hs.hs_host_register(arr, n)
                self.registered.append(arr)
        dev = torch.device(device)
        G, B = GUARD_ROWS, wl.B
        self._dev_full = []
        self.dev = []
        for m in dev_init:
            full = torch.full(((wl.device_rows + 2 * G) * B,), CANARY, dtype=torch.uint8, device=dev)
            inner = full[G * B:(G + wl.device_rows) * B]
            inner.copy_(torch.from_numpy(np.ascontiguousarray(m)))
            self._dev_full.append(full)
            self.dev.append(inner)
        self.hcl = torch.from_numpy(wl.host_cache_locs).to(dev)
        self.dbl = torch.from_numpy(wl.device_buffer_locs).to(dev)
        self.rp = None if wl.resident_pages is None else torch.from_numpy(wl.resident_pages).to(dev)
        tok, st, clk = wl.initial_state()
        self.tok = torch.from_numpy(tok).to(dev)
        self.st = torch.from_numpy(st).to(dev)
        self.clk = torch.from_numpy(clk).to(dev)
        io = (lambda t: t.pin_memory()) if host_io else (lambda t: t.to(dev))
        self.out = io(torch.full((wl.R, wl.K), -7, dtype=torch.int32))
        self.miss = io(torch.full((wl.R,), -7, dtype=torch.int32))
        self.tk = io(torch.empty((wl.R, wl.K), dtype=torch.int32))
        self.sl = io(torch.empty((wl.R,), dtype=torch.int32))
        stride = wl.host_row_stride if wl.cfg.host_layout == "page_first" else 0
        self.cfg = hs.make_config(wl.R, wl.K, wl.H, wl.B, wl.L, wl.ps, wl.max_context, wl.max_pages, stride)
        nws = hs.hs_workspace_bytes(self.cfg)
        self._ws_full = torch.full((nws + WS_GUARD,), CANARY, dtype=torch.uint8, device=dev)
        self.ws = self._ws_full[:nws]
        self.h = hs.hs_create(self.cfg, host, self.dev, wl.host_rows, wl.device_rows, self.ws)

    def close(self):
        if self.h is not None:
            hs.hs_destroy(self.h)
            self.h = None
        for p in self.registered:
            hs.hs_host_unregister(p)
        self.registered = []

    def check_guards(self, what: str = "") -> None:
        """No byte outside the pools and the workspace the library was given has changed."""
        G, B, R = GUARD_ROWS, self.wl.B, self.wl.device_rows
        for layer, full in enumerate(self._dev_full):
            head, tail = full[:G * B], full[(G + R) * B:]
            assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), \
                f"{what}: device pool {layer} written outside its rows"
        assert bool((self._ws_full[self.ws.numel():] == CANARY).all()), f"{what}: written past the workspace"
        for i, p in enumerate(self.host_bases):
            assert guards_intact(p), f"{what}: host pool {i} written outside its rows"

    def write_newest(self, step: int):
        rq, tk, rows = newest_writes(self.wl, step)
        idx = torch.from_numpy(rows).to(self.dev[0].device)
        for layer, pool in enumerate(self.dev):
            data = np.concatenate([self.wl.rows(layer, int(r), [int(t)]) for r, t in zip(rq, tk)])
            pool.view(-1, self.wl.B)[idx] = torch.from_numpy(data).to(pool.device)

    def upload(self, step: int, top_k=None, seq_lens=None):
        wl = self.wl
        self.tk.copy_(torch.from_numpy(wl.top_k_tokens(step) if top_k is None else top_k))
        self.sl.copy_(torch.from_numpy(wl.seq_lens(step) if seq_lens is None else seq_lens))

    def resolve(self, stream=None, num_requests=None):
        hs.hs_resolve(self.h, self.wl.R if num_requests is None else num_requests, self.tk, self.sl, self.hcl,
                      self.dbl, self.tok, self.st, self.clk, self.rp, self.out, self.miss, stream)

    def backup(self, stream=None, num_requests=None):
        hs.hs_backup(self.h, self.wl.R if num_requests is None else num_requests, self.sl, self.hcl, self.dbl,
                     self.rp, stream)

    def state(self):
        return dict(out=self.out.cpu().numpy(), miss=self.miss.cpu().numpy(), tokens=self.tok.cpu().numpy(),
                    stamps=self.st.cpu().numpy(), clock=self.clk.cpu().numpy())


def resolved_rows_ok(wl: W.Workload, gpu: GpuSim, top_k: np.ndarray, out: np.ndarray, what: str = "") -> int:
    """Every row the step resolved, in every layer of the GPU's device pools, holds the exact
    bytes the seeded generator gives its token (regenerated here, not taken from the oracle).
    Returns the number of rows checked."""
    checked = 0
    for layer in range(wl.L):
        pool = gpu.dev[layer].view(-1, wl.B)
        valid = out >= 0
        rows = torch.from_numpy(out[valid].astype(np.int64)).to(pool.device)
        got = pool[rows].cpu().numpy()
        want = np.concatenate([wl.rows(layer, r, top_k[r][valid[r]]) for r in range(out.shape[0])]) \
            if got.shape[0] else got
        if not np.array_equal(got, want):
            bad = np.nonzero((got != want).any(1))[0]
            raise AssertionError(f"{what}: layer {layer}: {len(bad)} resolved rows hold wrong bytes")
        checked += got.shape[0]
    return checked


def make_pair(wl: W.Workload, host_io: bool = False):
    """An oracle run with its own host pools and a GPU run with guarded, pinned ones.
    Returns (orc, gpu); close with close_pair."""
    from harness import OracleSim
    host, bases = host_pools(wl)
    orc = OracleSim(wl)
    gpu = GpuSim(wl, host, orc.dev, host_io=host_io, host_bases=bases)
    return orc, gpu


def close_pair(gpu: GpuSim) -> None:
    gpu.close()
    free_host(gpu.host_bases)


def final_host_check(orc, gpu: GpuSim, what: str = "") -> None:
    """Whole host pools: the GPU's (written only by the backups) equal the oracle's own copies,
    and no guard changed."""
    for i, (g, o) in enumerate(zip(gpu.host_bases, orc.host_bases)):
        if not np.array_equal(g, o):
            B = gpu.wl.host_row_stride
            bad = np.nonzero((g[: g.size // B * B].reshape(-1, B) != o[: o.size // B * B].reshape(-1, B)).any(1))[0]
            raise AssertionError(f"{what}: host pool {i} differs from the oracle's in {len(bad)} rows, e.g. {bad[:8]}")
    gpu.check_guards(what)
