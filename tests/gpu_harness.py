"""GPU side of the step driver: the library called through its C ABI binding.

Host pools are page-aligned anonymous mappings, registered (pinned + mapped) with
hs_host_register and shared with the oracle run, which reads the same bytes.
"""
from __future__ import annotations

import numpy as np
import torch

import hierarchical_sparse_attention_gb300 as hs
import workloads as W
from harness import newest_writes


_POOLS = {}  # data address -> workloads.HostPool (keeps the memory alive, knows how it was pinned)


def alloc_host(nbytes: int) -> np.ndarray:
    """Host bytes for a KV pool (huge pages when the host gives the whole pool, else
    driver-pinned memory; see workloads.HostPool)."""
    pool = W.HostPool(nbytes)
    _POOLS[pool.array.ctypes.data] = pool
    return pool.array


def needs_register(arr: np.ndarray) -> bool:
    pool = _POOLS.get(arr.ctypes.data)
    return True if pool is None else pool.needs_register


def host_pools(wl: W.Workload, nthreads: int = 0):
    pools = []
    for layer in range(wl.L):
        p = alloc_host(wl.host_rows * wl.B)
        wl.fill_host_pool(layer, p, nthreads)
        pools.append(p)
    return pools


class GpuSim:
    def __init__(self, wl: W.Workload, host, dev_init, device: str = "cuda", host_io: bool = False):
        """host_io: the step's top-k, seq_lens, row table and miss counts live in pinned host
        memory, which the kernels read and write directly (zero-copy step I/O)."""
        self.wl = wl
        self.host = host
        self.registered = []
        for p in host:
            if needs_register(p):
                hs.hs_host_register(p)
                self.registered.append(p)
        dev = torch.device(device)
        self.dev = [torch.from_numpy(np.ascontiguousarray(m)).to(dev) for m in dev_init]
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
        self.cfg = hs.make_config(wl.R, wl.K, wl.H, wl.B, wl.L, wl.ps, wl.max_context, wl.max_pages)
        self.ws = torch.zeros(hs.hs_workspace_bytes(self.cfg), dtype=torch.uint8, device=dev)
        self.h = hs.hs_create(self.cfg, host, self.dev, wl.host_rows, wl.device_rows, self.ws)

    def close(self):
        hs.hs_destroy(self.h)
        for p in self.registered:
            hs.hs_host_unregister(p)
        self.registered = []

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
