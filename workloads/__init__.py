"""Seeded synthetic workloads for the HiSparse decode-step resolver.

This module is input generation only: it holds none of the resolver's method.
It produces, as pure functions of a seed,

* the per-step indexer top-k token positions (with the reuse / window / residency
  mixes of the five workloads below),
* the sequence lengths, the token -> host-row table (``host_cache_locs``), the
  slot -> device-row table (``device_buffer_locs``) and the resident page table,
* the bytes of every KV row (``rowgen.c``), so both the CUDA path and the CPU
  oracle read identical host pools and a check can regenerate any row.

Both the oracle side and the GPU side consume these inputs; neither imports the
other.

Workload shapes (sizes from the vLLM and SGLang HiSparse pages):

=========== ===== ========================= ====== ===== ======= ====== =======
name        R     seq_len at step 0         K      H     B       L      steps
=========== ===== ========================= ====== ===== ======= ====== =======
tiny        2     8192, 100                 64     128   576 u8  1      16
dsa         32    131072                    2048   4096  656     1      64
mixed1m     16    1048576 (page 64, last    2048   4096  656     1      32
                  256 pages GPU-resident)
indexshare  256   U[32768, 65536]           2048   4096  656     4      32
sweep       64    262144                    2048   {2048,4096,6144} x reuse
                                                         {0.5,0.8,0.95,0.99}
                                                         1152 bf16  1   32
=========== ===== ========================= ====== ===== ======= ====== =======
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

FMT_U8, FMT_FP8MLA, FMT_BF16 = 0, 1, 2
FMT_NAMES = {FMT_U8: "u8", FMT_FP8MLA: "fp8mla", FMT_BF16: "bf16"}

HOST_PAGE = 64  # host pool page granularity used to scatter token rows
POISON_HOST = 0x5A  # written over a host row the step's backup must restore
POISON_DEVICE = 0xA5  # fill of device rows nobody has written

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "librowgen.so")
_lib = None


def build_rowgen(force: bool = False) -> str:
    """Compile rowgen.c into librowgen.so next to it (gcc, no -march flags)."""
    src = os.path.join(_HERE, "rowgen.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-pthread", src, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _rowgen():
    global _lib
    if _lib is None:
        build_rowgen()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        lib.rowgen_rows.argtypes = [u64, i32, i32, i32, i32, P, i64, P]
        lib.rowgen_rows.restype = None
        lib.rowgen_scatter.argtypes = [u64, i32, i32, i32, P, P, P, i64, P]
        lib.rowgen_scatter.restype = None
        lib.rowgen_fill_pool.argtypes = [u64, i32, i32, i32, i32, P, P, i32, P, i32, i64]
        lib.rowgen_fill_pool.restype = i32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# --------------------------------------------------------------------------------------
# host pool memory
# --------------------------------------------------------------------------------------
_HUGE = 0


def _huge_page_bytes() -> int:
    global _HUGE
    if not _HUGE:
        try:
            _HUGE = int(open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size").read())
        except (OSError, ValueError):
            _HUGE = 2 << 20
    return _HUGE


def _huge_backed_bytes(addr: int, nbytes: int) -> int:
    """AnonHugePages of the mapping that starts at addr (from /proc/self/smaps)."""
    try:
        lines = open("/proc/self/smaps").read().splitlines()
    except OSError:
        return 0
    inside = False
    for ln in lines:
        head = ln.split()[0] if ln else ""
        if "-" in head and ":" not in head:
            lo = int(head.split("-")[0], 16)
            inside = lo == addr
        elif inside and ln.startswith("AnonHugePages:"):
            return int(ln.split()[1]) * 1024
    return 0


class _CudaRt:
    lib = None

    @classmethod
    def get(cls):
        if cls.lib is None:
            for name in ("libcudart.so", "libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
                try:
                    cls.lib = ctypes.CDLL(name)
                    break
                except OSError:
                    continue
            if cls.lib is None:
                raise OSError("libcudart not found")
        return cls.lib


class HostPool:
    """Host memory for one layer's KV pool, pinned and mapped for the GPU.

    The GPU reads random rows of a host pool fastest when the pool sits on huge pages:
    with ordinary pages its translations thrash, and when the host cannot give the whole
    pool transparent huge pages the fallback regions do. So the pool is an anonymous
    mapping advised onto transparent huge pages, and if the kernel does not back every
    byte with them it is replaced by driver-pinned memory (cudaHostAlloc, mapped and
    portable). `array` is the bytes; `needs_register` tells whether the caller must still
    page-lock it (hs_host_register), i.e. the huge-page path."""

    def __init__(self, nbytes: int, before_fault=None):
        """before_fault(addr, nbytes): called on the fresh mapping before any of its pages is
        touched (to set its memory policy: place it on a memory node)."""
        import mmap
        self.nbytes = int(nbytes)
        self._mmap = None
        self._cuda_ptr = None
        huge = _huge_page_bytes()
        m = mmap.mmap(-1, max(self.nbytes, 1), flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        arr = np.frombuffer(m, dtype=np.uint8, count=self.nbytes)
        if before_fault is not None and self.nbytes:
            before_fault(arr.ctypes.data, len(m))
        ok = False
        try:
            m.madvise(mmap.MADV_HUGEPAGE)
            arr[::huge] = 0  # fault every huge page in
            ok = _huge_backed_bytes(arr.ctypes.data, self.nbytes) >= (self.nbytes // huge) * huge
        except (AttributeError, OSError, ValueError):
            ok = False
        if ok or self.nbytes < huge:
            self._mmap = m
            self.array = arr
            self.needs_register = True
            return
        del arr
        m.close()
        rt = _CudaRt.get()
        ptr = ctypes.c_void_p()
        # cudaHostAllocPortable | cudaHostAllocMapped
        err = rt.cudaHostAlloc(ctypes.byref(ptr), ctypes.c_size_t(self.nbytes), ctypes.c_uint(1 | 2))
        if err != 0 or not ptr.value:
            raise MemoryError(f"cudaHostAlloc of {self.nbytes} bytes failed ({err})")
        self._cuda_ptr = ptr.value
        self.array = np.ctypeslib.as_array((ctypes.c_uint8 * self.nbytes).from_address(ptr.value))
        self.needs_register = False

    def free(self):
        if self._cuda_ptr:
            _CudaRt.get().cudaFreeHost(ctypes.c_void_p(self._cuda_ptr))
            self._cuda_ptr = None
        self.array = None
        if self._mmap is not None:
            try:
                self._mmap.close()
            except BufferError:
                pass  # views still alive; the mapping goes with them
            self._mmap = None


# --------------------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------------------
@dataclass
class Config:
    name: str
    requests: int
    top_k: int
    hot_slots: int
    row_bytes: int
    fmt: int
    layers: int
    steps: int
    rule: str  # "reuse" | "window" | "mixed"
    reuse: float
    seq0: Sequence[int] = ()  # explicit per-request seq_len at step 0 (else seq_range)
    seq_range: Optional[tuple] = None  # (lo, hi) inclusive uniform draw per request
    window: int = 0  # "window": last `window` tokens always selected
    page_size: int = 0  # residency page size (0 = no residency)
    resident_tail_pages: int = 0  # "mixed": pages at the end of the step-0 sequence on the GPU
    resident_frac: float = 0.0  # "mixed": share of top-k drawn from the resident tail
    backup: bool = True  # run the eager backup every step
    host_layout: str = "layer_first"  # "layer_first": one host pool per layer; "page_first": one
    # pool whose row h holds every layer's bytes of a token (layer l at l * row_bytes)


CONFIGS: Dict[str, Config] = {
    "tiny": Config("tiny", 2, 64, 128, 576, FMT_U8, 1, 16, "reuse", 0.7, seq0=(8192, 100)),
    "dsa": Config("dsa", 32, 2048, 4096, 656, FMT_FP8MLA, 1, 64, "window", 0.9,
                  seq0=(131072,) * 32, window=64),
    "mixed1m": Config("mixed1m", 16, 2048, 4096, 656, FMT_FP8MLA, 1, 32, "mixed", 0.7,
                      seq0=(1048576,) * 16, page_size=64, resident_tail_pages=256, resident_frac=0.2),
    "indexshare": Config("indexshare", 256, 2048, 4096, 656, FMT_FP8MLA, 4, 32, "reuse", 0.85,
                         seq_range=(32768, 65536)),
    "sweep": Config("sweep", 64, 2048, 4096, 1152, FMT_BF16, 1, 32, "reuse", 0.8,
                    seq0=(262144,) * 64),
}
SWEEP_HOT = (2048, 4096, 6144)
SWEEP_REUSE = (0.5, 0.8, 0.95, 0.99)
_CONFIG_IDS = {"tiny": 1, "dsa": 2, "mixed1m": 3, "indexshare": 4, "sweep": 5}


def sweep_config(hot_slots: int, reuse: float) -> Config:
    c = dataclasses.replace(CONFIGS["sweep"], hot_slots=hot_slots, reuse=reuse)
    c.name = f"sweep_h{hot_slots}_f{reuse}"
    return c


def derive(cfg: Config, **kw) -> Config:
    """Copy of `cfg` with fields replaced; shrinking `requests` truncates `seq0`."""
    c = dataclasses.replace(cfg, **kw)
    if "requests" in kw and c.seq0:
        s = list(c.seq0)
        c.seq0 = tuple((s * ((c.requests + len(s) - 1) // len(s)))[: c.requests])
    return c


# --------------------------------------------------------------------------------------
# top-k generation
# --------------------------------------------------------------------------------------
def _uniform_excluding(rng: np.random.Generator, lo: int, hi: int, n: int, exclude: set) -> List[int]:
    """n distinct integers uniform over [lo, hi) \\ exclude (rejection sampling)."""
    if n <= 0:
        return []
    avail = (hi - lo) - sum(1 for x in exclude if lo <= x < hi)
    if n > avail:
        raise ValueError("not enough tokens to draw from")
    out: List[int] = []
    seen = set(exclude)
    if avail < 4 * n:  # dense draw: enumerate the candidates
        cand = np.array([x for x in range(lo, hi) if x not in seen], dtype=np.int64)
        return [int(x) for x in rng.choice(cand, size=n, replace=False)]
    while len(out) < n:
        draw = rng.integers(lo, hi, size=2 * (n - len(out)) + 8)
        for x in draw.tolist():
            if x not in seen:
                seen.add(x)
                out.append(x)
                if len(out) == n:
                    break
    return out


def _pick(rng: np.random.Generator, pool: Sequence[int], n: int) -> List[int]:
    n = min(n, len(pool))
    if n <= 0:
        return []
    idx = rng.choice(len(pool), size=n, replace=False)
    return [pool[i] for i in idx.tolist()]


class Workload:
    """All seeded inputs of one configuration.

    Tables use dense row-major int32 layouts:
      top_k_tokens[step]  [R, K]       token positions, -1 = padding
      seq_lens[step]      [R]
      host_cache_locs     [R, max_context]  token -> host row (-1 past the sequence)
      device_buffer_locs  [R, H+1]     slot -> device row; slot H is the newest-token row
      resident_pages      [R, max_pages] page -> device page (rows page*ps .. +ps), -1 = host only
    """

    def __init__(self, cfg: Config, seed: int = 0):
        self.cfg = cfg
        self.seed = int(seed)
        c = cfg
        self.R, self.K, self.H, self.B, self.L = c.requests, c.top_k, c.hot_slots, c.row_bytes, c.layers
        self.steps = c.steps
        self.ps = c.page_size
        base = np.random.default_rng([self.seed, _CONFIG_IDS.get(c.name.split("_")[0], 9), 0])
        if c.seq0:
            assert len(c.seq0) == self.R
            self.seq0 = np.asarray(c.seq0, dtype=np.int64)
        else:
            lo, hi = c.seq_range
            self.seq0 = base.integers(lo, hi + 1, size=self.R).astype(np.int64)
        self.seq_max = (self.seq0 + self.steps).astype(np.int32)  # tokens 0..seq_max-1 ever exist
        self.max_context = int(self.seq_max.max())

        # token -> host row: host pages (HOST_PAGE tokens) scattered by a seeded permutation
        npages = (self.seq_max.astype(np.int64) + HOST_PAGE - 1) // HOST_PAGE
        total_pages = int(npages.sum())
        perm = base.permutation(total_pages).astype(np.int64)
        self.host_rows = total_pages * HOST_PAGE
        hcl = np.full((self.R, self.max_context), -1, dtype=np.int32)
        pb = 0
        for r in range(self.R):
            t = np.arange(int(self.seq_max[r]), dtype=np.int64)
            hcl[r, : len(t)] = (perm[pb + t // HOST_PAGE] * HOST_PAGE + t % HOST_PAGE).astype(np.int32)
            pb += int(npages[r])
        self.host_cache_locs = hcl

        # slot -> device row: a seeded permutation of the hot region
        hot_rows = self.R * (self.H + 1)
        self.device_buffer_locs = base.permutation(hot_rows).astype(np.int32).reshape(self.R, self.H + 1)
        self.device_rows = hot_rows

        # resident tail (mixed residency)
        self.resident_pages = None
        self.tail0 = None
        if c.page_size > 0 and c.resident_tail_pages > 0:
            ps = c.page_size
            self.max_pages = (self.max_context + ps - 1) // ps
            first_page = self.seq0 // ps - c.resident_tail_pages  # per request
            self.tail0 = (first_page * ps).astype(np.int64)
            last_page = (self.seq_max.astype(np.int64) + ps - 1) // ps  # exclusive
            per_req = (last_page - first_page).astype(np.int64)
            base_page = (hot_rows + ps - 1) // ps
            n_res = int(per_req.sum())
            slot_perm = base.permutation(n_res).astype(np.int64)
            rp = np.full((self.R, self.max_pages), -1, dtype=np.int32)
            k = 0
            for r in range(self.R):
                for p in range(int(first_page[r]), int(last_page[r])):
                    rp[r, p] = int(base_page + slot_perm[k])
                    k += 1
            self.resident_pages = rp
            self.device_rows = int((base_page + n_res) * ps)
        else:
            self.max_pages = 0

        self._topk: List[np.ndarray] = []
        self._rngs = [np.random.default_rng([self.seed, _CONFIG_IDS.get(c.name.split("_")[0], 9), 1, r])
                      for r in range(self.R)]
        self._prev: List[List[int]] = [[] for _ in range(self.R)]

    # ---- per-step inputs -------------------------------------------------------------
    def seq_lens(self, step: int) -> np.ndarray:
        return (self.seq0 + step).astype(np.int32)

    def top_k_tokens(self, step: int) -> np.ndarray:
        while len(self._topk) <= step:
            self._topk.append(self._gen_step(len(self._topk)))
        return self._topk[step]

    def _gen_step(self, step: int) -> np.ndarray:
        c, K = self.cfg, self.K
        out = np.full((self.R, K), -1, dtype=np.int32)
        for r in range(self.R):
            rng = self._rngs[r]
            S = int(self.seq0[r]) + step
            newest = S - 1
            prev = self._prev[r]
            if c.rule == "window":
                w0 = max(0, S - c.window)
                chosen = list(range(w0, S))
                cs = set(chosen)
                n_reuse = int(np.floor(c.reuse * K)) if step > 0 else 0
                n_reuse = min(n_reuse, max(0, min(K, S) - len(chosen)))
                chosen += _pick(rng, [x for x in prev if x not in cs], n_reuse)
                cs = set(chosen)
                chosen += _uniform_excluding(rng, 0, S, min(K, S) - len(chosen), cs)
                self._prev[r] = chosen
            elif c.rule == "mixed":
                t0 = int(self.tail0[r])
                n_res = int(np.floor(c.resident_frac * K))
                res = [newest] + _uniform_excluding(rng, t0, newest, n_res - 1, set())
                n_host = K - n_res
                n_reuse = int(np.floor(c.reuse * K)) if step > 0 else 0
                host = _pick(rng, prev, n_reuse)
                host += _uniform_excluding(rng, 0, t0, n_host - len(host), set(host))
                self._prev[r] = host
                chosen = res + host
            else:  # "reuse"
                chosen = [newest]
                n_reuse = int(np.floor(c.reuse * K)) if step > 0 else 0
                n_reuse = min(n_reuse, max(0, min(K, S) - 1))
                chosen += _pick(rng, [x for x in prev if x != newest], n_reuse)
                chosen += _uniform_excluding(rng, 0, S, min(K, S) - len(chosen), set(chosen))
                self._prev[r] = chosen
            row = np.full(K, -1, dtype=np.int32)
            row[: len(chosen)] = chosen
            out[r] = row[rng.permutation(K)]
        return out

    # ---- caller-side layout helpers (the forward pass / allocator stand-in) -----------
    def resident_row(self, r: int, t: int) -> int:
        """Device row of token t if its page is GPU-resident, else -1."""
        if self.resident_pages is None:
            return -1
        p = self.resident_pages[r, t // self.ps]
        return -1 if p < 0 else int(p) * self.ps + t % self.ps

    def newest_device_row(self, r: int, seq_len: int) -> int:
        """Where the forward pass writes the newest token's KV row before the resolve:
        its resident row, else buffer slot seq_len-1 while the whole sequence fits the
        buffer, else the reserved slot H (padded buffer page, SGLang HiSparse analysis)."""
        t = seq_len - 1
        rr = self.resident_row(r, t)
        if rr >= 0:
            return rr
        if seq_len <= self.H:
            return int(self.device_buffer_locs[r, t])
        return int(self.device_buffer_locs[r, self.H])

    def initial_state(self):
        """(device_buffer_tokens [R,H], lru_slots [R,H], lru_clock [R]) at step 0.
        Requests that fit the buffer hold token s in slot s for every token before the
        newest one; the others start empty."""
        tok = np.full((self.R, self.H), -1, dtype=np.int32)
        for r in range(self.R):
            S = int(self.seq0[r])
            if S <= self.H:
                tok[r, : S - 1] = np.arange(S - 1, dtype=np.int32)
        return tok, np.zeros((self.R, self.H), dtype=np.int32), np.zeros(self.R, dtype=np.int32)

    def warm_slot_state(self, seed: int, fill: float = 0.8, clock: int = 50):
        """A seeded mid-decode slot map for requests past the fast path: a `fill` share of
        the slots hold distinct tokens below seq_len - 1 (the most recent positions first,
        as a decode's working set), stamps in [1, clock]; clock [R] = clock. Requests that
        fit the buffer keep the initial identity map."""
        rng = np.random.default_rng(seed)
        tok, st, _ = self.initial_state()
        for r in range(self.R):
            S = int(self.seq0[r])
            if S <= self.H:
                continue
            n = min(int(fill * self.H), S - 1)
            recent = np.arange(S - 1 - 4 * n, S - 1) if S - 1 >= 4 * n else np.arange(S - 1)
            held = rng.choice(recent, size=n, replace=False).astype(np.int32)
            slots = rng.permutation(self.H)[:n]
            tok[r, slots] = held
            st[r, slots] = rng.integers(1, clock + 1, size=n)
        return tok, st, np.full(self.R, clock, dtype=np.int32)

    def rewritten_positions(self, count: int):
        """CSR lists of the `count` positions before the newest one, per request: the rows a
        chunk of prefill (or a rejected speculative draft) rewrote on the host."""
        offs, toks = [0], []
        for r in range(self.R):
            S = int(self.seq0[r])
            t = np.arange(max(0, S - 1 - count), max(0, S - 1), dtype=np.int32)
            toks.append(t)
            offs.append(offs[-1] + t.size)
        return np.array(offs, dtype=np.int32), np.concatenate(toks) if toks else np.zeros(0, np.int32)

    def queries_bf16(self, step: int, heads: int, dims: int = 576) -> np.ndarray:
        """Seeded decode queries [R, heads, dims] as bfloat16 bit patterns, ~N(0, 1) (round to
        nearest even from float32)."""
        rng = np.random.default_rng((self.seed, 0x51, step, heads))
        x = rng.standard_normal((self.R, heads, dims)).astype(np.float32).view(np.uint32).astype(np.uint64)
        x = (x + 0x7FFF + ((x >> 16) & 1)) >> 16
        return x.astype(np.uint16)

    def initial_device_writes(self):
        """(requests, tokens, device rows) the caller writes before step 0: the fast-path
        buffer contents and the resident pages' rows (all tokens before the newest)."""
        rq, tk, rows = [], [], []
        for r in range(self.R):
            S = int(self.seq0[r])
            if S <= self.H:
                t = np.arange(S - 1, dtype=np.int64)
                rq.append(np.full(len(t), r)); tk.append(t)
                rows.append(self.device_buffer_locs[r, : S - 1].astype(np.int64))
            if self.resident_pages is not None:
                t = np.arange(int(self.tail0[r]), S - 1, dtype=np.int64)
                p = self.resident_pages[r, t // self.ps].astype(np.int64)
                rq.append(np.full(len(t), r)); tk.append(t); rows.append(p * self.ps + t % self.ps)
        if not rq:
            z = np.zeros(0, dtype=np.int64)
            return z.astype(np.int32), z.astype(np.int32), z
        return (np.concatenate(rq).astype(np.int32), np.concatenate(tk).astype(np.int32),
                np.concatenate(rows).astype(np.int64))

    # ---- bytes -----------------------------------------------------------------------
    def rows(self, layer: int, request: int, tokens) -> np.ndarray:
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(-1))
        out = np.empty((len(t), self.B), dtype=np.uint8)
        _rowgen().rowgen_rows(self.seed, self.cfg.fmt, self.B, layer, request, _ptr(t), len(t), _ptr(out))
        return out

    def scatter_rows(self, layer: int, requests, tokens, dst_rows, pool: np.ndarray) -> None:
        rq = np.ascontiguousarray(np.asarray(requests, dtype=np.int32))
        tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        dr = np.ascontiguousarray(np.asarray(dst_rows, dtype=np.int64))
        assert pool.dtype == np.uint8 and pool.flags.c_contiguous
        assert len(rq) == len(tk) == len(dr)
        if len(dr):
            assert dr.min() >= 0 and (dr.max() + 1) * self.B <= pool.size
        _rowgen().rowgen_scatter(self.seed, self.cfg.fmt, self.B, layer, _ptr(rq), _ptr(tk), _ptr(dr),
                                 len(dr), _ptr(pool))

    # ---- host pool layout ----------------------------------------------------------
    @property
    def host_row_stride(self) -> int:
        """Bytes from one host row to the next inside a layer's pool."""
        return self.L * self.B if self.cfg.host_layout == "page_first" else self.B

    @property
    def host_pool_bytes(self) -> int:
        """Bytes of one layer's pool (layer first) or of the one shared pool (page first)."""
        return self.host_rows * self.B * (self.L if self.cfg.host_layout == "page_first" else 1)

    def host_layer_views(self, base: np.ndarray) -> List[np.ndarray]:
        """Per-layer pool views of one page-first pool: layer l starts l * B bytes in."""
        assert self.cfg.host_layout == "page_first"
        return [base[layer * self.B:] for layer in range(self.L)]

    def host_row_bytes_of(self, pool: np.ndarray, row: int) -> np.ndarray:
        """The B bytes of host row `row` in one layer's pool (view)."""
        s = self.host_row_stride
        return pool[row * s: row * s + self.B]

    def fill_host_pool(self, layer: int, pool: np.ndarray, nthreads: int = 0) -> None:
        """Write every token's row of `layer` into its host row of `pool` (one layer's pool,
        or that layer's view of a page-first pool)."""
        assert pool.dtype == np.uint8 and pool.flags.c_contiguous
        assert pool.size >= (self.host_rows - 1) * self.host_row_stride + self.B
        if nthreads <= 0:
            nthreads = max(1, len(os.sched_getaffinity(0)))
        sm = np.ascontiguousarray(self.seq_max, dtype=np.int32)
        _rowgen().rowgen_fill_pool(self.seed, self.cfg.fmt, self.B, layer, self.R, _ptr(sm),
                                   _ptr(self.host_cache_locs), self.max_context, _ptr(pool), nthreads,
                                   self.host_row_stride)


def make(name: str, seed: int = 0, **overrides) -> Workload:
    if name.startswith("sweep_h"):
        h, f = name[len("sweep_h"):].split("_f")
        cfg = sweep_config(int(h), float(f))
    else:
        cfg = CONFIGS[name]
    if overrides:
        cfg = derive(cfg, **overrides)
    return Workload(cfg, seed)
