"""Benchmark of the HiSparse decode-step resolver / swap-in on GB300.

One step = one decode step of the whole hot path for the batch: hs_resolve (classify,
hit / LRU refresh, victim pick, miss-row copies from pinned host memory, row table) and
hs_backup (newest-token row back to host). Default workload: IndexShare -- 256 requests at
seq_len uniform in [32768, 65536] (+1 per step), one top-k of 2048 shared by 4 sparse-MLA
layers, 4096 hot slots, 656-byte FP8 MLA rows, top-k 85 % reused step to step plus the newest
token, eager backup every step; the four layers' host rows interleaved in one pinned pool
(--host-layout). --config dsa is the DSA decode shape (32 requests at seq_len 131072, one
layer). Inputs are seeded and synthetic and sit in device memory (host pool: pinned host
memory) before timing starts; L2 is flushed (256 MiB write) between timed steps.

Prints one JSON line. --impl reference times the CPU oracle (the plain policy
definition) on the same workload and steps instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "top-k rows resolved/s"
_HOST_POOLS = {}  # registered host pools kept across runs that share a host layout
UNIT = "rows/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=None,
                    help="workload (default: indexshare for the decode step and the split, the largest "
                         "configuration on one GPU; dsa for the other ops)")
    ap.add_argument("--host-layout", default="auto", choices=["auto", "layer_first", "page_first"],
                    help="host KV pool layout: one pool per layer, or one pool whose row holds every layer's "
                         "bytes of a token (auto: page_first for a layer group of more than one layer)")
    ap.add_argument("--rehearsal", default="disjoint", choices=["disjoint", "timed", "none"],
                    help="untimed steps replayed before timing: steps after the timed range (disjoint), the "
                         "timed steps' own inputs (timed), or none")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--op", default="step",
                    choices=["step", "invalidate_tokens", "invalidate_host_rows", "split", "spec", "mla", "e2e"],
                    help="step: the decode step (default); invalidate_*: one hot-slot invalidation call; "
                         "split: leader resolve + follower gathers on a copy stream vs the fused step")
    ap.add_argument("--sweep", action="store_true",
                    help="run every miss-rate sweep point (hot slots x reuse), one JSON line each")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.idx = device_index
        self.enabled = enabled
        self.proc = None

    def __enter__(self):
        if self.enabled:
            try:
                self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                              "--format=csv,noheader,nounits", "-lms", "100"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
            if self.proc is not None:
                import atexit
                atexit.register(self._stop)  # an exception before __exit__ must not leave it running
        return self

    def _stop(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), max=float(f[2]), hw=f[5], hwt=f[6], swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                            ("pcap", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------------------------------
def dist_init(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


_POOL_OBJS = []  # workloads.HostPool objects behind the arrays in use


def alloc_host(nbytes: int, bind=None):
    """Host pool bytes: huge pages when the host gives the whole pool, else driver-pinned
    memory (workloads.HostPool: the GPU reads random host rows fastest from huge pages).
    bind(addr, nbytes): places the mapping on a memory node before its pages are touched.
    Returns (array, needs hs_host_register)."""
    import workloads as W
    pool = W.HostPool(nbytes, before_fault=bind)
    _POOL_OBJS.append(pool)
    return pool.array, pool.needs_register


def host_device_ptr(arr) -> int:
    """Device-side address of driver-pinned, mapped host memory."""
    import ctypes
    import workloads as W
    dp = ctypes.c_void_p()
    err = W._CudaRt.get().cudaHostGetDevicePointer(ctypes.byref(dp), ctypes.c_void_p(arr.ctypes.data), 0)
    if err != 0:
        raise RuntimeError(f"cudaHostGetDevicePointer failed ({err})")
    return dp.value


class _DeviceView:
    """__cuda_array_interface__ over a mapped host range, so torch can read it from the GPU."""

    def __init__(self, ptr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes // 8,), "typestr": "<i8", "data": (ptr, False),
                                         "version": 3}


TOUCH_PASSES = 8
LINK_WARM_BYTES = 2 << 30  # host-pool bytes the GPU reads right before each timed pass


def touch_host_pool_from_gpu(dev_ptr: int, nbytes: int) -> None:
    """Read the whole registered host pool from the GPU, TOUCH_PASSES times (set-up,
    outside timing), so the timed steps see a host pool whose mappings the GPU has already
    used. One pass is not enough: regions first reached by the resolve kernel's random row
    reads then cost ~0.5 ms once each in the first few dozen steps; eight passes (or ~64
    warm-up steps) leave none."""
    import torch
    v = torch.as_tensor(_DeviceView(dev_ptr, nbytes), device="cuda")
    for _ in range(TOUCH_PASSES):
        v[::8].sum().item()


def newest_rows(wl, step):
    """Device rows and bytes the forward pass writes for the newest tokens of `step`."""
    S = wl.seq_lens(step)
    rows = np.array([wl.newest_device_row(r, int(S[r])) for r in range(wl.R)], dtype=np.int64)
    data = [np.concatenate([wl.rows(l, r, [int(S[r]) - 1]) for r in range(wl.R)]) for l in range(wl.L)]
    return rows, data


def ncu_traffic(config: str) -> dict:
    """Per-launch traffic of the workload's dominant kernel from the committed ncu capture,
    when one was taken on this workload and on the kernel source as it is now; else {}."""
    try:
        recs = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["records"]
        for rec in recs:
            if rec.get("workload") == config and \
                    kernel_code_hash(os.path.join(ROOT, rec["kernel_source"])) == rec.get("code_sha256_16"):
                return rec
    except (OSError, ValueError, KeyError, TypeError):
        pass
    return {}


def kernel_code_hash(path: str) -> str:
    """sha256[:16] of a CUDA source with its // comments and all whitespace removed, so a
    comment edit does not retire a profile of the same code."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    code = re.sub(r"//[^\n]*", "", text)
    return hashlib.sha256(re.sub(r"\s+", "", code).encode()).hexdigest()[:16]


# ------------------------------------------------------------------------------------------
def config_of(name: str):
    import workloads as W
    if name.startswith("sweep_h"):
        h, f = name[len("sweep_h"):].split("_f")
        return W.sweep_config(int(h), float(f))
    return W.CONFIGS[name]


def host_layout_for(args) -> str:
    """The host pool layout of the run: as asked, or for "auto" every layer's bytes of a token
    in one host row when the layer group has several layers (the layout the pair gather reads
    as one span per miss), else one pool per layer."""
    if args.host_layout != "auto":
        return args.host_layout
    return "page_first" if config_of(args.config).layers > 1 else "layer_first"


def make_workload(args, rank: int, steps: int):
    import workloads as W
    return W.make(args.config, args.seed + 1000 * rank, steps=steps, host_layout=host_layout_for(args))


def total_steps_of(args) -> int:
    """Warm-up, timed, and (for a disjoint rehearsal) K more steps after the timed range."""
    return args.warmup + args.steps + (args.steps if args.rehearsal == "disjoint" else 0)


def workload_desc(args, wl) -> str:
    """The workload string both arms print, from the configuration alone."""
    c = wl.cfg
    seq = (f"seq_len U[{c.seq_range[0]}, {c.seq_range[1]}]+1/step" if c.seq_range
           else f"seq_len {int(wl.seq0[0])}+1/step")
    return (f"{args.config}: {wl.R} requests x {seq}, top_k {wl.K}, {wl.H} hot slots, {wl.B}-byte rows, "
            f"{wl.L} layer(s), host pools {c.host_layout.replace('_', '-')}, seed {args.seed}, "
            f"timed steps {args.warmup}..{args.warmup + args.steps - 1} after {args.warmup} warm-up steps")


def cpu_oracle_run(wl, host, warm_steps, timed_steps, nthreads=1):
    """Time the CPU oracle over decode steps [warm_steps, warm_steps + timed_steps) (resolve +
    backup, bytes included) after running steps [0, warm_steps) untimed, so it times the same
    steps the GPU does. Requests are split over `nthreads` Python threads (ctypes drops the
    GIL). `host` are the per-layer host pools of wl's layout."""
    import oracle
    from_state = wl.initial_state()
    dev = []
    rq, tk0, rows0 = wl.initial_device_writes()
    for l in range(wl.L):
        p = np.full(wl.device_rows * wl.B, 0xA5, dtype=np.uint8)
        wl.scatter_rows(l, rq, tk0, rows0, p)
        dev.append(p)
    tokens, stamps, clock = from_state
    out = np.zeros((wl.R, wl.K), dtype=np.int32)
    miss = np.zeros(wl.R, dtype=np.int32)
    stride = wl.host_row_stride if wl.cfg.host_layout == "page_first" else 0
    orc = oracle.Oracle(wl.K, wl.H, wl.B, wl.L, wl.max_context, wl.host_rows, wl.device_rows, wl.ps, wl.max_pages,
                        stride)
    shards = np.array_split(np.arange(wl.R), nthreads)
    elapsed = 0.0
    rows_done = 0
    for step in range(warm_steps + timed_steps):
        nr, nd = newest_rows(wl, step)
        for l in range(wl.L):
            dev[l].reshape(-1, wl.B)[nr] = nd[l]
        tk = wl.top_k_tokens(step)
        S = wl.seq_lens(step)

        def work(ix):
            a, b = int(ix[0]), int(ix[-1]) + 1
            sl = slice(a, b)
            rp = None if wl.resident_pages is None else np.ascontiguousarray(wl.resident_pages[sl])
            orc.resolve(np.ascontiguousarray(tk[sl]), np.ascontiguousarray(S[sl]),
                        np.ascontiguousarray(wl.host_cache_locs[sl]), np.ascontiguousarray(wl.device_buffer_locs[sl]),
                        tokens[sl], stamps[sl], clock[sl], rp, out[sl], miss[sl], host, dev)

        # views of contiguous row blocks are contiguous, so the oracle writes in place
        t0 = time.perf_counter()
        if nthreads == 1:
            work(shards[0])
        else:
            th = [threading.Thread(target=work, args=(ix,)) for ix in shards if len(ix)]
            for t in th:
                t.start()
            for t in th:
                t.join()
        orc.backup(S, wl.host_cache_locs, wl.device_buffer_locs, wl.resident_pages, host, dev)
        if step >= warm_steps:
            elapsed += time.perf_counter() - t0
            rows_done += int((tk >= 0).sum())
    return rows_done, elapsed


def oracle_host_pools(wl):
    """Plain host pools of wl's layout for a CPU-only oracle run."""
    if wl.cfg.host_layout == "page_first":
        base = np.zeros(wl.host_pool_bytes, dtype=np.uint8)
        views = wl.host_layer_views(base)
        for l, v in enumerate(views):
            wl.fill_host_pool(l, v)
        return views
    host = [np.zeros(wl.host_rows * wl.B, dtype=np.uint8) for _ in range(wl.L)]
    for l in range(wl.L):
        wl.fill_host_pool(l, host[l])
    return host


# ------------------------------------------------------------------------------------------
def run_reference(args, ws, rank):
    """The reference arm: the CPU oracle, as it stands, on this machine's host cores, timed over
    the same steps of the same workload as our arm (the warm-up steps run untimed first)."""
    if rank != 0:
        return
    wl = make_workload(args, 0, total_steps_of(args))
    host = oracle_host_pools(wl)
    for s in range(args.warmup + args.steps):
        wl.top_k_tokens(s)
    rows, sec = cpu_oracle_run(wl, host, args.warmup, args.steps)
    value = rows / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": workload_desc(args, wl), "global_batch": wl.R * args.gpus,
                   "seq_len": int(wl.seq0[0]), "parallelism": "cpu"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"decode steps {args.warmup}..{args.warmup + args.steps - 1} of the workload "
                                   f"(after {args.warmup} untimed warm-up steps), single-threaded C oracle, "
                                   "resolve + row copies + backup"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
def rank_numa_node(local_rank: int, query=None) -> int:
    """The host memory node for this rank's host pools: the one nearest its GPU ("Hierarchical
    Sparse Attention" (Alibaba Tair KVCache), 2.4.4: the per-GPU host copy rate depends on NUMA
    binding). query(device) -> node defaults to hs_host_numa_node; -1: leave the placement to
    the kernel's default policy."""
    if query is None:
        import hierarchical_sparse_attention_gb300 as hs
        query = hs.hs_host_numa_node
    try:
        return int(query(local_rank))
    except Exception:  # noqa: BLE001 - no device or no answer: default placement
        return -1


def alloc_host_pools(wl, node: int = -1):
    """Host pools of wl's layout, placed on memory node `node` (-1: default) before their pages
    are touched, then filled. Returns (per-layer pool views, [(array, needs registering)])."""
    import hierarchical_sparse_attention_gb300 as hs
    bind = None
    if node is not None and node >= 0:
        bind = lambda addr, n: hs.hs_host_bind_node(addr, n, node)  # noqa: E731
    if wl.cfg.host_layout == "page_first":
        arr, reg = alloc_host(wl.host_pool_bytes, bind)
        views = wl.host_layer_views(arr)
        for l, v in enumerate(views):
            wl.fill_host_pool(l, v)
        return views, [(arr, reg)]
    pools = [alloc_host(wl.host_rows * wl.B, bind) for _ in range(wl.L)]
    for l, (arr, reg) in enumerate(pools):
        wl.fill_host_pool(l, arr)
    return [arr for arr, _ in pools], pools


def host_mem_available() -> int:
    """MemAvailable of /proc/meminfo in bytes (0 when it cannot be read)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return 0


HOST_MEM_FRACTION = 0.85  # of MemAvailable, for all of one host's ranks' host pools together


def build_host_pools(wl, hs, node: int = -1):
    """alloc_host_pools, then each pool registered (pinned and mapped) and read from the GPU
    TOUCH_PASSES times. Refuses to start, like a serving process whose host pool does not fit
    ("vLLM Hybrid HiSparse source implementation analysis": start-up checks the host memory),
    when this host's ranks' pools together would take more than HOST_MEM_FRACTION of the
    available memory, instead of driving the host out of memory."""
    need = wl.host_pool_bytes if wl.cfg.host_layout == "page_first" else wl.host_rows * wl.B * wl.L
    ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = host_mem_available()
    if avail and ranks * need > HOST_MEM_FRACTION * avail:
        raise MemoryError(f"host pools need {ranks} x {need / 1e9:.1f} GB on this host, more than "
                          f"{HOST_MEM_FRACTION:.0%} of the {avail / 1e9:.0f} GB available")
    views, pools = alloc_host_pools(wl, node)
    for arr, reg in pools:
        touch_host_pool_from_gpu(hs.hs_host_register(arr) if reg else host_device_ptr(arr), arr.nbytes)
    return views, pools


STALL_RATIO = 2.0
SLOW_RATIO = 3.0  # a later pass whose median step exceeds this x the graph-replayed pass's median
SLOW_FLOOR_MS = 0.2  # (or this, if larger: host-synchronised steps of tiny workloads are longer)
MAX_ATTEMPTS = 6
STALL_PAUSE_S = 5.0  # after a stalled pass the GPU spins this long (clocks stay up) before the next
# Host-pool readiness before timing: the busiest step of the warm-up replay must move its miss
# rows across the link at COLD_FRAC of the in-run ceiling at least (on a warm host ~0.55 at the
# dsa shape, whose first step fills an empty buffer with 43 MB, and ~0.8 at IndexShare; on a cold
# one 0.01-0.15); otherwise wait COLD_SLEEP_S and replay again, for COLD_WAIT_S at most.
COLD_FRAC, COLD_SLEEP_S, COLD_WAIT_S = 0.35, 10.0, 240.0


def stalled(ms, ws: int, ref_ms: float = 0.0) -> bool:
    """A timed pass with a step above STALL_RATIO x its median, or (ref_ms > 0) a median above
    SLOW_RATIO x ref_ms (a pass slow from end to end), on any rank."""
    med = float(np.median(ms))
    bad = float(np.max(ms)) > STALL_RATIO * med or (ref_ms > 0.0 and med > SLOW_RATIO * ref_ms)
    return max_over_ranks(1.0 if bad else 0.0, ws) > 0.0


def pick_pass(passes, clean: bool, ws: int) -> int:
    """The pass to report: the last one if it is clean, else (every pass stalled) the one with
    the lowest median step over the ranks' medians (the same index on every rank)."""
    if clean:
        return len(passes) - 1
    meds = [max_over_ranks(float(np.median(ms)), ws) for ms in passes]
    return int(np.argmin(meds))


def stall_pause() -> None:
    """Let a wave of host-side stalls pass before the next attempt: the GPU spins (its clocks
    stay where a loaded GPU runs them) for STALL_PAUSE_S."""
    import torch
    torch.cuda._sleep(int(2.0e9 * STALL_PAUSE_S))
    torch.cuda.synchronize()


def job_throughput(rows_this_rank: int, seconds_this_rank: float, ws: int) -> float:
    """Whole-job rows/s: every rank resolves a batch of the same shape (weak scaling), so the
    job resolves ws x its rows in the slowest rank's time."""
    return ws * rows_this_rank / max_over_ranks(seconds_this_rank, ws)


def release_host_pools(hs, pools):
    for arr, reg in pools:
        if reg:
            hs.hs_host_unregister(arr)
    for obj in _POOL_OBJS:
        obj.free()
    _POOL_OBJS.clear()


def run_ours(args, ws, rank, local):
    import torch
    import hierarchical_sparse_attention_gb300 as hs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    W_, K_ = args.warmup, args.steps
    total_steps = total_steps_of(args)
    wl = make_workload(args, rank, total_steps)
    R, K, H, B, L = wl.R, wl.K, wl.H, wl.B, wl.L
    layout = wl.cfg.host_layout
    numa_node = rank_numa_node(local)

    # ---- inputs: host pools (pinned, mapped, on the GPU's host memory node), device pools,
    # tables, all steps' top-k. The sweep points share one host layout, so their host pools
    # are built once.
    key = (args.config.split("_")[0], args.seed + 1000 * rank, wl.host_rows, B, L, total_steps, layout)
    if key not in _HOST_POOLS:
        for old in list(_HOST_POOLS):
            release_host_pools(hs, _HOST_POOLS.pop(old)[1])
        _HOST_POOLS[key] = build_host_pools(wl, hs, numa_node)
    host, pool_objs = _HOST_POOLS[key]
    # Right before each timed pass the GPU reads LINK_WARM_BYTES of the host pools (queued after
    # the spin that covers the host's queueing of the steps, so no step is timed behind it): on
    # some boxes a pass that began after tens of ms without host reads ran its first ~20 steps
    # at 20-50 ms each, ramping back to ~1.1 ms, while passes straight after host reads did not.
    link_views = [torch.as_tensor(_DeviceView(host_device_ptr(arr), arr.nbytes), device="cuda")
                  for arr, _ in pool_objs]

    def link_warm():
        left = LINK_WARM_BYTES // 8
        for v in link_views:
            n = min(left, v.numel())
            if n > 0:
                v[:n].sum()
            left -= n

    dpool = []
    rq, tk0, rows0 = wl.initial_device_writes()
    for l in range(L):
        init = np.full(wl.device_rows * B, 0xA5, dtype=np.uint8)
        wl.scatter_rows(l, rq, tk0, rows0, init)
        dpool.append(torch.from_numpy(init).to(dev))
    topk_all = torch.from_numpy(np.stack([wl.top_k_tokens(s) for s in range(total_steps)])).to(dev)
    seq_all = torch.from_numpy(np.stack([wl.seq_lens(s) for s in range(total_steps)])).to(dev)
    valid_rows = int((topk_all[W_:W_ + K_] >= 0).sum().item()) // K_  # per timed step (no padding here)
    newest = [newest_rows(wl, s) for s in range(total_steps)]
    newest_idx = torch.from_numpy(np.stack([n[0] for n in newest])).to(dev)
    newest_dat = [torch.from_numpy(np.stack([n[1][l] for n in newest])).to(dev) for l in range(L)]
    hcl = torch.from_numpy(wl.host_cache_locs).to(dev)
    dbl = torch.from_numpy(wl.device_buffer_locs).to(dev)
    rp = None if wl.resident_pages is None else torch.from_numpy(wl.resident_pages).to(dev)
    tok0, st0, clk0 = wl.initial_state()
    tok, st, clk = (torch.from_numpy(x).to(dev) for x in (tok0, st0, clk0))
    tk_buf = torch.empty((R, K), dtype=torch.int32, device=dev)  # the step's inputs, fixed addresses
    sl_buf = torch.empty((R,), dtype=torch.int32, device=dev)
    out = torch.empty((R, K), dtype=torch.int32, device=dev)
    miss = torch.empty((R,), dtype=torch.int32, device=dev)
    miss_acc = torch.zeros((total_steps, R), dtype=torch.int64, device=dev)
    stride = wl.host_row_stride if layout == "page_first" else 0
    cfg = hs.make_config(R, K, H, B, L, wl.ps, wl.max_context, wl.max_pages, stride)
    wsp = torch.zeros(hs.hs_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = hs.hs_create(cfg, host, dpool, wl.host_rows, wl.device_rows, wsp)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    copy_ctas, launches_per_resolve = hs.hs_launch_shape(h)

    def forward_stand_in(s):
        """What the forward pass leaves before the resolve: the newest token's row written to
        its device location and the step's top-k / seq_lens in the input buffers."""
        for l in range(L):
            dpool[l].view(-1, B).index_copy_(0, newest_idx[s], newest_dat[l][s])
        tk_buf.copy_(topk_all[s])
        sl_buf.copy_(seq_all[s])

    def resolve(strm):
        hs.hs_resolve(h, R, tk_buf, sl_buf, hcl, dbl, tok, st, clk, rp, out, miss, strm)

    def backup(strm):
        hs.hs_backup(h, R, sl_buf, hcl, dbl, rp, strm)

    warm_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(W_)]

    def reset_state_and_warm():
        """The warm-up steps from the initial state; returns the highest host-link rate of a
        warm-up step (GB/s of its miss rows over its resolve + backup)."""
        tok.copy_(torch.from_numpy(tok0)); st.copy_(torch.from_numpy(st0)); clk.copy_(torch.from_numpy(clk0))
        hs.hs_reset_hints(h, stream)  # the slot map changed outside the library
        for s in range(W_):
            forward_stand_in(s)
            warm_ev[s][0].record(stream)
            resolve(stream)
            backup(stream)
            warm_ev[s][1].record(stream)
            miss_acc[s].copy_(miss)
        torch.cuda.synchronize()
        if W_ == 0:
            return 0.0
        moved = miss_acc[:W_].sum(dim=1).cpu().numpy().astype(np.float64) * B * L
        return max(float(moved[s]) / (warm_ev[s][0].elapsed_time(warm_ev[s][1]) * 1e-3) / 1e9 for s in range(W_))

    # ---- H2D ceiling in the same process: pinned cudaMemcpy, 1 GiB, best of 12
    ceil_n = 1 << 30
    hsrc = torch.empty(ceil_n, dtype=torch.uint8, pin_memory=True)
    ddst = torch.empty(ceil_n, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(12):
        e0.record(stream)
        ddst.copy_(hsrc, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    h2d_ceiling = ceil_n / (best * 1e-3) / 1e9
    del hsrc, ddst

    # ---- one decode step (resolve + eager backup) captured as a CUDA graph, as decode runs
    reset_state_and_warm()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        resolve(torch.cuda.current_stream())
        backup(torch.cuda.current_stream())
    stream.wait_stream(cap)
    # Rehearsal, untimed, then the state is reset: the GPU's first reads of host-pool regions
    # can stall ~0.5 ms each (more so after other processes churned host memory); a serving
    # process pays that once at start-up, so the timed steps should not. "disjoint" replays the
    # K steps after the timed range (other rows of the same sequences), never the timed steps'
    # own inputs; "timed" replays the timed steps themselves (kept for comparison only).
    # Host-pool readiness: on a freshly started GPU host the GPU's reads of the registered
    # pools have run ~75x below the link's rate for the first minutes (steps of 80 ms instead
    # of 1.1 ms, whole processes long), and in waves later (another tenant of the host's
    # memory). Time each step of the warm-up replay until the busiest one moves its miss rows
    # across the link at COLD_FRAC of the ceiling; every probe is reported.
    ready_probes = []
    t_ready = time.perf_counter()
    while W_ > 0:
        ready_probes.append(round(reset_state_and_warm(), 1))
        ready = max_over_ranks(0.0 if ready_probes[-1] >= COLD_FRAC * h2d_ceiling else 1.0, ws) == 0.0
        late = time.perf_counter() - t_ready + COLD_SLEEP_S > COLD_WAIT_S
        if ready or max_over_ranks(1.0 if late else 0.0, ws) > 0.0:  # every rank leaves together
            break
        time.sleep(COLD_SLEEP_S)
    host_ready = {"busiest_warmup_step_gbs": ready_probes, "waited_s": round(time.perf_counter() - t_ready, 1),
                  "rule": f"the warm-up replay's busiest step moves its miss rows at >= "
                          f"{COLD_FRAC} x the ceiling before timing, replayed every {COLD_SLEEP_S:.0f} s "
                          f"for {COLD_WAIT_S:.0f} s at most", "ready": ready if W_ > 0 else None}
    rehearsal = {"disjoint": range(W_ + K_, W_ + 2 * K_), "timed": range(W_, W_ + K_), "none": range(0)}[args.rehearsal]
    if len(rehearsal):
        reset_state_and_warm()
        for s in rehearsal:
            forward_stand_in(s)
            graph.replay()
        torch.cuda.synchronize()
    reset_state_and_warm()

    # ---- timed region A: K graph-replayed steps, per-step events, L2 flushed between steps.
    # A pass in which some step took more than STALL_RATIO x the pass's median is measured
    # again (at most MAX_ATTEMPTS passes, the state reset before each): on this platform the
    # GPU's reads of a registered host pool sometimes stall for milliseconds for a while
    # (more often after another process released tens of GB of pinned memory), a property of
    # the host side that a serving process sees once at start-up. Every attempt is reported.
    def region_a():
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K_)]
        barrier(ws)
        torch.cuda.synchronize()
        # keep the GPU busy while the host queues every timed step, so the per-step events
        # measure device time, not Python call overhead between launches
        torch.cuda._sleep(int(2e6 * (5 + K_ // 4)))
        link_warm()
        for i in range(K_):
            s = W_ + i
            forward_stand_in(s)
            flush.zero_()
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
            miss_acc[s].copy_(miss)
        torch.cuda.synchronize()
        barrier(ws)
        return [e[0].elapsed_time(e[1]) for e in evs]

    attempts_a, passes_a, clean_a = [], [], False
    # clocks are sampled over both timed passes (A and B below): pass A alone is ~0.1 s
    clocks = ClockSampler(local, enabled=not args.no_clocks).__enter__()
    for attempt in range(MAX_ATTEMPTS):
        if attempt:
            stall_pause()
            reset_state_and_warm()
        step_ms = region_a()
        passes_a.append(step_ms)
        attempts_a.append({"p50_step_us": 1e3 * float(np.median(step_ms)),
                           "max_step_us": 1e3 * float(np.max(step_ms))})
        clean_a = not stalled(step_ms, ws)
        if clean_a:
            break
    reported_a = pick_pass(passes_a, clean_a, ws)
    step_ms = passes_a[reported_a]
    err = hs.hs_get_error(h, clear=True)
    misses = miss_acc[W_:W_ + K_].sum(dim=1).cpu().numpy()  # per timed step, all requests
    rows_timed = valid_rows * K_
    value = job_throughput(rows_timed, sum(step_ms) * 1e-3, ws)

    # ---- pass B: the same steps eagerly, with events around the dominant kernel. With copy
    # CTAs that is the one resolve launch. Without them hs_resolve is the resolve, the grouping
    # by host region and the pair gather; the same four kernels are issued here as
    # hs_resolve_layers(copy_layers = 0) (resolve + grouping) and hs_gather of every layer
    # (the gather alone), so the gather's own duration is measured. Stalled passes are
    # measured again, as above.
    split = launches_per_resolve > 1

    def pass_b():
        reset_state_and_warm()
        evb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K_)]
        torch.cuda._sleep(int(2e6 * (5 + K_ // 4)))
        link_warm()
        for i in range(K_):
            s = W_ + i
            forward_stand_in(s)
            flush.zero_()
            evb[i][0].record(stream)
            if split:
                hs.hs_resolve_layers(h, R, tk_buf, sl_buf, hcl, dbl, tok, st, clk, rp, out, miss, 0, stream)
                evb[i][1].record(stream)
                hs.hs_gather(h, R, hcl, 0, L, stream)
            else:
                resolve(stream)
                evb[i][1].record(stream)
            evb[i][2].record(stream)
            backup(stream)
            evb[i][3].record(stream)
            miss_acc[s].copy_(miss)
        torch.cuda.synchronize()
        if not np.array_equal(miss_acc[W_:W_ + K_].sum(dim=1).cpu().numpy(), misses):
            raise RuntimeError("pass B resolved different miss counts from the timed pass")
        return evb

    attempts_b, passes_b, evbs, clean_b = [], [], [], False
    for attempt in range(MAX_ATTEMPTS):
        if attempt:
            stall_pause()
        evb = pass_b()
        dom_try = [e[1 if split else 0].elapsed_time(e[2]) for e in evb]
        evbs.append(evb)
        passes_b.append(dom_try)
        attempts_b.append({"p50_dominant_us": 1e3 * float(np.median(dom_try)),
                           "max_dominant_us": 1e3 * float(np.max(dom_try))})
        clean_b = not stalled(dom_try, ws, max(float(np.median(step_ms)), SLOW_FLOOR_MS))
        if clean_b:
            break
    reported_b = pick_pass(passes_b, clean_b, ws)
    evb = evbs[reported_b]
    clocks.__exit__(None, None, None)
    res_ms = [e[0].elapsed_time(e[2]) for e in evb]     # the whole hs_resolve work
    dom_ms = [e[1 if split else 0].elapsed_time(e[2]) for e in evb]  # the dominant kernel alone
    bak_ms = [e[2].elapsed_time(e[3]) for e in evb]
    miss_bytes = misses.astype(np.float64) * B * L  # host-link bytes read per resolve (all layers)
    dom_s = np.array(dom_ms) * 1e-3
    res_s = np.array(res_ms) * 1e-3
    link_gbs = float(miss_bytes.sum() / dom_s.sum() / 1e9)
    call_gbs = float(miss_bytes.sum() / res_s.sum() / 1e9)
    # HBM algorithmic bytes of the resolve's work: top-k, seq_lens, slot map + stamps read,
    # host-row lookups for misses, slot->row table, state writes, row table, the residency
    # bitmap row of each request, miss rows written
    bit_row_bytes = (wl.max_context + 127) // 128 * 16
    hbm_bytes = (4 * R * K + 4 * R + 8 * R * H + 32 * misses + 4 * R * (H + 1) + 8 * R * K + 4 * R * K
                 + R * bit_row_bytes + miss_bytes).astype(np.float64)
    hbm_gbs = float(hbm_bytes.sum() / res_s.sum() / 1e9)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    traffic = ncu_traffic(f"{args.config}/{layout}")

    # ---- end to end through the C ABI with host buffers, as a serving loop runs it: one pinned
    # input block (the step's top-k rows and seq_lens) that the host scheduler refills before each
    # step (outside the timed region: it is the scheduler's work), one pinned output block (row
    # table and miss counts), and one CUDA graph replayed every step; a stream sync ends it.
    #   zero-copy (the line's value): the kernels read the inputs and write the outputs over the
    #     host link themselves (the ABI takes pinned host pointers for these four arrays);
    #   copies: one H2D copy of the inputs into device buffers, the calls, one D2H copy back.
    e2e_steps = min(K_, 16)
    io_steps = torch.from_numpy(np.stack([np.concatenate([wl.top_k_tokens(s).reshape(-1), wl.seq_lens(s)])
                                          for s in range(total_steps)]))
    io_pin = torch.empty((R * K + R,), dtype=torch.int32).pin_memory()
    out_pin = torch.empty((R * K + R,), dtype=torch.int32).pin_memory()
    io_in = torch.empty((R * K + R,), dtype=torch.int32, device=dev)
    io_out = torch.empty((R * K + R,), dtype=torch.int32, device=dev)
    pin_tk, pin_sl = io_pin[:R * K].view(R, K), io_pin[R * K:]
    pout_v, pmiss_v = out_pin[:R * K].view(R, K), out_pin[R * K:]
    in_tk, in_sl = io_in[:R * K].view(R, K), io_in[R * K:]
    out_v, miss_v = io_out[:R * K].view(R, K), io_out[R * K:]

    def e2e_calls(strm, zero_copy):
        if zero_copy:
            hs.hs_resolve(h, R, pin_tk, pin_sl, hcl, dbl, tok, st, clk, rp, pout_v, pmiss_v, strm)
            hs.hs_backup(h, R, pin_sl, hcl, dbl, rp, strm)
        else:
            io_in.copy_(io_pin, non_blocking=True)
            hs.hs_resolve(h, R, in_tk, in_sl, hcl, dbl, tok, st, clk, rp, out_v, miss_v, strm)
            hs.hs_backup(h, R, in_sl, hcl, dbl, rp, strm)
            out_pin.copy_(io_out, non_blocking=True)

    def e2e_pass(zero_copy):
        g_e = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(g_e, stream=cap):
            e2e_calls(torch.cuda.current_stream(), zero_copy)
        stream.wait_stream(cap)
        reset_state_and_warm()
        ms = []
        for i in range(e2e_steps):
            s = W_ + i
            for l in range(L):
                dpool[l].view(-1, B).index_copy_(0, newest_idx[s], newest_dat[l][s])
            flush.zero_()
            io_pin.copy_(io_steps[s])  # the scheduler's inputs for this step
            torch.cuda.synchronize()
            t0 = time.perf_counter()  # wall clock: graph launch, kernels (and copies), final sync
            g_e.replay()
            stream.synchronize()
            ms.append((time.perf_counter() - t0) * 1e3)
            if int(out_pin[R * K:].sum()) != int(miss_acc[s].sum()):  # the step's outputs reached the host
                raise RuntimeError(f"end-to-end step {s}: miss counts read back differ from the timed run")
        return ws * valid_rows * e2e_steps / max_over_ranks(sum(ms) * 1e-3, ws), ms

    def e2e_measured(zero_copy):  # the stall rule of the timed passes
        tries, runs, clean = [], [], False
        for attempt in range(MAX_ATTEMPTS):
            if attempt:
                stall_pause()
            v, ms = e2e_pass(zero_copy)
            runs.append((v, ms))
            tries.append(round(1e3 * float(np.median(ms)), 1))
            clean = not stalled(ms, ws, max(float(np.median(step_ms)), SLOW_FLOOR_MS))
            if clean:
                break
        v, ms = runs[pick_pass([m for _, m in runs], clean, ws)]
        return v, ms, tries

    e2e_copy_value, e2e_copy_ms, e2e_copy_tries = e2e_measured(False)
    e2e_value, e2e_ms, e2e_tries = e2e_measured(True)
    h2d_b = 4 * R * K + 4 * R
    d2h_b = 4 * R * K + 4 * R
    dominant = "resolve_kernel" if not split else "gather_pairs_kernel"

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K_, "warmup": W_,
        "ms_per_step": float(np.mean(step_ms)), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32", "data": "synthetic",
        "config": {"workload": workload_desc(args, wl),
                   "global_batch": R * ws, "seq_len": int(wl.seq0[0]), "parallelism": f"requests sharded, dp{ws}",
                   "l2": "flushed between timed steps (256 MiB write)",
                   "step": "hs_resolve + hs_backup replayed as one CUDA graph",
                   "host_layout": layout,
                   "rehearsal": {"disjoint": f"before timing, steps {W_ + K_}..{W_ + 2 * K_ - 1} (after the timed "
                                             "range) replayed once untimed, state reset",
                                 "timed": "before timing, the K timed steps' inputs replayed once untimed, state reset",
                                 "none": "none"}[args.rehearsal]},
        "p50_step_us": 1e3 * float(np.median(step_ms)), "p90_step_us": 1e3 * float(np.percentile(step_ms, 90)),
        "p50_resolve_us": 1e3 * float(np.median(res_ms)), "p90_resolve_us": 1e3 * float(np.percentile(res_ms, 90)),
        "p50_backup_us": 1e3 * float(np.median(bak_ms)),
        "p50_dominant_kernel_us": 1e3 * float(np.median(dom_ms)),
        "resolve_timing": "eager launches, CUDA events around the resolve work alone (without copy CTAs: "
                          "hs_resolve_layers(0) + hs_gather of every layer, the same four kernels as hs_resolve)",
        "host_pool_readiness": host_ready,
        "timed_attempts": attempts_a,
        "dominant_kernel_attempts": attempts_b,
        "attempt_rule": f"a pass with a step above {STALL_RATIO} x its median (the eager and end-to-end "
                        f"passes also: a median above {SLOW_RATIO} x the graph-replayed pass's, at least "
                        f"{SLOW_FLOOR_MS} ms) is measured again after a {STALL_PAUSE_S:.0f} s pause, at most "
                        f"{MAX_ATTEMPTS} passes; the first clean pass is reported, else (every pass stalled) "
                        f"the one with the lowest median",
        "reported_attempts": {"timed": reported_a, "dominant_kernel": reported_b},
        "step_us_per_step": [round(1e3 * x, 1) for x in step_ms],
        "dominant_kernel_us_per_step": [round(1e3 * x, 1) for x in dom_ms],
        "misses_per_step": float(misses.mean()), "miss_h2d_gbs": link_gbs, "h2d_ceiling_gbs": h2d_ceiling,
        "miss_h2d_frac_of_ceiling": link_gbs / h2d_ceiling,
        "miss_h2d_gbs_whole_call": call_gbs,
        "roofline": {"bound": "host_link", "achieved": link_gbs, "peak": h2d_ceiling, "unit": "GB/s",
                     "frac": link_gbs / h2d_ceiling,
                     "traffic": traffic.get("sysmem_read_bytes_per_launch"),
                     "traffic_metric": "ncu syslts sysmem read sectors x 32 B per launch (null: kernel changed)",
                     "algorithmic_bytes_per_launch": float(miss_bytes.mean()),
                     "kernel": dominant,
                     "kernel_timing": "CUDA events around the kernel's own launch on the launching stream, "
                                      "eager pass over the timed steps",
                     "copy_ctas_per_request": copy_ctas,
                     "peak_source": "pinned cudaMemcpy H2D, 1 GiB, best of 12, measured in this run",
                     "hbm": {"achieved": hbm_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": hbm_gbs / hbm_peak,
                             "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)",
                             "traffic": (traffic["dram_read_bytes_per_launch"] + traffic["dram_write_bytes_per_launch"])
                             if traffic else None,
                             "algorithmic_bytes_per_launch": float(hbm_bytes.mean()),
                             "timing": "the whole resolve work (all its launches)"}},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
                "steps": e2e_steps, "p50_step_us": 1e3 * float(np.median(e2e_ms)),
                "attempts_p50_step_us": e2e_tries, "copies_attempts_p50_step_us": e2e_copy_tries,
                "timing": "wall clock per step, graph launch to stream sync; the step's inputs are in one "
                          "pinned host block the host refills before each step and its outputs go to one "
                          "pinned host block: hs_resolve reads the top-k rows and seq_lens and writes the row "
                          "table and miss counts over the host link (zero-copy step I/O), hs_backup reads "
                          "seq_lens there; one graph replayed every step",
                "copies_value": e2e_copy_value, "copies_p50_step_us": 1e3 * float(np.median(e2e_copy_ms)),
                "copies_timing": "the same step with one H2D copy of the inputs into device buffers and one D2H "
                                 "copy of the outputs in the graph"},
        "host_pool": ("huge pages, hs_host_register" if pool_objs[0][1]
                      else "cudaHostAlloc (host could not back the pool with huge pages)"),
        "host_numa_node": numa_node,
        "gpu_launches": (launches_per_resolve + 1) * K_,
        "device_flags": err,
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        wl_cpu = make_workload(args, 0, W_ + K_)
        rows_c, sec_c = cpu_oracle_run(wl_cpu, host, W_, K_)
        line["cpu_baseline"] = {"value": rows_c / sec_c, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"the timed decode steps {W_}..{W_ + K_ - 1} of the same workload "
                                          f"(after {W_} untimed warm-up steps), single-threaded C oracle "
                                          "(resolve + row copies + backup)"}
        ncores = len(os.sched_getaffinity(0))
        rows_m, sec_m = cpu_oracle_run(make_workload(args, 0, W_ + K_), host, W_, K_, nthreads=ncores)
        line["cpu_baseline_threaded"] = {"value": rows_m / sec_m, "unit": UNIT, "cores": ncores,
                                         "kind": "oracle sharded by request over threads"}
    hs.hs_destroy(h)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
def measured_hbm_peak() -> float:
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("hbm_gbs", 6800.0))
    except (OSError, ValueError):
        return 6800.0


REWRITTEN = 64  # positions per request a prefill chunk rewrote on the host


def run_invalidate(args, ws, rank, local):
    """One hot-slot invalidation call per timed iteration on a seeded mid-decode slot map of
    the workload's shape: by token (each request drops the REWRITTEN positions before its
    newest token) or by host row (the sorted host rows of the same positions). The state is
    restored and L2 flushed before each call, outside the timed events."""
    import torch
    import hierarchical_sparse_attention_gb300 as hs
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.make(args.config, args.seed + 1000 * rank, steps=1)
    R, K, H, B, L = wl.R, wl.K, wl.H, wl.B, wl.L
    tok0, st0, _ = wl.warm_slot_state(args.seed + 1000 * rank)
    offs, toks = wl.rewritten_positions(REWRITTEN)
    S = wl.seq_lens(0)
    rows = np.unique(np.concatenate([wl.host_cache_locs[r, toks[offs[r]:offs[r + 1]]] for r in range(R)]))
    rows = rows.astype(np.int32)
    g_tok0, g_st0 = torch.from_numpy(tok0).to(dev), torch.from_numpy(st0).to(dev)
    tok, st = g_tok0.clone(), g_st0.clone()
    g_S, g_offs, g_toks = (torch.from_numpy(x).to(dev) for x in (S, offs, toks))
    g_hcl, g_rows = torch.from_numpy(wl.host_cache_locs).to(dev), torch.from_numpy(rows).to(dev)
    cfg = hs.make_config(R, K, H, B, L, wl.ps, wl.max_context, wl.max_pages)
    wsp = torch.zeros(hs.hs_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    hostp = [np.zeros(16 * B, dtype=np.uint8) for _ in range(L)]
    for p in hostp:
        hs.hs_host_register(p)
    devp = [torch.zeros(16 * B, dtype=torch.uint8, device=dev) for _ in range(L)]
    h = hs.hs_create(cfg, hostp, devp, 16, 16, wsp)  # the invalidation never touches pools
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def call():
        if args.op == "invalidate_tokens":
            hs.hs_invalidate_tokens(h, R, g_S, g_offs, g_toks, tok, st, stream)
        else:
            hs.hs_invalidate_host_rows(h, R, g_S, g_hcl, g_rows, rows.size, tok, st, stream)

    for _ in range(args.warmup):
        tok.copy_(g_tok0); st.copy_(g_st0)
        call()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local, enabled=not args.no_clocks) as clocks:
        for i in range(args.steps):
            tok.copy_(g_tok0); st.copy_(g_st0)
            flush.zero_()
            evs[i][0].record(stream)
            call()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    ms = [e[0].elapsed_time(e[1]) for e in evs]
    err = hs.hs_get_error(h, clear=True)
    cleared = int((tok != g_tok0).sum().item())
    hs.hs_destroy(h)
    for p in hostp:
        hs.hs_host_unregister(p)
    mean_s = max_over_ranks(sum(ms) / len(ms) * 1e-3, ws)
    # algorithmic bytes per call: the slot maps read, the list(s) read, cleared slots written
    # (token + stamp, and the hint), plus the host-row lookups of held tokens in the row form
    slots_read = int(((S > H) * H).sum()) * 4
    held = int((tok0 >= 0).sum())
    list_bytes = (toks.size + R + 1) * 4 if args.op == "invalidate_tokens" else rows.size * 4 + held * 4
    alg = slots_read + list_bytes + cleared * 10
    hbm = measured_hbm_peak()
    line = {
        "metric": f"{args.op.replace('invalidate_', 'hs_invalidate_')} latency", "value": 1e6 * mean_s,
        "unit": "us", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean_s,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": f"{args.config}: {R} requests x {H} hot slots, seq {int(S.max())}, "
                               f"{REWRITTEN} rewritten positions per request"
                               + (f" ({rows.size} sorted host rows)" if args.op != "invalidate_tokens" else ""),
                   "l2": "flushed between timed calls (256 MiB write)", "parallelism": f"requests sharded, dp{ws}"},
        "p50_us": 1e3 * float(np.median(ms)), "slots_cleared": cleared,
        "roofline": {"bound": "hbm", "achieved": alg / mean_s / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": alg / mean_s / 1e9 / hbm, "traffic": None, "algorithmic_bytes_per_launch": alg,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)",
                     "note": "one CTA per request over a few KB of state each: launch latency, not HBM, bounds it"},
        "gpu_launches": args.steps, "device_flags": err, "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_split(args, ws, rank, local):
    """A layer group's decode step two ways over the same steps: fused (hs_resolve copies
    every layer) and split (hs_resolve_layers copies layer 0, then hs_gather copies each
    follower layer on a copy stream behind its own event). Per step it times, from the
    step's start: layer 0 ready, each follower ready, all layers ready."""
    import torch
    import hierarchical_sparse_attention_gb300 as hs
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    W_, K_ = args.warmup, args.steps
    total = W_ + K_
    wl = make_workload(args, rank, total)
    R, K, H, B, L = wl.R, wl.K, wl.H, wl.B, wl.L
    assert L >= 2, "the split needs at least two layers"
    host, pools = build_host_pools(wl, hs, rank_numa_node(local))
    dpool = []
    for l in range(L):
        init = np.full(wl.device_rows * B, 0xA5, dtype=np.uint8)
        rq, tk0, rows0 = wl.initial_device_writes()
        wl.scatter_rows(l, rq, tk0, rows0, init)
        dpool.append(torch.from_numpy(init).to(dev))
    topk_all = torch.from_numpy(np.stack([wl.top_k_tokens(s) for s in range(total)])).to(dev)
    seq_all = torch.from_numpy(np.stack([wl.seq_lens(s) for s in range(total)])).to(dev)
    newest = [newest_rows(wl, s) for s in range(total)]
    newest_idx = torch.from_numpy(np.stack([n[0] for n in newest])).to(dev)
    newest_dat = [torch.from_numpy(np.stack([n[1][l] for n in newest])).to(dev) for l in range(L)]
    hcl = torch.from_numpy(wl.host_cache_locs).to(dev)
    dbl = torch.from_numpy(wl.device_buffer_locs).to(dev)
    rp = None if wl.resident_pages is None else torch.from_numpy(wl.resident_pages).to(dev)
    tok0, st0, clk0 = wl.initial_state()
    tk_buf = torch.empty((R, K), dtype=torch.int32, device=dev)
    sl_buf = torch.empty((R,), dtype=torch.int32, device=dev)
    out = torch.empty((R, K), dtype=torch.int32, device=dev)
    miss = torch.empty((R,), dtype=torch.int32, device=dev)
    cfg = hs.make_config(R, K, H, B, L, wl.ps, wl.max_context, wl.max_pages,
                         wl.host_row_stride if wl.cfg.host_layout == "page_first" else 0)
    wsps = {v: torch.zeros(hs.hs_workspace_bytes(cfg), dtype=torch.uint8, device=dev) for v in ("fused", "split", "split0")}
    handles = {v: hs.hs_create(cfg, host, dpool, wl.host_rows, wl.device_rows, wsps[v]) for v in wsps}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def forward_stand_in(s):
        for l in range(L):
            dpool[l].view(-1, B).index_copy_(0, newest_idx[s], newest_dat[l][s])
        tk_buf.copy_(topk_all[s])
        sl_buf.copy_(seq_all[s])

    # two copies of the slot state, one per variant; both variants see the same inputs, so
    # they make the same decisions and write the same rows
    states = {v: tuple(torch.from_numpy(x).to(dev) for x in (tok0, st0, clk0)) for v in ("fused", "split", "split0")}

    def one_step(s, variant, evs):
        tok, st, clk = states[variant]
        h = handles[variant]  # each variant keeps its own hints and plan
        forward_stand_in(s)
        flush.zero_()
        if evs is not None:
            evs[0].record(stream)
        if variant in ("split", "split0"):
            if variant == "split":
                hs.hs_resolve_layers(h, R, tk_buf, sl_buf, hcl, dbl, tok, st, clk, rp, out, miss, 1, stream)
            else:  # the resolve copies nothing; layer 0 is gathered right behind it
                hs.hs_resolve_layers(h, R, tk_buf, sl_buf, hcl, dbl, tok, st, clk, rp, out, miss, 0, stream)
                hs.hs_gather(h, R, hcl, 0, 1, stream)
            if evs is not None:
                evs[1].record(stream)  # layer 0 ready
            lead = torch.cuda.Event()
            lead.record(stream)
            copy.wait_event(lead)
            for l in range(1, L):
                hs.hs_gather(h, R, hcl, l, 1, copy)
                if evs is not None:
                    evs[1 + l].record(copy)  # layer l ready
            done = torch.cuda.Event()
            done.record(copy)
            stream.wait_event(done)
        else:
            hs.hs_resolve(h, R, tk_buf, sl_buf, hcl, dbl, tok, st, clk, rp, out, miss, stream)
            if evs is not None:
                for l in range(L):
                    evs[1 + l].record(stream)  # every layer ready at once
        hs.hs_backup(h, R, sl_buf, hcl, dbl, rp, stream)

    # steps interleave the variants on the same step's inputs, so all meet the host pool in the
    # same state; the order rotates each step, since the first to read a step's rows pays for
    # the host pages it is first to reach
    variants = ("fused", "split", "split0")

    def rotated(s):
        k = s % len(variants)
        return variants[k:] + variants[:k]

    for s in range(W_):
        for v in rotated(s):
            one_step(s, v, None)
    torch.cuda.synchronize()
    evs = {v: [[torch.cuda.Event(enable_timing=True) for _ in range(L + 1)] for _ in range(K_)]
           for v in ("fused", "split", "split0")}
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(K_):
        for v in rotated(W_ + i):
            one_step(W_ + i, v, evs[v][i])
    torch.cuda.synchronize()
    barrier(ws)
    res = {v: np.array([[e[0].elapsed_time(e[1 + l]) * 1e3 for l in range(L)] for e in evs[v]]) for v in evs}
    err = 0
    copy_ctas, per_resolve = hs.hs_launch_shape(handles["fused"])
    order = 2  # the two kernels that group the plan by host region before follower gathers
    split_launches = (per_resolve if copy_ctas == 0 else 1 + order) + (L - 1) + 1
    split0_launches = 1 + order + 1 + (L - 1) + 1
    for h in handles.values():
        err |= hs.hs_get_error(h, clear=True)
        hs.hs_destroy(h)
    for arr, reg in pools:
        if reg:
            hs.hs_host_unregister(arr)
    f, sp, s0 = res["fused"], res["split"], res["split0"]
    line = {
        "metric": "time to first layer ready (leader resolve + follower gathers)", "value": float(sp[:, 0].mean()),
        "unit": "us", "n_gpus": ws, "steps": K_, "warmup": W_, "ms_per_step": float(sp[:, -1].mean()) / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": f"{args.config}: {R} requests, top_k {K}, {H} hot slots, {B}-byte rows, {L} layers, "
                               f"host pools {wl.cfg.host_layout.replace('_', '-')}",
                   "l2": "flushed between timed steps (256 MiB write)",
                   "split": "hs_resolve_layers(copy_layers=1) then hs_gather(l, 1) for l = 1..L-1 on a copy stream"},
        "split_layer_ready_us_mean": [float(x) for x in sp.mean(0)],
        "split_layer_ready_us_p50": [float(x) for x in np.median(sp, 0)],
        "fused_all_layers_ready_us_p50": float(np.median(f[:, -1])),
        "fused_all_layers_ready_us_mean": float(f[:, -1].mean()),
        "split_all_layers_ready_us_mean": float(sp.max(1).mean()),
        "first_layer_ready_speedup": float(f[:, -1].mean() / sp[:, 0].mean()),
        "split0_layer_ready_us_p50": [float(x) for x in np.median(s0, 0)],
        "split0": "hs_resolve_layers(copy_layers=0), hs_gather(0, 1) on the same stream, followers on the copy stream",
        "misses_per_step": float(miss.sum().item()),
        "gpu_launches": K_ * ((per_resolve + 1) + split_launches + split0_launches), "device_flags": err,
        "copy_ctas_per_request": copy_ctas,
        "host_pool": "huge pages, hs_host_register" if pools[0][1] else "cudaHostAlloc",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


MLA_HEADS = 128  # query heads per request on one GPU (attention data-parallel)


def measured_bf16_peak(sustained: bool = False) -> float:
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d.get("bf16_tflops_sustained" if sustained else "bf16_tflops", 1900.0))
    except (OSError, ValueError):
        return 1900.0


def run_mla(args, ws, rank, local):
    """The synthetic consumer alone: sparse-MLA decode attention (hs_sparse_mla_decode) over
    a row table of the workload's shape -- each request's top_k distinct rows drawn from its
    own part of the device pool (its hot buffer), MLA_HEADS query heads. Times each split
    count (1, 2, 4) with L2 flushed between calls and reports the fastest as the line."""
    import torch
    import hierarchical_sparse_attention_gb300 as hs
    import workloads as W
    from collections import OrderedDict

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    wl = W.make(args.config, args.seed + 1000 * rank, steps=2)
    R, K, H, B = wl.R, wl.K, wl.H, wl.B
    assert B == 656, "the consumer reads fp8 MLA rows"
    Hq = MLA_HEADS
    rng = np.random.default_rng(args.seed + 5)
    # the device pool holds real rows: each request's buffer rows carry some token's bytes
    pool = np.empty(wl.device_rows * B, dtype=np.uint8)
    for r in range(R):
        toks = rng.integers(0, int(wl.seq0[r]) - 1, size=H + 1)
        rows = wl.device_buffer_locs[r]
        data = wl.rows(0, r, [int(t) for t in toks])
        pool.reshape(-1, B)[rows] = data.reshape(-1, B)
    out_rows = np.stack([rng.permutation(wl.device_buffer_locs[r][:H])[:K] for r in range(R)]).astype(np.int32)
    q = wl.queries_bf16(0, Hq)
    g_pool = torch.from_numpy(pool).to(dev)
    g_rows = torch.from_numpy(out_rows).to(dev)
    g_q = torch.from_numpy(q.view(np.int16)).to(dev)
    o = torch.empty((R, Hq, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((R, Hq), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sm_scale = 1.0 / 1400.0  # about unit-spread scores on the synthetic fp8 rows
    flops = 2.0 * R * Hq * K * (576 + 512)  # S = Q K^T and O = P V, algorithmic
    bytes_alg = R * K * B + q.nbytes + o.numel() * 4 + lse.numel() * 4 + out_rows.nbytes
    res = OrderedDict()
    for splits in (1, 2, 4):
        wsb = hs.hs_sparse_mla_workspace_bytes(R, Hq, splits)
        wsp = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)

        def call():
            hs.hs_sparse_mla_decode(R, Hq, K, splits, g_q, g_pool, wl.device_rows, g_rows, sm_scale, o, lse, wsp,
                                    wsb, err, stream)

        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        barrier(ws)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            call()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        ms = [e[0].elapsed_time(e[1]) for e in evs]
        res[splits] = (max_over_ranks(sum(ms) / len(ms) * 1e-3, ws), float(np.median(ms)) * 1e3)
    best = min(res, key=lambda k: res[k][0])
    t = res[best][0]
    peak = measured_bf16_peak()
    line = {
        "metric": "sparse-MLA decode attention over the row table (TFLOP/s)", "value": ws * flops / t / 1e12,
        "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"{args.config}: {R} requests x {Hq} heads x top_k {K} rows of {B} B (fp8 MLA), "
                               f"576-dim keys, 512-dim values, splits {best}",
                   "l2": "flushed between timed calls (256 MiB write)"},
        "per_split_count_us": {str(k): {"mean": 1e6 * v[0], "p50": v[1]} for k, v in res.items()},
        "roofline": {"bound": "tensor", "achieved": flops / t / 1e12, "peak": peak, "unit": "TFLOP/s",
                     "frac": flops / t / 1e12 / peak, "traffic": None,
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops (of measured); fp16 and bf16 share the "
                                    "nominal dense rate, so the bf16 figure stands for the fp16 operands",
                     "hbm": {"achieved": bytes_alg / t / 1e9, "peak": measured_hbm_peak(), "unit": "GB/s",
                             "algorithmic_bytes_per_launch": bytes_alg}},
        "gpu_launches": args.steps * hs.hs_sparse_mla_launches(R, Hq, best), "device_flags": int(err.item()),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, ws, rank, local):
    """The decode step with its consumer: hs_resolve + hs_backup, then the synthetic sparse-MLA
    attention (hs_sparse_mla_decode, MLA_HEADS heads, 2 splits) over the rows the resolve
    returned, on layer 0's device pool. Three timed passes over the same steps, each from the
    same state: resolve + backup (graph), attention alone, the whole step (one graph)."""
    import torch
    import hierarchical_sparse_attention_gb300 as hs
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    W_, K_ = args.warmup, args.steps
    total = W_ + K_
    wl = W.make(args.config, args.seed + 1000 * rank, steps=total)
    R, K, H, B, L = wl.R, wl.K, wl.H, wl.B, wl.L
    assert B == 656, "the consumer reads fp8 MLA rows"
    pools = [alloc_host(wl.host_rows * B) for _ in range(L)]
    for l, (arr, reg) in enumerate(pools):
        wl.fill_host_pool(l, arr)
        touch_host_pool_from_gpu(hs.hs_host_register(arr) if reg else host_device_ptr(arr), arr.nbytes)
    host = [arr for arr, _ in pools]
    dpool = []
    for l in range(L):
        init = np.full(wl.device_rows * B, 0xA5, dtype=np.uint8)
        rq, tk0, rows0 = wl.initial_device_writes()
        wl.scatter_rows(l, rq, tk0, rows0, init)
        dpool.append(torch.from_numpy(init).to(dev))
    topk_all = torch.from_numpy(np.stack([wl.top_k_tokens(s) for s in range(total)])).to(dev)
    seq_all = torch.from_numpy(np.stack([wl.seq_lens(s) for s in range(total)])).to(dev)
    newest = [newest_rows(wl, s) for s in range(total)]
    newest_idx = torch.from_numpy(np.stack([n[0] for n in newest])).to(dev)
    newest_dat = [torch.from_numpy(np.stack([n[1][l] for n in newest])).to(dev) for l in range(L)]
    hcl = torch.from_numpy(wl.host_cache_locs).to(dev)
    dbl = torch.from_numpy(wl.device_buffer_locs).to(dev)
    tok0, st0, clk0 = wl.initial_state()
    tok, st, clk = (torch.from_numpy(x).to(dev) for x in (tok0, st0, clk0))
    tk_buf = torch.empty((R, K), dtype=torch.int32, device=dev)
    sl_buf = torch.empty((R,), dtype=torch.int32, device=dev)
    out = torch.empty((R, K), dtype=torch.int32, device=dev)
    miss = torch.empty((R,), dtype=torch.int32, device=dev)
    cfg = hs.make_config(R, K, H, B, L, wl.ps, wl.max_context, wl.max_pages)
    wsp = torch.zeros(hs.hs_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = hs.hs_create(cfg, host, dpool, wl.host_rows, wl.device_rows, wsp)
    resolve_launches = hs.hs_launch_shape(h)[1]
    Hq, splits = MLA_HEADS, 2  # two splits: 64 CTA pairs on 128 SMs (one cluster of four per request)
    qs = [torch.from_numpy(wl.queries_bf16(i, Hq).view(np.int16)).to(dev) for i in range(4)]
    q_buf = torch.empty_like(qs[0])
    o = torch.empty((R, Hq, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((R, Hq), dtype=torch.float32, device=dev)
    mwsb = hs.hs_sparse_mla_workspace_bytes(R, Hq, splits)
    mws = torch.zeros(max(mwsb, 16), dtype=torch.uint8, device=dev)
    merr = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def forward_stand_in(s):
        for l in range(L):
            dpool[l].view(-1, B).index_copy_(0, newest_idx[s], newest_dat[l][s])
        tk_buf.copy_(topk_all[s])
        sl_buf.copy_(seq_all[s])
        q_buf.copy_(qs[s % 4])

    def resolve_backup(strm):
        hs.hs_resolve(h, R, tk_buf, sl_buf, hcl, dbl, tok, st, clk, None, out, miss, strm)
        hs.hs_backup(h, R, sl_buf, hcl, dbl, None, strm)

    def attention(strm):
        hs.hs_sparse_mla_decode(R, Hq, K, splits, q_buf, dpool[0], wl.device_rows, out, 1.0 / 1400.0, o, lse, mws,
                                mwsb, merr, strm)

    def reset():
        tok.copy_(torch.from_numpy(tok0)); st.copy_(torch.from_numpy(st0)); clk.copy_(torch.from_numpy(clk0))
        hs.hs_reset_hints(h, stream)
        for s in range(W_):
            forward_stand_in(s)
            resolve_backup(stream)
            attention(stream)
        torch.cuda.synchronize()

    graphs = {}
    for name, fns in (("resolve", (resolve_backup,)), ("step", (resolve_backup, attention))):
        reset()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for fn in fns:
                fn(torch.cuda.current_stream())
        stream.wait_stream(cap)
        graphs[name] = g
    times = {}
    for name in ("resolve", "attention", "step"):
        reset()
        for i in range(K_):  # rehearsal, untimed (host-pool first access)
            forward_stand_in(W_ + i)
            if name == "attention":
                resolve_backup(stream)
                attention(stream)
            else:
                graphs[name].replay()
        torch.cuda.synchronize()
        reset()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K_)]
        barrier(ws)
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e6 * (5 + K_ // 4)))
        for i in range(K_):
            forward_stand_in(W_ + i)
            if name == "attention":
                resolve_backup(stream)  # untimed: the rows this step's attention reads
            flush.zero_()
            evs[i][0].record(stream)
            if name == "attention":
                attention(stream)
            else:
                graphs[name].replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        ms = [e[0].elapsed_time(e[1]) for e in evs]
        times[name] = (max_over_ranks(sum(ms) * 1e-3, ws), float(np.median(ms)) * 1e3)
    err = hs.hs_get_error(h, clear=True)
    hs.hs_destroy(h)
    for arr, reg in pools:
        if reg:
            hs.hs_host_unregister(arr)
    rows = int((topk_all[W_:] >= 0).sum().item())
    t_step = times["step"][0]
    line = {
        "metric": "decode steps/s with the sparse-MLA consumer (resolve + backup + attention)",
        "value": ws * K_ / t_step, "unit": "steps/s", "n_gpus": ws, "steps": K_, "warmup": W_,
        "ms_per_step": 1e3 * t_step / K_, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32+f16", "data": "synthetic",
        "config": {"workload": f"{args.config}: {R} requests, top_k {K}, {H} hot slots, {B}-byte fp8 MLA rows; "
                               f"attention {Hq} heads x 576/512 dims, {splits} split(s)",
                   "l2": "flushed between timed steps (256 MiB write)"},
        "p50_us": {k: v[1] for k, v in times.items()},
        "mean_us": {k: 1e6 * v[0] / K_ for k, v in times.items()},
        "top_k_rows_resolved_per_s_in_step": ws * rows / t_step,
        "gpu_launches": K_ * (resolve_launches + 1 + hs.hs_sparse_mla_launches(R, Hq, splits)),
        "device_flags": err, "attention_flags": int(merr.item()),
        "host_pool": "huge pages, hs_host_register" if pools[0][1] else "cudaHostAlloc",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


SPEC_QUERIES = 4  # n_spec = 3 draft tokens (MTP3) + the sampled one


def run_spec(args, ws, rank, local):
    """Speculative batches at the workload's shape: Q = SPEC_QUERIES verify steps per batch,
    H = (Q + 1) * top_k hot slots (the buffer the pages size for n_spec + 2), every position
    accepted. Per batch the forward stand-in writes the Q new rows, then hs_resolve_spec
    (one launch for the Q verify steps when each request has copy CTAs) and hs_backup_spec
    run; events bracket resolve + backup. Top-k rows keep 90 % of the previous verify step's
    row and draw the rest over the step's length."""
    import torch
    import hierarchical_sparse_attention_gb300 as hs
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    Q = SPEC_QUERIES
    W_, K_ = args.warmup, args.steps
    nb = W_ + K_
    wl = W.make(args.config, args.seed + 1000 * rank, steps=nb * Q + 2)
    R, K, B, L = wl.R, wl.K, wl.B, wl.L
    H = (Q + 1) * K
    pools = [alloc_host(wl.host_rows * B) for _ in range(L)]
    for l, (arr, reg) in enumerate(pools):
        wl.fill_host_pool(l, arr)
        touch_host_pool_from_gpu(hs.hs_host_register(arr) if reg else host_device_ptr(arr), arr.nbytes)
    host = [arr for arr, _ in pools]
    dev_rows = R * (H + Q)
    dpool = [torch.full((dev_rows * B,), 0xA5, dtype=torch.uint8, device=dev) for _ in range(L)]
    dbl_np = np.arange(dev_rows, dtype=np.int32).reshape(R, H + Q)
    S0 = (wl.seq0 - 1).astype(np.int32)
    assert int(S0.min()) + 1 > H, "every request starts past the fast path"
    rng = np.random.default_rng(args.seed + 77)
    tks, s0s = [], []
    prev = [rng.choice(int(S0[r]), size=K, replace=False).astype(np.int32) for r in range(R)]
    for b in range(nb):
        tk = np.empty((Q, R, K), np.int32)
        for q in range(Q):
            for r in range(R):
                S = int(S0[r]) + q + 1
                keep = rng.permutation(prev[r])[: int(0.9 * K)]
                fresh = np.setdiff1d(rng.integers(0, S, size=2 * K).astype(np.int32), keep)
                fresh = rng.permutation(fresh)[: K - keep.size]
                row = np.concatenate([keep, fresh])
                if row.size < K:
                    row = np.concatenate([row, np.full(K - row.size, -1, np.int32)])
                tk[q, r] = rng.permutation(row)
                prev[r] = row[row >= 0]
        tks.append(tk)
        s0s.append(S0.copy())
        S0 = S0 + Q
    g_tk = torch.from_numpy(np.stack(tks)).to(dev)
    g_s0 = torch.from_numpy(np.stack(s0s)).to(dev)
    acc = torch.full((R,), Q, dtype=torch.int32, device=dev)
    # the forward writes: batch b's position S0 + j of request r goes to reserved row H + j
    new_rows = torch.from_numpy(dbl_np[:, H:].reshape(-1).astype(np.int64)).to(dev)
    new_dat = [torch.from_numpy(np.concatenate([wl.rows(l, r, list(range(int(s0s[0][r]), int(s0s[0][r]) + Q)))
                                                for r in range(R)])).to(dev) for l in range(L)]
    hcl = torch.from_numpy(wl.host_cache_locs).to(dev)
    dbl = torch.from_numpy(dbl_np).to(dev)
    tok = torch.full((R, H), -1, dtype=torch.int32, device=dev)
    st = torch.zeros((R, H), dtype=torch.int32, device=dev)
    clk = torch.zeros((R,), dtype=torch.int32, device=dev)
    out = torch.empty((Q, R, K), dtype=torch.int32, device=dev)
    miss = torch.empty((Q, R), dtype=torch.int32, device=dev)
    cfg = hs.make_config(R, K, H, B, L, wl.ps, wl.max_context, wl.max_pages)
    wsp = torch.zeros(hs.hs_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    h = hs.hs_create(cfg, host, dpool, wl.host_rows, dev_rows, wsp)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    miss_acc = torch.zeros((nb, Q, R), dtype=torch.int64, device=dev)

    def batch(b, evs):
        for l in range(L):  # the forward pass's new rows (their bytes do not matter here)
            dpool[l].view(-1, B).index_copy_(0, new_rows, new_dat[l])
        flush.zero_()
        if evs is not None:
            evs[0].record(stream)
        hs.hs_resolve_spec(h, R, Q, g_tk[b], g_s0[b], hcl, dbl, tok, st, clk, None, out, miss, stream)
        hs.hs_backup_spec(h, R, Q, g_s0[b], acc, hcl, dbl, None, stream)
        if evs is not None:
            evs[1].record(stream)
        miss_acc[b].copy_(miss)

    for b in range(W_):
        batch(b, None)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K_)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local, enabled=not args.no_clocks) as clocks:
        torch.cuda._sleep(int(2e6 * (5 + K_ // 4)))
        for i in range(K_):
            batch(W_ + i, evs[i])
        torch.cuda.synchronize()
    barrier(ws)
    ms = [e[0].elapsed_time(e[1]) for e in evs]
    err = hs.hs_get_error(h, clear=True)
    copy_ctas, _ = hs.hs_launch_shape(h)
    # one resolve launch per batch; without copy CTAs each step's plan is then grouped by host
    # region (two launches) and gathered (one)
    per_batch = 1 + (0 if copy_ctas > 0 else 3 * Q) + 1
    hs.hs_destroy(h)
    for arr, reg in pools:
        if reg:
            hs.hs_host_unregister(arr)
    total_s = max_over_ranks(sum(ms) * 1e-3, ws)
    rows = int((np.stack(tks[W_:]) >= 0).sum())
    misses = miss_acc[W_:].sum(dim=2).float().mean(dim=0).cpu().numpy()  # per verify step
    line = {
        "metric": "top-k rows resolved/s (speculative batches)", "value": ws * rows / total_s, "unit": "rows/s",
        "n_gpus": ws, "steps": K_, "warmup": W_, "ms_per_step": 1e3 * total_s / K_, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"{args.config}: {R} requests, top_k {K}, {Q} verify steps per batch "
                               f"(n_spec {Q - 1}), H = (n_spec + 2) * top_k = {H} slots, {B}-byte rows, "
                               "every draft accepted",
                   "l2": "flushed between timed batches (256 MiB write)",
                   "step": "hs_resolve_spec (the Q verify steps in one launch) + hs_backup_spec"},
        "p50_batch_us": 1e3 * float(np.median(ms)), "p50_per_verify_step_us": 1e3 * float(np.median(ms)) / Q,
        "misses_per_verify_step": [float(x) for x in misses],
        "gpu_launches": K_ * per_batch, "copy_ctas_per_request": copy_ctas, "device_flags": err,
        "clocks": clocks.summary(),
        "host_pool": "huge pages, hs_host_register" if pools[0][1] else "cudaHostAlloc",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.config is None:
        args.config = "indexshare" if args.op in ("step", "split") else "dsa"
    ws, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.op == "e2e":
        run_e2e(args, ws, rank, local)
    elif args.op == "mla":
        run_mla(args, ws, rank, local)
    elif args.op == "spec":
        run_spec(args, ws, rank, local)
    elif args.op == "split":
        run_split(args, ws, rank, local)
    elif args.op != "step":
        run_invalidate(args, ws, rank, local)
    elif args.sweep and ws == 1:
        # One process per point, as a serving process holds one pool for its lifetime:
        # tearing down and rebuilding tens of GB of pinned host memory inside one process
        # leaves later points on fragmented memory (no huge pages) or with host-link stalls.
        import workloads as W
        fwd = ["--steps", str(args.steps), "--warmup", str(args.warmup), "--seed", str(args.seed)]
        fwd += ["--no-cpu-baseline"] * args.no_cpu_baseline + ["--no-clocks"] * args.no_clocks
        for hot in W.SWEEP_HOT:
            for reuse in W.SWEEP_REUSE:
                r = subprocess.run([sys.executable, os.path.abspath(__file__), "--config",
                                    f"sweep_h{hot}_f{reuse}"] + fwd)
                if r.returncode != 0:
                    sys.exit(r.returncode)
    elif args.sweep:
        import workloads as W
        for hot in W.SWEEP_HOT:
            for reuse in W.SWEEP_REUSE:
                args.config = f"sweep_h{hot}_f{reuse}"
                run_ours(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
