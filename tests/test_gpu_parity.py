"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit-exact.

Each step, both sides get the same seeded inputs; the test compares the physical row
table, the miss counts, the slot map, the stamps, the clock and the error flags every
step, the eager backup's host rows every step, and the whole device pools (hot rows,
reserved rows, resident pages) at intervals and at the end. All comparisons are exact:
the path is integer bookkeeping and byte copies.

The two sides share no memory: the oracle fills and keeps its own host pools, the GPU gets
pinned pools with guard rows around them (and around its device pools and workspace). So
besides agreeing with the oracle, every row a GPU step resolved must hold the bytes the seeded
generator gives its token (regenerated, in every layer), and at the end the GPU's whole host
pools -- written only by its backups -- must equal the oracle's, with every guard intact.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from harness import OracleSim, host_newest_ok, poison_host_newest  # noqa: E402

pytestmark = pytest.mark.gpu

ROWS_EVERY_STEP = 1 << 20  # check the resolved rows every step when a step has at most this many


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hierarchical_sparse_attention_gb300 as hs  # noqa: F401
    import gpu_harness
    return gpu_harness


def compare_step(gpu, orc, what):
    import hierarchical_sparse_attention_gb300 as hs
    g = gpu.state()
    np.testing.assert_array_equal(g["out"], orc.out, err_msg=f"{what}: out_rows")
    np.testing.assert_array_equal(g["miss"], orc.miss, err_msg=f"{what}: miss_counts")
    np.testing.assert_array_equal(g["tokens"], orc.tokens, err_msg=f"{what}: device_buffer_tokens")
    np.testing.assert_array_equal(g["stamps"], orc.stamps, err_msg=f"{what}: lru_slots")
    np.testing.assert_array_equal(g["clock"], orc.clock, err_msg=f"{what}: lru_clock")
    return hs.hs_get_error(gpu.h, clear=True)


def compare_pools(gpu, orc, what):
    for layer in range(len(gpu.dev)):
        d = gpu.dev[layer].cpu().numpy()
        if not np.array_equal(d, orc.dev[layer]):
            rows = np.nonzero((d.reshape(-1, orc.wl.B) != orc.dev[layer].reshape(-1, orc.wl.B)).any(1))[0]
            raise AssertionError(f"{what}: device pool layer {layer} differs in {len(rows)} rows, e.g. {rows[:8]}")


def run_parity(wl, pools=None, steps=None, pool_every=8, graph_from=None, host_io=False):
    """pools: (gpu host pools, their base arrays, oracle host pools) to reuse across runs of
    one host layout; by default each side gets fresh ones."""
    gh = _gpu()
    if pools is None:
        host, bases = gh.host_pools(wl)
        orc = OracleSim(wl)
        own = True
    else:
        host, bases, orc_host = pools
        orc = OracleSim(wl, host_pools=orc_host)
        own = False
    gpu = gh.GpuSim(wl, host, orc.dev, host_io=host_io, host_bases=bases)
    steps = wl.steps if steps is None else steps
    rows_every = 1 if wl.R * wl.K * wl.L <= ROWS_EVERY_STEP else pool_every
    graph = None
    try:
        for step in range(steps):
            gpu.write_newest(step)
            orc.write_newest(step)
            poison_host_newest(wl, step, gpu.host)
            poison_host_newest(wl, step, orc.host)
            gpu.upload(step)
            if graph_from is not None and step >= graph_from:
                if graph is None:
                    graph = torch.cuda.CUDAGraph()
                    s = torch.cuda.Stream()
                    s.wait_stream(torch.cuda.current_stream())
                    with torch.cuda.graph(graph, stream=s):
                        gpu.resolve(stream=torch.cuda.current_stream())
                        gpu.backup(stream=torch.cuda.current_stream())
                    torch.cuda.current_stream().wait_stream(s)
                graph.replay()  # inputs were refreshed in place by upload()
            else:
                gpu.resolve()
                gpu.backup()
            torch.cuda.synchronize()
            what = f"{wl.cfg.name} step {step}"
            assert host_newest_ok(wl, step, gpu.host), f"{what}: backup did not restore the newest host rows"
            oerr = orc.resolve(step)
            oerr |= orc.backup(step)
            gerr = compare_step(gpu, orc, what)
            assert gerr == oerr, f"{what}: flags gpu {gerr} oracle {oerr}"
            last = step == steps - 1
            if (step + 1) % rows_every == 0 or last:
                gh.resolved_rows_ok(wl, gpu, wl.top_k_tokens(step), gpu.state()["out"], what)
            if (step + 1) % pool_every == 0 or last:
                compare_pools(gpu, orc, what)
        gh.final_host_check(orc, gpu, f"{wl.cfg.name} after {steps} steps")
    finally:
        gpu.close()
        if own:
            gh.free_host(bases)
    return orc


def test_tiny():
    orc = run_parity(W.make("tiny"), pool_every=1)
    assert orc.miss[0] > 0


def test_tiny_fast_to_slow_transition():
    wl = W.make("tiny", seq0=(8192, 120))  # request 1 outgrows the 128-slot buffer at step 9
    run_parity(wl, pool_every=1)


def test_dsa_decode_shape():
    run_parity(W.make("dsa"), pool_every=16)


def test_mixed_residency_1m():
    run_parity(W.make("mixed1m"), pool_every=16)


def test_indexshare_4_layers():
    run_parity(W.make("indexshare"), pool_every=32)


def test_no_copy_ctas_resolve_and_gather_in_a_graph():
    """80 requests leave no SM for copy CTAs, so hs_resolve is four launches: the resolve
    (recording its plan, copying nothing), the two kernels that group the plan by host region,
    and a gather of all 3 layers. Eager for two steps, then the four replayed from a CUDA
    graph; every layer's rows match the oracle."""
    import hierarchical_sparse_attention_gb300 as hs
    gh = _gpu()
    wl = W.make("indexshare", 9, requests=80, top_k=64, hot_slots=128, steps=6, layers=3, seq_range=(1000, 3000))
    orc, gpu = gh.make_pair(wl)
    try:
        assert hs.hs_launch_shape(gpu.h) == (0, 4)
    finally:
        gh.close_pair(gpu)
    run_parity(wl, graph_from=2)
    few = W.make("indexshare", 9, requests=4, top_k=64, hot_slots=128, steps=1, layers=3, seq_range=(1000, 3000))
    orc, gpu = gh.make_pair(few)
    try:
        copy_ctas, launches = hs.hs_launch_shape(gpu.h)
        assert copy_ctas > 0 and launches == 1
    finally:
        gh.close_pair(gpu)


def test_no_copy_ctas_edges():
    """Without copy CTAs: every request on the fast path (an empty plan, no pairs to copy), and
    the largest top_k with a ragged sequence mix."""
    run_parity(W.make("indexshare", 10, requests=80, top_k=64, hot_slots=128, steps=4, layers=2,
                      seq_range=(60, 100)), pool_every=1)
    run_parity(W.make("indexshare", 11, requests=80, top_k=4096, hot_slots=4096, steps=3, layers=2,
                      seq_range=(3000, 9000)), pool_every=1)


def test_miss_rate_sweep():
    from harness import host_pools_for
    gh = _gpu()
    base = W.make("sweep_h4096_f0.8")
    # token rows and host layout do not depend on the sweep point: one set of pools per side
    host, bases = gh.host_pools(base)
    orc_host = host_pools_for(base)
    try:
        for h in W.SWEEP_HOT:
            for f in W.SWEEP_REUSE:
                wl = W.make(f"sweep_h{h}_f{f}")
                assert wl.host_rows == base.host_rows
                run_parity(wl, pools=(host, bases, orc_host), pool_every=32)
    finally:
        gh.free_host(bases)


@pytest.mark.parametrize("shape", [
    dict(requests=3, top_k=1000, hot_slots=3001, row_bytes=100, layers=3, seq0=(9000, 2000, 2500)),  # 4-byte path
    dict(requests=2, top_k=77, hot_slots=131, row_bytes=37, layers=2, seq0=(5000, 90)),  # byte path
    dict(requests=5, top_k=1, hot_slots=1, row_bytes=48, layers=1, seq0=(40, 1, 2, 3, 500)),  # K = H = 1
    dict(requests=4, top_k=2, hot_slots=2, row_bytes=32, layers=2, seq0=(40, 1, 2, 300)),  # K = H = 2
    dict(requests=2, top_k=2048, hot_slots=2048, row_bytes=656, layers=1, seq0=(300000, 2100)),  # H = K
    # the largest top_k: the top-k hash half full; > 1024 victims a step (the bitonic sort)
    dict(requests=2, top_k=4096, hot_slots=4096, row_bytes=656, layers=1, seq0=(200000, 4100)),
    dict(requests=2, top_k=4096, hot_slots=8192, row_bytes=656, layers=1, seq0=(200000, 9000)),  # row table global
])
def test_ragged_shapes(shape):
    kw = dict(shape)
    kw.setdefault("steps", 10)
    wl = W.make("tiny", fmt=W.FMT_U8, **kw)
    run_parity(wl, pool_every=1)


def test_graph_capture_replay():
    run_parity(W.make("dsa", requests=8, steps=12), pool_every=4, graph_from=2)


def test_zero_copy_step_io():
    """top_k_tokens, seq_lens, out_rows and miss_counts in pinned host memory: the kernels read
    and write them over the host link (copy CTAs, the fast path and graph replay included)."""
    run_parity(W.make("dsa", requests=8, steps=10, seq0=(6000, 9000, 300, 7000, 8000, 4100, 20000, 5000)),
               pool_every=2, graph_from=4, host_io=True)
    run_parity(W.make("mixed1m", requests=4, steps=6), pool_every=3, host_io=True)
    # 80 requests, no copy CTAs: the grouping and gather kernels behind a resolve that read
    # the step's inputs from host memory
    run_parity(W.make("indexshare", 9, requests=80, top_k=64, hot_slots=128, steps=4, layers=2,
                      seq_range=(1000, 3000)), pool_every=1, graph_from=2, host_io=True)


def test_graph_capture_replay_indexshare():
    run_parity(W.make("indexshare", requests=16, steps=8, layers=2), pool_every=4, graph_from=1)


def test_large_buffer_row_table_in_global():
    """H = 5 x top_k = 10,240 slots at top_k 2048 (the speculative sizing): the resolve CTA's
    shared memory cannot hold the slot -> row table too, so it reads it from global memory."""
    run_parity(W.make("dsa", 8, requests=3, hot_slots=10240, steps=8, seq0=(40000, 52000, 30000)))


def test_page_first_host_layout():
    """One host pool whose row h holds every layer's bytes of a token (host_row_stride =
    L x B, layer l at l x B): copy CTAs reading a miss's layers as one span, the resolve
    without copy CTAs followed by the pair gather in span mode (eager, then from a graph), and
    the backup writing into the strided rows."""
    run_parity(W.make("indexshare", 12, requests=8, top_k=256, hot_slots=512, steps=6, layers=3,
                      seq_range=(3000, 9000), host_layout="page_first"), pool_every=1)
    run_parity(W.make("indexshare", 13, requests=80, top_k=64, hot_slots=128, steps=6, layers=3,
                      seq_range=(1000, 3000), host_layout="page_first"), pool_every=1, graph_from=2)


@pytest.mark.parametrize("shape", [
    dict(requests=3, top_k=300, hot_slots=700, row_bytes=100, layers=3, seq0=(9000, 2000, 400)),  # 4-byte path
    dict(requests=2, top_k=77, hot_slots=131, row_bytes=37, layers=2, seq0=(5000, 90)),  # byte path
    dict(requests=90, top_k=40, hot_slots=64, row_bytes=48, layers=2, seq0=tuple(range(50, 950, 10))),
])
def test_page_first_ragged(shape):
    run_parity(W.make("tiny", fmt=W.FMT_U8, steps=6, host_layout="page_first", **shape), pool_every=1)


def test_indexshare_page_first():
    """The IndexShare workload at full size with its four layers' host caches interleaved
    row by row in one pool."""
    run_parity(W.make("indexshare", host_layout="page_first"), pool_every=32)
