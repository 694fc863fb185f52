"""GPU parity of the leader/follower split (hs_resolve_layers + hs_gather) against the
oracle, bit-exact: the leader resolve copies only its layers and records the miss plan;
follower gathers replay it, on the same stream or on a copy stream behind per-layer
events, or inside a CUDA graph. Every step the slot state, row table and every layer's
pool must equal the oracle's fused step, and the recorded plan the oracle's plan."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from harness import host_newest_ok, poison_host_newest  # noqa: E402
from test_gpu_parity import _gpu, compare_pools, compare_step  # noqa: E402

pytestmark = pytest.mark.gpu


def _plan_views(gpu):
    """The plan region of the workspace, as hs.h lays it out after the residency bitmap."""
    wl = gpu.wl
    off = 256 + ((wl.R * ((wl.max_context + 127) // 128) * 16 + 255) & ~255)
    RK = wl.R * wl.K
    words = gpu.ws[off: off + 4 * (2 * RK + wl.R)].view(torch.int32)
    return words[:RK].view(wl.R, wl.K), words[RK:2 * RK].view(wl.R, wl.K), words[2 * RK:]


def run_split(wl, copy_layers, gathers, mode="same", steps=None, check_plan=True):
    """mode: 'same' stream, 'side' (a copy stream behind per-layer events), or 'graph'."""
    import hierarchical_sparse_attention_gb300 as hs
    gh = _gpu()
    orc, gpu = gh.make_pair(wl)
    oplan = orc.orc.new_plan(wl.R)
    side = torch.cuda.Stream()
    graph = None

    def gpu_step(stream):
        hs.hs_resolve_layers(gpu.h, wl.R, gpu.tk, gpu.sl, gpu.hcl, gpu.dbl, gpu.tok, gpu.st, gpu.clk, gpu.rp,
                             gpu.out, gpu.miss, copy_layers, stream)
        if mode == "side":
            done = torch.cuda.Event()
            done.record(stream)
            side.wait_event(done)
            for first, n in gathers:
                hs.hs_gather(gpu.h, wl.R, gpu.hcl, first, n, side)
                ev = torch.cuda.Event()
                ev.record(side)  # layer(s) ready: the attention of these layers would wait here
                stream.wait_event(ev)
        else:
            for first, n in gathers:
                hs.hs_gather(gpu.h, wl.R, gpu.hcl, first, n, stream)
        gpu.backup(stream)

    try:
        for step in range(wl.steps if steps is None else steps):
            gpu.write_newest(step)
            orc.write_newest(step)
            poison_host_newest(wl, step, gpu.host)
            poison_host_newest(wl, step, orc.host)
            gpu.upload(step)
            cur = torch.cuda.current_stream()
            if mode == "graph":
                if graph is None:
                    graph = torch.cuda.CUDAGraph()
                    s = torch.cuda.Stream()
                    s.wait_stream(cur)
                    with torch.cuda.graph(graph, stream=s):
                        gpu_step(torch.cuda.current_stream())
                    cur.wait_stream(s)
                graph.replay()
            else:
                gpu_step(cur)
            torch.cuda.synchronize()
            assert host_newest_ok(wl, step, gpu.host)
            oerr = orc.orc.resolve(wl.top_k_tokens(step), wl.seq_lens(step), wl.host_cache_locs,
                                   wl.device_buffer_locs, orc.tokens, orc.stamps, orc.clock, wl.resident_pages,
                                   orc.out, orc.miss, orc.host, orc.dev, copy_layers=wl.L, plan=oplan)
            oerr |= orc.backup(step)
            gerr = compare_step(gpu, orc, f"{wl.cfg.name} split step {step}")
            assert gerr == oerr, f"step {step}: flags gpu {gerr} oracle {oerr}"
            compare_pools(gpu, orc, f"{wl.cfg.name} split step {step}")
            if check_plan:
                pt, pd, pc = _plan_views(gpu)
                pc = pc.cpu().numpy()
                np.testing.assert_array_equal(pc, oplan.count, err_msg=f"step {step}: plan counts")
                pt, pd = pt.cpu().numpy(), pd.cpu().numpy()
                for r in range(wl.R):
                    m = int(pc[r])
                    np.testing.assert_array_equal(pt[r, :m], oplan.tokens[r, :m], err_msg=f"step {step} r {r}")
                    np.testing.assert_array_equal(pd[r, :m], oplan.dst[r, :m], err_msg=f"step {step} r {r}")
            gh.resolved_rows_ok(wl, gpu, wl.top_k_tokens(step), gpu.state()["out"], f"split step {step}")
        gh.final_host_check(orc, gpu, f"{wl.cfg.name} split")
    finally:
        gh.close_pair(gpu)


def _indexshare_small(**kw):
    base = dict(requests=4, top_k=64, hot_slots=128, steps=8, layers=3, seq_range=(1000, 3000))
    base.update(kw)
    return W.make("indexshare", 5, **base)


def test_split_leader_one_layer_followers_each():
    run_split(_indexshare_small(), 1, [(1, 1), (2, 1)])


def test_split_followers_on_copy_stream():
    run_split(_indexshare_small(), 1, [(1, 1), (2, 1)], mode="side")


def test_split_in_cuda_graph():
    run_split(_indexshare_small(), 1, [(1, 2)], mode="graph")


def test_split_without_copy_ctas():
    # 80 requests leave no SM for copy CTAs: the resolve CTA copies the leader layer itself
    run_split(W.make("indexshare", 6, requests=80, top_k=64, hot_slots=128, steps=5, layers=3,
                     seq_range=(1000, 3000)), 1, [(1, 2)], check_plan=True)


def test_full_resolve_then_regather_in_miss_order():
    """A full hs_resolve with copy CTAs copies every layer and keeps its plan in miss order (no
    host-region grouping); hs_gather of every layer then replays it with the same bytes."""
    run_split(_indexshare_small(), 3, [(0, 3)])


def test_split_page_first_host_rows():
    """Every layer's bytes of a token in one host row: the followers' gather copies each miss's
    follower layers as one span, on the same stream and inside a graph, with and without copy
    CTAs."""
    run_split(_indexshare_small(host_layout="page_first"), 1, [(1, 2)])
    run_split(_indexshare_small(host_layout="page_first"), 1, [(1, 1), (2, 1)], mode="graph")
    run_split(W.make("indexshare", 8, requests=80, top_k=64, hot_slots=128, steps=4, layers=3,
                     seq_range=(1000, 3000), host_layout="page_first"), 2, [(2, 1)], mode="side")


def test_split_four_layers_dsa_rows():
    run_split(W.make("indexshare", 7, requests=6, top_k=256, hot_slots=512, steps=6, layers=4,
                     seq_range=(4000, 9000)), 2, [(2, 1), (3, 1)], mode="side")


def test_leader_only_step_matches_the_oracle():
    """copy_layers = 1 and no gather: the followers' pools keep their old rows, exactly as the
    oracle's leader-only step leaves them."""
    import hierarchical_sparse_attention_gb300 as hs
    gh = _gpu()
    wl = _indexshare_small(steps=3)
    orc, gpu = gh.make_pair(wl)
    try:
        for step in range(wl.steps):
            gpu.write_newest(step)
            orc.write_newest(step)
            gpu.upload(step)
            hs.hs_resolve_layers(gpu.h, wl.R, gpu.tk, gpu.sl, gpu.hcl, gpu.dbl, gpu.tok, gpu.st, gpu.clk, gpu.rp,
                                 gpu.out, gpu.miss, 1)
            torch.cuda.synchronize()
            oerr = orc.orc.resolve(wl.top_k_tokens(step), wl.seq_lens(step), wl.host_cache_locs,
                                   wl.device_buffer_locs, orc.tokens, orc.stamps, orc.clock, wl.resident_pages,
                                   orc.out, orc.miss, orc.host, orc.dev, copy_layers=1)
            assert compare_step(gpu, orc, f"leader only, step {step}") == oerr
            compare_pools(gpu, orc, f"leader only, step {step}")
        # invalid layer ranges are refused on the host
        with pytest.raises(hs.HsError):
            hs.hs_gather(gpu.h, wl.R, gpu.hcl, 2, 2)
        with pytest.raises(hs.HsError):
            hs.hs_resolve_layers(gpu.h, wl.R, gpu.tk, gpu.sl, gpu.hcl, gpu.dbl, gpu.tok, gpu.st, gpu.clk, gpu.rp,
                                 gpu.out, gpu.miss, wl.L + 1)
        # the plan was grouped by host region over all the resolve's requests: a gather of
        # fewer is refused; after a speculative batch (which records no plan) any gather is
        hs.hs_gather(gpu.h, wl.R, gpu.hcl, 1, 1)
        with pytest.raises(hs.HsError):
            hs.hs_gather(gpu.h, wl.R - 1, gpu.hcl, 1, 1)
        committed = (gpu.sl - 1).contiguous()
        hs.hs_resolve_spec(gpu.h, wl.R, 1, gpu.tk, committed, gpu.hcl, gpu.dbl, gpu.tok, gpu.st, gpu.clk, gpu.rp,
                           gpu.out, gpu.miss)
        with pytest.raises(hs.HsError):
            hs.hs_gather(gpu.h, wl.R, gpu.hcl, 1, 1)
        torch.cuda.synchronize()
        gpu.check_guards("leader only")
    finally:
        gh.close_pair(gpu)
