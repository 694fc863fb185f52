"""GPU parity of speculative batches (hs_resolve_spec + hs_backup_spec) against the oracle,
bit-exact: every verify step's row table and miss counts, the slot state after each batch,
the accepted positions' host rows after each backup, and the whole device pools. Inputs come
from the oracle-side driver of tests/test_oracle_spec.py (seeded top-k rows, forward-pass
writes, accepted counts); both sides see the same ones."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from test_gpu_parity import _gpu  # noqa: E402
from test_oracle_spec import SpecRun, _spec_workload  # noqa: E402

pytestmark = pytest.mark.gpu


class GpuSpec:
    """The library side of a SpecRun: its own pools, state and handle over the same geometry."""

    def __init__(self, run: SpecRun):
        import hierarchical_sparse_attention_gb300 as hs
        _gpu()
        self.run, wl = run, run.wl
        self.host = [p.copy() for p in run.host]
        for p in self.host:
            hs.hs_host_register(p)
        self.dev = [torch.from_numpy(p.copy()).cuda() for p in run.dev]
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        self.hcl, self.dbl = t(wl.host_cache_locs), t(run.dbl)
        self.rp = None if wl.resident_pages is None else t(wl.resident_pages)
        self.tok, self.st, self.clk = t(run.tok), t(run.st), t(run.clk)
        self.cfg = hs.make_config(wl.R, wl.K, run.H, wl.B, wl.L, wl.ps, wl.max_context, wl.max_pages)
        self.ws = torch.zeros(hs.hs_workspace_bytes(self.cfg), dtype=torch.uint8, device="cuda")
        self.h = hs.hs_create(self.cfg, self.host, self.dev, wl.host_rows, run.device_rows, self.ws)

    def close(self):
        import hierarchical_sparse_attention_gb300 as hs
        hs.hs_destroy(self.h)
        for p in self.host:
            hs.hs_host_unregister(p)

    def forward(self, writes):
        wl = self.run.wl
        for r, t, row, h in writes:
            for layer in range(wl.L):
                self.dev[layer].view(-1, wl.B)[row] = torch.from_numpy(wl.rows(layer, r, [t])[0]).cuda()
                self.host[layer][h * wl.B:(h + 1) * wl.B] = 0xEE

    def resolve(self, tk, S0, copy_layers=None, side=False):
        """The batch through hs_resolve_spec, or, with copy_layers, through
        hs_resolve_spec_layers and then every verify step's hs_gather_spec for the follower
        layers in step order (on a side stream behind an event when `side`)."""
        import hierarchical_sparse_attention_gb300 as hs
        wl, Q = self.run.wl, tk.shape[0]
        g_tk = torch.from_numpy(tk).cuda()
        out = torch.full((Q, wl.R, wl.K), -7, dtype=torch.int32, device="cuda")
        miss = torch.full((Q, wl.R), -7, dtype=torch.int32, device="cuda")
        args = (self.h, wl.R, Q, g_tk, torch.from_numpy(S0).cuda(), self.hcl, self.dbl, self.tok, self.st,
                self.clk, self.rp, out, miss)
        if copy_layers is None:
            hs.hs_resolve_spec(*args)
        else:
            stream = torch.cuda.current_stream()
            hs.hs_resolve_spec_layers(*args, copy_layers, stream)
            gs = torch.cuda.Stream() if side else stream
            if side:
                ev = torch.cuda.Event()
                ev.record(stream)
                gs.wait_event(ev)
            if copy_layers < wl.L:
                for q in range(Q):
                    hs.hs_gather_spec(self.h, wl.R, self.hcl, q, copy_layers, wl.L - copy_layers, gs)
        torch.cuda.synchronize()
        return out.cpu().numpy(), miss.cpu().numpy()

    def backup(self, S0, acc):
        import hierarchical_sparse_attention_gb300 as hs
        wl = self.run.wl
        hs.hs_backup_spec(self.h, wl.R, self.run.Q, torch.from_numpy(S0).cuda(), torch.from_numpy(acc).cuda(),
                          self.hcl, self.dbl, self.rp)
        torch.cuda.synchronize()


def run_spec_parity(name, Q, batches, hot_slots=None, fixed_accept=None, steps=40, copy_layers=None, side=False,
                    wl=None, expect_copy_ctas=None):
    """GPU batches against the oracle's full batches (hs_resolve_spec; the oracle pins that a
    leader-only batch plus per-step follower gathers equals it)."""
    import hierarchical_sparse_attention_gb300 as hs
    wl = _spec_workload(name, steps) if wl is None else wl
    run = SpecRun(wl, Q, seed=5, hot_slots=(Q + 1) * wl.K if hot_slots is None else hot_slots)
    gpu = GpuSpec(run)
    if expect_copy_ctas is not None:
        assert (hs.hs_launch_shape(gpu.h)[0] > 0) == expect_copy_ctas
    try:
        for b in range(batches):
            writes = run.forward()
            gpu.forward(writes)
            tk = run.topk()
            S0 = run.S0.copy()
            out, miss = gpu.resolve(tk, S0, copy_layers, side)
            o_out, o_miss, oerr = run.resolve(tk)
            np.testing.assert_array_equal(out, o_out, err_msg=f"batch {b}: out_rows")
            np.testing.assert_array_equal(miss, o_miss, err_msg=f"batch {b}: miss_counts")
            np.testing.assert_array_equal(gpu.tok.cpu().numpy(), run.tok, err_msg=f"batch {b}: slots")
            np.testing.assert_array_equal(gpu.st.cpu().numpy(), run.st, err_msg=f"batch {b}: stamps")
            np.testing.assert_array_equal(gpu.clk.cpu().numpy(), run.clk, err_msg=f"batch {b}: clock")
            assert hs.hs_get_error(gpu.h, clear=True) == oerr
            acc = None if fixed_accept is None else np.full(wl.R, fixed_accept, np.int32)
            acc, S0b, oerr = run.accept(acc)
            gpu.backup(S0b, acc)
            assert hs.hs_get_error(gpu.h, clear=True) == oerr
            for layer in range(wl.L):
                np.testing.assert_array_equal(gpu.host[layer], run.host[layer], err_msg=f"batch {b}: host {layer}")
                np.testing.assert_array_equal(gpu.dev[layer].cpu().numpy(), run.dev[layer],
                                              err_msg=f"batch {b}: device pool {layer}")
    finally:
        gpu.close()


def test_spec_dsa_small_q4():
    run_spec_parity("dsa_small", 4, 6)


def test_spec_mixed_residency_q3():
    run_spec_parity("mixed_small", 3, 6)


def test_spec_indexshare_layers_q2():
    run_spec_parity("indexshare_small", 2, 6)


def test_spec_tiny_fast_path_and_transition():
    # tiny: one request long, one inside the buffer (seq 100, H 256), which leaves the fast
    # path after ~52 batches of three accepted positions
    run_spec_parity("tiny", 3, 60, fixed_accept=3, steps=200)


def test_spec_one_query_matches_plain_steps():
    """Q = 1 batches through the spec entry points against the oracle's plain steps."""
    run_spec_parity("dsa_small", 1, 8, fixed_accept=1)


def test_spec_indexshare_leader_then_step_gathers():
    """IndexShare under MTP: each verify step copies layer 0 and records its plan; the
    followers replay every step's plan in step order."""
    run_spec_parity("indexshare_small", 2, 6, copy_layers=1)


def test_spec_indexshare_no_leader_copies_side_stream():
    run_spec_parity("indexshare_small", 3, 6, copy_layers=0, side=True)


def _wide_indexshare(steps=40):
    import workloads as W
    return W.make("indexshare", 12, requests=80, top_k=64, hot_slots=128, steps=steps, layers=3,
                  seq_range=(1000, 3000))


def test_spec_without_copy_ctas():
    """80 requests leave no SM for copy CTAs: every verify step is the resolve without copies,
    the grouping by host region and the gather, for the full batch and the split one."""
    run_spec_parity(None, 2, 4, wl=_wide_indexshare(), expect_copy_ctas=False)
    run_spec_parity(None, 2, 4, wl=_wide_indexshare(), copy_layers=1, expect_copy_ctas=False)


def test_gather_spec_misuse():
    import hierarchical_sparse_attention_gb300 as hs
    wl = _spec_workload("indexshare_small")
    Q = 2
    run = SpecRun(wl, Q, seed=5, hot_slots=(Q + 1) * wl.K)
    gpu = GpuSpec(run)
    try:
        with pytest.raises(hs.HsError):  # no batch yet
            hs.hs_gather_spec(gpu.h, wl.R, gpu.hcl, 0, 1, 1)
        gpu.forward(run.forward())
        tk = run.topk()
        gpu.resolve(tk, run.S0.copy(), copy_layers=1)
        hs.hs_gather_spec(gpu.h, wl.R, gpu.hcl, Q - 1, 1, 2)
        for bad in ((wl.R, Q, 1, 1), (wl.R, -1, 1, 1), (wl.R - 1, 0, 1, 1), (wl.R, 0, 2, 2)):
            with pytest.raises(hs.HsError):
                hs.hs_gather_spec(gpu.h, bad[0], gpu.hcl, bad[1], bad[2], bad[3])
        with pytest.raises(hs.HsError):  # a batch's plans are replayed per step
            hs.hs_gather(gpu.h, wl.R, gpu.hcl, 1, 1)
        with pytest.raises(hs.HsError):
            hs.hs_resolve_spec_layers(gpu.h, wl.R, Q, torch.from_numpy(tk).cuda(), torch.from_numpy(run.S0).cuda(),
                                      gpu.hcl, gpu.dbl, gpu.tok, gpu.st, gpu.clk, gpu.rp,
                                      torch.empty((Q, wl.R, wl.K), dtype=torch.int32, device="cuda"), None,
                                      wl.L + 1)
        torch.cuda.synchronize()
    finally:
        gpu.close()
