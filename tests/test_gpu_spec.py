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

    def resolve(self, tk, S0):
        import hierarchical_sparse_attention_gb300 as hs
        wl, Q = self.run.wl, tk.shape[0]
        g_tk = torch.from_numpy(tk).cuda()
        out = torch.full((Q, wl.R, wl.K), -7, dtype=torch.int32, device="cuda")
        miss = torch.full((Q, wl.R), -7, dtype=torch.int32, device="cuda")
        hs.hs_resolve_spec(self.h, wl.R, Q, g_tk, torch.from_numpy(S0).cuda(), self.hcl, self.dbl, self.tok, self.st,
                           self.clk, self.rp, out, miss)
        torch.cuda.synchronize()
        return out.cpu().numpy(), miss.cpu().numpy()

    def backup(self, S0, acc):
        import hierarchical_sparse_attention_gb300 as hs
        wl = self.run.wl
        hs.hs_backup_spec(self.h, wl.R, self.run.Q, torch.from_numpy(S0).cuda(), torch.from_numpy(acc).cuda(),
                          self.hcl, self.dbl, self.rp)
        torch.cuda.synchronize()


def run_spec_parity(name, Q, batches, hot_slots=None, fixed_accept=None, steps=40):
    import hierarchical_sparse_attention_gb300 as hs
    wl = _spec_workload(name, steps)
    run = SpecRun(wl, Q, seed=5, hot_slots=(Q + 1) * wl.K if hot_slots is None else hot_slots)
    gpu = GpuSpec(run)
    try:
        for b in range(batches):
            writes = run.forward()
            gpu.forward(writes)
            tk = run.topk()
            S0 = run.S0.copy()
            out, miss = gpu.resolve(tk, S0)
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
